// Sampling verification on sm_103a: one streaming pass over the logits plus a
// per-row finisher.
//
// Speculative sampling, Algorithm 1 Phases 3-4 (Leviathan, Kalman & Matias,
// "Fast Inference from Transformers via Speculative Decoding"; paper-graph-ui
// teardown §2.3 "Algorithm Walkthrough", multigrid.ai "The algorithm",
// fullstackaihub §3 "The Algorithm at Position i"), with temperature
// standardisation p = softmax(l / T) (§2.2).
//
// Streaming pass.  CTA (b, i, s) reads vocabulary slice s of target row
// (b, i) and, for i < gamma_b, of draft row (b, i) once, with 16-byte loads
// that do not allocate in L1, and keeps an online softmax normaliser per row:
// the running max m and S = sum 2^((l - m) log2(e)/T), rescaled when m grows
// (one exp per element).  It writes (m, S) for p and q to the workspace, and
// the CTA holding the draft token x_i also records l_p(x_i), l_q(x_i).
//
// Row finisher.  The last CTA of batch row b to finish (an atomic arrival
// counter; nothing waits) combines the slice normalisers of every position,
// computes p_i(x_i), q_i(x_i) and the accept decisions u_i <= min(1, p/q)
// (with p(x) > 0), and finds the first rejection n.  It then re-reads the one
// or two rows the draw needs -- target and draft row n for the residual
// max(0, p_n - q_n) (p_n when that mass is <= 1e-15), target row gamma_b for
// the bonus draw from p -- which the streaming pass has just brought through
// L2, sums the weights in 32-lane chunks, locates the chunk holding
// u_final * (total weight) by a block prefix scan over the chunk sums, and the
// token by a warp scan inside that chunk.  p and q are never written to
// memory; HBM traffic is the read-once logits plus at most two rows per batch
// row that miss L2.
#include "common.cuh"
#include "kernels.h"

namespace specv {

namespace {

constexpr int kST = kStreamThreads;
constexpr int kSW = kST / 32;
constexpr int kMaxChunks = kMaxVocab / 128;  // fp32 chunks of 32 lanes x 4 elements

// Online normaliser update with a group of cnt raw logits (cnt is a compile-time vector width).
template <int kCnt>
__device__ __forceinline__ void online(float& m, float& s, float& raw, const float* f, float sc) {
  float vm = f[0];
#pragma unroll
  for (int j = 1; j < kCnt; ++j) vm = max_nan(vm, f[j]);
  raw = max_nan(raw, vm);
  if (vm > -INFINITY) {
    if (vm > m) {
      s *= exp2f((m - vm) * sc);
      m = vm;
    }
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kCnt; ++j) acc += exp2f((f[j] - m) * sc);
    s += acc;
  }
}

// Merge normaliser (om, os) into (m, s).
__device__ __forceinline__ void merge(float& m, float& s, float om, float os, float sc) {
  const float M = fmaxf(m, om);
  if (!(M > -INFINITY)) return;  // both empty
  const float a = m > -INFINITY ? s * exp2f((m - M) * sc) : 0.f;
  const float c = om > -INFINITY ? os * exp2f((om - M) * sc) : 0.f;
  s = a + c;
  m = M;
}

struct FinishSmem {
  float mp[kMaxGamma + 1], sp[kMaxGamma + 1], mq[kMaxGamma + 1], sq[kMaxGamma + 1];
  int acc[kMaxGamma + 1];
  float W[2][kMaxChunks];  // per-chunk residual mass and p mass of the drawn row(s)
  float red[kSW];
  int n, invalid;
  uint32_t err;
  int chunk;
  float prefix;
  int lastc;
};

// Weights of one lane's kV elements of chunk c of the drawn row(s): p, and w =
// max(0, p - q) for a residual draw (w = p otherwise).  Elements past V weigh 0.
template <typename T>
__device__ __forceinline__ void chunk_weights(const T* tr, const T* dr, bool resid, int V, bool vec, int c, int lane,
                                              float mp, float ip, float mq, float iq, float sc,
                                              float (&p)[Elems<T>::kVec], float (&w)[Elems<T>::kVec]) {
  constexpr int kV = Elems<T>::kVec;
  const int base = c * 32 * kV + lane * kV;
  float lt[kV], ld[kV];
  if (vec && base + kV <= V) {
    Elems<T>::widen(ldg_stream(tr + base), lt);
    if (resid) Elems<T>::widen(ldg_stream(dr + base), ld);
  } else {
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      lt[j] = base + j < V ? Elems<T>::one(tr, base + j) : -INFINITY;
      ld[j] = (resid && base + j < V) ? Elems<T>::one(dr, base + j) : -INFINITY;
    }
  }
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    p[j] = exp2f((lt[j] - mp) * sc) * ip;
    if (resid) {
      const float q = exp2f((ld[j] - mq) * sc) * iq;
      w[j] = fmaxf(p[j] - q, 0.f);
    } else {
      w[j] = p[j];
    }
  }
}

template <int kV>
__device__ __forceinline__ float lane_sum(const float (&w)[kV]) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kV; ++j) s += w[j];
  return s;
}

// Block-wide: total of W[0..nc) and the chunk holding target t (smallest c with
// running sum > t among positive chunks; else the last positive chunk).
__device__ void locate_chunk(const float* W, int nc, float u, FinishSmem& sm, float& total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nc + kST - 1) / kST;
  const int c0 = min(nc, tid * per), c1 = min(nc, c0 + per);
  float ts = 0.f;
  int lastpos = -1;
  for (int c = c0; c < c1; ++c) {
    ts += W[c];
    if (W[c] > 0.f) lastpos = c;
  }
  // block exclusive scan of thread sums
  const float inc = warp_inclusive_scan(ts, lane);
  if (lane == 31) sm.red[warp] = inc;
  if (tid == 0) {
    sm.chunk = 0x7fffffff;
    sm.lastc = -1;
  }
  __syncthreads();
  float wbase = 0.f, tot = 0.f;
  for (int w = 0; w < kSW; ++w) {
    if (w < warp) wbase += sm.red[w];
    tot += sm.red[w];
  }
  total = tot;
  const float t = u * tot;
  float cum = wbase + inc - ts;
  int found = -1;
  float pre = 0.f;
  for (int c = c0; c < c1; ++c) {
    const float v = W[c];
    if (v > 0.f && cum + v > t) {
      found = c;
      pre = cum;
      break;
    }
    cum += v;
  }
  if (found >= 0) atomicMin(&sm.chunk, found);
  if (lastpos >= 0) atomicMax(&sm.lastc, lastpos);
  __syncthreads();
  if (found >= 0 && found == sm.chunk) sm.prefix = pre;
  __syncthreads();
}

template <typename T>
__device__ void finish_row(const SampleParams& a, int b, int gb, FinishSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = a.G + 1;
  const int NS = a.nslices;
  const float sc = a.scale;
  const float4* part = reinterpret_cast<const float4*>(a.ws.part) + (size_t)b * G1 * NS;

  // 1. per-position normalisers from the slice partials (fixed combination order)
  for (int i = warp; i <= gb; i += kSW) {
    float4 pr = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    if (lane < NS) pr = __ldcg(part + (size_t)i * NS + lane);
    const float Mp = warp_max_nan(pr.x);
    const float Mq = warp_max_nan(pr.z);
    const float tp = (pr.x > -INFINITY && Mp < INFINITY) ? pr.y * exp2f((pr.x - Mp) * sc) : 0.f;
    const float tq = (pr.z > -INFINITY && Mq < INFINITY) ? pr.w * exp2f((pr.z - Mq) * sc) : 0.f;
    float Sp = 0.f, Sq = 0.f;
    for (int r = 0; r < NS; ++r) {
      Sp += __shfl_sync(0xffffffffu, tp, r);
      Sq += __shfl_sync(0xffffffffu, tq, r);
    }
    if (lane == 0) {
      sm.mp[i] = Mp;
      sm.sp[i] = Sp;
      sm.mq[i] = Mq;
      sm.sq[i] = Sq;
    }
  }
  __syncthreads();

  // 2. validity and accept decisions, one thread per position
  const float* U = a.uniforms + (size_t)b * G1;
  uint32_t err = 0;
  if (tid <= gb) {
    const int i = tid;
    const bool bad_p = !(sm.mp[i] > -INFINITY && sm.mp[i] < INFINITY);
    int code = 1;
    if (bad_p) {
      err |= kErrNonfinite;
      code = -1;
    }
    if (i < gb) {
      const bool bad_q = !(sm.mq[i] > -INFINITY && sm.mq[i] < INFINITY);
      const int x = __ldg(a.ids + (size_t)b * a.G + i);
      const float ui = __ldg(U + i);
      if (bad_q) err |= kErrNonfinite;
      if (x < 0 || x >= a.V) err |= kErrToken;
      if (!(ui >= 0.f && ui < 1.f)) err |= kErrArg;
      if (err) {
        code = -1;
      } else {
        const float2 xl = __ldcg(reinterpret_cast<const float2*>(a.ws.xl) + (size_t)b * a.G + i);
        const float px = exp2f((xl.x - sm.mp[i]) * sc) / sm.sp[i];
        const float qx = exp2f((xl.y - sm.mq[i]) * sc) / sm.sq[i];
        const float ratio = px >= qx ? 1.f : px / qx;  // min(1, p/q); q = 0 < p gives 1
        code = (px > 0.f && ui <= ratio) ? 1 : 0;
      }
    }
    sm.acc[i] = code;
  }
  if (tid == 0) {
    const float uf = __ldg(U + a.G);
    if (!(uf >= 0.f && uf < 1.f)) err |= kErrArg;
    sm.err = 0;
  }
  __syncthreads();
  if (err) atomicOr(&sm.err, err);
  // every partial and logit slot this row used goes back to zero: workspaces are shared by calls of any shape
  float4* partw = reinterpret_cast<float4*>(a.ws.part) + (size_t)b * G1 * NS;
  for (int k = tid; k < (gb + 1) * NS; k += kST) partw[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = tid; k < gb; k += kST) reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + k] = make_float2(0.f, 0.f);
  __syncthreads();
  if (tid == 0) {
    int n = gb;
    for (int i = 0; i < gb; ++i) {
      if (sm.acc[i] == 0) {
        n = i;
        break;
      }
    }
    sm.n = n;
    sm.invalid = sm.err != 0;
  }
  __syncthreads();
  int32_t* e = a.emitted + (size_t)b * G1;
  if (sm.invalid) {
    if (tid == 0) {
      for (int j = 0; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = -1;
      atomicOr(a.ws.err, sm.err);
      a.ws.ticket[b] = 0u;
    }
    return;
  }

  // 3. the draw: residual at the first rejection, or the bonus token
  constexpr int kV = Elems<T>::kVec;
  const int n = sm.n;
  const bool resid = n < gb;
  const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + n) * a.V;
  const T* dr = resid ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + n) * a.V : tr;
  const float mp = sm.mp[n], ip = 1.f / sm.sp[n];
  const float mq = resid ? sm.mq[n] : 0.f, iq = resid ? 1.f / sm.sq[n] : 0.f;
  const int nc = (a.V + 32 * kV - 1) / (32 * kV);
  const bool vec = a.vec != 0;
  constexpr int U2 = 4;
  for (int c0 = warp; c0 < nc; c0 += U2 * kSW) {
    float lw[U2], lp[U2];
#pragma unroll
    for (int u = 0; u < U2; ++u) {
      const int c = c0 + u * kSW;
      lw[u] = lp[u] = 0.f;
      if (c < nc) {
        float pv[kV], wv[kV];
        chunk_weights<T>(tr, dr, resid, a.V, vec, c, lane, mp, ip, mq, iq, sc, pv, wv);
        lw[u] = lane_sum<kV>(wv);
        lp[u] = lane_sum<kV>(pv);
      }
    }
#pragma unroll
    for (int u = 0; u < U2; ++u) {
      const int c = c0 + u * kSW;
      if (c < nc) {
        const float cw = warp_sum(lw[u]);
        const float cp = resid ? warp_sum(lp[u]) : cw;
        if (lane == 0) {
          sm.W[0][c] = cw;
          sm.W[1][c] = cp;
        }
      }
    }
  }
  __syncthreads();
  const float uf = __ldg(U + a.G);
  float total;
  int which = resid ? 0 : 1;
  locate_chunk(sm.W[which], nc, uf, sm, total);
  if (resid && !(total > kZFloor)) {  // degenerate residual: draw from p instead
    which = 1;
    locate_chunk(sm.W[1], nc, uf, sm, total);
  }
  const bool use_p = which == 1;
  bool fallback = sm.chunk == 0x7fffffff;
  const int c = fallback ? sm.lastc : sm.chunk;
  if (c < 0) {  // no weight anywhere (cannot happen for a valid row): report, never index
    if (tid == 0) {
      for (int j = 0; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = -1;
      atomicOr(a.ws.err, kErrNonfinite);
      a.ws.ticket[b] = 0u;
    }
    return;
  }
  if (warp == 0) {
    float pv[kV], wv[kV];
    chunk_weights<T>(tr, dr, resid && !use_p, a.V, vec, c, lane, mp, ip, mq, iq, sc, pv, wv);
    const float ls = lane_sum<kV>(wv);
    const float inc = warp_inclusive_scan(ls, lane);
    float exc = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) exc = 0.f;
    const float tt = fallback ? 0.f : uf * total - sm.prefix;
    int lastj = -1;
#pragma unroll
    for (int j = 0; j < kV; ++j)
      if (wv[j] > 0.f) lastj = j;
    const int base = c * 32 * kV + lane * kV;
    int tok = -1;
    const unsigned hit = fallback ? 0u : __ballot_sync(0xffffffffu, ls > 0.f && inc > tt);
    if (hit) {
      const int l = __ffs(hit) - 1;
      if (lane == l) {
        float cum = exc;
        for (int j = 0; j < kV; ++j) {
          cum += wv[j];
          if (wv[j] > 0.f && cum > tt) {
            tok = base + j;
            break;
          }
        }
        if (tok < 0) tok = base + lastj;
      }
      tok = __shfl_sync(0xffffffffu, tok, l);
    } else {
      const unsigned nz = __ballot_sync(0xffffffffu, ls > 0.f);
      const int l = 31 - __clz(nz);
      if (lane == l) tok = base + lastj;
      tok = __shfl_sync(0xffffffffu, tok, l);
    }
    if (lane == 0) {
      for (int j = 0; j < n; ++j) e[j] = __ldg(a.ids + (size_t)b * a.G + j);
      e[n] = tok;
      for (int j = n + 1; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = n;
      a.ws.ticket[b] = 0u;
    }
  }
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_stream_kernel(const SampleParams a) {
  __shared__ FinishSmem sm;
  __shared__ float red[4][kSW];
  __shared__ int last;
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NS = a.nslices;
  const int s = blockIdx.x % NS;
  const int pos = blockIdx.x / NS;
  const int G1 = a.G + 1;
  const int b = pos / G1;
  const int i = pos - b * G1;
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  if (gb < 0 || gb > a.G) {
    if (i == 0 && s == 0 && tid == 0) {
      int32_t* e = a.emitted + (size_t)b * G1;
      for (int j = 0; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = -1;
      atomicOr(a.ws.err, kErrArg);
    }
    return;
  }
  if (i > gb) return;  // padded target row: never read
  const bool has_q = i < gb;
  const float sc = a.scale;
  const int lo = s * a.slice;
  const int n = min(a.V, lo + a.slice) - lo;
  const T* tp = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + i) * a.V + lo;
  const T* dp = has_q ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + i) * a.V + lo : tp;

  float mp = -INFINITY, sp = 0.f, rp = -INFINITY;
  float mq = -INFINITY, sq = 0.f, rq = -INFINITY;
  int done = 0;
  if (a.vec) {
    const int nv = n / kV;
    const uint4* t4 = reinterpret_cast<const uint4*>(tp);
    const uint4* d4 = reinterpret_cast<const uint4*>(dp);
    int v = tid;
    if (has_q) {
      for (; v + (U - 1) * kST < nv; v += U * kST) {
        uint4 r0[U], r1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = ldg_stream(t4 + v + u * kST);
#pragma unroll
        for (int u = 0; u < U; ++u) r1[u] = ldg_stream(d4 + v + u * kST);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float f[kV];
          Elems<T>::widen(r0[u], f);
          online<kV>(mp, sp, rp, f, sc);
          Elems<T>::widen(r1[u], f);
          online<kV>(mq, sq, rq, f, sc);
        }
      }
      for (; v < nv; v += kST) {
        float f[kV];
        Elems<T>::widen(ldg_stream(t4 + v), f);
        online<kV>(mp, sp, rp, f, sc);
        Elems<T>::widen(ldg_stream(d4 + v), f);
        online<kV>(mq, sq, rq, f, sc);
      }
    } else {
      for (; v + (U - 1) * kST < nv; v += U * kST) {
        uint4 r0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = ldg_stream(t4 + v + u * kST);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float f[kV];
          Elems<T>::widen(r0[u], f);
          online<kV>(mp, sp, rp, f, sc);
        }
      }
      for (; v < nv; v += kST) {
        float f[kV];
        Elems<T>::widen(ldg_stream(t4 + v), f);
        online<kV>(mp, sp, rp, f, sc);
      }
    }
    done = nv * kV;
  }
  for (int k = done + tid; k < n; k += kST) {
    float f[1] = {Elems<T>::one(tp, k)};
    online<1>(mp, sp, rp, f, sc);
    if (has_q) {
      f[0] = Elems<T>::one(dp, k);
      online<1>(mq, sq, rq, f, sc);
    }
  }

  // block merge of the normalisers (fixed order, identical for p and q)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mp, o), os = __shfl_xor_sync(0xffffffffu, sp, o);
    const float qm = __shfl_xor_sync(0xffffffffu, mq, o), qs = __shfl_xor_sync(0xffffffffu, sq, o);
    merge(mp, sp, om, os, sc);
    merge(mq, sq, qm, qs, sc);
  }
  rp = warp_max_nan(rp);
  rq = warp_max_nan(rq);
  if (lane == 0) {
    red[0][warp] = mp;
    red[1][warp] = sp;
    red[2][warp] = mq;
    red[3][warp] = sq;
    sm.red[warp] = max_nan(rp, rq);
  }
  __syncthreads();
  if (tid == 0) {
    float Mp = red[0][0], Sp = red[1][0], Mq = red[2][0], Sq = red[3][0], raw = sm.red[0];
    for (int w = 1; w < kSW; ++w) {
      merge(Mp, Sp, red[0][w], red[1][w], sc);
      merge(Mq, Sq, red[2][w], red[3][w], sc);
      raw = max_nan(raw, sm.red[w]);
    }
    const bool bad = !(raw < INFINITY);               // NaN or +inf in this slice
    float4 out = make_float4(bad ? NAN : Mp, Sp, bad ? NAN : Mq, Sq);
    reinterpret_cast<float4*>(a.ws.part)[(size_t)pos * NS + s] = out;
    if (has_q) {
      const int x = __ldg(a.ids + (size_t)b * a.G + i);
      if (x >= lo && x < lo + n)
        reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + i] =
            make_float2(Elems<T>::one(tp, x - lo), Elems<T>::one(dp, x - lo));
    }
    __threadfence();
    const unsigned prev = atomicAdd(a.ws.ticket + b, 1u);
    last = prev == static_cast<unsigned>(NS * (gb + 1) - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  finish_row<T>(a, b, gb, sm);
}

cudaError_t sample_launch(const SampleParams& p, int dtype, cudaStream_t stream) {
  const long long ctas = (long long)p.B * (p.G + 1) * p.nslices;
  const dim3 grid(static_cast<unsigned>(ctas)), block(kStreamThreads);
  if (dtype == 0) {
    verify_stream_kernel<float><<<grid, block, 0, stream>>>(p);
  } else {
    verify_stream_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace specv
