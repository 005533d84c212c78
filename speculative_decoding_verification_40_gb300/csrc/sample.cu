// Sampling verification on sm_103a: a streaming pass over the logits, then a
// draw pass over the rows the draws need.
//
// Speculative sampling, Algorithm 1 Phases 3-4 (Leviathan, Kalman & Matias,
// "Fast Inference from Transformers via Speculative Decoding"; paper-graph-ui
// teardown §2.3 "Algorithm Walkthrough", multigrid.ai "The algorithm",
// fullstackaihub §3 "The Algorithm at Position i"), with temperature
// standardisation p = softmax(l / T) (§2.2).
//
// Stream kernel, one CTA per (batch row b, position i, vocabulary slice s):
//   reads slice s of target row (b, i) and, for i < gamma_b, of draft row
//   (b, i) once, with 16-byte loads that do not allocate in L1, keeping online
//   softmax normalisers -- the running max m and S = sum 2^((l - m) log2(e)/T),
//   rescaled when m grows, one hardware exp2 per element -- and writes (m, S)
//   for p and q; the CTA holding the draft token x_i records l_p(x_i),
//   l_q(x_i).  No CTA waits for or signals another.
// Draw kernel, one CTA per (batch row b, draw slice d), rows in reverse order
//   so the rows the stream kernel read last are still in L2:
//   every CTA of row b combines the slice normalisers, takes the accept
//   decisions u_i <= min(1, p_i(x_i)/q_i(x_i)) (with p(x) > 0) and finds the
//   first rejection n -- the same arithmetic in every CTA, so they agree bit
//   for bit -- then, over slice d of target row n (and of draft row n for a
//   residual draw), writes the mass of w = max(0, p_n - q_n) and of p_n per
//   chunk.  The last CTA of row b (atomic arrival counter) picks, from
//   u_final * (total mass), the slice, then the chunk from the stored chunk
//   masses, then the token by warp scans over that chunk's recomputed
//   weights: the residual draw, the draw from p_n when the residual mass is
//   <= 1e-15, or the bonus draw from p_{gamma_b} when nothing was rejected.
//   It writes the row's outputs and returns every slot the row used to zero.
// p and q are never written to memory; HBM traffic is the logits read once
// plus at most the two drawn rows per batch row that have left L2.
#include "common.cuh"
#include "kernels.h"
#include "softmax.cuh"

namespace specv {

namespace {

constexpr int kST = kStreamThreads;
constexpr int kSW = kST / 32;
constexpr int kR = 4;  // 16-byte vectors per lane in one draw chunk

enum : int { kRowInvalid = 1, kRowResid = 2 };

struct RowState {
  int n, flags;
  uint32_t err;
  float mp, ip, mq, iq;
};

// Weights of one lane's kV elements starting at `base` of the drawn row(s): p, and w = max(0, p - q)
// for a residual draw (w = p otherwise); elements past V weigh 0.  The mass pass and the final scan
// both use this arithmetic, so they see identical weights.
template <typename T>
__device__ __forceinline__ void seg_weights(const T* tr, const T* dr, bool resid, int V, bool vec, int base,
                                            const RowState& st, float sc, float (&p)[Elems<T>::kVec],
                                            float (&w)[Elems<T>::kVec]) {
  constexpr int kV = Elems<T>::kVec;
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
    p[j] = fast_exp2((lt[j] - st.mp) * sc) * st.ip;
    w[j] = resid ? fmaxf(p[j] - fast_exp2((ld[j] - st.mq) * sc) * st.iq, 0.f) : p[j];
  }
}

template <int kV>
__device__ __forceinline__ float lane_sum(const float (&w)[kV]) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kV; ++j) s += w[j];
  return s;
}

struct DrawSmem {
  float mp[kMaxGamma + 1], sp[kMaxGamma + 1], mq[kMaxGamma + 1], sq[kMaxGamma + 1];
  int acc[kMaxGamma + 1];
  float2 cs[kMaxChunksPerSlice];  // chunk masses of this CTA's slice, then of the chosen slice (w, p)
  float2 ds[kMaxSlices];          // slice masses of the drawn row (w, p)
  uint32_t err;
  int last, pick, mode;
  float t, pre;
};

// Accept decisions of row b from the slice normalisers: the same arithmetic in every CTA of the row.
__device__ RowState decide_row(const SampleParams& a, int b, int gb, DrawSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = a.G + 1;
  const int NS = a.nslices;
  const float sc = a.scale;
  const float4* part = reinterpret_cast<const float4*>(a.ws.part) + (size_t)b * G1 * NS;
  // per-position normalisers from the slice partials (fixed combination order)
  for (int i = warp; i <= gb; i += kSW) {
    float4 pr = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    if (lane < NS) pr = __ldcg(part + (size_t)i * NS + lane);
    const float Mp = warp_max_nan(pr.x);
    const float Mq = warp_max_nan(pr.z);
    const float tp = (pr.x > -INFINITY && Mp < INFINITY) ? pr.y * fast_exp2((pr.x - Mp) * sc) : 0.f;
    const float tq = (pr.z > -INFINITY && Mq < INFINITY) ? pr.w * fast_exp2((pr.z - Mq) * sc) : 0.f;
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
  if (tid == 0) sm.err = 0;
  __syncthreads();
  // validity and accept decisions, one thread per position
  const float* U = a.uniforms + (size_t)b * G1;
  uint32_t err = 0;
  if (tid <= gb) {
    const int i = tid;
    int code = 1;
    if (!(sm.mp[i] > -INFINITY && sm.mp[i] < INFINITY)) err |= kErrNonfinite;
    if (i < gb) {
      const int x = __ldg(a.ids + (size_t)b * a.G + i);
      const float ui = __ldg(U + i);
      if (!(sm.mq[i] > -INFINITY && sm.mq[i] < INFINITY)) err |= kErrNonfinite;
      if (x < 0 || x >= a.V) err |= kErrToken;
      if (!(ui >= 0.f && ui < 1.f)) err |= kErrArg;
      if (!err) {
        const float2 xl = __ldcg(reinterpret_cast<const float2*>(a.ws.xl) + (size_t)b * a.G + i);
        const float px = fast_exp2((xl.x - sm.mp[i]) * sc) / sm.sp[i];
        const float qx = fast_exp2((xl.y - sm.mq[i]) * sc) / sm.sq[i];
        const float ratio = px >= qx ? 1.f : px / qx;  // min(1, p/q); q = 0 < p gives 1
        code = (px > 0.f && ui <= ratio) ? 1 : 0;
      }
    }
    sm.acc[i] = err ? -1 : code;
  }
  if (tid == 0) {
    const float uf = __ldg(U + a.G);
    if (!(uf >= 0.f && uf < 1.f)) err |= kErrArg;
  }
  if (err) atomicOr(&sm.err, err);
  __syncthreads();
  RowState st = {};
  int n = gb;
  for (int i = 0; i < gb; ++i) {
    if (sm.acc[i] == 0) {
      n = i;
      break;
    }
  }
  st.n = n;
  st.err = sm.err;
  if (st.err) {
    st.flags = kRowInvalid;
  } else {
    st.flags = n < gb ? kRowResid : 0;
    st.mp = sm.mp[n];
    st.ip = 1.f / sm.sp[n];
    if (n < gb) {
      st.mq = sm.mq[n];
      st.iq = 1.f / sm.sq[n];
    }
  }
  return st;
}

// Last CTA of row b: slice, chunk and token of the draw; the row's outputs; every slot back to zero.
template <typename T>
__device__ void resolve_row(const SampleParams& a, int b, int gb, const RowState& st, DrawSmem& sm) {
  constexpr int kV = Elems<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31;
  const int G1 = a.G + 1;
  const int ND = a.ndslices;
  const int seg = 32 * kV;
  const int cpc = kR * seg;
  const int cps = a.dslice / cpc;
  const int nc = (a.V + cpc - 1) / cpc;
  float2* dsum = reinterpret_cast<float2*>(a.ws.dsum) + (size_t)b * ND;
  float2* dch = reinterpret_cast<float2*>(a.ws.dch) + (size_t)b * ND * cps;
  int32_t* e = a.emitted + (size_t)b * G1;
  const bool resid = st.flags & kRowResid;
  const bool failed = st.flags & kRowInvalid;
  if (!failed && tid < ND) sm.ds[tid] = __ldcg(dsum + tid);
  __syncthreads();
  if (!failed && tid == 0) {
    // total mass in slice order; the residual, or p when the residual mass is degenerate
    const float uf = __ldg(a.uniforms + (size_t)b * G1 + a.G);
    float Z = 0.f, P = 0.f;
    for (int d = 0; d < ND; ++d) {
      Z += sm.ds[d].x;
      P += sm.ds[d].y;
    }
    const bool use_p = !resid || !(Z > kZFloor);
    const float tot = use_p ? P : Z;
    const float t = uf * tot;
    int sd = -1, lastd = -1;
    float cum = 0.f, pre = 0.f, lastpre = 0.f;
    for (int d = 0; d < ND; ++d) {
      const float v = use_p ? sm.ds[d].y : sm.ds[d].x;
      if (v > 0.f) {
        if (sd < 0 && cum + v > t) {
          sd = d;
          pre = cum;
        }
        lastd = d;
        lastpre = cum;
      }
      cum += v;
    }
    const bool fallback = sd < 0;
    if (fallback) {
      sd = lastd;
      pre = lastpre;
    }
    sm.pick = sd;
    sm.mode = (use_p ? 1 : 0) | (fallback ? 2 : 0);
    sm.t = t;
    sm.pre = pre;
  }
  if (failed && tid == 0) sm.pick = -1;
  __syncthreads();
  // chunk within the chosen slice: stage its chunk masses, then one thread scans them
  const int sd = sm.pick;
  if (sd >= 0) {
    const int c0 = sd * cps, c1 = min(c0 + cps, nc);
    for (int c = c0 + tid; c < c1; c += kST) sm.cs[c - c0] = __ldcg(dch + (size_t)sd * cps + (c - c0));
    __syncthreads();
    if (tid == 0) {
      const bool use_p = sm.mode & 1;
      bool fallback = sm.mode & 2;
      const float t = sm.t;
      int pc = -1, lastc = -1;
      float cum2 = sm.pre, cpre = 0.f;
      for (int c = c0; c < c1; ++c) {
        const float v = use_p ? sm.cs[c - c0].y : sm.cs[c - c0].x;
        if (v > 0.f) {
          if (!fallback && pc < 0 && cum2 + v > t) {
            pc = c;
            cpre = cum2;
          }
          lastc = c;
        }
        cum2 += v;
      }
      if (pc < 0) {
        pc = lastc;
        fallback = true;
      }
      sm.pick = pc;
      sm.mode = (use_p ? 1 : 0) | (fallback ? 2 : 0);
      sm.pre = cpre;
    }
    __syncthreads();
  }
  const int pc = sd >= 0 ? sm.pick : -1;
  if (pc >= 0 && tid < 32) {  // warp 0: the token inside the chunk, segment by segment
    const bool use_p = sm.mode & 1;
    const bool fallback = sm.mode & 2;
    const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + st.n) * a.V;
    const T* dr = resid ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + st.n) * a.V : tr;
    float tt = sm.t - sm.pre;
    int tok = -1, lasttok = -1;
    for (int r = 0; r < kR && tok < 0; ++r) {
      const int base = pc * cpc + r * seg + lane * kV;
      float pv[kV], wv[kV];
      seg_weights<T>(tr, dr, resid && !use_p, a.V, a.vec != 0, base, st, a.scale, pv, wv);
      const float ls = lane_sum<kV>(wv);
      const float inc = warp_inclusive_scan(ls, lane);
      float exc = __shfl_up_sync(0xffffffffu, inc, 1);
      if (lane == 0) exc = 0.f;
      int lastj = -1;
#pragma unroll
      for (int j = 0; j < kV; ++j)
        if (wv[j] > 0.f) lastj = j;
      const unsigned nz = __ballot_sync(0xffffffffu, ls > 0.f);
      if (nz) {  // last positive weight so far: the fallback when rounding leaves t past the total
        const int l = 31 - __clz(nz);
        lasttok = __shfl_sync(0xffffffffu, base + lastj, l);
      }
      const unsigned hit = fallback ? 0u : __ballot_sync(0xffffffffu, ls > 0.f && inc > tt);
      if (hit) {
        const int l = __ffs(hit) - 1;
        int k = -1;
        if (lane == l) {
          float c = exc;
          for (int j = 0; j < kV; ++j) {
            c += wv[j];
            if (wv[j] > 0.f && c > tt) {
              k = base + j;
              break;
            }
          }
          if (k < 0) k = base + lastj;
        }
        tok = __shfl_sync(0xffffffffu, k, l);
      } else {
        tt -= __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    if (tok < 0) tok = lasttok;
    if (lane == 0) {
      if (tok >= 0) {
        for (int j = 0; j < st.n; ++j) e[j] = __ldg(a.ids + (size_t)b * a.G + j);
        e[st.n] = tok;
        for (int j = st.n + 1; j < G1; ++j) e[j] = -1;
        a.n_acc[b] = st.n;
      } else {  // no weight anywhere (cannot happen for a valid row): report, never index
        for (int j = 0; j < G1; ++j) e[j] = -1;
        a.n_acc[b] = -1;
        atomicOr(a.ws.err, kErrNonfinite);
      }
    }
  } else if (tid == 0) {
    for (int j = 0; j < G1; ++j) e[j] = -1;
    a.n_acc[b] = -1;
    atomicOr(a.ws.err, failed ? st.err : kErrNonfinite);
  }
  // every slot of this row back to zero for the next call
  const int NS = a.nslices;
  float4* part = reinterpret_cast<float4*>(a.ws.part) + (size_t)b * G1 * NS;
  for (int k = tid; k < (gb + 1) * NS; k += kST) part[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = tid; k < gb; k += kST) reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + k] = make_float2(0.f, 0.f);
  for (int k = tid; k < ND * cps; k += kST) dch[k] = make_float2(0.f, 0.f);
  for (int k = tid; k < ND; k += kST) dsum[k] = make_float2(0.f, 0.f);
  if (tid == 0) a.ws.ticket[b] = 0u;
}

}  // namespace

// ----------------------------------------------------------------------------- stream kernel

template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_stream_kernel(const SampleParams a) {
  __shared__ float red[4][kSW];
  __shared__ float rawr[kSW];
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the draw kernel may be scheduled once every stream CTA is running; it waits for their results
  asm volatile("griddepcontrol.launch_dependents;");
  const int NS = a.nslices;
  const int s = blockIdx.x % NS;
  const int pos = blockIdx.x / NS;
  const int G1 = a.G + 1;
  const int b = pos / G1;
  const int i = pos - b * G1;
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  if (gb < 0 || gb > a.G || i > gb) return;  // invalid length (the draw kernel reports it) or padding
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
        online_group<T, U>(mp, sp, rp, r0, sc);
        online_group<T, U>(mq, sq, rq, r1, sc);
      }
      for (; v < nv; v += kST) {
        const uint4 r0[1] = {ldg_stream(t4 + v)};
        const uint4 r1[1] = {ldg_stream(d4 + v)};
        online_group<T, 1>(mp, sp, rp, r0, sc);
        online_group<T, 1>(mq, sq, rq, r1, sc);
      }
    } else {
      for (; v + (U - 1) * kST < nv; v += U * kST) {
        uint4 r0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = ldg_stream(t4 + v + u * kST);
        online_group<T, U>(mp, sp, rp, r0, sc);
      }
      for (; v < nv; v += kST) {
        const uint4 r0[1] = {ldg_stream(t4 + v)};
        online_group<T, 1>(mp, sp, rp, r0, sc);
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
  rp = warp_max_nan(max_nan(rp, rq));
  if (lane == 0) {
    red[0][warp] = mp;
    red[1][warp] = sp;
    red[2][warp] = mq;
    red[3][warp] = sq;
    rawr[warp] = rp;
  }
  __syncthreads();
  if (tid == 32 && has_q) {  // the logits at the draft token, if this slice holds it
    const int x = __ldg(a.ids + (size_t)b * a.G + i);
    if (x >= lo && x < lo + n)
      reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + i] =
          make_float2(Elems<T>::one(tp, x - lo), Elems<T>::one(dp, x - lo));
  }
  if (tid == 0) {
    float Mp = red[0][0], Sp = red[1][0], Mq = red[2][0], Sq = red[3][0], raw = rawr[0];
    for (int w = 1; w < kSW; ++w) {
      merge(Mp, Sp, red[0][w], red[1][w], sc);
      merge(Mq, Sq, red[2][w], red[3][w], sc);
      raw = max_nan(raw, rawr[w]);
    }
    const bool bad = !(raw < INFINITY);  // NaN or +inf in this slice
    reinterpret_cast<float4*>(a.ws.part)[(size_t)pos * NS + s] = make_float4(bad ? NAN : Mp, Sp, bad ? NAN : Mq, Sq);
  }
}

// ----------------------------------------------------------------------------- draw kernel

template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_draw_kernel(const SampleParams a) {
  __shared__ DrawSmem sm;
  constexpr int kV = Elems<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ND = a.ndslices;
  const int b = a.B - 1 - static_cast<int>(blockIdx.x / ND);  // last-streamed rows first: still in L2
  const int d = static_cast<int>(blockIdx.x % ND);
  const int G1 = a.G + 1;
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  // launched as a programmatic dependent of the stream kernel: wait for all of it (and its writes)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (gb < 0 || gb > a.G) {  // invalid draft length: nothing was streamed for this row
    if (d == 0 && tid == 0) {
      int32_t* e = a.emitted + (size_t)b * G1;
      for (int j = 0; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = -1;
      atomicOr(a.ws.err, kErrArg);
    }
    return;
  }
  const RowState st = decide_row(a, b, gb, sm);
  if (!(st.flags & kRowInvalid)) {
    const bool resid = st.flags & kRowResid;
    const bool vec = a.vec != 0;
    const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + st.n) * a.V;
    const T* dr = resid ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + st.n) * a.V : tr;
    const int seg = 32 * kV;                     // elements per segment
    const int cpc = kR * seg;                    // elements per chunk
    const int cps = a.dslice / cpc;              // chunks per slice
    const int c0 = d * cps;
    const int c1 = min(c0 + cps, (a.V + cpc - 1) / cpc);
    const float sc = a.scale;
    for (int c = c0 + warp; c < c1; c += kSW) {
      float lw = 0.f, lp = 0.f;
      if (vec && (c + 1) * cpc <= a.V) {
        uint4 rt[kR], rd[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) {  // every load of the chunk in flight at once
          rt[r] = ldg_stream(tr + c * cpc + r * seg + lane * kV);
          if (resid) rd[r] = ldg_stream(dr + c * cpc + r * seg + lane * kV);
        }
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          float lt[kV], ld[kV];
          Elems<T>::widen(rt[r], lt);
          if (resid) Elems<T>::widen(rd[r], ld);
          float sw = 0.f, spp = 0.f;
#pragma unroll
          for (int j = 0; j < kV; ++j) {
            const float p = fast_exp2((lt[j] - st.mp) * sc) * st.ip;
            const float w = resid ? fmaxf(p - fast_exp2((ld[j] - st.mq) * sc) * st.iq, 0.f) : p;
            sw += w;
            spp += p;
          }
          lw += sw;
          lp += spp;
        }
      } else {
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          float pv[kV], wv[kV];
          seg_weights<T>(tr, dr, resid, a.V, vec, c * cpc + r * seg + lane * kV, st, sc, pv, wv);
          lw += lane_sum<kV>(wv);
          lp += lane_sum<kV>(pv);
        }
      }
      const float cw = warp_sum(lw);
      const float cp = resid ? warp_sum(lp) : cw;
      if (lane == 0) sm.cs[c - c0] = make_float2(cw, cp);
    }
    __syncthreads();
    if (tid == 0) {  // slice masses: the chunk masses summed in chunk order
      float2* dch = reinterpret_cast<float2*>(a.ws.dch) + ((size_t)b * ND + d) * cps;
      float W = 0.f, P = 0.f;
      for (int c = 0; c < c1 - c0; ++c) {
        const float2 v = sm.cs[c];
        dch[c] = v;
        W += v.x;
        P += v.y;
      }
      reinterpret_cast<float2*>(a.ws.dsum)[(size_t)b * ND + d] = make_float2(W, P);
    }
  }
  if (tid == 0) {
    __threadfence();
    sm.last = atomicAdd(a.ws.ticket + b, 1u) == static_cast<unsigned>(ND - 1);
  }
  __syncthreads();
  if (sm.last) {
    __threadfence();
    resolve_row<T>(a, b, gb, st, sm);
  }
}

template <typename T>
static cudaError_t launch_draw(const SampleParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.B * p.ndslices));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_draw_kernel<T>, p);
}

cudaError_t sample_launch(const SampleParams& p, int dtype, int phases, cudaStream_t stream) {
  const dim3 block(kStreamThreads);
  const dim3 g1(static_cast<unsigned>((long long)p.B * (p.G + 1) * p.nslices));
  cudaError_t e = cudaSuccess;
  if (dtype == 0) {
    if (phases & 1) verify_stream_kernel<float><<<g1, block, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (phases & 2) e = launch_draw<float>(p, stream);
  } else {
    if (phases & 1) verify_stream_kernel<__nv_bfloat16><<<g1, block, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (phases & 2) e = launch_draw<__nv_bfloat16>(p, stream);
  }
  return e;
}

}  // namespace specv
