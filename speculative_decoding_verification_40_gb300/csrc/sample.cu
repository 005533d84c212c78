// Sampling verification on sm_103a: one persistent launch that streams the
// logits once and spreads the final draw over the whole GPU.
//
// Speculative sampling, Algorithm 1 Phases 3-4 (Leviathan, Kalman & Matias,
// "Fast Inference from Transformers via Speculative Decoding"; paper-graph-ui
// teardown §2.3 "Algorithm Walkthrough", multigrid.ai "The algorithm",
// fullstackaihub §3 "The Algorithm at Position i"), with temperature
// standardisation p = softmax(l / T) (§2.2).
//
// A grid of co-resident CTAs (cooperative launch) takes work items in a fixed
// order from one shared counter.  Per batch row b there are
//   stream items (b, i, s): vocabulary slice s of target row (b, i) and, for
//     i < gamma_b, of draft row (b, i), read once with 16-byte loads that do
//     not allocate in L1.  Keeps online softmax normalisers per row -- the
//     running max m and S = sum 2^((l - m) log2(e)/T), rescaled when m grows,
//     one hardware exp2 per element -- and writes (m, S) for p and q.  The CTA
//     holding the draft token x_i records l_p(x_i), l_q(x_i).  The last stream
//     item of row b (atomic arrival counter) combines the normalisers, takes
//     the accept decisions u_i <= min(1, p_i(x_i)/q_i(x_i)) (with p(x) > 0),
//     finds the first rejection n, and publishes the row's draw parameters;
//   draw items (b, d), ordered after the stream items of row b + K, so the row
//     is decided and the rows it needs are still in L2: slice d of target row
//     n (and of draft row n for a residual draw); writes the mass of
//     w = max(0, p_n - q_n) and of p_n per 32-lane chunk.  The last draw item
//     of row b picks, from u_final * (total mass), the slice, then the chunk
//     from the stored chunk masses, then the token by a warp scan over that
//     chunk's recomputed weights: the residual draw, the draw from p_n when the
//     residual mass is <= 1e-15, or the bonus draw from p_{gamma_b} when
//     nothing was rejected.
// A draw item waits (bounded, SPEC_ERR_TIMEOUT) until its row is published.
// A CTA takes its next item only once its current item can no longer wait,
// so it never holds an unstarted item that others depend on.
// p and q are never written to memory; HBM traffic is the logits read once
// plus the drawn rows that have left L2.  Every counter and slot a row used is
// zero again when the row is done.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace specv {

namespace {

constexpr int kST = kStreamThreads;
constexpr int kSW = kST / 32;
constexpr unsigned kSpinLimit = 1u << 20;  // about a second of 256 ns sleeps, then SPEC_ERR_TIMEOUT

enum : int { kRowInvalid = 1, kRowResid = 2, kRowTimeout = 4 };

struct __align__(16) RowState {
  int n, flags;
  float mp, ip, mq, iq;
  int pad0, pad1;
};

// Row state as written by another CTA: read through L2 (two 16-byte loads).
__device__ __forceinline__ RowState load_state(const RowState* p) {
  const int4* q = reinterpret_cast<const int4*>(p);
  const int4 x = __ldcg(q), y = __ldcg(q + 1);
  RowState s;
  s.n = x.x;
  s.flags = x.y;
  s.mp = __int_as_float(x.z);
  s.ip = __int_as_float(x.w);
  s.mq = __int_as_float(y.x);
  s.iq = __int_as_float(y.y);
  s.pad0 = s.pad1 = 0;
  return s;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Work item codes past the end: the CTA leaves.
__device__ __forceinline__ void publish(const Workspace& ws, int b) {
  __threadfence();
  atomicExch(ws.ready + b, 1u);
}

// Online normaliser update with a group of raw logits.
template <int kCnt>
__device__ __forceinline__ void online(float& m, float& s, float& raw, const float* f, float sc) {
  float vm = f[0];
#pragma unroll
  for (int j = 1; j < kCnt; ++j) vm = max_nan(vm, f[j]);
  raw = max_nan(raw, vm);
  if (vm > -INFINITY) {
    if (vm > m) {
      s *= fast_exp2((m - vm) * sc);
      m = vm;
    }
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kCnt; ++j) acc += fast_exp2((f[j] - m) * sc);
    s += acc;
  }
}

// Merge normaliser (om, os) into (m, s).
__device__ __forceinline__ void merge(float& m, float& s, float om, float os, float sc) {
  const float M = fmaxf(m, om);
  if (!(M > -INFINITY)) return;  // both empty
  const float x = m > -INFINITY ? s * fast_exp2((m - M) * sc) : 0.f;
  const float y = om > -INFINITY ? os * fast_exp2((om - M) * sc) : 0.f;
  s = x + y;
  m = M;
}

struct Smem {
  float red[4][kSW];
  float raw[kSW];
  float mp[kMaxGamma + 1], sp[kMaxGamma + 1], mq[kMaxGamma + 1], sq[kMaxGamma + 1];
  int acc[kMaxGamma + 1];
  float2 cs[kMaxChunksPerSlice];  // chunk masses of one draw slice (w, p)
  float2 ds[kMaxSlices];          // slice masses of one drawn row (w, p)
  unsigned long long next;        // the item this CTA takes after the current one
  uint32_t err;
  int last, ok, pick, n;
  float t, pre;
  RowState st;
};

// Weights of one lane's kV elements of chunk c (32 lanes x kV elements) of the
// drawn row(s): p, and w = max(0, p - q) for a residual draw (w = p otherwise).
// Elements past V weigh 0.  The same arithmetic serves the mass pass and the
// final scan, so both see identical weights.
template <typename T>
__device__ __forceinline__ void chunk_weights(const T* tr, const T* dr, bool resid, int V, bool vec, int c, int lane,
                                              const RowState& st, float sc, float (&p)[Elems<T>::kVec],
                                              float (&w)[Elems<T>::kVec]) {
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

// ----------------------------------------------------------------------------- stream items

template <typename T>
__device__ __noinline__ void row_decide(const SampleParams& a, int b, int gb, Smem& sm);

template <typename T>
__device__ void stream_item(const SampleParams& a, int b, int i, int s, Smem& sm) {
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = a.G + 1;
  const int NS = a.nslices;
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  if (gb < 0 || gb > a.G) {  // invalid draft length: publish an invalid row once
    if (i == 0 && s == 0 && tid == 0) {
      RowState* st = reinterpret_cast<RowState*>(a.ws.rowstate) + b;
      st->flags = kRowInvalid;
      atomicOr(a.ws.err, kErrArg);
      publish(a.ws, b);
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
  rp = warp_max_nan(max_nan(rp, rq));
  if (lane == 0) {
    sm.red[0][warp] = mp;
    sm.red[1][warp] = sp;
    sm.red[2][warp] = mq;
    sm.red[3][warp] = sq;
    sm.raw[warp] = rp;
  }
  __syncthreads();
  // from here on this item cannot wait: take the next one while thread 0 finishes
  if (tid == 32) sm.next = atomicAdd(a.ws.fetch, 1ull);
  if (tid == 0) {
    float Mp = sm.red[0][0], Sp = sm.red[1][0], Mq = sm.red[2][0], Sq = sm.red[3][0], raw = sm.raw[0];
    for (int w = 1; w < kSW; ++w) {
      merge(Mp, Sp, sm.red[0][w], sm.red[1][w], sc);
      merge(Mq, Sq, sm.red[2][w], sm.red[3][w], sc);
      raw = max_nan(raw, sm.raw[w]);
    }
    const bool bad = !(raw < INFINITY);  // NaN or +inf in this slice
    reinterpret_cast<float4*>(a.ws.part)[((size_t)b * G1 + i) * NS + s] =
        make_float4(bad ? NAN : Mp, Sp, bad ? NAN : Mq, Sq);
    if (has_q) {
      const int x = __ldg(a.ids + (size_t)b * a.G + i);
      if (x >= lo && x < lo + n)
        reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + i] =
            make_float2(Elems<T>::one(tp, x - lo), Elems<T>::one(dp, x - lo));
    }
    __threadfence();
    const unsigned prev = atomicAdd(a.ws.ticket + b, 1u);
    sm.last = prev == static_cast<unsigned>(NS * (gb + 1) - 1);
  }
  __syncthreads();
  if (sm.last) {
    __threadfence();
    row_decide<T>(a, b, gb, sm);
  }
}

// Last stream item of row b: normalisers, accept decisions, first rejection; publishes the draw.
template <typename T>
__device__ __noinline__ void row_decide(const SampleParams& a, int b, int gb, Smem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = a.G + 1;
  const int NS = a.nslices;
  const float sc = a.scale;
  float4* part = reinterpret_cast<float4*>(a.ws.part) + (size_t)b * G1 * NS;

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
  // the partials and logit slots are consumed: back to zero
  for (int k = tid; k < (gb + 1) * NS; k += kST) part[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = tid; k < gb; k += kST) reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + k] = make_float2(0.f, 0.f);
  if (tid == 0) {
    int n = gb;
    for (int i = 0; i < gb; ++i) {
      if (sm.acc[i] == 0) {
        n = i;
        break;
      }
    }
    RowState st = {};
    st.n = n;
    if (sm.err) {
      st.flags = kRowInvalid;
      atomicOr(a.ws.err, sm.err);
    } else {
      st.flags = n < gb ? kRowResid : 0;
      st.mp = sm.mp[n];
      st.ip = 1.f / sm.sp[n];
      if (n < gb) {
        st.mq = sm.mq[n];
        st.iq = 1.f / sm.sq[n];
      }
    }
    reinterpret_cast<RowState*>(a.ws.rowstate)[b] = st;
    publish(a.ws, b);
  }
}

// ----------------------------------------------------------------------------- draw items

template <typename T>
__device__ __noinline__ void resolve_row(const SampleParams& a, int b, Smem& sm);

template <typename T>
__device__ __noinline__ void draw_item(const SampleParams& a, int b, int d, Smem& sm) {
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = a.G + 1;
  const int ND = a.nslices;
  if (tid == 0) {
    unsigned v = 0, spins = 0;
    while ((v = ld_acquire(a.ws.ready + b)) == 0u && ++spins < kSpinLimit) __nanosleep(256);
    sm.ok = v != 0u;
    if (v) {
      sm.st = load_state(reinterpret_cast<const RowState*>(a.ws.rowstate) + b);
    } else {
      atomicOr(&reinterpret_cast<RowState*>(a.ws.rowstate)[b].flags, kRowTimeout);
      atomicOr(a.ws.err, kErrTimeout);
    }
  }
  __syncthreads();
  const bool ok = sm.ok;
  const RowState st = sm.st;
  if (tid == 32) sm.next = atomicAdd(a.ws.fetch, 1ull);  // past the wait: nothing left to block on
  float2* dsum = reinterpret_cast<float2*>(a.ws.dsum) + (size_t)b * ND;
  if (ok && !(st.flags & kRowInvalid)) {
    const bool resid = st.flags & kRowResid;
    const bool vec = a.vec != 0;
    const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + st.n) * a.V;
    const T* dr = resid ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + st.n) * a.V : tr;
    const int cpc = 32 * kV;                     // elements per chunk
    const int cps = a.slice / cpc;               // chunks per slice
    const int c0 = d * cps;
    const int c1 = min(c0 + cps, (a.V + cpc - 1) / cpc);
    const float sc = a.scale;
    for (int cb = c0 + warp; cb < c1; cb += U * kSW) {
      uint4 rt[U], rd[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {  // loads of U whole chunks in flight
        const int c = cb + u * kSW;
        if (vec && c < c1 && (c + 1) * cpc <= a.V) {
          rt[u] = ldg_stream(tr + c * cpc + lane * kV);
          if (resid) rd[u] = ldg_stream(dr + c * cpc + lane * kV);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = cb + u * kSW;
        if (c >= c1) break;  // uniform across the warp
        float pv[kV], wv[kV];
        if (vec && (c + 1) * cpc <= a.V) {
          float lt[kV], ld[kV];
          Elems<T>::widen(rt[u], lt);
          if (resid) Elems<T>::widen(rd[u], ld);
#pragma unroll
          for (int j = 0; j < kV; ++j) {
            pv[j] = fast_exp2((lt[j] - st.mp) * sc) * st.ip;
            wv[j] = resid ? fmaxf(pv[j] - fast_exp2((ld[j] - st.mq) * sc) * st.iq, 0.f) : pv[j];
          }
        } else {
          chunk_weights<T>(tr, dr, resid, a.V, vec, c, lane, st, sc, pv, wv);
        }
        const float cw = warp_sum(lane_sum<kV>(wv));
        const float cp = resid ? warp_sum(lane_sum<kV>(pv)) : cw;
        if (lane == 0) sm.cs[c - c0] = make_float2(cw, cp);
      }
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
      dsum[d] = make_float2(W, P);
    }
  }
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(a.ws.dticket + b, 1u);
    sm.last = prev == static_cast<unsigned>(ND - 1);
  }
  __syncthreads();
  if (sm.last) {
    __threadfence();
    resolve_row<T>(a, b, sm);
  }
}

// Last draw item of row b: slice, chunk and token of the draw; the row's outputs; reset.
template <typename T>
__device__ __noinline__ void resolve_row(const SampleParams& a, int b, Smem& sm) {
  constexpr int kV = Elems<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31;
  const int G1 = a.G + 1;
  const int ND = a.nslices;
  const int cpc = 32 * kV;
  const int cps = a.slice / cpc;
  const int nc = (a.V + cpc - 1) / cpc;
  RowState* rs = reinterpret_cast<RowState*>(a.ws.rowstate) + b;
  float2* dsum = reinterpret_cast<float2*>(a.ws.dsum) + (size_t)b * ND;
  float2* dch = reinterpret_cast<float2*>(a.ws.dch) + (size_t)b * ND * cps;
  int32_t* e = a.emitted + (size_t)b * G1;
  if (tid == 0) {
    sm.st = load_state(rs);
    sm.pick = -1;
  }
  __syncthreads();
  const RowState st = sm.st;
  const bool resid = st.flags & kRowResid;
  const bool failed = st.flags & (kRowInvalid | kRowTimeout);
  const float uf = failed ? 0.f : __ldg(a.uniforms + (size_t)b * G1 + a.G);
  if (!failed && tid < ND) sm.ds[tid] = __ldcg(dsum + tid);
  __syncthreads();
  if (!failed && tid == 0) {
    // total mass in slice order; the residual, or p when the residual mass is degenerate
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
    sm.n = (use_p ? 1 : 0) | (fallback ? 2 : 0);
    sm.t = t;
    sm.pre = pre;
  }
  __syncthreads();
  // chunk within the chosen slice: stage its chunk masses, then one thread scans them
  const int sd = sm.pick;
  if (!failed && sd >= 0) {
    const int c0 = sd * cps, c1 = min(c0 + cps, nc);
    for (int c = c0 + tid; c < c1; c += kST) sm.cs[c - c0] = __ldcg(dch + (size_t)sd * cps + (c - c0));
    __syncthreads();
    if (tid == 0) {
      const bool use_p = sm.n & 1;
      bool fallback = sm.n & 2;
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
      sm.n = (use_p ? 1 : 0) | (fallback ? 2 : 0);
      sm.pre = cpre;
    }
  } else if (tid == 0) {
    sm.pick = -1;
  }
  __syncthreads();
  const int pc = sm.pick;
  if (!failed && pc >= 0 && tid < 32) {  // warp 0: the token inside the chunk
    const bool use_p = sm.n & 1;
    const bool fallback = sm.n & 2;
    const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + st.n) * a.V;
    const T* dr = resid ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + st.n) * a.V : tr;
    float pv[kV], wv[kV];
    chunk_weights<T>(tr, dr, resid && !use_p, a.V, a.vec != 0, pc, lane, st, a.scale, pv, wv);
    const float ls = lane_sum<kV>(wv);
    const float inc = warp_inclusive_scan(ls, lane);
    float exc = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) exc = 0.f;
    const float tt = sm.t - sm.pre;
    int lastj = -1;
#pragma unroll
    for (int j = 0; j < kV; ++j)
      if (wv[j] > 0.f) lastj = j;
    const int base = pc * cpc + lane * kV;
    int tok = -1;
    const unsigned hit = fallback ? 0u : __ballot_sync(0xffffffffu, ls > 0.f && inc > tt);
    if (hit) {
      const int l = __ffs(hit) - 1;
      if (lane == l) {
        float c = exc;
        for (int j = 0; j < kV; ++j) {
          c += wv[j];
          if (wv[j] > 0.f && c > tt) {
            tok = base + j;
            break;
          }
        }
        if (tok < 0) tok = base + lastj;
      }
      tok = __shfl_sync(0xffffffffu, tok, l);
    } else {
      const unsigned nz = __ballot_sync(0xffffffffu, ls > 0.f);
      if (nz) {
        const int l = 31 - __clz(nz);
        if (lane == l) tok = base + lastj;
        tok = __shfl_sync(0xffffffffu, tok, l);
      }
    }
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
    if (!failed) atomicOr(a.ws.err, kErrNonfinite);
  }
  // every slot of this row back to zero for the next call
  const int nch = ND * cps;
  for (int k = tid; k < nch; k += kST) dch[k] = make_float2(0.f, 0.f);
  for (int k = tid; k < ND; k += kST) dsum[k] = make_float2(0.f, 0.f);
  if (tid == 0) {
    *rs = RowState{};
    a.ws.ready[b] = 0u;
    a.ws.ticket[b] = 0u;
    a.ws.dticket[b] = 0u;
  }
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_fused_kernel(const SampleParams a) {
  __shared__ Smem sm;
  const int tid = threadIdx.x;
  const long long SS = (long long)(a.G + 1) * a.nslices;  // stream items per batch row
  const long long ND = a.nslices;                         // draw items per batch row
  const long long K = a.lag;                              // draw items trail stream items by K rows
  const long long B = a.B;
  const long long head = K * SS;                          // units 0..K-1: stream items only
  const long long body = head + (B - K) * (SS + ND);      // units K..B-1: stream then draw items
  const unsigned long long total = body + K * ND;         // units B..B+K-1: draw items only
  constexpr unsigned long long kUnset = ~0ull;
  if (tid == 0) sm.next = atomicAdd(a.ws.fetch, 1ull);
  __syncthreads();
  for (;;) {
    const unsigned long long it = sm.next;
    if (it >= total) break;
    __syncthreads();  // every thread has read sm.next
    if (tid == 0) sm.next = kUnset;
    __syncthreads();
    const long long x0 = static_cast<long long>(it);
    if (x0 < head) {
      const long long r = x0 / SS, j = x0 - r * SS;
      stream_item<T>(a, static_cast<int>(r), static_cast<int>(j / ND), static_cast<int>(j % ND), sm);
    } else if (x0 < body) {
      const long long x = x0 - head;
      const long long u = x / (SS + ND);
      const long long j = x - u * (SS + ND);
      if (j >= SS)
        draw_item<T>(a, static_cast<int>(u), static_cast<int>(j - SS), sm);
      else
        stream_item<T>(a, static_cast<int>(K + u), static_cast<int>(j / ND), static_cast<int>(j % ND), sm);
    } else {
      const long long x = x0 - body;
      draw_item<T>(a, static_cast<int>(B - K + x / ND), static_cast<int>(x % ND), sm);
    }
    __syncthreads();  // shared memory is reused by the next item
    if (tid == 0 && sm.next == kUnset) sm.next = atomicAdd(a.ws.fetch, 1ull);  // items that returned early
    __syncthreads();
  }
  // the last CTA to leave returns the counters to zero for the next call
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.ws.done, 1u) == gridDim.x - 1) {
      *a.ws.fetch = 0ull;
      *a.ws.done = 0u;
    }
  }
}

cudaError_t sample_occupancy(int dtype, int* ctas_per_sm) {
  if (dtype == 0)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, verify_fused_kernel<float>, kStreamThreads, 0);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, verify_fused_kernel<__nv_bfloat16>,
                                                       kStreamThreads, 0);
}

cudaError_t sample_launch(const SampleParams& p, int dtype, int grid, cudaStream_t stream) {
  void* args[] = {const_cast<SampleParams*>(&p)};
  if (dtype == 0)
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(verify_fused_kernel<float>), dim3(grid),
                                       dim3(kStreamThreads), args, 0, stream);
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(verify_fused_kernel<__nv_bfloat16>), dim3(grid),
                                     dim3(kStreamThreads), args, 0, stream);
}

}  // namespace specv
