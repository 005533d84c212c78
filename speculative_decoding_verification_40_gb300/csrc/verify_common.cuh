// Device helpers shared by the sampling kernels: the online softmax pass over a slice of a logit row,
// the combination of slice normalisers, the accept test, and the draw weights.
//
// Speculative sampling, Algorithm 1 Phases 3-4 (Leviathan, Kalman & Matias; paper-graph-ui teardown
// §2.3 "Algorithm Walkthrough"), with temperature standardisation p = softmax(l / T) (§2.2).
#pragma once

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
  float uf;      // the final draw's uniform (thread 0 only)
  int x;         // draft id x_i of this thread's position i = thread index (i < gamma_b)
  float cp, cq;  // p = 2^(l log2(e)/T + cp), cp = -m_p log2(e)/T - log2 S_p; q likewise (times the lenience)
  float tt, dt;  // standardisation thresholds of the drawn target / draft row (-inf: none)
};

// p and w = max(0, p - q) (w = p unless resid) from widened logits: one FFMA and one exp2 per
// probability; the chunk-mass pass, scalar or packed, computes exactly these.
template <int kV>
__device__ __forceinline__ void weights_of(const float (&lt)[kV], const float (&ld)[kV], bool resid,
                                           const RowState& st, float sc, float (&p)[kV], float (&w)[kV]) {
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    p[j] = fast_exp2(fmaf(masked(lt[j], st.tt), sc, st.cp));
    w[j] = resid ? fmaxf(p[j] - fast_exp2(fmaf(masked(ld[j], st.dt), sc, st.cq)), 0.f) : p[j];
  }
}

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
  weights_of<kV>(lt, ld, resid, st, sc, p, w);
}

template <int kV>
__device__ __forceinline__ float lane_sum(const float (&w)[kV]) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kV; ++j) s += w[j];
  return s;
}

// Row normalisers of one position from its NS slice partials (m_p, S_p, m_q, S_q), combined by one warp
// in a fixed order, so every caller gets the same values bit for bit.  Every lane returns them.
// pr: lane r < NS holds slice r's partial (m_p, S_p, m_q, S_q), the other lanes (-inf, 0, -inf, 0).
__device__ __forceinline__ float4 combine_partials(float4 pr, int NS, float sc) {
  const float Mp = warp_max_nan(pr.x);
  const float Mq = warp_max_nan(pr.z);
  const float tp = (pr.x > -INFINITY && Mp < INFINITY) ? pr.y * fast_exp2((pr.x - Mp) * sc) : 0.f;
  const float tq = (pr.z > -INFINITY && Mq < INFINITY) ? pr.w * fast_exp2((pr.z - Mq) * sc) : 0.f;
  float Sp = 0.f, Sq = 0.f;
  for (int r = 0; r < NS; ++r) {
    Sp += __shfl_sync(0xffffffffu, tp, r);
    Sq += __shfl_sync(0xffffffffu, tq, r);
  }
  return make_float4(Mp, Sp, Mq, Sq);
}

__device__ __forceinline__ float4 load_partial(const float4* __restrict__ part_pos, int NS) {
  float4 pr = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  if ((threadIdx.x & 31) < NS) pr = __ldcg(part_pos + (threadIdx.x & 31));
  return pr;
}

__device__ __forceinline__ float4 position_norm(const float4* __restrict__ part_pos, int NS, float sc) {
  return combine_partials(load_partial(part_pos, NS), NS, sc);
}

// Accept test of guess i < gamma_b of row b, u_i <= min(1, p(x_i)/q(x_i)) with p(x_i) > 0, from the
// position's normalisers and the logits at the draft token; err collects what makes the row invalid.
// x = x_i, ui = u_i and xl = (l_p(x_i), l_q(x_i)) are passed in, so callers can load them early.
__device__ __forceinline__ int accept_test(const SampleParams& a, float4 nm, int x, float ui, float2 xl,
                                           uint32_t& err) {
  if (!(nm.x > -INFINITY && nm.x < INFINITY)) err |= kErrNonfinite;
  if (!(nm.z > -INFINITY && nm.z < INFINITY)) err |= kErrNonfinite;
  if (x < 0 || x >= a.V) err |= kErrToken;
  if (!(ui >= 0.f && ui < 1.f)) err |= kErrArg;
  if (err) return 0;
  const float sc = a.scale;
  const float px = fast_exp2((xl.x - nm.x) * sc) / nm.y;
  const float qx = fast_exp2((xl.y - nm.z) * sc) / nm.w * a.lq;  // l q(x) (l = 1 unless lenient)
  const float ratio = px >= qx ? 1.f : px / qx;  // min(1, p/q); q = 0 < p gives 1
  return (px > 0.f && ui <= ratio) ? 1 : 0;
}

}  // namespace

// A 16-byte vector of -inf logits (the padding of a thread's last, partial group of loads).
template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec() {
  return sizeof(T) == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                        : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}

// Online normalisers (m, S) of n logits of one row (and of a second row when has_q), this thread's
// share: 16-byte vectors when vec, in groups of U per row in flight, then a scalar tail.  raw tracks the
// NaN-propagating maximum of the raw logits (NaN / +inf detection).
template <typename T, bool kMask>
__device__ __forceinline__ void slice_normalisers(const T* __restrict__ tp, const T* __restrict__ dp, bool has_q,
                                                  int n, bool vec, float sc, float tt, float dt, float& mp,
                                                  float& sp, float& rp, float& mq, float& sq, float& rq) {
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 4;
  const int tid = threadIdx.x;
  int done = 0;
  if (vec) {
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
        online_group<T, U, kMask>(mp, sp, rp, r0, sc, tt);
        online_group<T, U, kMask>(mq, sq, rq, r1, sc, dt);
      }
      // the thread's last (at most U - 1) vectors as one group whose missing vectors read as -inf, so all
      // of their loads are in flight at once (a 64 KB bfloat16 row of 4000 vectors leaves three)
      if (v < nv) {
        uint4 r0[U], r1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = v + u * kST < nv ? ldg_stream(t4 + v + u * kST) : neg_inf_vec<T>();
#pragma unroll
        for (int u = 0; u < U; ++u) r1[u] = v + u * kST < nv ? ldg_stream(d4 + v + u * kST) : neg_inf_vec<T>();
        online_group<T, U, kMask>(mp, sp, rp, r0, sc, tt);
        online_group<T, U, kMask>(mq, sq, rq, r1, sc, dt);
      }
    } else {
      for (; v + (U - 1) * kST < nv; v += U * kST) {
        uint4 r0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = ldg_stream(t4 + v + u * kST);
        online_group<T, U, kMask>(mp, sp, rp, r0, sc, tt);
      }
      if (v < nv) {
        uint4 r0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = v + u * kST < nv ? ldg_stream(t4 + v + u * kST) : neg_inf_vec<T>();
        online_group<T, U, kMask>(mp, sp, rp, r0, sc, tt);
      }
    }
    done = nv * kV;
  }
  for (int k = done + tid; k < n; k += kST) {
    float f[1] = {Elems<T>::one(tp, k)};
    online<1, kMask>(mp, sp, rp, f, sc, tt);
    if (has_q) {
      f[0] = Elems<T>::one(dp, k);
      online<1, kMask>(mq, sq, rq, f, sc, dt);
    }
  }
}

}  // namespace specv
