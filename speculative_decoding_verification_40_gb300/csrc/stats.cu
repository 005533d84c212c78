// Per-position acceptance statistics on sm_103a.
//
// Definition 3.2, Lemma 3.3 and Theorem 3.5 of Leviathan, Kalman & Matias,
// "Fast Inference from Transformers via Speculative Decoding" (paper-graph-ui
// teardown, "Computing alpha from p and q"): for each position i < gamma_b,
// beta = sum_x min(p(x), q(x)), the residual mass sum_x max(0, p(x) - q(x)),
// and p(x_i), q(x_i), min(1, p(x_i)/q(x_i)) at the draft token, with p and q
// the temperature softmaxes of the target and draft rows (§2.2).
//
// beta needs the row normalisers of p and q before any element can be
// compared.  One thread-block cluster of CS CTAs per (batch row b, position
// i); CTA r of the cluster owns the vocabulary slice [r*L, r*L + L) of target
// and draft row (b, i).  Each CTA
//   1. streams its two slices from HBM (16-byte loads, no L1 allocation),
//      keeping online softmax normalisers (running max m,
//      S = sum 2^((l - m) log2(e)/T)) for p and q;
//   2. pushes its (m, S) pair into every CTA of the cluster (distributed
//      shared memory stores) and meets them at a cluster barrier, so every CTA
//      combines the same values in the same order;
//   3. reads its slices again -- microseconds later, from L2 -- with
//      p = 2^(l log2(e)/T - c_p), c_p = m log2(e)/T + log2 S (likewise q),
//      summing min(p, q) and p; the residual mass is
//      sum p - sum min(p, q) = sum max(0, p - q);
//   4. pushes those sums, and p(x_i), q(x_i) if it owns x_i, to rank 0, which
//      writes the position's statistics after a second cluster barrier.
// HBM traffic is the logits once (the second read hits L2: the slices a whole
// GPU of resident CTAs holds between the two reads are a few tens of MB); no
// CTA touches another's shared memory after the second barrier.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "softmax.cuh"

namespace specv {

namespace {

constexpr int kT = kStatsThreads;
constexpr int kW = kT / 32;
constexpr int kU = 4;  // 16-byte loads in flight per thread and row
constexpr int kMinBlocks = 4;  // resident CTAs per SM the register budget is sized for

// Adds min(p, q) and p over kV elements of each row, p = 2^(l_p sc + ncp), q = 2^(l_q sc + ncq).
template <int kV>
__device__ __forceinline__ void overlap(const float* f, const float* g, float sc, float ncp, float ncq, float& tmin,
                                        float& tp) {
  if constexpr (kV == 8) {
    // bfloat16 rows: (p, q) and (min, p) pairs through the packed f32x2 FMA / add, the same rounding as
    // the scalar operations
    const unsigned long long sc2 = pack2(sc, sc), nc2 = pack2(ncp, ncq);
    unsigned long long acc = pack2(tmin, tp);
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      float ep, eq;
      unpack2(fma2(pack2(f[j], g[j]), sc2, nc2), ep, eq);
      const float p = fast_exp2(ep), q = fast_exp2(eq);
      acc = add2(acc, pack2(fminf(p, q), p));
    }
    unpack2(acc, tmin, tp);
  } else {
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      const float p = fast_exp2(fmaf(f[j], sc, ncp));
      const float q = fast_exp2(fmaf(g[j], sc, ncq));
      tmin += fminf(p, q);
      tp += p;
    }
  }
}

__device__ __forceinline__ void write_stats(const VerifyParams& a, size_t o, float beta, float px, float qx, float ap,
                                            float z) {
  if (a.beta) a.beta[o] = beta;
  if (a.p_draft) a.p_draft[o] = px;
  if (a.q_draft) a.q_draft[o] = qx;
  if (a.accept_prob) a.accept_prob[o] = ap;
  if (a.resid) a.resid[o] = z;
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kT, kMinBlocks) stats_rows_kernel(const VerifyParams a) {
  __shared__ __align__(16) float x1[kMaxCluster][4];  // (m_p, S_p, m_q, S_q) of every CTA; NaN maxima if bad
  __shared__ __align__(16) float x2[kMaxCluster][4];  // rank 0: sum min(p,q), sum max(0,p-q), p(x), q(x)
  __shared__ float red[5][kW];
  __shared__ float bc[4];
  constexpr int kV = Elems<T>::kVec;

  const int CS = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int pos = blockIdx.x / CS;  // b * G + i
  const int b = pos / a.G;
  const int i = pos - b * a.G;
  const int G1 = a.G + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  if (gb < 0 || gb > a.G || i >= gb) {  // the whole cluster leaves together; padded positions are never read
    if (rank == 0 && tid == 0) {
      write_stats(a, pos, NAN, NAN, NAN, NAN, NAN);
      if (gb < 0 || gb > a.G) atomicOr(a.ws.err, kErrArg);
    }
    return;
  }
  const int lo = rank * a.L;
  const int n = max(0, min(a.V, lo + a.L) - lo);
  // uniform over the cluster (the same sizes in every CTA), so the whole cluster leaves together
  if (!bounds_ok(pos < a.B * a.G && CS <= kMaxCluster && (long long)CS * a.L >= a.V, a.ws.err)) return;
  const float sc = a.scale;
  const T* tp = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + i) * a.V + lo;
  const T* dp = reinterpret_cast<const T*>(a.draft) + (size_t)pos * a.V + lo;
  const uint4* t4 = reinterpret_cast<const uint4*>(tp);
  const uint4* d4 = reinterpret_cast<const uint4*>(dp);
  const int nv = a.vec ? n / kV : 0;  // 16-byte vectors (rows on a 16-byte boundary); scalar tail after them
  const int x = __ldg(a.ids + pos);
  const bool owner = x >= lo && x < lo + n;
  float lpx = 0.f, lqx = 0.f;  // logits at the draft token, loaded early by the thread that reports them
  if (tid == 0 && owner) {
    lpx = Elems<T>::one(tp, x - lo);
    lqx = Elems<T>::one(dp, x - lo);
  }

  // 1. online normalisers of the slices, streamed from HBM
  float mp = -INFINITY, sp = 0.f, rp = -INFINITY;
  float mq = -INFINITY, sq = 0.f, rq = -INFINITY;
  {
    int v = tid;
    for (; v + (kU - 1) * kT < nv; v += kU * kT) {
      uint4 r0[kU], r1[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) r0[u] = ldg_stream(t4 + v + u * kT);
#pragma unroll
      for (int u = 0; u < kU; ++u) r1[u] = ldg_stream(d4 + v + u * kT);
      online_group<T, kU>(mp, sp, rp, r0, sc);
      online_group<T, kU>(mq, sq, rq, r1, sc);
    }
    for (; v < nv; v += kT) {
      const uint4 r0[1] = {ldg_stream(t4 + v)};
      const uint4 r1[1] = {ldg_stream(d4 + v)};
      online_group<T, 1>(mp, sp, rp, r0, sc);
      online_group<T, 1>(mq, sq, rq, r1, sc);
    }
    for (int k = nv * kV + tid; k < n; k += kT) {
      float f[1] = {Elems<T>::one(tp, k)};
      online<1>(mp, sp, rp, f, sc);
      f[0] = Elems<T>::one(dp, k);
      online<1>(mq, sq, rq, f, sc);
    }
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mp, s), os = __shfl_xor_sync(0xffffffffu, sp, s);
    const float qm = __shfl_xor_sync(0xffffffffu, mq, s), qs = __shfl_xor_sync(0xffffffffu, sq, s);
    merge(mp, sp, om, os, sc);
    merge(mq, sq, qm, qs, sc);
  }
  rp = warp_max_nan(max_nan(rp, rq));
  if (lane == 0) {
    red[0][warp] = mp;
    red[1][warp] = sp;
    red[2][warp] = mq;
    red[3][warp] = sq;
    red[4][warp] = rp;
  }
  __syncthreads();
  if (warp == 0) {  // merge the warps' normalisers, then push the slice's pair to every CTA of the cluster
    float Mp = lane < kW ? red[0][lane] : -INFINITY, Sp = lane < kW ? red[1][lane] : 0.f;
    float Mq = lane < kW ? red[2][lane] : -INFINITY, Sq = lane < kW ? red[3][lane] : 0.f;
    float raw = lane < kW ? red[4][lane] : -INFINITY;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, Mp, s), os = __shfl_xor_sync(0xffffffffu, Sp, s);
      const float qm = __shfl_xor_sync(0xffffffffu, Mq, s), qs = __shfl_xor_sync(0xffffffffu, Sq, s);
      merge(Mp, Sp, om, os, sc);
      merge(Mq, Sq, qm, qs, sc);
    }
    raw = warp_max_nan(raw);
    const bool bad = !(raw < INFINITY);  // NaN or +inf in this slice
    if (lane < CS)
      dsmem_st_v4(dsmem_map(smem_addr(&x1[rank][0]), static_cast<uint32_t>(lane)), bad ? NAN : Mp, Sp,
                  bad ? NAN : Mq, Sq);
  }

  // 2. cluster barrier A: every CTA now holds every slice's normalisers
  cluster_sync();
  if (warp == 0) {
    const float m0 = lane < CS ? x1[lane][0] : -INFINITY, s0 = lane < CS ? x1[lane][1] : 0.f;
    const float m1 = lane < CS ? x1[lane][2] : -INFINITY, s1 = lane < CS ? x1[lane][3] : 0.f;
    const float gmp = warp_max_nan(m0);
    const float gmq = warp_max_nan(m1);
    // NaN or +inf anywhere, or a row that is entirely -inf
    const bool bad = !(gmp < INFINITY && gmp > -INFINITY) || !(gmq < INFINITY && gmq > -INFINITY);
    float Sp = 0.f, Sq = 0.f;
    if (!bad) {
      const float tpv = m0 > -INFINITY ? s0 * fast_exp2((m0 - gmp) * sc) : 0.f;
      const float tqv = m1 > -INFINITY ? s1 * fast_exp2((m1 - gmq) * sc) : 0.f;
      for (int r = 0; r < CS; ++r) {  // fixed order: identical sums in every CTA
        Sp += __shfl_sync(0xffffffffu, tpv, r);
        Sq += __shfl_sync(0xffffffffu, tqv, r);
      }
    }
    if (lane == 0) {
      bc[0] = bad ? NAN : -gmp * sc;
      bc[1] = bad ? NAN : Sp;
      bc[2] = bad ? NAN : -gmq * sc;
      bc[3] = bad ? NAN : Sq;
    }
  }
  __syncthreads();
  const float ncp0 = bc[0], Sp = bc[1], ncq0 = bc[2], Sq = bc[3];
  const bool bad = !(Sp > 0.f);
  const float ncp = ncp0 - __log2f(Sp), ncq = ncq0 - __log2f(Sq);

  // 3. overlaps over the slice, read again (from L2)
  float tmin = 0.f, tpp = 0.f;
  if (!bad) {
    int v = tid;
    for (; v + (kU - 1) * kT < nv; v += kU * kT) {
      uint4 r0[kU], r1[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) r0[u] = ldg_stream(t4 + v + u * kT);
#pragma unroll
      for (int u = 0; u < kU; ++u) r1[u] = ldg_stream(d4 + v + u * kT);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        float f[kV], g[kV];
        Elems<T>::widen(r0[u], f);
        Elems<T>::widen(r1[u], g);
        overlap<kV>(f, g, sc, ncp, ncq, tmin, tpp);
      }
    }
    for (; v < nv; v += kT) {
      float f[kV], g[kV];
      Elems<T>::widen(ldg_stream(t4 + v), f);
      Elems<T>::widen(ldg_stream(d4 + v), g);
      overlap<kV>(f, g, sc, ncp, ncq, tmin, tpp);
    }
    for (int k = nv * kV + tid; k < n; k += kT) {
      const float f[1] = {Elems<T>::one(tp, k)};
      const float g[1] = {Elems<T>::one(dp, k)};
      overlap<1>(f, g, sc, ncp, ncq, tmin, tpp);
    }
  }
  tpp = warp_sum(tpp - tmin);  // sum max(0, p - q) = sum p - sum min(p, q)
  tmin = warp_sum(tmin);
  if (lane == 0) {
    red[0][warp] = tmin;
    red[1][warp] = tpp;
  }
  __syncthreads();
  if (warp == 0) {
    float bt = lane < kW ? red[0][lane] : 0.f, zt = lane < kW ? red[1][lane] : 0.f;
    for (int s = 16; s > 0; s >>= 1) {
      bt += __shfl_xor_sync(0xffffffffu, bt, s);
      zt += __shfl_xor_sync(0xffffffffu, zt, s);
    }
    if (lane == 0) {
      float px = -1.f, qx = -1.f;
      if (!bad && owner) {
        px = fast_exp2(fmaf(lpx, sc, ncp0)) / Sp;
        qx = fast_exp2(fmaf(lqx, sc, ncq0)) / Sq;
      }
      dsmem_st_v4(dsmem_map(smem_addr(&x2[rank][0]), 0u), bt, zt, px, qx);
    }
  }

  // 4. cluster barrier B; rank 0 combines the slices in rank order and writes the statistics
  cluster_sync();
  if (rank == 0 && warp == 0) {
    float Bt = 0.f, Zt = 0.f;
    const float rb = lane < CS ? x2[lane][0] : 0.f, rz = lane < CS ? x2[lane][1] : 0.f;
    for (int r = 0; r < CS; ++r) {
      Bt += __shfl_sync(0xffffffffu, rb, r);
      Zt += __shfl_sync(0xffffffffu, rz, r);
    }
    const bool xok = x >= 0 && x < a.V;
    if (lane == 0) {
      if (bad || !xok) {
        write_stats(a, pos, NAN, NAN, NAN, NAN, NAN);
        atomicOr(a.ws.err, bad ? kErrNonfinite : kErrToken);
      } else {
        const int owner = x / a.L;
        const float pxr = x2[owner][2], qxr = x2[owner][3];
        const float ratio = pxr >= qxr ? 1.f : pxr / qxr;  // min(1, p/q); q = 0 < p gives 1
        write_stats(a, pos, Bt, pxr, qxr, pxr > 0.f ? ratio : 0.f, Zt);
      }
    }
  }
}

template <typename T>
static cudaError_t launch_one(const VerifyParams& p, int cs, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.B * p.G * cs), 1, 1);
  cfg.blockDim = dim3(kT, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stats_rows_kernel<T>, p);
}

template <typename T>
static cudaError_t prepare_one() {
  return cudaFuncSetAttribute(stats_rows_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename T>
static cudaError_t clusters_one(int cs, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs * 1024), 1, 1);
  cfg.blockDim = dim3(kT, 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, stats_rows_kernel<T>, &cfg);
}

cudaError_t stats_prepare(int dtype) { return dtype == 0 ? prepare_one<float>() : prepare_one<__nv_bfloat16>(); }

cudaError_t stats_max_active_clusters(int dtype, int cs, int* out) {
  return dtype == 0 ? clusters_one<float>(cs, out) : clusters_one<__nv_bfloat16>(cs, out);
}

cudaError_t stats_launch(const VerifyParams& p, int dtype, int cs, cudaStream_t stream) {
  return dtype == 0 ? launch_one<float>(p, cs, stream) : launch_one<__nv_bfloat16>(p, cs, stream);
}

}  // namespace specv
