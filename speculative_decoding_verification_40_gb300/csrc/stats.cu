// Per-position acceptance statistics on sm_103a.
//
// Definition 3.2, Lemma 3.3 and Theorem 3.5 of Leviathan, Kalman & Matias,
// "Fast Inference from Transformers via Speculative Decoding" (paper-graph-ui
// teardown, "Computing alpha from p and q"): for each position i < gamma_b,
// beta = sum_x min(p(x), q(x)), the residual mass sum_x max(0, p(x) - q(x)),
// and p(x_i), q(x_i), min(1, p(x_i)/q(x_i)) at the draft token, with p and q
// the temperature softmaxes of the target and draft rows (§2.2).
//
// Work decomposition.  One thread-block cluster of CS CTAs per (batch row b,
// position i); CTA r of the cluster owns the vocabulary slice [r*L, r*L + L)
// of target and draft row (b, i).  Each CTA
//   1. streams its slices from HBM into shared memory as float32 (16-byte
//      loads, no L1 allocation) and takes the slice max;
//   2. replaces each logit by 2^((l - m_slice) * log2(e)/T) and sums them;
//   3. exchanges (max, sum) with the other CTAs through distributed shared
//      memory, so every CTA holds the row normalisers and its own scale
//      a_r = 2^((m_slice - m_row) log2(e)/T) / S_row (p = e * a_r);
//   4. sums min(p, q) and max(0, p - q) over its slice;
//   5. exchanges those sums; the CTA owning x_i supplies p(x_i), q(x_i), and
//      rank 0 writes the position's statistics.
// Every logit is read from HBM once; p and q never leave shared memory.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace specv {

namespace {

struct Xch1 {  // per-CTA slice normalisers
  float mp, sp, mq, sq;
};
struct Xch2 {  // per-CTA slice overlaps and the values at the draft token
  float beta, z, psum, px, qx;
};

// Copies n logits of one row (and of a second row when two_rows) to shared
// memory as float32 and returns this thread's NaN-propagating maxima.  Entries
// [n, fill_to) are set to -inf.
template <typename T>
__device__ __forceinline__ void load_rows(const T* __restrict__ src0, const T* __restrict__ src1, bool two_rows,
                                          int n, int fill_to, bool vec, float* __restrict__ dst0,
                                          float* __restrict__ dst1, float& m0, float& m1) {
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 4;
  const int tid = threadIdx.x;
  m0 = -INFINITY;
  m1 = -INFINITY;
  int done = 0;
  if (vec) {
    const int nv = n / kV;
    const uint4* s0 = reinterpret_cast<const uint4*>(src0);
    const uint4* s1 = reinterpret_cast<const uint4*>(src1);
    int v = tid;
    if (two_rows) {
      for (; v + (U - 1) * kThreads < nv; v += U * kThreads) {
        uint4 r0[U], r1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = ldg_stream(s0 + v + u * kThreads);
#pragma unroll
        for (int u = 0; u < U; ++u) r1[u] = ldg_stream(s1 + v + u * kThreads);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float f[kV], g[kV];
          Elems<T>::widen(r0[u], f);
          Elems<T>::widen(r1[u], g);
#pragma unroll
          for (int j = 0; j < kV; ++j) {
            m0 = max_nan(m0, f[j]);
            m1 = max_nan(m1, g[j]);
          }
          store_f32<kV>(dst0 + (v + u * kThreads) * kV, f);
          store_f32<kV>(dst1 + (v + u * kThreads) * kV, g);
        }
      }
      for (; v < nv; v += kThreads) {
        const uint4 r0 = ldg_stream(s0 + v);
        const uint4 r1 = ldg_stream(s1 + v);
        float f[kV], g[kV];
        Elems<T>::widen(r0, f);
        Elems<T>::widen(r1, g);
#pragma unroll
        for (int j = 0; j < kV; ++j) {
          m0 = max_nan(m0, f[j]);
          m1 = max_nan(m1, g[j]);
        }
        store_f32<kV>(dst0 + v * kV, f);
        store_f32<kV>(dst1 + v * kV, g);
      }
    } else {
      for (; v + (U - 1) * kThreads < nv; v += U * kThreads) {
        uint4 r0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r0[u] = ldg_stream(s0 + v + u * kThreads);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float f[kV];
          Elems<T>::widen(r0[u], f);
#pragma unroll
          for (int j = 0; j < kV; ++j) m0 = max_nan(m0, f[j]);
          store_f32<kV>(dst0 + (v + u * kThreads) * kV, f);
        }
      }
      for (; v < nv; v += kThreads) {
        const uint4 r0 = ldg_stream(s0 + v);
        float f[kV];
        Elems<T>::widen(r0, f);
#pragma unroll
        for (int j = 0; j < kV; ++j) m0 = max_nan(m0, f[j]);
        store_f32<kV>(dst0 + v * kV, f);
      }
    }
    done = nv * kV;
  }
  for (int k = done + tid; k < n; k += kThreads) {
    const float f = Elems<T>::one(src0, k);
    m0 = max_nan(m0, f);
    dst0[k] = f;
    if (two_rows) {
      const float g = Elems<T>::one(src1, k);
      m1 = max_nan(m1, g);
      dst1[k] = g;
    }
  }
  for (int k = n + tid; k < fill_to; k += kThreads) {
    dst0[k] = -INFINITY;
    if (two_rows) dst1[k] = -INFINITY;
  }
}

// In-place e = 2^((l - m) * sc) over [0, len) (len a multiple of 4); returns this thread's sum.
__device__ __forceinline__ float exp_rows(float* __restrict__ s, int len, float m, float sc) {
  float acc = 0.f;
  if (!(m > -INFINITY) || !(m < INFINITY)) {  // empty / all -inf slice, or an invalid row
    for (int k = threadIdx.x * 4; k < len; k += kThreads * 4)
      *reinterpret_cast<float4*>(s + k) = make_float4(0.f, 0.f, 0.f, 0.f);
    return 0.f;
  }
  for (int k = threadIdx.x * 4; k < len; k += kThreads * 4) {
    float4 v = *reinterpret_cast<const float4*>(s + k);
    v.x = exp2f((v.x - m) * sc);
    v.y = exp2f((v.y - m) * sc);
    v.z = exp2f((v.z - m) * sc);
    v.w = exp2f((v.w - m) * sc);
    acc += (v.x + v.y) + (v.z + v.w);
    *reinterpret_cast<float4*>(s + k) = v;
  }
  return acc;
}

// Block reduction of N values (sum, or NaN-propagating max); every thread gets
// the result, combined in a fixed order so all CTAs agree bit for bit.
template <int N, bool kMax>
__device__ __forceinline__ void block_reduce(float (&v)[N], float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = kMax ? warp_max_nan(v[j]) : warp_sum(v[j]);
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < N; ++j) red[warp * N + j] = v[j];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < N; ++j) {
    float a = red[j];
    for (int w = 1; w < kWarps; ++w) a = kMax ? max_nan(a, red[w * N + j]) : a + red[w * N + j];
    v[j] = a;
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
__global__ void __launch_bounds__(kThreads, 2) stats_rows_kernel(const VerifyParams a) {
  extern __shared__ __align__(16) float smem[];
  __shared__ Xch1 x1;
  __shared__ Xch2 x2;
  __shared__ float red0[kWarps * 2];
  __shared__ float red1[kWarps * 2];
  __shared__ float red2[kWarps * 2];
  __shared__ float bc[4];

  const int CS = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int pos = blockIdx.x / CS;  // b * G + i
  const int b = pos / a.G;
  const int i = pos - b * a.G;
  const int G1 = a.G + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t o = (size_t)b * a.G + i;

  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  if (gb < 0 || gb > a.G || i >= gb) {  // the whole cluster leaves together; padded positions are never read
    if (rank == 0 && tid == 0) {
      write_stats(a, o, NAN, NAN, NAN, NAN, NAN);
      if (gb < 0 || gb > a.G) atomicOr(a.ws.err, kErrArg);
    }
    return;
  }
  const int lo = rank * a.L;
  const int n = max(0, min(a.V, lo + a.L) - lo);
  const int nch = (n + kChunk - 1) / kChunk;
  const int Lpad = static_cast<int>(align_up(a.L, kChunk));
  float* sP = smem;
  float* sQ = smem + Lpad;
  const float sc = a.scale;
  const T* tp = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + i) * a.V + lo;
  const T* dp = reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + i) * a.V + lo;

  // 1. slices to shared memory, slice maxima
  float m2[2];
  load_rows<T>(tp, dp, true, n, nch * kChunk, a.vec != 0, sP, sQ, m2[0], m2[1]);
  block_reduce<2, true>(m2, red0);
  const float Mp = m2[0], Mq = m2[1];

  // 2. exponentials relative to the slice max, slice sums
  float s2[2];
  s2[0] = exp_rows(sP, nch * kChunk, Mp, sc);
  s2[1] = exp_rows(sQ, nch * kChunk, Mq, sc);
  block_reduce<2, false>(s2, red1);

  // 3. cluster exchange of slice normalisers
  if (tid == 0) x1 = Xch1{Mp, s2[0], Mq, s2[1]};
  cluster_sync();
  if (warp == 0) {
    float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
    if (lane < CS) {
      const uint32_t base = dsmem_map(smem_addr(&x1), lane);
      mp = dsmem_ld_f32(base + 0);
      sp = dsmem_ld_f32(base + 4);
      mq = dsmem_ld_f32(base + 8);
      sq = dsmem_ld_f32(base + 12);
    }
    const float gmp = warp_max_nan(mp);
    const float gmq = warp_max_nan(mq);
    // NaN or +inf anywhere, or a row that is entirely -inf
    const bool bad = !(gmp < INFINITY && gmp > -INFINITY) || !(gmq < INFINITY && gmq > -INFINITY);
    float Sp = 0.f, Sq = 0.f;
    if (!bad) {
      const float tpv = mp > -INFINITY ? sp * exp2f((mp - gmp) * sc) : 0.f;
      const float tqv = mq > -INFINITY ? sq * exp2f((mq - gmq) * sc) : 0.f;
      for (int r = 0; r < CS; ++r) {  // fixed order: identical sums in every CTA
        Sp += __shfl_sync(0xffffffffu, tpv, r);
        Sq += __shfl_sync(0xffffffffu, tqv, r);
      }
    }
    if (lane == 0) {
      bc[0] = (!bad && Mp > -INFINITY) ? exp2f((Mp - gmp) * sc) / Sp : 0.f;
      bc[1] = (!bad && Mq > -INFINITY) ? exp2f((Mq - gmq) * sc) / Sq : 0.f;
      bc[2] = bad ? 1.f : 0.f;
    }
  }
  __syncthreads();
  const float ap = bc[0], aq = bc[1];
  const bool bad = bc[2] != 0.f;

  // 4. overlaps over the slice
  float t2[2] = {0.f, 0.f};  // sum min(p,q), sum max(0,p-q)
  if (!bad) {
    for (int k = tid * 4; k < nch * kChunk; k += kThreads * 4) {
      const float4 ep = *reinterpret_cast<const float4*>(sP + k);
      const float4 eq = *reinterpret_cast<const float4*>(sQ + k);
      const float p0 = ep.x * ap, p1 = ep.y * ap, p2 = ep.z * ap, p3 = ep.w * ap;
      const float q0 = eq.x * aq, q1 = eq.y * aq, q2 = eq.z * aq, q3 = eq.w * aq;
      t2[0] += (fminf(p0, q0) + fminf(p1, q1)) + (fminf(p2, q2) + fminf(p3, q3));
      t2[1] += (fmaxf(p0 - q0, 0.f) + fmaxf(p1 - q1, 0.f)) + (fmaxf(p2 - q2, 0.f) + fmaxf(p3 - q3, 0.f));
    }
  }
  block_reduce<2, false>(t2, red2);
  const int x = __ldg(a.ids + o);
  if (tid == 0) {
    float px = -1.f, qx = -1.f;
    if (!bad && x >= lo && x < lo + n) {
      px = sP[x - lo] * ap;
      qx = sQ[x - lo] * aq;
    }
    x2 = Xch2{t2[0], t2[1], 0.f, px, qx};
  }
  cluster_sync();

  // 5. combine and write (rank 0)
  if (rank == 0 && warp == 0) {
    float rb = 0.f, rz = 0.f;
    if (lane < CS) {
      const uint32_t base = dsmem_map(smem_addr(&x2), lane);
      rb = dsmem_ld_f32(base + 0);
      rz = dsmem_ld_f32(base + 4);
    }
    float Bt = 0.f, Zt = 0.f;
    for (int r = 0; r < CS; ++r) {
      Bt += __shfl_sync(0xffffffffu, rb, r);
      Zt += __shfl_sync(0xffffffffu, rz, r);
    }
    const bool xok = x >= 0 && x < a.V;
    if (lane == 0) {
      if (bad || !xok) {
        write_stats(a, o, NAN, NAN, NAN, NAN, NAN);
        atomicOr(a.ws.err, bad ? kErrNonfinite : kErrToken);
      } else {
        const uint32_t base = dsmem_map(smem_addr(&x2), static_cast<uint32_t>(x / a.L));
        const float px = dsmem_ld_f32(base + 12);
        const float qx = dsmem_ld_f32(base + 16);
        const float ratio = px >= qx ? 1.f : px / qx;  // min(1, p/q); q = 0 < p gives 1
        write_stats(a, o, Bt, px, qx, px > 0.f ? ratio : 0.f, Zt);
      }
    }
  }
  cluster_sync();  // keeps every CTA's shared memory alive until the cluster is done with it
}

template <typename T>
static cudaError_t launch_one(const VerifyParams& p, int cs, int smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.B * p.G * cs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
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
static cudaError_t prepare_one(int smem) {
  cudaError_t e = cudaFuncSetAttribute(stats_rows_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(stats_rows_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename T>
static cudaError_t clusters_one(int cs, int smem, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs * 1024), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, stats_rows_kernel<T>, &cfg);
}

cudaError_t stats_prepare(int dtype, int smem) {
  return dtype == 0 ? prepare_one<float>(smem) : prepare_one<__nv_bfloat16>(smem);
}

cudaError_t stats_max_active_clusters(int dtype, int cs, int smem, int* out) {
  return dtype == 0 ? clusters_one<float>(cs, smem, out) : clusters_one<__nv_bfloat16>(cs, smem, out);
}

cudaError_t stats_launch(const VerifyParams& p, int dtype, int cs, int smem, cudaStream_t stream) {
  return dtype == 0 ? launch_one<float>(p, cs, smem, stream) : launch_one<__nv_bfloat16>(p, cs, smem, stream);
}

}  // namespace specv
