// Sampling verification and acceptance statistics on sm_103a.
//
// Speculative sampling, Algorithm 1 Phases 3-4 (Leviathan, Kalman & Matias,
// "Fast Inference from Transformers via Speculative Decoding"; paper-graph-ui
// teardown §2.3 "Algorithm Walkthrough", fullstackaihub §3 "The Algorithm at
// Position i"), with temperature standardisation (§2.2).
//
// Work decomposition.  One thread-block cluster of CS CTAs per (batch row b,
// position i); CTA r of the cluster owns the vocabulary slice [r*L, r*L + L)
// of target row (b, i) and, for i < gamma_b, of draft row (b, i).  Each CTA
//   1. streams its slice(s) from HBM into shared memory as float32 (16-byte
//      loads, no L1 allocation) and takes the slice max;
//   2. replaces each logit by 2^((l - m_slice) * log2(e)/T) and sums them;
//   3. exchanges (max, sum) with the other CTAs through distributed shared
//      memory, so every CTA holds the row normalisers and its own scale
//      a_r = 2^((m_slice - m_row) log2(e)/T) / S_row (p = e * a_r);
//   4. computes, over its slice, sum min(p, q), sum max(0, p - q), sum p, and
//      the residual / p mass of every 128-element chunk;
//   5. exchanges those sums; the CTA owning x_i supplies p(x_i), q(x_i).
// In sampling mode every position also draws, from the row's final uniform,
// the token it would emit if the walk stopped there: the residual
// max(0, p_i - q_i) (p_i if that mass is <= 1e-15) for i < gamma_b, p_i for the
// bonus position i = gamma_b.  The slice is picked from the prefix of the
// cluster's slice masses, the chunk from the prefix of chunk masses, the token
// by a warp scan inside the chunk -- so p and q are never written to HBM and
// every logit is read from HBM exactly once.  The last position cluster of row
// b to finish (an atomic arrival counter, no waiting) walks the accept
// decisions up to the first rejection and writes emitted[b] and n_accepted[b].
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

__device__ __forceinline__ void write_invalid_row(const VerifyParams& a, int b) {
  int32_t* e = a.emitted + (size_t)b * (a.G + 1);
  for (int j = 0; j <= a.G; ++j) e[j] = -1;
  a.n_acc[b] = -1;
}

__device__ __forceinline__ void write_stats(const VerifyParams& a, size_t o, float beta, float px, float qx, float ap,
                                            float z) {
  if (a.beta) a.beta[o] = beta;
  if (a.p_draft) a.p_draft[o] = px;
  if (a.q_draft) a.q_draft[o] = qx;
  if (a.accept_prob) a.accept_prob[o] = ap;
  if (a.resid) a.resid[o] = z;
}

// Last arrival of row b: first rejection and the row's outputs; resets the counter.
__device__ void finalize_row(const VerifyParams& a, int b, int gb) {
  const int G1 = a.G + 1;
  const int32_t* acc = a.ws.acc + (size_t)b * G1;
  bool inv = false;
  for (int j = 0; j <= gb; ++j) inv |= __ldcg(acc + j) < 0;
  int32_t* e = a.emitted + (size_t)b * G1;
  if (inv) {
    for (int j = 0; j < G1; ++j) e[j] = -1;
    a.n_acc[b] = -1;
  } else {
    int n = gb;
    for (int j = 0; j < gb; ++j) {
      if (__ldcg(acc + j) == 0) {
        n = j;
        break;
      }
    }
    for (int j = 0; j < n; ++j) e[j] = __ldg(a.ids + (size_t)b * a.G + j);
    e[n] = __ldcg(a.ws.tok + (size_t)b * G1 + n);
    for (int j = n + 1; j < G1; ++j) e[j] = -1;
    a.n_acc[b] = n;
  }
  // leave every slot this row used at zero: workspaces are shared by calls of any shape
  for (int j = 0; j <= gb; ++j) {
    a.ws.acc[(size_t)b * G1 + j] = 0;
    a.ws.tok[(size_t)b * G1 + j] = 0;
  }
  a.ws.ticket[b] = 0u;
}

}  // namespace

template <typename T, bool kStats>
__global__ void __launch_bounds__(kThreads, 2) verify_rows_kernel(const VerifyParams a) {
  extern __shared__ __align__(16) float smem[];
  __shared__ Xch1 x1;
  __shared__ Xch2 x2;
  __shared__ float red0[kWarps * 2];
  __shared__ float red1[kWarps * 2];
  __shared__ float red2[kWarps * 3];
  __shared__ float bc[4];

  const int CS = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int PR = kStats ? a.G : a.G + 1;  // grid positions per batch row
  const int pos = blockIdx.x / CS;
  const int b = pos / PR;
  const int i = pos - b * PR;
  const int G1 = a.G + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  if (gb < 0 || gb > a.G) {  // the whole cluster leaves together
    if (rank == 0 && tid == 0) {
      if (kStats) {
        write_stats(a, (size_t)b * a.G + i, NAN, NAN, NAN, NAN, NAN);
      } else if (i == 0) {
        write_invalid_row(a, b);
      }
      atomicOr(a.ws.err, kErrArg);
    }
    return;
  }
  if (kStats ? (i >= gb) : (i > gb)) {  // padded position: never read
    if (kStats && rank == 0 && tid == 0) write_stats(a, (size_t)b * a.G + i, NAN, NAN, NAN, NAN, NAN);
    return;
  }
  const bool has_q = i < gb;
  const int lo = rank * a.L;
  const int n = max(0, min(a.V, lo + a.L) - lo);
  const int nch = (n + kChunk - 1) / kChunk;
  const int Lpad = static_cast<int>(align_up(a.L, kChunk));
  float* sP = smem;
  float* sQ = smem + Lpad;
  float* Wr = sQ + Lpad;           // per-chunk residual mass
  float* Wp = Wr + Lpad / kChunk;  // per-chunk p mass
  const float sc = a.scale;

  const T* tp = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + i) * a.V + lo;
  const T* dp = has_q ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + i) * a.V + lo : tp;

  // 1. slice(s) to shared memory, slice maxima
  float m2[2];
  load_rows<T>(tp, dp, has_q, n, nch * kChunk, a.vec != 0, sP, sQ, m2[0], m2[1]);
  block_reduce<2, true>(m2, red0);
  const float Mp = m2[0], Mq = m2[1];

  // 2. exponentials relative to the slice max, slice sums
  float s2[2];
  s2[0] = exp_rows(sP, nch * kChunk, Mp, sc);
  s2[1] = has_q ? exp_rows(sQ, nch * kChunk, Mq, sc) : 0.f;
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
    const bool bad = !(gmp < INFINITY && gmp > -INFINITY) || (has_q && !(gmq < INFINITY && gmq > -INFINITY));
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
      bc[1] = (!bad && has_q && Mq > -INFINITY) ? exp2f((Mq - gmq) * sc) / Sq : 0.f;
      bc[2] = bad ? 1.f : 0.f;
    }
  }
  __syncthreads();
  const float ap = bc[0], aq = bc[1];
  const bool bad = bc[2] != 0.f;

  // 4. overlaps over the slice, chunk masses for the draw
  float t3[3] = {0.f, 0.f, 0.f};  // sum min(p,q), sum max(0,p-q), sum p
  if (!bad) {
    for (int c = warp; c < nch; c += kWarps) {
      const int k = c * kChunk + lane * 4;
      const float4 ep = *reinterpret_cast<const float4*>(sP + k);
      const float p0 = ep.x * ap, p1 = ep.y * ap, p2 = ep.z * ap, p3 = ep.w * ap;
      const float lp = (p0 + p1) + (p2 + p3);
      float lw;
      if (has_q) {
        const float4 eq = *reinterpret_cast<const float4*>(sQ + k);
        const float q0 = eq.x * aq, q1 = eq.y * aq, q2 = eq.z * aq, q3 = eq.w * aq;
        t3[0] += (fminf(p0, q0) + fminf(p1, q1)) + (fminf(p2, q2) + fminf(p3, q3));
        lw = (fmaxf(p0 - q0, 0.f) + fmaxf(p1 - q1, 0.f)) + (fmaxf(p2 - q2, 0.f) + fmaxf(p3 - q3, 0.f));
      } else {
        lw = lp;
      }
      t3[1] += lw;
      t3[2] += lp;
      if (!kStats) {
        const float cw = warp_sum(lw);
        const float cp = has_q ? warp_sum(lp) : cw;
        if (lane == 0) {
          Wr[c] = cw;
          Wp[c] = cp;
        }
      }
    }
  }
  block_reduce<3, false>(t3, red2);
  int x = 0;
  if (has_q) x = __ldg(a.ids + (size_t)b * a.G + i);
  if (tid == 0) {
    float px = -1.f, qx = -1.f;
    if (has_q && !bad && x >= lo && x < lo + n) {
      px = sP[x - lo] * ap;
      qx = sQ[x - lo] * aq;
    }
    x2 = Xch2{t3[0], t3[1], t3[2], px, qx};
  }
  cluster_sync();

  // 5. combine; accept decision; the draw this position would make
  if (warp == 0) {
    float rb = 0.f, rz = 0.f, rp = 0.f;
    if (lane < CS) {
      const uint32_t base = dsmem_map(smem_addr(&x2), lane);
      rb = dsmem_ld_f32(base + 0);
      rz = dsmem_ld_f32(base + 4);
      rp = dsmem_ld_f32(base + 8);
    }
    float Bt = 0.f, Zt = 0.f, Pt = 0.f;
    for (int r = 0; r < CS; ++r) {
      Bt += __shfl_sync(0xffffffffu, rb, r);
      Zt += __shfl_sync(0xffffffffu, rz, r);
      Pt += __shfl_sync(0xffffffffu, rp, r);
    }
    const bool xok = !has_q || (x >= 0 && x < a.V);
    float px = 0.f, qx = 0.f;
    if (has_q && xok && !bad) {
      const uint32_t base = dsmem_map(smem_addr(&x2), static_cast<uint32_t>(x / a.L));
      px = dsmem_ld_f32(base + 12);
      qx = dsmem_ld_f32(base + 16);
    }
    const float ratio = px >= qx ? 1.f : px / qx;  // min(1, p/q); q = 0 < p gives 1
    const float aprob = px > 0.f ? ratio : 0.f;

    if (kStats) {
      if (rank == 0 && lane == 0) {
        const size_t o = (size_t)b * a.G + i;
        if (bad || !xok) {
          write_stats(a, o, NAN, NAN, NAN, NAN, NAN);
          atomicOr(a.ws.err, bad ? kErrNonfinite : kErrToken);
        } else {
          write_stats(a, o, Bt, px, qx, aprob, Zt);
        }
      }
    } else {
      const float* U = a.uniforms + (size_t)b * G1;
      const float uf = __ldg(U + a.G);
      const float ui = has_q ? __ldg(U + i) : 0.f;
      const bool uok = (uf >= 0.f && uf < 1.f) && (!has_q || (ui >= 0.f && ui < 1.f));
      const bool invalid = bad || !xok || !uok;
      if (!invalid) {
        // distribution of the draw: residual, or p (bonus position / degenerate residual)
        const bool use_p = !has_q || !(Zt > kZFloor);
        const float tot = use_p ? Pt : Zt;
        const float t = uf * tot;
        const float mine = use_p ? rp : rz;
        // owning CTA: first rank whose mass carries the running sum past t
        int owner = -1, last = -1;
        float pre = 0.f, last_pre = 0.f, cum = 0.f;
        for (int r = 0; r < CS; ++r) {
          const float v = __shfl_sync(0xffffffffu, mine, r);
          if (v > 0.f) {
            if (owner < 0 && cum + v > t) {
              owner = r;
              pre = cum;
            }
            last = r;
            last_pre = cum;
          }
          cum += v;
        }
        bool fallback = owner < 0;  // rounding left t at or past the total
        if (fallback) {
          owner = last;
          pre = last_pre;
        }
        if (owner == rank) {
          const float* W = use_p ? Wp : Wr;
          float tt = t - pre;
          int chunk = -1, lastc = -1;
          for (int base = 0; base < nch; base += 32) {
            const int c = base + lane;
            const float v = c < nch ? W[c] : 0.f;
            const float inc = warp_inclusive_scan(v, lane);
            float exc = __shfl_up_sync(0xffffffffu, inc, 1);
            if (lane == 0) exc = 0.f;
            const unsigned hit = __ballot_sync(0xffffffffu, v > 0.f && inc > tt);
            const unsigned nz = __ballot_sync(0xffffffffu, v > 0.f);
            if (!fallback && hit) {
              const int l = __ffs(hit) - 1;
              chunk = base + l;
              tt -= __shfl_sync(0xffffffffu, exc, l);
              break;
            }
            if (nz) lastc = base + 31 - __clz(nz);
            tt -= __shfl_sync(0xffffffffu, inc, 31);
          }
          if (chunk < 0) {
            chunk = lastc;
            fallback = true;
          }
          // weights of this lane's 4 elements, recomputed exactly as in step 4
          const int k = chunk * kChunk + lane * 4;
          const float4 ep = *reinterpret_cast<const float4*>(sP + k);
          float w[4] = {ep.x * ap, ep.y * ap, ep.z * ap, ep.w * ap};
          if (has_q && !use_p) {
            const float4 eq = *reinterpret_cast<const float4*>(sQ + k);
            w[0] = fmaxf(w[0] - eq.x * aq, 0.f);
            w[1] = fmaxf(w[1] - eq.y * aq, 0.f);
            w[2] = fmaxf(w[2] - eq.z * aq, 0.f);
            w[3] = fmaxf(w[3] - eq.w * aq, 0.f);
          }
          const float ls = (w[0] + w[1]) + (w[2] + w[3]);
          const float inc = warp_inclusive_scan(ls, lane);
          float exc = __shfl_up_sync(0xffffffffu, inc, 1);
          if (lane == 0) exc = 0.f;
          int lastj = -1;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (w[j] > 0.f) lastj = j;
          int tok = -1;
          const unsigned hit = __ballot_sync(0xffffffffu, ls > 0.f && inc > tt);
          if (!fallback && hit) {
            const int l = __ffs(hit) - 1;
            if (lane == l) {
              float c = exc;
              for (int j = 0; j < 4; ++j) {
                c += w[j];
                if (w[j] > 0.f && c > tt) {
                  tok = k + j;
                  break;
                }
              }
              if (tok < 0) tok = k + lastj;
            }
            tok = __shfl_sync(0xffffffffu, tok, l);
          } else {
            const unsigned nz = __ballot_sync(0xffffffffu, ls > 0.f);
            const int l = 31 - __clz(nz);
            if (lane == l) tok = k + lastj;
            tok = __shfl_sync(0xffffffffu, tok, l);
          }
          if (lane == 0) {
            a.ws.tok[(size_t)b * G1 + i] = lo + tok;
            __threadfence();
          }
        }
      }
      if (rank == 0 && lane == 0) {
        int code;
        if (invalid) {
          code = -1;
          atomicOr(a.ws.err, bad ? kErrNonfinite : (!xok ? kErrToken : kErrArg));
        } else {
          code = has_q ? ((px > 0.f && ui <= ratio) ? 1 : 0) : 1;
        }
        a.ws.acc[(size_t)b * G1 + i] = code;
        __threadfence();
      }
    }
  }
  cluster_sync();  // keeps every CTA's shared memory alive until the cluster is done with it

  if (!kStats && rank == 0 && tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(a.ws.ticket + b, 1u);
    if (prev == static_cast<unsigned>(gb)) {  // gb + 1 positions report per row
      __threadfence();
      finalize_row(a, b, gb);
    }
  }
}

template <typename T, bool kStats>
static cudaError_t launch_one(const VerifyParams& p, int cs, int smem, cudaStream_t stream) {
  auto kern = verify_rows_kernel<T, kStats>;
  const int PR = kStats ? p.G : p.G + 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.B * PR * cs), 1, 1);
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
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T, bool kStats>
static cudaError_t prepare_one(int smem) {
  auto kern = verify_rows_kernel<T, kStats>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename T, bool kStats>
static cudaError_t clusters_one(int cs, int smem, int* out) {
  auto kern = verify_rows_kernel<T, kStats>;
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
  return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

#define SPECV_DISPATCH(fn, ...)                                                              \
  (dtype == 0 ? (stats ? fn<float, true>(__VA_ARGS__) : fn<float, false>(__VA_ARGS__))        \
              : (stats ? fn<__nv_bfloat16, true>(__VA_ARGS__) : fn<__nv_bfloat16, false>(__VA_ARGS__)))

cudaError_t verify_prepare(int dtype, bool stats, int smem) { return SPECV_DISPATCH(prepare_one, smem); }

cudaError_t verify_max_active_clusters(int dtype, bool stats, int cs, int smem, int* out) {
  return SPECV_DISPATCH(clusters_one, cs, smem, out);
}

cudaError_t verify_launch(const VerifyParams& p, int dtype, bool stats, int cs, int smem, cudaStream_t stream) {
  return SPECV_DISPATCH(launch_one, p, cs, smem, stream);
}

}  // namespace specv
