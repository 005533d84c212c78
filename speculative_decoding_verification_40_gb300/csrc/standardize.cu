// Top-k and nucleus (top-p) standardisation thresholds on sm_103a.
//
// Standardised sampling (Leviathan, Kalman & Matias, "Fast Inference from
// Transformers via Speculative Decoding", §2.2, as restated in the
// paper-graph-ui teardown "Standardized Sampling"): top-k keeps the k largest
// probabilities, nucleus sampling keeps the shortest descending prefix whose
// mass reaches top_p; both renormalise over the kept tokens.  Softmax is
// increasing in the logit, so either kept set is {x : l(x) >= tau} for one
// logit threshold tau per row (ties at tau are all kept); the verification and
// sampling entry points take tau and treat logits below it as -inf.
//
// One CTA per row.  Pass 0 takes the row max M.  Pass 1 histograms the row
// over 2048 bins of the distance from the max, floor((M - l) c) (c = 48 per
// unit of log2 probability, so a bin is an interval of logits and a lower bin
// holds larger logits; logits more than 42.6 units down, whose nucleus weight
// is below the 2^-40 fixed point, share the last bin, summed in registers):
// top-k counts elements, nucleus sums the weights 2^((l - M) log2(e)/T) in 2^-40
// fixed point (exact, order-independent integer adds: the same result in every
// run).  The bin holding the k-th element / the running mass top_p * total is
// found by a block scan; pass 2 gathers that bin's logits into shared memory
// and sorts them (bitonic), and the threshold is read off the sorted bin.  If
// the bin holds more than 8192 logits, an exact radix selection over the
// order-preserving 32-bit keys of the bin's logits (11 + 11 + 10 bits, one pass
// each) takes over.
#include <cuda_bf16.h>

#include "../../include/spec_verify.h"
#include "common.cuh"
#include "softmax.cuh"

namespace specv {

namespace {

constexpr int kTT = 512;
constexpr int kTW = kTT / 32;
constexpr int kBins = 2048;  // first two levels; the third uses 1024
constexpr float kFixF = 1099511627776.f;  // 2^40

// Order-preserving key: a < b as floats iff key(a) < key(b); -0 is folded onto +0.
__device__ __forceinline__ uint32_t fkey(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Calls fn(f) for every logit of the row (each thread a strided share), 16-byte loads when vec with
// four in flight per thread.
template <typename T, typename F>
__device__ __forceinline__ void for_each_logit(const T* __restrict__ row, int V, bool vec, F&& fn) {
  constexpr int kV = Elems<T>::kVec;
  int done = 0;
  if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int nv = V / kV;
    int v = threadIdx.x;
    for (; v + 3 * kTT < nv; v += 4 * kTT) {
      uint4 r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) r[u] = __ldg(r4 + v + u * kTT);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float f[kV];
        Elems<T>::widen(r[u], f);
#pragma unroll
        for (int j = 0; j < kV; ++j) fn(f[j]);
      }
    }
    for (; v < nv; v += kTT) {
      float f[kV];
      Elems<T>::widen(__ldg(r4 + v), f);
#pragma unroll
      for (int j = 0; j < kV; ++j) fn(f[j]);
    }
    done = nv * kV;
  }
  for (int k = done + threadIdx.x; k < V; k += kTT) fn(Elems<T>::one(row, k));
}

__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += y;
  }
  return v;
}

struct Pick {
  int bin;                  // the bin holding the need-th unit from the top
  unsigned long long above; // units in the bins above it
  unsigned long long total; // units in every bin
};

// A histogram of 64-bit sums kept as two arrays of 32-bit words, so that every update is a native
// 32-bit shared-memory atomic: bin b holds hi[b] * 2^32 + lo[b] (hi may be null: 32-bit counts).
struct Hist {
  unsigned int* lo;
  unsigned int* hi;
  __device__ __forceinline__ unsigned long long get(int b) const {
    return (hi ? (static_cast<unsigned long long>(hi[b]) << 32) : 0ull) + lo[b];
  }
  // adds v (< 2^41) to bin b; a wrap of the low word carries into the high word
  __device__ __forceinline__ void add(int b, unsigned long long v) const {
    const unsigned int l = static_cast<unsigned int>(v);
    if (!hi) {
      atomicAdd(lo + b, l);
      return;
    }
    const unsigned int old = atomicAdd(lo + b, l);
    const unsigned int carry = (old + l < old) ? 1u : 0u;
    const unsigned int h = static_cast<unsigned int>(v >> 32) + carry;
    if (h) atomicAdd(hi + b, h);
  }
  __device__ __forceinline__ void zero(int nb) const {
    for (int k = threadIdx.x; k < nb; k += kTT) {
      lo[k] = 0u;
      if (hi) hi[k] = 0u;
    }
    __syncthreads();
  }
};

// Over the nb bins of h read from the highest bin down: the bin where the running sum first reaches
// need (1 <= need <= total), the sum above that bin, and the total.  Every thread gets the result.
__device__ Pick pick_from_top(const Hist& h, int nb, unsigned long long need, unsigned long long* wsum, Pick* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nb / kTT;  // bins per thread, thread 0 holding the highest
  unsigned long long local = 0;
  for (int j = 0; j < per; ++j) local += h.get(nb - 1 - (tid * per + j));
  const unsigned long long incl_w = warp_incl_u64(local, lane);
  if (lane == 31) wsum[warp] = incl_w;
  __syncthreads();
  unsigned long long before = 0, total = 0;
  for (int w = 0; w < kTW; ++w) {
    if (w < warp) before += wsum[w];
    total += wsum[w];
  }
  const unsigned long long incl = before + incl_w;
  const unsigned long long excl = incl - local;
  if (excl < need && need <= incl) {
    unsigned long long run = excl;
    for (int j = 0; j < per; ++j) {
      const int bin = nb - 1 - (tid * per + j);
      const unsigned long long v = h.get(bin);
      if (run + v >= need) {
        out->bin = bin;
        out->above = run;
        break;
      }
      run += v;
    }
  }
  if (tid == 0) out->total = total;
  __syncthreads();
  const Pick p = *out;
  __syncthreads();
  return p;
}

}  // namespace

constexpr int kCap = 8192;          // logits of the selected bin sorted in shared memory (a power of two)
static_assert(kCap * sizeof(float) >= kBins * sizeof(unsigned long long), "the gather buffer holds the histogram");
constexpr float kBinsPerUnit = 48.f;  // bins per unit of log2 probability (the last bin starts 42.6 units down)

__device__ __forceinline__ int dist_bin(float f, float M, float scale) {
  const float d = (M - f) * scale * kBinsPerUnit;  // >= 0, nondecreasing as f decreases
  return d < static_cast<float>(kBins - 1) ? static_cast<int>(d) : kBins - 1;
}

// Exact radix selection over the order-preserving keys of the logits in distance bin `db`: the key at
// which the running count (top-k) or fixed-point mass (nucleus) from the largest logit down first
// reaches `need`.
template <typename T, bool kTopP, typename W>
__device__ uint32_t radix_select(const T* row, int V, bool vec, float M, float scale, int db, unsigned long long need,
                                 const Hist& h, unsigned long long* wsum, Pick* pk, W&& weight) {
  h.zero(kBins);
  for_each_logit<T>(row, V, vec, [&](float f) {
    if (f > -INFINITY && dist_bin(f, M, scale) == db) h.add(fkey(f) >> 21, kTopP ? weight(f) : 1ull);
  });
  __syncthreads();
  const Pick p1 = pick_from_top(h, kBins, need, wsum, pk);
  const uint32_t b1 = static_cast<uint32_t>(p1.bin);
  const unsigned long long need2 = need - p1.above;
  h.zero(kBins);
  for_each_logit<T>(row, V, vec, [&](float f) {
    if (f > -INFINITY && dist_bin(f, M, scale) == db) {
      const uint32_t key = fkey(f);
      if ((key >> 21) == b1) h.add((key >> 10) & 0x7ffu, kTopP ? weight(f) : 1ull);
    }
  });
  __syncthreads();
  const Pick p2 = pick_from_top(h, kBins, need2, wsum, pk);
  const uint32_t hi = (b1 << 11) | static_cast<uint32_t>(p2.bin);
  const unsigned long long need3 = need2 - p2.above;
  h.zero(kBins);
  for_each_logit<T>(row, V, vec, [&](float f) {
    if (f > -INFINITY && dist_bin(f, M, scale) == db) {
      const uint32_t key = fkey(f);
      if ((key >> 10) == hi) h.add(key & 0x3ffu, kTopP ? weight(f) : 1ull);
    }
  });
  __syncthreads();
  const Pick p3 = pick_from_top(h, 1024, need3, wsum, pk);
  return (hi << 10) | static_cast<uint32_t>(p3.bin);
}

// Descending bitonic sort of cand[0, n2) (n2 a power of two, padded with -inf) by the whole CTA.
__device__ void sort_desc(float* cand, int n2) {
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n2 / 2; i += kTT) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const float a = cand[lo], b = cand[hi];
        if (desc ? (a < b) : (a > b)) {
          cand[lo] = b;
          cand[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

// Top-k (kTopP = false: k) or nucleus (kTopP = true: top_p, temperature scale) threshold of one row.
template <typename T, bool kTopP>
__global__ void __launch_bounds__(kTT) threshold_kernel(const void* __restrict__ logits, int V, int k, float scale,
                                                        float top_p, int vec, float* __restrict__ thr) {
  // the histogram and the gathered bin share one buffer: the bin is gathered after the histogram is read
  __shared__ __align__(16) unsigned char buf[kCap * sizeof(float)];
  const Hist hist{reinterpret_cast<unsigned int*>(buf), kTopP ? reinterpret_cast<unsigned int*>(buf) + kBins : nullptr};
  float* cand = reinterpret_cast<float*>(buf);
  __shared__ unsigned long long wsum[kTW];
  __shared__ float red[kTW];
  __shared__ Pick pk;
  __shared__ int cnt;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T* row = reinterpret_cast<const T*>(logits) + (size_t)blockIdx.x * V;
  const bool vv = vec != 0;
  // top-k bins in units of the logit itself (any positive scale orders them the same way)
  const float bscale = kTopP ? scale : 1.4426950408889634f;

  // pass 0: the row max (NaN-propagating)
  float m = -INFINITY;
  for_each_logit<T>(row, V, vv, [&](float f) { m = max_nan(m, f); });
  m = warp_max_nan(m);
  if (lane == 0) red[warp] = m;
  if (tid == 0) cnt = 0;
  __syncthreads();
  float M = red[0];
  for (int w = 1; w < kTW; ++w) M = max_nan(M, red[w]);
  if (!(M < INFINITY)) {  // NaN or +inf in the row
    if (tid == 0) thr[blockIdx.x] = NAN;
    return;
  }
  if (!(M > -INFINITY)) {  // nothing finite: top-k keeps everything, nucleus has no distribution
    if (tid == 0) thr[blockIdx.x] = kTopP ? NAN : -INFINITY;
    return;
  }
  if (kTopP && top_p >= 1.f) {
    if (tid == 0) thr[blockIdx.x] = -INFINITY;
    return;
  }
  const float nm = -M * scale;
  // the weight in (0, 1] times 2^40 is exact in float (a power-of-two scale); its integer part is the
  // fixed-point weight
  auto weight = [&](float f) -> unsigned long long {
    return __float2ull_rz(fast_exp2(fmaf(f, scale, nm)) * kFixF);
  };

  // pass 1: histogram over the distance from the max (stored high bin first: index kBins-1-bin); the far
  // bin, where most logits of a long row land, is summed in registers instead of by contended atomics
  hist.zero(kBins);
  unsigned long long tail = 0;
  for_each_logit<T>(row, V, vv, [&](float f) {
    if (f > -INFINITY) {
      const int bin = dist_bin(f, M, bscale);
      const unsigned long long u = kTopP ? weight(f) : 1ull;
      if (bin == kBins - 1)
        tail += u;
      else
        hist.add(kBins - 1 - bin, u);
    }
  });
  tail = warp_incl_u64(tail, lane);
  if (lane == 31) wsum[warp] = tail;
  __syncthreads();
  if (tid == 0) {
    unsigned long long t = 0;
    for (int w = 0; w < kTW; ++w) t += wsum[w];
    hist.lo[0] = static_cast<unsigned int>(t);
    if (kTopP) hist.hi[0] = static_cast<unsigned int>(t >> 32);
  }
  __syncthreads();
  Pick p = pick_from_top(hist, kBins, 1ull, wsum, &pk);
  unsigned long long need;
  if (kTopP) {
    need = static_cast<unsigned long long>(ceil(static_cast<double>(top_p) * static_cast<double>(p.total)));  // once
    if (need < 1) need = 1;
    if (need > p.total) need = p.total;
  } else {
    if (static_cast<unsigned long long>(k) > p.total) {  // fewer than k finite logits
      if (tid == 0) thr[blockIdx.x] = -INFINITY;
      return;
    }
    need = static_cast<unsigned long long>(k);
  }
  p = pick_from_top(hist, kBins, need, wsum, &pk);
  const int db = kBins - 1 - p.bin;
  const unsigned long long need2 = need - p.above;

  // pass 2: the bin's logits into shared memory
  for_each_logit<T>(row, V, vv, [&](float f) {
    if (f > -INFINITY && dist_bin(f, M, bscale) == db) {
      const int at = atomicAdd(&cnt, 1);
      if (at < kCap) cand[at] = f;
    }
  });
  __syncthreads();
  const int n = cnt;
  if (n > kCap) {  // too many to sort here: exact radix selection over the bin
    const uint32_t key = radix_select<T, kTopP>(row, V, vv, M, bscale, db, need2, hist, wsum, &pk, weight);
    if (tid == 0) thr[blockIdx.x] = key_float(key);
    return;
  }
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  for (int i = n + tid; i < n2; i += kTT) cand[i] = -INFINITY;
  __syncthreads();
  sort_desc(cand, n2);
  if (!kTopP) {
    if (tid == 0) thr[blockIdx.x] = cand[need2 - 1];
    return;
  }
  // nucleus: the first sorted logit at which the running fixed-point mass reaches need2 (block scan)
  constexpr int kPer = kCap / kTT;
  unsigned long long local = 0;
  for (int j = 0; j < kPer; ++j) {
    const int i = tid * kPer + j;
    if (i < n) local += weight(cand[i]);
  }
  const unsigned long long incl_w = warp_incl_u64(local, lane);
  if (lane == 31) wsum[warp] = incl_w;
  __syncthreads();
  unsigned long long before = 0;
  for (int w = 0; w < warp; ++w) before += wsum[w];
  const unsigned long long excl = before + incl_w - local;
  unsigned long long run = excl;
  if (excl < need2 && need2 <= excl + local) {
    for (int j = 0; j < kPer; ++j) {
      const int i = tid * kPer + j;
      run += weight(cand[i]);
      if (run >= need2) {
        thr[blockIdx.x] = cand[i];
        break;
      }
    }
  }
}

cudaError_t topk_threshold_launch(const void* logits, int dtype, int R, int V, int k, int vec, float* thr,
                                  cudaStream_t stream) {
  if (dtype == 0)
    threshold_kernel<float, false><<<R, kTT, 0, stream>>>(logits, V, k, 1.f, 1.f, vec, thr);
  else
    threshold_kernel<__nv_bfloat16, false><<<R, kTT, 0, stream>>>(logits, V, k, 1.f, 1.f, vec, thr);
  return cudaGetLastError();
}

cudaError_t topp_threshold_launch(const void* logits, int dtype, int R, int V, float scale, float top_p, int vec,
                                  float* thr, cudaStream_t stream) {
  if (dtype == 0)
    threshold_kernel<float, true><<<R, kTT, 0, stream>>>(logits, V, 0, scale, top_p, vec, thr);
  else
    threshold_kernel<__nv_bfloat16, true><<<R, kTT, 0, stream>>>(logits, V, 0, scale, top_p, vec, thr);
  return cudaGetLastError();
}

}  // namespace specv
