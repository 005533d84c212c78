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
// One CTA per row.  Logits are binned by their distance from a reference R,
// floor((R - l) c) over 2048 bins (c = 48 per unit of log2 probability, so a
// bin is an interval of logits and a lower bin holds larger logits; logits
// more than 42.6 units down, whose nucleus weight is below the 2^-40 fixed
// point, share the last bin, counted in registers).  Nucleus masses are sums
// of the weights 2^((l - R) log2(e)/T) in 2^-40 fixed point: exact,
// order-independent integer adds, the same result in every run.
//   Rows of at most 128 KB: R is the row max (pass 0); pass 1 counts (top-k)
//   or sums the fixed-point weights (nucleus) per bin; the bin holding the
//   k-th logit / the running mass top_p * total is found by a block scan; pass
//   2 gathers it, and the threshold is read off its logits in descending
//   order.
//   Longer rows: R is the max of the row's first sixteenth, so pass 1 (counts
//   per bin, the logits above R set aside) also finds the true max, and the
//   row is read twice in all.  Top-k proceeds as above; the nucleus brackets
//   the bins its threshold can lie in from the counts (a bin's count bounds its
//   mass within 1.6 %), gathers them in pass 2 while summing every weight in
//   float, and takes the threshold the exact fixed-point sums give wherever the
//   float sums' error bounds leave one candidate (else one exact pass decides).
// A selected bin of more than 4096 logits takes an exact radix selection over
// the order-preserving 32-bit keys of its logits (11 + 11 + 10 bits, one pass
// each).
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "../../include/spec_verify.h"
#include "common.cuh"
#include "softmax.cuh"

namespace specv {

namespace {

constexpr int kTT = 512;
constexpr int kTW = kTT / 32;
constexpr int kBins = 2048;  // first two levels; the third uses 1024

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

// A histogram of 64-bit sums kept as three arrays of 32-bit words, bits 0-13, 14-27 and 28 up of every
// added value, so that every update is a 32-bit shared-memory atomic whose result is not waited for (a
// returned old value, needed to carry between two words, would stall each thread on every update).  With
// at most 2^18 adds of values below 2^60 per bin, none of the words can wrap: 2^18 (2^14 - 1) < 2^32, and
// the high words sum the values' bits 28 up.  mid and hi null: plain 32-bit counts.
struct Hist {
  unsigned int* lo;
  unsigned int* mid;
  unsigned int* hi;
  __device__ __forceinline__ unsigned long long get(int b) const {
    if (!mid) return lo[b];
    return (static_cast<unsigned long long>(hi[b]) << 28) + (static_cast<unsigned long long>(mid[b]) << 14) + lo[b];
  }
  __device__ __forceinline__ void add(int b, unsigned long long v) const {
    if (!mid) {
      atomicAdd(lo + b, static_cast<unsigned int>(v));
      return;
    }
    const unsigned int l = static_cast<unsigned int>(v) & 0x3fffu;
    const unsigned int m = static_cast<unsigned int>(v >> 14) & 0x3fffu;
    const unsigned int h = static_cast<unsigned int>(v >> 28);
    if (l) atomicAdd(lo + b, l);
    if (m) atomicAdd(mid + b, m);
    if (h) atomicAdd(hi + b, h);
  }
  __device__ __forceinline__ void zero(int nb) const {
    for (int k = threadIdx.x; k < nb; k += kTT) {
      lo[k] = 0u;
      if (mid) {
        mid[k] = 0u;
        hi[k] = 0u;
      }
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

constexpr int kCap = 4096;  // logits of the selected bin sorted in shared memory (a power of two)
// the histogram (three words per bin) and the gathered logits share one buffer
constexpr int kBufBytes = 3 * kBins * sizeof(unsigned int);
static_assert(kBufBytes >= kCap * sizeof(float), "the buffer holds the gathered logits");
constexpr float kBinsPerUnit = 48.f;  // bins per unit of log2 probability (the last bin starts 42.6 units down)

// floor(d) for d in [0, kBins - 1], kBins - 1 above: a round-toward-zero add of 2^23 leaves floor(d) in the
// low mantissa bits (plain FP32 and integer operations, no conversion instruction).
// s48 = scale * kBinsPerUnit.
__device__ __forceinline__ int dist_bin(float f, float M, float s48) {
  const float d = fminf((M - f) * s48, static_cast<float>(kBins - 1));  // >= 0
  return __float_as_int(__fadd_rz(d, 8388608.f)) & 0x7fffff;
}

// trunc(w * 2^40) for a float w in [0, 2^23), from w's bits: the 24-bit significand shifted by its exponent
// (the same integer as the truncating float-to-64-bit conversion, with integer shifts instead).
__device__ __forceinline__ unsigned long long fixed40(float w) {
  const uint32_t u = __float_as_uint(w);
  const int e = static_cast<int>(u >> 23) - 110;  // w * 2^40 = significand * 2^(biased exponent - 150 + 40)
  const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
  if (u < 0x00800000u) return 0ull;  // zero (exp2 flushes subnormals)
  return e >= 0 ? m << e : (e > -24 ? m >> -e : 0ull);
}

// Exact radix selection over the order-preserving keys of the logits l <= M in distance bin `db` (M the
// reference the bins are measured from): the key at which the running count (top-k) or fixed-point mass
// (nucleus) from the largest logit down first reaches `need`.
template <typename T, bool kTopP, typename W>
__device__ uint32_t radix_select(const T* row, int V, bool vec, float M, float s48, int db, unsigned long long need,
                                 const Hist& h, unsigned long long* wsum, Pick* pk, W&& weight) {
  h.zero(kBins);
  for_each_logit<T>(row, V, vec, [&](float f) {
    if (f > -INFINITY && f <= M && dist_bin(f, M, s48) == db) h.add(fkey(f) >> 21, kTopP ? weight(f) : 1ull);
  });
  __syncthreads();
  const Pick p1 = pick_from_top(h, kBins, need, wsum, pk);
  const uint32_t b1 = static_cast<uint32_t>(p1.bin);
  const unsigned long long need2 = need - p1.above;
  h.zero(kBins);
  for_each_logit<T>(row, V, vec, [&](float f) {
    if (f > -INFINITY && f <= M && dist_bin(f, M, s48) == db) {
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
    if (f > -INFINITY && f <= M && dist_bin(f, M, s48) == db) {
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

constexpr int kOver = 512;           // logits above the provisional max kept for the selection
constexpr float kOverUnits = 10.f;   // largest M - R (log2 units) whose overflow weights the fixed point holds
constexpr int kSampleRowBytes = 131072;  // longer rows take the provisional max from a prefix

// Logits the reference R of a long row is the max of: the row's first sixteenth, at least 4096.
__device__ __forceinline__ int sample_len(int V) { return min(V, max(4096, V / 16)); }

// Block-wide NaN-propagating maximum; every thread gets it.
__device__ __forceinline__ float block_max_nan(float m, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  m = warp_max_nan(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float M = red[0];
  for (int w = 1; w < kTW; ++w) M = max_nan(M, red[w]);
  __syncthreads();
  return M;
}

// Block-wide sum of the threads' values; every thread gets it.
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_incl_u64(v, lane);
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kTW; ++w) t += wsum[w];
  __syncthreads();
  return t;
}

// Block-wide maximum of the threads' values; every thread gets it.
__device__ __forceinline__ unsigned int block_max_u32(unsigned int v, unsigned long long* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_max_sync(0xffffffffu, v);
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  unsigned int m = 0;
  for (int w = 0; w < kTW; ++w) m = max(m, static_cast<unsigned int>(wsum[w]));
  __syncthreads();
  return m;
}

// The first index of s[0, n) (n <= kPer * kTT, largest logit first) at which the running sum of units from
// index 0 reaches need, 1 <= need <= the sum over s[0, n); every thread gets it.
template <int kPer, typename U>
__device__ int first_reaching(const float* s, int n, unsigned long long need, U&& units, unsigned long long* wsum,
                              int* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long local = 0;
  for (int j = 0; j < kPer; ++j) {
    const int i = tid * kPer + j;
    if (i < n) local += units(s[i]);
  }
  const unsigned long long incl_w = warp_incl_u64(local, lane);
  if (lane == 31) wsum[warp] = incl_w;
  __syncthreads();
  unsigned long long before = 0;
  for (int w = 0; w < warp; ++w) before += wsum[w];
  const unsigned long long excl = before + incl_w - local;
  if (excl < need && need <= excl + local) {
    unsigned long long run = excl;
    for (int j = 0; j < kPer; ++j) {
      const int i = tid * kPer + j;
      run += units(s[i]);
      if (run >= need) {
        *out = i;
        break;
      }
    }
  }
  __syncthreads();
  const int r = *out;
  __syncthreads();
  return r;
}

// Among n <= kTT gathered logits (in any order): the logit at which the running sum of units, taken from the
// largest down (ties by index), first reaches need_a, and the one for need_b.  Thread t sums the units
// of the logits that come before cand[t] in that order, so no sort or scan is needed; w holds the units
// (kTT slots).  found_a / found_b = 0 if the whole sum stays below the need.  Every thread gets the results.
struct Reached {
  float a, b;
  int found_a, found_b;
};

template <typename U>
__device__ Reached reach_small(const float* cand, int n, unsigned long long need_a, unsigned long long need_b,
                               U&& units, unsigned long long* w, Reached* out) {
  const int t = threadIdx.x;
  if (t == 0) {
    out->found_a = 0;
    out->found_b = 0;
  }
  if (t < n) w[t] = units(cand[t]);
  __syncthreads();
  if (t < n) {
    const float f = cand[t];
    unsigned long long pre = 0;
    for (int j = 0; j < n; ++j) {
      const float g = cand[j];
      if (g > f || (g == f && j < t)) pre += w[j];
    }
    const unsigned long long post = pre + w[t];
    if (pre < need_a && need_a <= post) {
      out->a = f;
      out->found_a = 1;
    }
    if (pre < need_b && need_b <= post) {
      out->b = f;
      out->found_b = 1;
    }
  }
  __syncthreads();
  const Reached r = *out;
  __syncthreads();
  return r;
}

// Over s[0, n) (n <= kPer * kTT, largest first) with units(s[i]): the first index whose running sum reaches
// need_a, the same for need_b (-1 where the whole sum stays below), and the whole sum.  Every thread gets
// them.  One block scan.
struct Reach {
  int a, b;
  unsigned long long total;
};

template <int kPer, typename U>
__device__ Reach reach_two(const float* s, int n, unsigned long long need_a, unsigned long long need_b, U&& units,
                           unsigned long long* wsum, Reach* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    out->a = -1;
    out->b = -1;
  }
  unsigned long long v[kPer], local = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = tid * kPer + j;
    v[j] = i < n ? units(s[i]) : 0ull;
    local += v[j];
  }
  const unsigned long long incl_w = warp_incl_u64(local, lane);
  if (lane == 31) wsum[warp] = incl_w;
  __syncthreads();
  unsigned long long run = 0, total = 0;
  for (int w = 0; w < kTW; ++w) {
    if (w < warp) run += wsum[w];
    total += wsum[w];
  }
  run += incl_w - local;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = tid * kPer + j;
    if (run < need_a && run + v[j] >= need_a) out->a = i;
    if (run < need_b && run + v[j] >= need_b) out->b = i;
    run += v[j];
  }
  __syncthreads();
  const Reach r{out->a, out->b, total};
  __syncthreads();
  return r;
}

// Pass 1 over the row against the reference R: the logits in (-inf, R] counted per distance bin
// floor((R - l) s48), stored high bin first (index kBins - 1 - bin), the far bin, where most logits of a
// long row land, counted in registers instead of by contended atomics.  kAbove: the finite logits above R
// are appended to over[] (*nover counts them all, and may pass kOver), their max is returned in *omax, and
// whether a NaN or +inf was seen is returned, block-wide; the common case, a finite logit at or below R,
// takes one comparison before its bin.  Without kAbove R is the row max and the row holds no NaN or +inf.
// A -inf logit lands in the far bin (the fminf in dist_bin), which counts only finite logits -- unless
// kNoFar: the far bin's count is not used (the nucleus: its weights truncate to 0), and counts -inf too.
template <typename T, bool kAbove, bool kNoFar>
__device__ bool count_pass(const T* row, int V, bool vv, float R, float s48, const Hist& hist, float* over,
                           int* nover, unsigned long long* wsum, float* red, float* omax) {
  hist.zero(kBins);
  unsigned int tail = 0;
  float om = -INFINITY;
  int bad = 0;
  for_each_logit<T>(row, V, vv, [&](float f) {
    if (kAbove && !(f <= R)) {
      if (f < INFINITY) {  // finite, above R
        om = fmaxf(om, f);
        const int at = atomicAdd(nover, 1);
        if (at < kOver) over[at] = f;
      } else {  // NaN or +inf
        bad = 1;
      }
    } else {
      const int bin = dist_bin(f, R, s48);
      if (bin == kBins - 1)
        tail += (kNoFar || f > -INFINITY) ? 1u : 0u;
      else
        atomicAdd(hist.lo + (kBins - 1 - bin), 1u);
    }
  });
  const unsigned long long t = block_sum_u64(tail, wsum);
  if (threadIdx.x == 0) hist.add(0, t);
  if (!kAbove) {
    __syncthreads();
    *omax = -INFINITY;
    return false;
  }
  *omax = block_max_nan(om, red);  // its barriers also complete the histogram
  return __syncthreads_or(bad) != 0;
}

// The weighted histogram over the logits in (-inf, R]: exact fixed-point masses per distance bin (the far
// bin's weights are below 2^-42 and truncate to 0).
template <typename T, typename W>
__device__ void mass_pass(const T* row, int V, bool vv, float R, float s48, const Hist& hist, W&& weight) {
  hist.zero(kBins);
  for_each_logit<T>(row, V, vv, [&](float f) {
    if (f <= R && f > -INFINITY) {
      const int bin = dist_bin(f, R, s48);
      if (bin < kBins - 1) hist.add(kBins - 1 - bin, weight(f));
    }
  });
  __syncthreads();
}

// Fixed-point weight bounds of a logit in distance bin b (nucleus, bins of 1/48 log2 unit): every weight
// 2^(-(R - l) log2(e)/T) * 2^40 of a logit binned at b lies in [lo, hi].  The bin and the weight round
// their exponents apart by far less than the 1/16 of a bin each bound is widened by.
__device__ __forceinline__ void bin_bounds(int b, unsigned long long& lo, unsigned long long& hi) {
  const float w_lo = exp2f(-(static_cast<float>(b) + 1.0625f) / kBinsPerUnit) * 0.999999f;
  const float w_hi = exp2f(-(static_cast<float>(b) - 0.0625f) / kBinsPerUnit) * 1.000001f;
  lo = fixed40(w_lo);
  hi = fixed40(w_hi) + 2ull;  // the truncation, and one unit of margin
}

// ceil(top_p * total) clamped to [1, total] (in double, once: monotone in total).
__device__ __forceinline__ unsigned long long nucleus_need(float top_p, unsigned long long total) {
  unsigned long long need = static_cast<unsigned long long>(ceil(static_cast<double>(top_p) * static_cast<double>(total)));
  if (need < 1) need = 1;
  if (need > total) need = total;
  return need;
}

// Nucleus bracket from the count histogram.  With base = the overflow's exact mass, the total mass lies
// in [tlo, thi] = base + sum_b count_b [lo_b, hi_b], so the running mass to reach, need, lies in
// [nlo, nhi] = [need(tlo), need(thi)]; the threshold's bin lies between the first distance bin whose upper
// cumulative bound reaches nlo and the first whose lower cumulative bound reaches nhi (the last binned
// distance if none).  Also the logits in the bins of that range.  Every thread gets the results.
struct Bracket {
  int first, last;
  unsigned long long count;
};

__device__ Bracket nucleus_bracket(const Hist& h, unsigned long long base, float top_p, unsigned long long* wsum,
                                   unsigned long long* wsum2, Bracket* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = kBins / kTT;  // nearest bins first: thread t holds bins t*kPer ..
  // the far bin (the last) carries no fixed-point mass: its weights are below 2^-42
  auto count = [&](int b) -> unsigned long long { return b < kBins - 1 ? h.get(kBins - 1 - b) : 0ull; };
  unsigned long long cl = 0, ch = 0;
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    unsigned long long lo, hi;
    bin_bounds(b, lo, hi);
    const unsigned long long c = count(b);
    cl += c * lo;
    ch += c * hi;
  }
  if (tid == 0) {
    out->first = kBins - 2;
    out->last = kBins - 2;
  }
  const unsigned long long il = warp_incl_u64(cl, lane), ih = warp_incl_u64(ch, lane);
  if (lane == 31) {
    wsum[warp] = il;
    wsum2[warp] = ih;
  }
  __syncthreads();
  unsigned long long rl = base, rh = base, tlo = base, thi = base;
  for (int w = 0; w < kTW; ++w) {
    if (w < warp) {
      rl += wsum[w];
      rh += wsum2[w];
    }
    tlo += wsum[w];
    thi += wsum2[w];
  }
  const unsigned long long nlo = nucleus_need(top_p, tlo), nhi = nucleus_need(top_p, thi);
  rl += il - cl;
  rh += ih - ch;
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    if (b > kBins - 2) break;
    unsigned long long lo, hi;
    bin_bounds(b, lo, hi);
    const unsigned long long c = count(b);
    rl += c * lo;
    rh += c * hi;
    if (rh >= nlo) atomicMin(&out->first, b);
    if (rl >= nhi) atomicMin(&out->last, b);
  }
  __syncthreads();
  const int f = out->first, l = out->last;
  unsigned long long n = 0;
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    if (b >= f && b <= l) n += count(b);
  }
  n = block_sum_u64(n, wsum);
  return Bracket{f, l, n};
}

// Top-k (kTopP = false: k) or nucleus (kTopP = true: top_p, temperature scale) threshold of one row.
//
// kWhole (rows of at most kSampleRowBytes): R is the row max, taken by a pass of its own; then pass 1 and
// the gather as in the file comment (the nucleus weighted per bin at once).
// Otherwise the distance bins and the nucleus weights take as reference R the max of the row's first
// sixteenth.  Pass 1 counts the logits per distance bin and sets aside the few above R (the "overflow", at
// most kOver); these rank above every binned logit, so the selection walks the sorted overflow first, then
// the bins from the top.
//   top-k: the bin of the k-th logit from the counts; pass 2 gathers it, and the logit's rank among the
//     gathered (or, past kCap logits, the radix selection) gives the threshold.
//   nucleus: a bin's count bounds its mass within about 1.6 %, so the counts bracket the bins the running
//     mass top_p * total can end in; pass 2 gathers the logits of a logit interval holding those bins and
//     sums every weight in float: the total, and the mass above the interval.  Each candidate's exact
//     fixed-point weight, with those of the candidates ranked above it, then locates the running mass
//     top_p * total taken at both ends of the sums' error bounds: if both ends stop at the same logit,
//     that logit is the threshold the exact fixed-point sums give; otherwise (rare: 5 to 7 of 1280-1536
//     c3 rows) a pass of exact fixed-point sums decides.  A bracket of more than kCap logits (top_p
//     within a few percent of 1) takes the weighted histogram instead: exact fixed-point masses per bin,
//     then the gather.
// So a long row is read twice, apart from its prefix and those fallbacks.  If more than kOver logits lie
// above R, or the nucleus weights of the overflow could leave the fixed point (M - R above kOverUnits),
// pass 1 is run again against R = M, where nothing lies above the reference.
template <typename T, bool kTopP, bool kWhole>
__global__ void __launch_bounds__(kTT, 3) threshold_kernel(const void* __restrict__ logits, int V, int k, float scale,
                                                           float top_p, int vec, int path, float* __restrict__ thr) {
  // the histogram and the gathered logits share one buffer: the logits are gathered after the histogram
  // is read
  __shared__ __align__(16) unsigned char buf[kBufBytes];
  unsigned int* hw = reinterpret_cast<unsigned int*>(buf);
  const Hist counts{hw, nullptr, nullptr};
  const Hist masses{hw, hw + kBins, hw + 2 * kBins};
  float* cand = reinterpret_cast<float*>(buf);
  __shared__ float over[kOver];
  __shared__ unsigned long long wsum[kTW], wsum2[kTW];
  __shared__ float red[kTW];
  __shared__ Pick pk;
  __shared__ Bracket bk;
  __shared__ Reach rc;
  __shared__ Reached rs;
  __shared__ int cnt, nover, sel;
  const int tid = threadIdx.x;
  const T* row = reinterpret_cast<const T*>(logits) + (size_t)blockIdx.x * V;
  const bool vv = vec != 0;
  // top-k bins in units of the logit itself (any positive scale orders them the same way)
  const float bscale = kTopP ? scale : 1.4426950408889634f;
  const float b48 = bscale * kBinsPerUnit;
  if (tid == 0) {
    cnt = 0;
    nover = 0;
  }

  // the reference: the max of the row's prefix (NaN-propagating)
  float m = -INFINITY;
  for_each_logit<T>(row, kWhole ? V : sample_len(V), vv, [&](float f) { m = max_nan(m, f); });
  float R = block_max_nan(m, red);
  if (!(R < INFINITY)) {  // NaN or +inf in the row
    if (tid == 0) thr[blockIdx.x] = NAN;
    return;
  }
  float nm = -R * scale;
  // the weight 2^((l - R) log2(e)/T) in (0, 2^kOverUnits] in 2^-40 fixed point (truncated)
  auto weight = [&](float f) -> unsigned long long { return fixed40(fast_exp2(fmaf(f, scale, nm))); };
  auto units = [&](float f) -> unsigned long long { return kTopP ? weight(f) : 1ull; };

  // a row read whole for R has no logit above R: the nucleus takes the weighted histogram at once (for
  // rows this short the count pass and the bracket cost more steps than the per-logit weights they save)
  constexpr bool whole = kWhole;
  if (kTopP && whole) {
    if (!(R > -INFINITY)) {  // nothing finite: no distribution
      if (tid == 0) thr[blockIdx.x] = NAN;
      return;
    }
    if (top_p >= 1.f) {
      if (tid == 0) thr[blockIdx.x] = -INFINITY;
      return;
    }
  }

  // pass 1: counts per distance bin against R, the overflow and its max
  float omax = -INFINITY;
  if (!(kTopP && whole) && count_pass<T, !kWhole, kTopP>(row, V, vv, R, b48, counts, over, &nover, wsum, red, &omax)) {
    if (tid == 0) thr[blockIdx.x] = NAN;  // NaN or +inf in the row
    return;
  }
  const float M = fmaxf(R, omax);
  if (!(M > -INFINITY)) {  // nothing finite: top-k keeps everything, nucleus has no distribution
    if (tid == 0) thr[blockIdx.x] = kTopP ? NAN : -INFINITY;
    return;
  }
  if (kTopP && top_p >= 1.f) {
    if (tid == 0) thr[blockIdx.x] = -INFINITY;
    return;
  }
  int no = nover;
  if (!whole && (no > kOver || (kTopP && !((M - R) * scale < kOverUnits)))) {
    // pass 1 again against the true max: no logit lies above it (nover is left as it is)
    R = M;
    nm = -R * scale;
    count_pass<T, !kWhole, kTopP>(row, V, vv, R, b48, counts, over, &nover, wsum, red, &omax);
    no = 0;
  }

  // the overflow, largest first, and its units (a count, or the exact fixed-point mass)
  if (!whole && no > 0) {
    int n2 = 1;
    while (n2 < no) n2 <<= 1;
    for (int i = no + tid; i < n2; i += kTT) over[i] = -INFINITY;
    __syncthreads();
    sort_desc(over, n2);
  }
  unsigned long long O = static_cast<unsigned long long>(no);
  if (kTopP) {
    unsigned long long local = 0;
    for (int i = tid; i < no; i += kTT) local += weight(over[i]);
    O = block_sum_u64(local, wsum);
  }

  int db = 0;                     // the distance bin (top-k, weighted nucleus) holding the threshold
  unsigned long long need2 = 0;   // units still needed inside the gathered logits
  if (!kTopP) {
    const Pick p0 = pick_from_top(counts, kBins, 1ull, wsum, &pk);
    const unsigned long long total = O + p0.total;
    if (static_cast<unsigned long long>(k) > total) {  // fewer than k finite logits
      if (tid == 0) thr[blockIdx.x] = -INFINITY;
      return;
    }
    if (static_cast<unsigned long long>(k) <= O) {  // the k-th largest is in the overflow
      if (tid == 0) thr[blockIdx.x] = over[k - 1];
      return;
    }
    const Pick p = pick_from_top(counts, kBins, static_cast<unsigned long long>(k) - O, wsum, &pk);
    db = kBins - 1 - p.bin;
    need2 = static_cast<unsigned long long>(k) - O - p.above;
    // pass 2: the bin's logits into shared memory.  dist_bin(l) = db gives x_lo <= l (half a bin of margin
    // for the bin's rounding), so one comparison passes over every other logit; the few at or above x_lo
    // take the exact test
    const float x_lo = db < kBins - 1 ? R - (static_cast<float>(db) + 1.5f) / b48 : -INFINITY;
    for_each_logit<T>(row, V, vv, [&](float f) {
      if (f >= x_lo && f <= R && f > -INFINITY && dist_bin(f, R, b48) == db) {
        const int at = atomicAdd(&cnt, 1);
        if (at < kCap) cand[at] = f;
      }
    });
    __syncthreads();
  } else {
    bool weighted = true;
    const Bracket br = whole ? Bracket{0, 0, ~0ull} : nucleus_bracket(counts, O, top_p, wsum, wsum2, &bk);
    if (!whole && path != 2 && br.count <= static_cast<unsigned long long>(kCap)) {
      // a logit interval holding the bracket's bins: dist_bin(l) in [first, last] gives x_lo <= l <= x_hi,
      // half a bin of margin at each end for the bins' rounding
      const float x_hi = R - (static_cast<float>(br.first) - 0.5f) / b48;
      const float x_lo = R - (static_cast<float>(br.last) + 1.5f) / b48;
      // pass 2: the interval's logits into shared memory, and every weight summed in float: below the
      // interval (the common case: one comparison and one add), inside it, and above it up to R (with
      // their term counts; the logits above R are the overflow, whose exact mass is O; -inf weighs 0)
      float tlow = 0.f, tin = 0.f, tab = 0.f;
      unsigned int nin = 0, nab = 0;
      for_each_logit<T>(row, V, vv, [&](float f) {
        const float w = fast_exp2(fmaf(f, scale, nm));
        if (f >= x_lo) {
          if (f <= R) {
            if (f > x_hi) {
              tab += w;
              ++nab;
            } else {
              tin += w;
              ++nin;
              const int at = atomicAdd(&cnt, 1);
              if (at < kCap) cand[at] = f;
            }
          }
        } else {
          tlow += w;
        }
      });
      // each thread's float sums to fixed point, then exact integer sums.  A float sum of n positive terms
      // is within (n - 1) 2^-24 of its exact value (relative): n is at most V / kTT + 64 for the sum below
      // the interval (the mass beyond the nucleus, a small part of the total for the usual top_p) and the
      // largest count of any thread for the other two; plus the conversions (one unit per thread and sum)
      // and the <= V weights the exact sum truncates.
      const unsigned long long le = block_sum_u64(fixed40(tlow), wsum);
      const unsigned long long ie = block_sum_u64(fixed40(tin), wsum);
      const unsigned long long ae = block_sum_u64(fixed40(tab), wsum);
      const double nmax = block_max_u32(max(nin, nab), wsum);
      const unsigned long long te = le + ie + ae;
      const double u = 5.9604644775390625e-8 * 1.01;
      const unsigned long long slack = static_cast<unsigned long long>(V) + 4 * kTT;
      const unsigned long long aerr = static_cast<unsigned long long>(static_cast<double>(ae) * nmax * u) + slack;
      const double nlow = static_cast<double>(V) / kTT + 64.0;
      const unsigned long long terr =
          static_cast<unsigned long long>(static_cast<double>(le) * nlow * u + static_cast<double>(ie + ae) * nmax * u) +
          slack;
      const unsigned long long nlo = nucleus_need(top_p, O + (te > terr ? te - terr : 0ull));
      const unsigned long long nhi = nucleus_need(top_p, O + te + terr);
      const int n = cnt;
      if (n <= kCap) {
        // more than kTT candidates: sorted, largest first (at most kTT: reach_small takes them as they are)
        const bool small = n <= kTT;
        unsigned long long* wbuf = reinterpret_cast<unsigned long long*>(cand + kCap / 2);
        if (!small) {
          int n2 = 1;
          while (n2 < n) n2 <<= 1;
          for (int i = n + tid; i < n2; i += kTT) cand[i] = -INFINITY;
          __syncthreads();
          sort_desc(cand, n2);
        }
        const unsigned long long alo = ae > aerr ? ae - aerr : 0ull, ahi = ae + aerr;
        if (path == 1) {
          // the exact pass below, whatever the bounds say
        } else if (nhi <= O) {  // inside the overflow, whatever the exact total
          const Reach r = reach_two<kOver / kTT>(over, no, nlo, nhi, units, wsum, &rc);
          if (over[r.a] == over[r.b]) {
            if (tid == 0) thr[blockIdx.x] = over[r.a];
            return;
          }
        } else if (nlo > O + ahi) {  // past the logits above the interval, whatever the exact sums
          if (small) {
            const Reached r = reach_small(cand, n, nlo - O - ahi, nhi - O - alo, units, wbuf, &rs);
            if (r.found_a && r.found_b && r.a == r.b) {
              if (tid == 0) thr[blockIdx.x] = r.a;
              return;
            }
          } else {
            const Reach r = reach_two<kCap / kTT>(cand, n, nlo - O - ahi, nhi - O - alo, units, wsum, &rc);
            if (r.a >= 0 && r.b >= 0 && cand[r.a] == cand[r.b]) {
              if (tid == 0) thr[blockIdx.x] = cand[r.a];
              return;
            }
          }
        }
        // undecided by the bounds: exact fixed-point sums over the same classes
        unsigned long long tx = 0, ax = 0;
        for_each_logit<T>(row, V, vv, [&](float f) {
          if (f <= R) {
            const unsigned long long v = weight(f);
            tx += v;
            if (f > x_hi) ax += v;
          }
        });
        tx = block_sum_u64(tx, wsum);
        ax = block_sum_u64(ax, wsum);
        const unsigned long long need = nucleus_need(top_p, O + tx);
        if (need <= O) {
          const int i = first_reaching<kOver / kTT>(over, no, need, units, wsum, &sel);
          if (tid == 0) thr[blockIdx.x] = over[i];
          return;
        }
        if (need > O + ax) {
          if (small) {
            const Reached r = reach_small(cand, n, need - O - ax, need - O - ax, units, wbuf, &rs);
            if (r.found_a) {
              if (tid == 0) thr[blockIdx.x] = r.a;
              return;
            }
          } else {
            const Reach r = reach_two<kCap / kTT>(cand, n, need - O - ax, need - O - ax, units, wsum, &rc);
            if (r.a >= 0) {
              if (tid == 0) thr[blockIdx.x] = cand[r.a];
              return;
            }
          }
        }
      }
      // more logits in the interval than the buffer holds, or a threshold outside it (not expected):
      // the weighted histogram
    }
    if (weighted) {
      // the weighted histogram: exact fixed-point masses per bin, then the bin's logits
      __syncthreads();
      if (tid == 0) cnt = 0;
      mass_pass<T>(row, V, vv, R, b48, masses, weight);
      const Pick p0 = pick_from_top(masses, kBins, 1ull, wsum, &pk);
      const unsigned long long need = nucleus_need(top_p, O + p0.total);
      if (need <= O) {
        const int i = first_reaching<kOver / kTT>(over, no, need, units, wsum, &sel);
        if (tid == 0) thr[blockIdx.x] = over[i];
        return;
      }
      const Pick p = pick_from_top(masses, kBins, need - O, wsum, &pk);
      db = kBins - 1 - p.bin;
      need2 = need - O - p.above;
      for_each_logit<T>(row, V, vv, [&](float f) {
        if (f <= R && f > -INFINITY && dist_bin(f, R, b48) == db) {
          const int at = atomicAdd(&cnt, 1);
          if (at < kCap) cand[at] = f;
        }
      });
      __syncthreads();
    }
  }
  const int n = cnt;
  if (!kTopP && n <= kTT) {  // the need2-th largest by rank, no sort
    if (tid < n) {
      const float f = cand[tid];
      int r = 0;
      for (int j = 0; j < n; ++j) {
        const float g = cand[j];
        r += (g > f || (g == f && j < tid)) ? 1 : 0;
      }
      if (r == static_cast<int>(need2) - 1) thr[blockIdx.x] = f;
    }
    return;
  }
  if (n > kCap) {  // too many to sort here: exact radix selection over the bin
    const uint32_t key = radix_select<T, kTopP>(row, V, vv, R, b48, db, need2, masses, wsum, &pk, weight);
    if (tid == 0) thr[blockIdx.x] = key_float(key);
    return;
  }
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  for (int i = n + tid; i < n2; i += kTT) cand[i] = -INFINITY;
  __syncthreads();
  sort_desc(cand, n2);
  // top-k: the need2-th largest of the bin; nucleus: the first sorted logit at which the running
  // fixed-point mass reaches need2
  const int i = kTopP ? first_reaching<kCap / kTT>(cand, n, need2, units, wsum, &sel) : static_cast<int>(need2) - 1;
  if (tid == 0) thr[blockIdx.x] = cand[i];
}

namespace {

// The nucleus selection of long rows: 0 = the float sums' bounds decide, the exact pass only where they
// leave two candidates; 1 = always the exact pass; 2 = always the weighted histogram.  All three give the
// same thresholds; SPECVERIFY_NUCLEUS_PATH=bounds / exact / weighted picks one (for tests).
int nucleus_path() {
  const char* env = std::getenv("SPECVERIFY_NUCLEUS_PATH");
  if (!env) return 0;
  if (std::strcmp(env, "exact") == 0) return 1;
  if (std::strcmp(env, "weighted") == 0) return 2;
  return 0;
}

// Rows of at most kSampleRowBytes take the kernel that reads the whole row for R (the exact max).
template <typename T, bool kTopP>
cudaError_t threshold_launch(const void* logits, int R, int V, int k, float scale, float top_p, int vec, float* thr,
                             cudaStream_t stream) {
  const int path = kTopP ? nucleus_path() : 0;
  if (static_cast<long long>(V) * sizeof(T) <= kSampleRowBytes)
    threshold_kernel<T, kTopP, true><<<R, kTT, 0, stream>>>(logits, V, k, scale, top_p, vec, path, thr);
  else
    threshold_kernel<T, kTopP, false><<<R, kTT, 0, stream>>>(logits, V, k, scale, top_p, vec, path, thr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t topk_threshold_launch(const void* logits, int dtype, int R, int V, int k, int vec, float* thr,
                                  cudaStream_t stream) {
  return dtype == 0 ? threshold_launch<float, false>(logits, R, V, k, 1.f, 1.f, vec, thr, stream)
                    : threshold_launch<__nv_bfloat16, false>(logits, R, V, k, 1.f, 1.f, vec, thr, stream);
}

cudaError_t topp_threshold_launch(const void* logits, int dtype, int R, int V, float scale, float top_p, int vec,
                                  float* thr, cudaStream_t stream) {
  return dtype == 0 ? threshold_launch<float, true>(logits, R, V, 0, scale, top_p, vec, thr, stream)
                    : threshold_launch<__nv_bfloat16, true>(logits, R, V, 0, scale, top_p, vec, thr, stream);
}

}  // namespace specv
