// Greedy (argmax) verification on sm_103a.
//
// Argmax standardisation (Leviathan, Kalman & Matias; paper-graph-ui teardown
// §2.2 "Standardized Sampling", multigrid.ai on sampling temperature): p_i is
// the one-hot vector at argmax of target row (b, i), so a guess is accepted
// exactly when it equals that argmax, and the emitted token at the first
// mismatch (or at the bonus position) is the argmax itself.  Only the target
// logits are read.
//
// Each CTA scans one slice of one target row with 16-byte streaming loads and
// keeps a (value, index) maximum with the lowest index on ties.  The CTA's
// result is folded into the position's 64-bit key with one atomicMax: the high
// word is the value mapped to an order-preserving unsigned integer, the low
// word is 0xffffffff - index, so a larger key means a larger value or, on a
// tie, a smaller index.  A NaN or +inf anywhere sets the key to all ones
// (invalid).  The last CTA of batch row b to finish (an atomic arrival
// counter) compares the argmaxes with the draft ids, writes the row's outputs,
// and resets the keys and the counter to zero for the next call.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace specv {

namespace {

constexpr unsigned long long kKeyInvalid = ~0ull;

__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long pack_key(float v, int idx) {
  return (static_cast<unsigned long long>(ordered_bits(v)) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(idx));
}

// Fold element x at index k into (best, bi): strictly larger wins, so the
// earliest index survives among equal values visited in increasing order.
__device__ __forceinline__ void consider(float x, int k, float& best, int& bi, bool& bad) {
  bad |= !(x < INFINITY);       // NaN or +inf
  x = (x == 0.f) ? 0.f : x;     // -0 and +0 compare equal: one canonical zero
  if (x > best) {
    best = x;
    bi = k;
  }
}

__device__ __forceinline__ void pick(float& best, int& bi, float ob, int oi) {
  if (ob > best || (ob == best && oi < bi)) {
    best = ob;
    bi = oi;
  }
}

__device__ void finalize_greedy(const GreedyParams& a, int b, int gb) {
  const int G1 = a.G + 1;
  unsigned long long* key = a.ws.key + (size_t)b * G1;
  bool nonfinite = false, badtok = false;
  for (int j = 0; j <= gb; ++j) {
    const unsigned long long k = __ldcg(key + j);
    if (k == kKeyInvalid || static_cast<uint32_t>(k >> 32) == ordered_bits(-INFINITY)) nonfinite = true;
  }
  for (int j = 0; j < gb; ++j) {
    const int x = __ldg(a.ids + (size_t)b * a.G + j);
    if (x < 0 || x >= a.V) badtok = true;
  }
  int32_t* e = a.emitted + (size_t)b * G1;
  if (nonfinite || badtok) {
    for (int j = 0; j < G1; ++j) e[j] = -1;
    a.n_acc[b] = -1;
    atomicOr(a.ws.err, nonfinite ? kErrNonfinite : kErrToken);
  } else {
    int n = gb;
    for (int j = 0; j < gb; ++j) {
      const int am = static_cast<int>(0xffffffffu - static_cast<uint32_t>(__ldcg(key + j)));
      if (am != __ldg(a.ids + (size_t)b * a.G + j)) {
        n = j;
        break;
      }
    }
    for (int j = 0; j < n; ++j) e[j] = __ldg(a.ids + (size_t)b * a.G + j);
    e[n] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(__ldcg(key + n)));
    for (int j = n + 1; j < G1; ++j) e[j] = -1;
    a.n_acc[b] = n;
  }
  for (int j = 0; j <= gb; ++j) key[j] = 0ull;
  a.ws.ticket[b] = 0u;
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kGreedyThreads) greedy_rows_kernel(const GreedyParams a) {
  constexpr int kW = kGreedyThreads / 32;
  __shared__ float rv[kW];
  __shared__ int ri[kW];
  __shared__ int rbad[kW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x % a.nslices;
  const int pos = blockIdx.x / a.nslices;
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

  const int lo = s * a.slice;
  const int n = min(a.V, lo + a.slice) - lo;
  if (!bounds_ok(b < a.B && n > 0 && lo + n <= a.V, a.ws.err)) return;
  const T* src = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + i) * a.V + lo;
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 4;
  float best = -INFINITY;
  int bi = INT_MAX;
  bool bad = false;
  int done = 0;
  if (a.vec) {
    const int nv = n / kV;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    int v = tid;
    for (; v + (U - 1) * kGreedyThreads < nv; v += U * kGreedyThreads) {
      uint4 r[U];
#pragma unroll
      for (int u = 0; u < U; ++u) r[u] = ldg_stream(s4 + v + u * kGreedyThreads);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[kV];
        Elems<T>::widen(r[u], f);
#pragma unroll
        for (int j = 0; j < kV; ++j) consider(f[j], lo + (v + u * kGreedyThreads) * kV + j, best, bi, bad);
      }
    }
    for (; v < nv; v += kGreedyThreads) {
      float f[kV];
      Elems<T>::widen(ldg_stream(s4 + v), f);
#pragma unroll
      for (int j = 0; j < kV; ++j) consider(f[j], lo + v * kV + j, best, bi, bad);
    }
    done = nv * kV;
  }
  for (int k = done + tid; k < n; k += kGreedyThreads) consider(Elems<T>::one(src, k), lo + k, best, bi, bad);

#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    pick(best, bi, ob, oi);
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    rv[warp] = best;
    ri[warp] = bi;
    rbad[warp] = bad ? 1 : 0;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kW; ++w) {
      pick(best, bi, rv[w], ri[w]);
      bad |= rbad[w] != 0;
    }
    atomicMax(a.ws.key + pos, bad ? kKeyInvalid : pack_key(best, bi));
    __threadfence();
    const unsigned prev = atomicAdd(a.ws.ticket + b, 1u);
    if (prev == static_cast<unsigned>(a.nslices * (gb + 1) - 1)) {
      __threadfence();
      finalize_greedy(a, b, gb);
    }
  }
}

cudaError_t greedy_launch(const GreedyParams& p, int dtype, cudaStream_t stream) {
  const long long ctas = (long long)p.B * (p.G + 1) * p.nslices;
  const dim3 grid(static_cast<unsigned>(ctas)), block(kGreedyThreads);
  if (dtype == 0) {
    greedy_rows_kernel<float><<<grid, block, 0, stream>>>(p);
  } else {
    greedy_rows_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace specv
