// Online softmax normalisers shared by the streaming kernels: the running max m
// and S = sum 2^((l - m) log2(e)/T) of a run of logits, rescaled when m grows,
// one hardware exp2 (ex2.approx) per element.
#pragma once

#include "common.cuh"

namespace specv {

// Packed pairs of float32 (sm_100 family f32x2 arithmetic): lane 0 in the low word.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}

__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Online normaliser update with a group of raw logits.
// With kMask, logits below thr count as -inf in the sum (a standardised row: top-k / nucleus); the
// running max and the raw max still see every logit (the max is always kept, so it is a valid shift).
__device__ __forceinline__ float masked(float f, float thr) { return f < thr ? -INFINITY : f; }

template <int kCnt, bool kMask = false>
__device__ __forceinline__ void online(float& m, float& s, float& raw, const float* f, float sc,
                                       float thr = -INFINITY) {
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
    for (int j = 0; j < kCnt; ++j) acc += fast_exp2(((kMask ? masked(f[j], thr) : f[j]) - m) * sc);
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

// NaN-propagating max of U 16-byte vectors of raw logits, as float32.
template <typename T, int U>
struct GroupMax;

template <int U>
struct GroupMax<float, U> {
  __device__ static __forceinline__ float get(const uint4 (&r)[U]) {
    float m = __uint_as_float(r[0].x);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      m = max_nan(m, __uint_as_float(r[u].x));
      m = max_nan(m, __uint_as_float(r[u].y));
      m = max_nan(m, __uint_as_float(r[u].z));
      m = max_nan(m, __uint_as_float(r[u].w));
    }
    return m;
  }
};

template <int U>
struct GroupMax<__nv_bfloat16, U> {
  // pairs of bf16 compared two at a time on the packed words, then the last pair widened
  __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ static __forceinline__ float get(const uint4 (&r)[U]) {
    uint32_t m = max2(max2(r[0].x, r[0].y), max2(r[0].z, r[0].w));
#pragma unroll
    for (int u = 1; u < U; ++u) m = max2(m, max2(max2(r[u].x, r[u].y), max2(r[u].z, r[u].w)));
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
};

// Online normaliser update with U 16-byte vectors of raw logits: one max and one rescale per group,
// then 2^((l - m) log2(e)/T) per element as a single FFMA and a hardware exp2.
template <typename T, int U, bool kMask = false>
__device__ __forceinline__ void online_group(float& m, float& s, float& raw, const uint4 (&r)[U], float sc,
                                             float thr = -INFINITY) {
  constexpr int kV = Elems<T>::kVec;
  const float vm = GroupMax<T, U>::get(r);
  raw = max_nan(raw, vm);
  if (vm > -INFINITY) {
    if (vm > m) {
      s *= fast_exp2((m - vm) * sc);
      m = vm;
    }
    const float nc = -m * sc;
    float a0 = 0.f, a1 = 0.f;  // even elements accumulate in a0, odd in a1
    if constexpr (sizeof(T) == 2) {
      // bfloat16 carries twice the elements per byte: pairs go through the packed f32x2 FMA / add (two
      // float32 lanes, the same rounding as two scalar operations), fewer instructions per element
      const unsigned long long sc2 = pack2(sc, sc), nc2 = pack2(nc, nc);
      unsigned long long acc = 0ull;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[kV];
        Elems<T>::widen(r[u], f);
#pragma unroll
        for (int j = 0; j < kV; j += 2) {
          const unsigned long long x =
              pack2(kMask ? masked(f[j], thr) : f[j], kMask ? masked(f[j + 1], thr) : f[j + 1]);
          float t0, t1;
          unpack2(fma2(x, sc2, nc2), t0, t1);
          acc = add2(acc, pack2(fast_exp2(t0), fast_exp2(t1)));
        }
      }
      unpack2(acc, a0, a1);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[kV];
        Elems<T>::widen(r[u], f);
#pragma unroll
        for (int j = 0; j < kV; j += 2) {
          a0 += fast_exp2(fmaf(kMask ? masked(f[j], thr) : f[j], sc, nc));
          a1 += fast_exp2(fmaf(kMask ? masked(f[j + 1], thr) : f[j + 1], sc, nc));
        }
      }
    }
    s += a0 + a1;
  }
}

}  // namespace specv
