// Device-side building blocks shared by the verification kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

// ---------------------------------------------------------------- launch constants
constexpr int kStatsThreads = 256;     // threads per CTA of the statistics kernel
constexpr int kMaxCluster = 16;        // largest thread-block cluster (non-portable size)
constexpr int kGreedyThreads = 256;    // threads per CTA of the greedy kernel
constexpr int kGreedySlice = 8192;     // target-row elements per greedy CTA
constexpr int kStreamThreads = 256;    // threads per CTA of the sampling kernels
constexpr int kStreamSliceBytes = 65536;  // bytes of one logit row per sampling work item
constexpr int kMaxVocab = 262144;      // SPEC_MAX_VOCAB
constexpr int kMaxGamma = 64;          // SPEC_MAX_GAMMA

// Device error word: bit k is set for spec_status_t k.
constexpr uint32_t kErrArg = 1u << 1;
constexpr uint32_t kErrNonfinite = 1u << 4;
constexpr uint32_t kErrToken = 1u << 5;
constexpr uint32_t kErrTimeout = 1u << 6;
constexpr uint32_t kErrBounds = 1u << 8;   // debug-bounds builds: an index check failed (access skipped)

#ifdef SPEC_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// Residual-mass floor below which the draw falls back to p (interactiveml correction rule).
constexpr float kZFloor = 1e-15f;

// ---------------------------------------------------------------- workspace
// Every region is zero when no call is running: each row's last work item
// returns the slots it used to zero, so workspaces can be shared by calls of
// any shape.  Only the error word keeps its value until it is read.
constexpr int kMaxSlices = 32;          // vocabulary slices per row in the sampling kernel
constexpr int kMaxChunksPerSlice = 128; // chunks per sampling slice
// Chunk slots of one drawn row (draw slices x chunks per slice): at most V / 512 + 128 = 640 for
// V <= 262144, since a draw slice holds at least V / 32 elements and a chunk at least 512.
constexpr int kMaxRowChunks = 640;

struct Workspace {
  uint32_t* err;             // error word (bits above)
  uint32_t* ticket;          // [B] arrivals per batch row: greedy slice CTAs, or draw CTAs
  unsigned long long* key;   // [B, G+1] greedy (value, index) argmax keys
  float* part;               // [B, G+1, kMaxSlices] float4 slice normalisers (m_p, S_p, m_q, S_q)
  float* xl;                 // [B, G] float2 target / draft logit at the draft token
  float* dch;                // [B, chunks] float2 mass of each chunk of the drawn row(s)
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Chunk records per row: enough for any slice length the host may choose (<= 128 chunks per slice).
__host__ __device__ inline size_t chunks_per_row(int V) { return (size_t)(V + 127) / 128 + kMaxChunksPerSlice; }

__host__ __device__ inline size_t ws_bytes_for(int B, int G, int V) {
  const size_t P = (size_t)B * (size_t)(G + 1);
  return 256 + align_up((size_t)B * 4, 256) + align_up(P * 8, 256) + align_up(P * kMaxSlices * 16, 256) +
         align_up((size_t)B * G * 8, 256) + align_up((size_t)B * chunks_per_row(V) * 8, 256);
}

inline Workspace ws_carve(void* base, int B, int G, int V) {
  const size_t P = (size_t)B * (size_t)(G + 1);
  char* p = static_cast<char*>(base);
  Workspace w;
  w.err = reinterpret_cast<uint32_t*>(p);
  p += 256;
  w.ticket = reinterpret_cast<uint32_t*>(p);
  p += align_up((size_t)B * 4, 256);
  w.key = reinterpret_cast<unsigned long long*>(p);
  p += align_up(P * 8, 256);
  w.part = reinterpret_cast<float*>(p);
  p += align_up(P * kMaxSlices * 16, 256);
  w.xl = reinterpret_cast<float*>(p);
  p += align_up((size_t)B * G * 8, 256);
  w.dch = reinterpret_cast<float*>(p);
  return w;
}

#ifdef __CUDACC__
// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Cluster-wide barrier; release/acquire orders shared-memory writes before it
// with distributed-shared-memory reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Split cluster barrier: arrive without ordering (at a CTA's start), wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Split cluster barrier with ordering: shared-memory writes (local or distributed) before the arrive are
// visible to every thread of the cluster after its matching wait.  Each thread alternates arrive / wait.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores into shared memory of a CTA of this cluster (address from dsmem_map).
__device__ __forceinline__ void dsmem_st_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void dsmem_st_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float a) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// 16-byte streaming load of read-only data: no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Index check of debug-bounds builds (-DSPEC_DEBUG_BOUNDS): a false condition records kErrBounds in the
// error word and returns false, and the caller skips the access.  In normal builds it is always true and
// compiles away.  Conditions are uniform over a CTA where the caller returns before a barrier.
__device__ __forceinline__ bool bounds_ok(bool cond, uint32_t* err) {
  if (kDebugBounds && !cond) {
    atomicOr(err, kErrBounds);
    return false;
  }
  return true;
}

// max that propagates NaN: a NaN anywhere in a row survives the reduction.
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Inclusive prefix sum across the warp's lanes.
__device__ __forceinline__ float warp_inclusive_scan(float v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += y;
  }
  return v;
}
// ---------------------------------------------------------------- logit element access
template <typename T>
struct Elems;

template <>
struct Elems<float> {
  static constexpr int kVec = 4;  // elements per 16-byte load
  __device__ static __forceinline__ void widen(const uint4& r, float* f) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
  __device__ static __forceinline__ float one(const float* p, int k) { return __ldg(p + k); }
};

template <>
struct Elems<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void widen(const uint4& r, float* f) {
    f[0] = __uint_as_float(r.x << 16);
    f[1] = __uint_as_float(r.x & 0xffff0000u);
    f[2] = __uint_as_float(r.y << 16);
    f[3] = __uint_as_float(r.y & 0xffff0000u);
    f[4] = __uint_as_float(r.z << 16);
    f[5] = __uint_as_float(r.z & 0xffff0000u);
    f[6] = __uint_as_float(r.w << 16);
    f[7] = __uint_as_float(r.w & 0xffff0000u);
  }
  __device__ static __forceinline__ float one(const __nv_bfloat16* p, int k) {
    const unsigned short bits = __ldg(reinterpret_cast<const unsigned short*>(p) + k);
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  }
};

template <int kVec>
__device__ __forceinline__ void store_f32(float* dst, const float* f) {
#pragma unroll
  for (int j = 0; j < kVec; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
}

#endif  // __CUDACC__

}  // namespace specv
