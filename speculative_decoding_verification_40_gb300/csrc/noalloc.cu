// spec_verify_sample_noalloc: sampling verification for callers that cannot
// allocate device memory.  The scratch the two sampling kernels need lives in
// one fixed array of this library instead of a caller-supplied workspace.
#include <mutex>

#include "../../include/spec_verify.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoallocBytes = static_cast<size_t>(SPEC_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

// Zero-initialised at module load on every device that loads the library, and kept until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

// Device address of g_noalloc_scratch on each device; the host-side symbol is only a stand-in.  Resolved
// once per device by the first call there; a cudaDeviceReset of that device invalidates it (the array's
// new address is not looked up again).
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {  // first call on this device: resolve the symbol with it current
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SPEC_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits, int dtype,
                                          const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                                          float temperature, int B, int gamma, int V, int32_t* emitted,
                                          int32_t* n_accepted, void* stream) {
  const size_t need = spec_workspace_size(B, gamma, V, dtype);
  if (need == 0) return (dtype != SPEC_F32 && dtype != SPEC_BF16) ? SPEC_ERR_DTYPE : SPEC_ERR_ARG;
  if (need > kNoallocBytes) return SPEC_ERR_WORKSPACE;  // beyond the fixed scratch: use spec_verify_sample
  if (B == 0) return SPEC_OK;
  // every argument check before the shared array is touched: a rejected call leaves it as it was
  int st = specv::check_sample_args(target_logits, draft_logits, dtype, draft_ids, uniforms, temperature, B, gamma,
                                    V, emitted, n_accepted);
  if (st != SPEC_OK) return st;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != SPEC_OK) return st;
  // The error word and the per-row arrival counters must start at zero; every other slot is either
  // written before it is read or left at zero by the previous call.
  const size_t head = 256 + specv::align_up(static_cast<size_t>(B) * 4, 256);
  if (cudaMemsetAsync(scratch, 0, head, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  return spec_verify_sample(target_logits, draft_logits, dtype, draft_ids, draft_len, uniforms, temperature, B,
                            gamma, V, emitted, n_accepted, scratch, kNoallocBytes, stream);
}
