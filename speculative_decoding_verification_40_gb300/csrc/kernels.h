// Parameters and host launchers of the verification kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace specv {

struct VerifyParams {
  const void* target;        // [B, G+1, V]
  const void* draft;         // [B, G, V]
  const int32_t* ids;        // [B, G]
  const int32_t* draft_len;  // [B] or nullptr
  float scale;               // log2(e) / T
  int B, G, V;
  int L;                     // vocabulary slice per CTA (multiple of 8)
  int vec;                   // every logit row starts on a 16-byte boundary
  float* beta;               // [B, G] statistics outputs (any may be nullptr)
  float* p_draft;
  float* q_draft;
  float* accept_prob;
  float* resid;
  Workspace ws;
};

struct GreedyParams {
  const void* target;        // [B, G+1, V]
  const int32_t* ids;        // [B, G]
  const int32_t* draft_len;  // [B] or nullptr
  int B, G, V;
  int slice;                 // target elements per CTA (multiple of 8)
  int nslices;               // CTAs per target row
  int vec;
  int32_t* emitted;
  int32_t* n_acc;
  Workspace ws;
};

struct SampleParams {
  const void* target;        // [B, G+1, V]
  const void* draft;         // [B, G, V]
  const int32_t* ids;        // [B, G]
  const int32_t* draft_len;  // [B] or nullptr
  const float* uniforms;     // [B, G+1]
  const float* tthr;         // [B, G+1] standardisation thresholds of the target rows, or nullptr
  const float* dthr;         // [B, G] standardisation thresholds of the draft rows, or nullptr
  float scale;               // log2(e) / T
  float lq;                  // lenience l in (0, 1]: q enters the accept test and the residual as l q
  int B, G, V;
  int slice;                 // vocabulary elements per work item (a multiple of 32 x elements per 16 bytes)
  int nslices;               // stream CTAs per logit row (<= kMaxSlices)
  int dslice;                // vocabulary elements per draw CTA (a multiple of the draw chunk)
  int ndslices;              // draw CTAs per batch row (<= kMaxSlices)
  int vec;                   // every logit row starts on a 16-byte boundary
  int cluster;               // draw kernel: the ndslices CTAs of a row form one thread-block cluster
  int rcs;                   // one-launch kernel: CTAs per batch row (thread-block cluster size, <= 16)
  int rslice;                // one-launch kernel: vocabulary elements per CTA (a multiple of 16 bytes)
  int sms;                   // streaming multiprocessors of the device (host side; 0 if unknown)
  int lazy;                  // draw kernel: early-exit validity (logit rows after the first rejection ignored)
  int32_t* emitted;          // [B, G+1]
  int32_t* n_acc;            // [B]
  Workspace ws;
};

// Host-side argument checks of the sampling entry points other than the workspace (sizes, dtype,
// temperature, pointers); a spec_status_t.
int check_sample_args(const void* target, const void* draft, int dtype, const int32_t* ids, const float* uniforms,
                      float temperature, int B, int gamma, int V, const int32_t* emitted, const int32_t* n_accepted);

// dtype: 0 = float32, 1 = bfloat16.  stats selects the statistics kernel.
cudaError_t stats_prepare(int dtype);
cudaError_t stats_max_active_clusters(int dtype, int cs, int* out);
cudaError_t stats_launch(const VerifyParams& p, int dtype, int cs, cudaStream_t stream);
// phases: 1 = stream kernel, 2 = draw kernel, 3 = both (or the short-row kernel for rows of at most 8 KB)
cudaError_t sample_launch(const SampleParams& p, int dtype, int phases, cudaStream_t stream);
// early exit: the one-launch kernel streaming each row only up to its first rejection
cudaError_t sample_early_exit_launch(SampleParams p, int dtype, cudaStream_t stream);
// the early exit's one-launch kernel: a thread-block cluster of p.rcs CTAs per batch row (slices of
// p.rslice elements) that streams a row's positions only up to its first rejection; pdl: launch as a
// programmatic dependent of the previous launch on the stream
cudaError_t rows_launch(const SampleParams& p, int dtype, cudaStream_t stream, bool pdl);
// clusters of cs CTAs of the early exit's one-launch kernel the device holds at once (0: cannot be
// scheduled), for draft width G
cudaError_t rows_max_active_clusters(int dtype, int G, int cs, int* out);
// stream kernel (gamma = 0) then one sampling CTA per row; emitted is the [B] token output
cudaError_t rows_sample_launch(const SampleParams& p, int dtype, cudaStream_t stream);
// one CTA per row: the logit threshold of top-k / nucleus standardisation
cudaError_t topk_threshold_launch(const void* logits, int dtype, int R, int V, int k, int vec, float* thr,
                                  cudaStream_t stream);
cudaError_t topp_threshold_launch(const void* logits, int dtype, int R, int V, float scale, float top_p, int vec,
                                  float* thr, cudaStream_t stream);
cudaError_t greedy_launch(const GreedyParams& p, int dtype, cudaStream_t stream);

}  // namespace specv
