// Planning helpers around the verification step: the expected tokens per step (Eq. 1), the walltime
// improvement (Theorem 3.8), the arithmetic-operations factor (Theorem 3.11), the optimal number of
// guesses (§3.5) and the corpus acceptance rate alpha = E[beta] (Corollary 3.6) -- Leviathan, Kalman &
// Matias, "Fast Inference from Transformers via Speculative Decoding", as restated in the paper-graph-ui
// teardown (§3.1-§3.5).  The first four are host functions; alpha is a one-CTA device reduction of the
// beta values spec_accept_stats writes.
#include <cmath>

#include "../../include/spec_verify.h"
#include "common.cuh"

namespace {

constexpr int kAlphaThreads = 1024;

// Mean of the finite entries of beta[0, n) and their count, in double, in a fixed order: thread t sums
// entries t, t + 1024, ... in turn, then the partial sums are added in thread order.
__global__ void __launch_bounds__(kAlphaThreads) alpha_mean_kernel(const float* __restrict__ beta, long long n,
                                                                   double* __restrict__ out) {
  __shared__ double ps[kAlphaThreads];
  __shared__ long long pc[kAlphaThreads];
  double s = 0.0;
  long long c = 0;
  for (long long k = threadIdx.x; k < n; k += kAlphaThreads) {
    const float b = __ldg(beta + k);
    if (isfinite(b)) {
      s += static_cast<double>(b);
      ++c;
    }
  }
  ps[threadIdx.x] = s;
  pc[threadIdx.x] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    double S = 0.0;
    long long C = 0;
    for (int t = 0; t < kAlphaThreads; ++t) {
      S += ps[t];
      C += pc[t];
    }
    out[0] = C > 0 ? S / static_cast<double>(C) : nan("");
    out[1] = static_cast<double>(C);
  }
}

}  // namespace

extern "C" {

double spec_expected_tokens(double alpha, int gamma) {
  if (!(alpha >= 0.0 && alpha <= 1.0) || gamma < 0) return nan("");
  if (alpha == 1.0) return static_cast<double>(gamma) + 1.0;
  return (1.0 - std::pow(alpha, gamma + 1)) / (1.0 - alpha);
}

double spec_walltime_improvement(double alpha, int gamma, double c) {
  if (!(c >= 0.0)) return nan("");
  return spec_expected_tokens(alpha, gamma) / (static_cast<double>(gamma) * c + 1.0);
}

double spec_operations_factor(double alpha, int gamma, double c_hat) {
  if (!(c_hat >= 0.0)) return nan("");
  return (static_cast<double>(gamma) * c_hat + static_cast<double>(gamma) + 1.0) / spec_expected_tokens(alpha, gamma);
}

int spec_optimal_gamma(double alpha, double c, int max_gamma, double* improvement) {
  if (!(alpha >= 0.0 && alpha <= 1.0) || !(c >= 0.0) || max_gamma < 1) return -1;
  int best = 1;
  double best_v = spec_walltime_improvement(alpha, 1, c);
  for (int g = 2; g <= max_gamma; ++g) {
    const double v = spec_walltime_improvement(alpha, g, c);
    if (v > best_v) {
      best = g;
      best_v = v;
    }
  }
  if (improvement) *improvement = best_v;
  return best;
}

int spec_alpha_mean(const float* beta, long long n, double* out, void* stream) {
  if (n < 0 || out == nullptr || (n > 0 && beta == nullptr)) return SPEC_ERR_ARG;
  alpha_mean_kernel<<<1, kAlphaThreads, 0, static_cast<cudaStream_t>(stream)>>>(beta, n, out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
