// C ABI of the verification library: argument checks, launch plan, launches.
// The operations are specified in include/spec_verify.h.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "../../include/spec_verify.h"
#include "common.cuh"
#include "kernels.h"

namespace {

using specv::align_up;

constexpr int kStatsSliceBytes = 64 * 1024;  // bytes of each row a statistics CTA streams
constexpr int kMaxDevices = 64;

struct Plan {
  int cs;     // CTAs per cluster (vocabulary slices per row)
  int L;      // slice length in elements
  int smem;   // dynamic shared memory per CTA
  int nclus;  // clusters the device holds at once (0 until checked on a device)
};

// Statistics kernel: CS CTAs per position, each streaming about 32 KB of each row (at most 16,
// the largest cluster); no dynamic shared memory.
Plan plan_for(int V, int cs, int dtype) {
  (void)dtype;
  Plan p;
  p.cs = cs;
  p.L = static_cast<int>(align_up((V + cs - 1) / cs, 8));
  p.smem = 0;
  p.nclus = 0;
  return p;
}

// SPECVERIFY_CLUSTER (1 to 16) overrides the cluster size.
bool choose_plan(int V, int dtype, Plan* out) {
  const long long esz = dtype == SPEC_F32 ? 4 : 2;
  long long slice = kStatsSliceBytes;
  if (const char* env = std::getenv("SPECVERIFY_STATS_SLICE")) {
    const long long want = std::atoll(env);
    if (want > 0) slice = want;
  }
  long long cs = (static_cast<long long>(V) * esz + slice - 1) / slice;
  if (cs < 1) cs = 1;
  if (cs > specv::kMaxCluster) cs = specv::kMaxCluster;
  if (const char* env = std::getenv("SPECVERIFY_CLUSTER")) {
    const int want = std::atoi(env);
    if (want >= 1 && want <= specv::kMaxCluster) cs = want;
  }
  *out = plan_for(V, static_cast<int>(cs), dtype);
  return true;
}

// Kernel attributes are per device; set them once per (device, kernel, dtype).
std::atomic<int> g_prepared[kMaxDevices][2];
std::mutex g_prep_mu;

int prepare(int dtype) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::atomic<int>& flag = g_prepared[dev][dtype];
  if (flag.load(std::memory_order_acquire)) return SPEC_OK;
  std::lock_guard<std::mutex> lk(g_prep_mu);
  if (!flag.load(std::memory_order_relaxed)) {
    if (specv::stats_prepare(dtype) != cudaSuccess) return SPEC_ERR_CUDA;
    flag.store(1, std::memory_order_release);
  }
  return SPEC_OK;
}

int device_sms();

// Fewest vocabulary elements a stream or draw CTA is given when a small batch halves the slices.
constexpr int kMinSlice = 4096;

// Vocabulary elements per sampling CTA and logit row: 64 KB of the row, at least V/32 so a row has
// at most 32 slices.  `positions` > 0 (the verification's B (gamma + 1)):
//  - a batch that would give fewer than two stream CTAs per SM has its slices halved, down to kMinSlice
//    elements, so that a latency-bound small batch still spreads over the GPU (c1, B = 8 and gamma = 4
//    over V = 32128: 320 CTAs of 4096 elements instead of 40 of 32768);
//  - a batch whose grid fits one wave of four CTAs per SM, with at least three per SM, when its slices are
//    larger (up to 256 KB of a row, the most a draw-chunk count allows) takes the largest such slice: the
//    whole stream pass then starts at once and has no partially filled last wave (c2, B = 64, gamma = 8,
//    V = 128256: 576 CTAs of a whole 250 KB row, 57.9 us per call against 60.4 us for 2304 CTAs of 64 KB).
// SPECVERIFY_SLICE (elements) overrides within the same limits.
int sample_slice(int V, int dtype, long long positions = 0) {
  const int chunk = 4 * 32 * (dtype == SPEC_F32 ? 4 : 8);  // elements per draw chunk (4 x 32 lanes x 16 B)
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  int slice = specv::kStreamSliceBytes / esz;
  if (positions > 0) {
    const long long sms = device_sms() > 0 ? device_sms() : 152;
    while (slice / 2 >= kMinSlice && positions * ((V + slice - 1) / slice) < 2 * sms) slice /= 2;
    for (int big = specv::kMaxChunksPerSlice * chunk; big > slice; big /= 2) {
      const long long ctas = positions * ((V + big - 1) / big);
      if (ctas <= 4 * sms && ctas >= 3 * sms) {
        slice = big;
        break;
      }
    }
  }
  if (const char* env = std::getenv("SPECVERIFY_SLICE")) {
    const int want = std::atoi(env);
    if (want > 0) slice = want;
  }
  const int lo = (V + specv::kMaxSlices - 1) / specv::kMaxSlices;
  if (slice < lo) slice = lo;
  slice = static_cast<int>(align_up(slice, chunk));
  if (slice > specv::kMaxChunksPerSlice * chunk) slice = specv::kMaxChunksPerSlice * chunk;
  return slice;
}

// Clusters of `cs` CTAs of the one-launch sampling kernel the current device holds at once (cached per
// device, dtype and size); 0 if it cannot schedule one, -1 if the query fails.
int rows_clusters(int dtype, int G, int cs) {
  struct Entry {
    int dev, dtype, G, cs, n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : cache)
      if (e.dev == dev && e.dtype == dtype && e.G == G && e.cs == cs) return e.n;
  }
  int n = 0;
  if (specv::rows_max_active_clusters(dtype, G, cs, &n) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() < 1024) cache.push_back(Entry{dev, dtype, G, cs, n});
  return n;
}

// Cluster size (CTAs per batch row) and slice length of the one-launch sampling kernel: slices of at
// most 64 KB of a row, so CS = ceil(row bytes / 64 KB); a batch that would give fewer than four CTAs per
// SM has its rows split further (CS doubled while slices stay at least 2 KB, at most 16 CTAs per row),
// so that a small batch still spreads over the GPU (c2, B = 64 rows of 250 KB: 16 CTAs of 16 KB; c1,
// B = 8: 16 CTAs of 4 KB).  A slice holds at most kMaxChunksPerSlice draw chunks, and the cluster size is
// one the device can co-schedule (halved otherwise).  SPECVERIFY_ROW_CLUSTER (1 to 16) overrides.
int rows_plan(int B, int G, int V, int dtype, int* cs_out, int* slice_out) {
  const long long esz = dtype == SPEC_F32 ? 4 : 2;
  const int kv = static_cast<int>(16 / esz);
  const int cpc = 4 * 32 * kv;  // elements per draw chunk
  const long long row = static_cast<long long>(V) * esz;
  int cs = static_cast<int>((row + specv::kStreamSliceBytes - 1) / specv::kStreamSliceBytes);
  if (cs < 1) cs = 1;
  const long long want = 4LL * (device_sms() > 0 ? device_sms() : 152);
  while (cs * 2 <= specv::kMaxCluster && static_cast<long long>(B) * cs < want && row / (cs * 2) >= 2048) cs *= 2;
  if (const char* env = std::getenv("SPECVERIFY_ROW_CLUSTER")) {
    const int w = std::atoi(env);
    if (w >= 1 && w <= specv::kMaxCluster) cs = w;
  }
  if (cs > specv::kMaxCluster) cs = specv::kMaxCluster;
  auto slice_of = [&](int c) { return static_cast<int>(align_up((V + c - 1) / c, kv)); };
  while (cs < specv::kMaxCluster && (slice_of(cs) + cpc - 1) / cpc > specv::kMaxChunksPerSlice) ++cs;
  for (;;) {
    const int n = rows_clusters(dtype, G, cs);
    if (n < 0) return SPEC_ERR_CUDA;
    if (n > 0) break;
    if (cs == 1) return SPEC_ERR_ARG;
    cs /= 2;
  }
  const int L = slice_of(cs);
  if ((L + cpc - 1) / cpc > specv::kMaxChunksPerSlice) return SPEC_ERR_ARG;
  *cs_out = cs;
  *slice_out = L;
  return SPEC_OK;
}

// Falls back to smaller clusters when the device cannot co-schedule the planned one.
int schedulable_plan(int V, int dtype, Plan* plan) {
  for (int tries = 0; tries < 5; ++tries) {
    int n = 0;
    if (specv::stats_max_active_clusters(dtype, plan->cs, &n) != cudaSuccess) {
      cudaGetLastError();
      return SPEC_ERR_CUDA;
    }
    if (n > 0) {
      plan->nclus = n;
      return SPEC_OK;
    }
    if (plan->cs == 1) return SPEC_ERR_ARG;
    *plan = plan_for(V, plan->cs / 2, dtype);
  }
  return SPEC_ERR_ARG;
}

// Plans already resolved on a device (the occupancy query costs tens of microseconds).
struct PlanEntry {
  int dev, V, dtype, env_cs;
  Plan plan;
};
std::mutex g_plan_mu;
std::vector<PlanEntry> g_plans;

int env_cluster() {
  const char* env = std::getenv("SPECVERIFY_CLUSTER");
  return env ? std::atoi(env) : 0;
}

int resolve_plan(int V, int dtype, Plan* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  const int env_cs = env_cluster();
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    for (const PlanEntry& e : g_plans) {
      if (e.dev == dev && e.V == V && e.dtype == dtype && e.env_cs == env_cs) {
        *out = e.plan;
        return SPEC_OK;
      }
    }
  }
  Plan plan;
  if (!choose_plan(V, dtype, &plan)) return SPEC_ERR_ARG;
  int st = prepare(dtype);
  if (st != SPEC_OK) return st;
  if ((st = schedulable_plan(V, dtype, &plan)) != SPEC_OK) return st;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  if (g_plans.size() < 4096) g_plans.push_back(PlanEntry{dev, V, dtype, env_cs, plan});
  *out = plan;
  return SPEC_OK;
}

// Streaming multiprocessors of the current device (cached per device), 0 if the query fails.
int device_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 0;
  }
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Vocabulary elements per draw CTA.  A draw CTA re-reads its slice of one row only if that row
// draws there, so wide slices cost little traffic; they are halved (32768 -> 16384) when the batch
// would otherwise give fewer than three draw CTAs per SM, and halved further, down to kMinSlice, while
// it gives fewer than two (small, latency-bound batches).  At least V/32 (at most 32 draw CTAs per
// row), a multiple of the draw chunk; SPECVERIFY_DSLICE (elements) overrides within the limits.
int draw_slice(int B, int V, int dtype) {
  const int chunk = 4 * 32 * (dtype == SPEC_F32 ? 4 : 8);
  const long long wide = 32768;
  const long long ctas = static_cast<long long>(B) * ((V + wide - 1) / wide);
  int slice = ctas >= 3LL * device_sms() ? 32768 : 16384;
  const long long want = 2LL * (device_sms() > 0 ? device_sms() : 152);
  while (slice / 2 >= kMinSlice && static_cast<long long>(B) * ((V + slice - 1) / slice) < want) slice /= 2;
  if (const char* env = std::getenv("SPECVERIFY_DSLICE")) {
    const int want = std::atoi(env);
    if (want > 0) slice = want;
  }
  const int lo = (V + specv::kMaxSlices - 1) / specv::kMaxSlices;
  if (slice < lo) slice = lo;
  slice = static_cast<int>(align_up(slice, chunk));
  if (slice > specv::kMaxChunksPerSlice * chunk) slice = specv::kMaxChunksPerSlice * chunk;
  return slice;
}

// Target elements per greedy CTA: kGreedySlice, halved (down to 2048) while the batch would give fewer
// than two CTAs per SM, as for the sampling slices.
int greedy_slice(int B, int gamma, int V) {
  int slice = specv::kGreedySlice;
  const long long want = 2LL * (device_sms() > 0 ? device_sms() : 152);
  const long long positions = static_cast<long long>(B) * (gamma + 1);
  while (slice / 2 >= 2048 && positions * ((V + slice - 1) / slice) < want) slice /= 2;
  return slice;
}

bool rows_aligned(const void* p, int V, int esz) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((static_cast<size_t>(V) * esz) % 16 == 0);
}

int check_sizes(int dtype, int B, int gamma, int V) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (B < 0 || gamma < 0 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_VOCAB) return SPEC_ERR_ARG;
  // grid size: B * (gamma+1) * max(cluster size, greedy CTAs per row) CTAs
  const long long per_row = SPEC_MAX_VOCAB / specv::kGreedySlice;
  if ((long long)B * (gamma + 1) * per_row > 0x7fffffffLL) return SPEC_ERR_ARG;
  return SPEC_OK;
}

}  // namespace

namespace specv {

// Host-side checks of the sampling entry points' arguments other than the workspace: sizes, dtype,
// temperature and the pointers a call with B > 0 dereferences.
int check_sample_args(const void* target, const void* draft, int dtype, const int32_t* ids, const float* uniforms,
                      float temperature, int B, int gamma, int V, const int32_t* emitted, const int32_t* n_accepted) {
  const int st = check_sizes(dtype, B, gamma, V);
  if (st != SPEC_OK) return st;
  if (!(std::isfinite(temperature) && temperature > 0.f)) return SPEC_ERR_ARG;
  if (B == 0) return SPEC_OK;
  if (target == nullptr || uniforms == nullptr || emitted == nullptr || n_accepted == nullptr) return SPEC_ERR_ARG;
  if (gamma > 0 && (draft == nullptr || ids == nullptr)) return SPEC_ERR_ARG;
  return SPEC_OK;
}

}  // namespace specv

namespace {

int check_common(int dtype, int B, int gamma, int V, const void* workspace, size_t ws_bytes) {
  const int st = check_sizes(dtype, B, gamma, V);
  if (st != SPEC_OK || B == 0) return st;
  if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SPEC_ERR_WORKSPACE;
  if (ws_bytes < specv::ws_bytes_for(B, gamma, V)) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return SPEC_OK;
  cudaGetLastError();
  return SPEC_ERR_CUDA;
}

// phases (sampling only): 1 = stream kernel, 2 = draw kernel, 3 = both.
int run_verify(const void* target, const void* draft, int dtype, const int32_t* ids, const int32_t* draft_len,
               const float* uniforms, float temperature, int B, int gamma, int V, int32_t* emitted,
               int32_t* n_accepted, float* beta, float* p_draft, float* q_draft, float* accept_prob,
               float* resid, void* workspace, size_t ws_bytes, void* stream, bool stats, int phases = 3,
               bool early_exit = false, const float* tthr = nullptr, const float* dthr = nullptr,
               float lenience = 1.f) {
  int st = check_common(dtype, B, gamma, V, workspace, ws_bytes);
  if (st != SPEC_OK) return st;
  if (!(std::isfinite(temperature) && temperature > 0.f)) return SPEC_ERR_ARG;
  if (!(lenience > 0.f && lenience <= 1.f)) return SPEC_ERR_ARG;
  if (B == 0 || (stats && gamma == 0)) return SPEC_OK;
  if (target == nullptr) return SPEC_ERR_ARG;
  if (gamma > 0 && (draft == nullptr || ids == nullptr)) return SPEC_ERR_ARG;
  if (!stats && (uniforms == nullptr || emitted == nullptr || n_accepted == nullptr)) return SPEC_ERR_ARG;
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const bool vec = rows_aligned(target, V, esz) && (gamma == 0 || rows_aligned(draft, V, esz));

  if (!stats) {
    specv::SampleParams p = {};
    p.target = target;
    p.draft = draft;
    p.ids = ids;
    p.draft_len = draft_len;
    p.uniforms = uniforms;
    p.tthr = tthr;
    p.dthr = gamma > 0 ? dthr : nullptr;
    p.scale = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    p.lq = lenience;
    p.B = B;
    p.G = gamma;
    p.V = V;
    p.slice = sample_slice(V, dtype, static_cast<long long>(B) * (gamma + 1));
    p.nslices = (V + p.slice - 1) / p.slice;
    p.dslice = draw_slice(B, V, dtype);
    p.ndslices = (V + p.dslice - 1) / p.dslice;
    p.sms = device_sms();
    // the resolving CTA gathers the chunk masses of a whole drawn row in shared memory
    if (p.ndslices * (p.dslice / (4 * 32 * (dtype == SPEC_F32 ? 4 : 8))) > specv::kMaxRowChunks) return SPEC_ERR_ARG;
    p.vec = vec ? 1 : 0;
    p.emitted = emitted;
    p.n_acc = n_accepted;
    p.ws = specv::ws_carve(workspace, B, gamma, V);
    // the early exit's one-launch plan; without one (a cluster the device cannot schedule) the early exit
    // takes the two-kernel path
    if (early_exit && rows_plan(B, gamma, V, dtype, &p.rcs, &p.rslice) != SPEC_OK) p.rcs = 0;
    if (early_exit) return launch_status(specv::sample_early_exit_launch(p, dtype, static_cast<cudaStream_t>(stream)));
    return launch_status(specv::sample_launch(p, dtype, phases, static_cast<cudaStream_t>(stream)));
  }

  Plan plan;
  if ((st = resolve_plan(V, dtype, &plan)) != SPEC_OK) return st;

  specv::VerifyParams p = {};
  p.target = target;
  p.draft = draft;
  p.ids = ids;
  p.draft_len = draft_len;
  p.scale = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  p.B = B;
  p.G = gamma;
  p.V = V;
  p.L = plan.L;
  p.vec = vec ? 1 : 0;
  p.beta = beta;
  p.p_draft = p_draft;
  p.q_draft = q_draft;
  p.accept_prob = accept_prob;
  p.resid = resid;
  p.ws = specv::ws_carve(workspace, B, gamma, V);
  return launch_status(specv::stats_launch(p, dtype, plan.cs, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

size_t spec_workspace_size(int B, int gamma, int V, int dtype) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return 0;
  if (B < 0 || gamma < 0 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_VOCAB) return 0;
  return specv::ws_bytes_for(B, gamma, V);
}

int spec_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (workspace == nullptr) return SPEC_ERR_WORKSPACE;
  return launch_status(cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

int spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_ids,
                       const int32_t* draft_len, const float* uniforms, float temperature, int B, int gamma, int V,
                       int32_t* emitted, int32_t* n_accepted, void* workspace, size_t ws_bytes, void* stream) {
  return run_verify(target_logits, draft_logits, dtype, draft_ids, draft_len, uniforms, temperature, B, gamma, V,
                    emitted, n_accepted, nullptr, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes, stream,
                    false);
}

int spec_verify_sample_stream(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                              float temperature, int B, int gamma, int V, int32_t* emitted, int32_t* n_accepted,
                              void* workspace, size_t ws_bytes, void* stream) {
  return run_verify(target_logits, draft_logits, dtype, draft_ids, draft_len, uniforms, temperature, B, gamma, V,
                    emitted, n_accepted, nullptr, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes, stream,
                    false, 1);
}

int spec_verify_sample_draw(const void* target_logits, const void* draft_logits, int dtype,
                            const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                            float temperature, int B, int gamma, int V, int32_t* emitted, int32_t* n_accepted,
                            void* workspace, size_t ws_bytes, void* stream) {
  return run_verify(target_logits, draft_logits, dtype, draft_ids, draft_len, uniforms, temperature, B, gamma, V,
                    emitted, n_accepted, nullptr, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes, stream,
                    false, 2);
}

int spec_accept_stats(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_ids,
                      const int32_t* draft_len, float temperature, int B, int gamma, int V, float* beta,
                      float* p_draft, float* q_draft, float* accept_prob, float* resid_mass, void* workspace,
                      size_t ws_bytes, void* stream) {
  return run_verify(target_logits, draft_logits, dtype, draft_ids, draft_len, nullptr, temperature, B, gamma, V,
                    nullptr, nullptr, beta, p_draft, q_draft, accept_prob, resid_mass, workspace, ws_bytes, stream,
                    true);
}

int spec_verify_sample_early_exit(const void* target_logits, const void* draft_logits, int dtype,
                                  const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                                  float temperature, int B, int gamma, int V, int32_t* emitted,
                                  int32_t* n_accepted, void* workspace, size_t ws_bytes, void* stream) {
  return run_verify(target_logits, draft_logits, dtype, draft_ids, draft_len, uniforms, temperature, B, gamma, V,
                    emitted, n_accepted, nullptr, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes, stream,
                    false, 3, true);
}

int spec_verify_sample_masked(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                              const float* target_thr, const float* draft_thr, float temperature, int B, int gamma,
                              int V, int32_t* emitted, int32_t* n_accepted, void* workspace, size_t ws_bytes,
                              void* stream) {
  return run_verify(target_logits, draft_logits, dtype, draft_ids, draft_len, uniforms, temperature, B, gamma, V,
                    emitted, n_accepted, nullptr, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes, stream,
                    false, 3, false, target_thr, draft_thr);
}

int spec_verify_sample_lenient(const void* target_logits, const void* draft_logits, int dtype,
                               const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                               float temperature, float lenience, int B, int gamma, int V, int32_t* emitted,
                               int32_t* n_accepted, void* workspace, size_t ws_bytes, void* stream) {
  return run_verify(target_logits, draft_logits, dtype, draft_ids, draft_len, uniforms, temperature, B, gamma, V,
                    emitted, n_accepted, nullptr, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes, stream,
                    false, 3, false, nullptr, nullptr, lenience);
}

int spec_topk_threshold(const void* logits, int dtype, int R, int V, int k, float* thr, void* stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (R < 0 || V < 1 || V > SPEC_MAX_VOCAB || k < 1) return SPEC_ERR_ARG;
  if (R == 0) return SPEC_OK;
  if (logits == nullptr || thr == nullptr) return SPEC_ERR_ARG;
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  return launch_status(specv::topk_threshold_launch(logits, dtype, R, V, k, rows_aligned(logits, V, esz) ? 1 : 0,
                                                    thr, static_cast<cudaStream_t>(stream)));
}

int spec_topp_threshold(const void* logits, int dtype, float temperature, float top_p, int R, int V, float* thr,
                        void* stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (R < 0 || V < 1 || V > SPEC_MAX_VOCAB) return SPEC_ERR_ARG;
  if (!(std::isfinite(temperature) && temperature > 0.f) || !(top_p > 0.f && top_p <= 1.f)) return SPEC_ERR_ARG;
  if (R == 0) return SPEC_OK;
  if (logits == nullptr || thr == nullptr) return SPEC_ERR_ARG;
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const float scale = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  return launch_status(specv::topp_threshold_launch(logits, dtype, R, V, scale, top_p,
                                                    rows_aligned(logits, V, esz) ? 1 : 0, thr,
                                                    static_cast<cudaStream_t>(stream)));
}

int spec_sample_rows_masked(const void* logits, int dtype, const float* uniforms, const float* thr,
                            float temperature, int R, int V, int32_t* tokens, void* workspace, size_t ws_bytes,
                            void* stream);

int spec_sample_rows(const void* logits, int dtype, const float* uniforms, float temperature, int R, int V,
                     int32_t* tokens, void* workspace, size_t ws_bytes, void* stream) {
  return spec_sample_rows_masked(logits, dtype, uniforms, nullptr, temperature, R, V, tokens, workspace, ws_bytes,
                                 stream);
}

int spec_sample_rows_masked(const void* logits, int dtype, const float* uniforms, const float* thr,
                            float temperature, int R, int V, int32_t* tokens, void* workspace, size_t ws_bytes,
                            void* stream) {
  int st = check_common(dtype, R, 0, V, workspace, ws_bytes);
  if (st != SPEC_OK) return st;
  if (!(std::isfinite(temperature) && temperature > 0.f)) return SPEC_ERR_ARG;
  if (R == 0) return SPEC_OK;
  if (logits == nullptr || uniforms == nullptr || tokens == nullptr) return SPEC_ERR_ARG;
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  specv::SampleParams p = {};
  p.target = logits;
  p.uniforms = uniforms;
  p.tthr = thr;
  p.scale = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  p.B = R;
  p.G = 0;
  p.V = V;
  p.slice = sample_slice(V, dtype);
  p.nslices = (V + p.slice - 1) / p.slice;
  p.dslice = p.slice;
  p.ndslices = p.nslices;
  p.vec = rows_aligned(logits, V, esz) ? 1 : 0;
  p.emitted = tokens;
  p.n_acc = nullptr;
  p.ws = specv::ws_carve(workspace, R, 0, V);
  return launch_status(specv::rows_sample_launch(p, dtype, static_cast<cudaStream_t>(stream)));
}

int spec_verify_greedy(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_ids,
                       const int32_t* draft_len, int B, int gamma, int V, int32_t* emitted, int32_t* n_accepted,
                       void* workspace, size_t ws_bytes, void* stream) {
  (void)draft_logits;
  int st = check_common(dtype, B, gamma, V, workspace, ws_bytes);
  if (st != SPEC_OK) return st;
  if (B == 0) return SPEC_OK;
  if (target_logits == nullptr || emitted == nullptr || n_accepted == nullptr) return SPEC_ERR_ARG;
  if (gamma > 0 && draft_ids == nullptr) return SPEC_ERR_ARG;
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  specv::GreedyParams p = {};
  p.target = target_logits;
  p.ids = draft_ids;
  p.draft_len = draft_len;
  p.B = B;
  p.G = gamma;
  p.V = V;
  p.slice = greedy_slice(B, gamma, V);
  p.nslices = (V + p.slice - 1) / p.slice;
  p.vec = rows_aligned(target_logits, V, esz) ? 1 : 0;
  p.emitted = emitted;
  p.n_acc = n_accepted;
  p.ws = specv::ws_carve(workspace, B, gamma, V);
  return launch_status(specv::greedy_launch(p, dtype, static_cast<cudaStream_t>(stream)));
}

int spec_check_status(void* workspace, void* stream) {
  if (workspace == nullptr) return SPEC_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  if (word == 0) return SPEC_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  for (int code = 1; code < 32; ++code)
    if (word & (1u << code)) return code;
  return SPEC_ERR_CUDA;
}

int spec_verify_plan(int B, int gamma, int V, int dtype, int* cluster_size, int* slice_len, int* smem_bytes,
                     int* greedy_ctas_per_row) {
  int st = check_sizes(dtype, B, gamma, V);
  if (st != SPEC_OK) return st;
  Plan plan;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    if ((st = resolve_plan(V, dtype, &plan)) != SPEC_OK) return st;
  } else {
    cudaGetLastError();  // no device: report the plan before the co-scheduling check
    if (!choose_plan(V, dtype, &plan)) return SPEC_ERR_ARG;
  }
  if (cluster_size) *cluster_size = plan.cs;
  if (slice_len) *slice_len = plan.L;
  if (smem_bytes) *smem_bytes = plan.smem;
  if (greedy_ctas_per_row) {
    const int gs = greedy_slice(B, gamma, V);
    *greedy_ctas_per_row = (V + gs - 1) / gs;
  }
  return SPEC_OK;
}

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_ARG: return "invalid argument";
    case SPEC_ERR_DTYPE: return "unknown dtype";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_NONFINITE: return "non-finite or all -inf logit row";
    case SPEC_ERR_TOKEN_RANGE: return "draft id outside [0, V)";
    case SPEC_ERR_TIMEOUT: return "timeout";
    case SPEC_ERR_WORKSPACE: return "workspace too small or misaligned";
    case SPEC_ERR_BOUNDS: return "index check failed";
    default: return "unknown status";
  }
}

}  // extern "C"
