/*
 * spec_verify.h -- C ABI of the batched verification step of speculative
 * sampling, for one NVIDIA GB300 (sm_103a).
 *
 * The method is Algorithm 1 of Leviathan, Kalman & Matias, "Fast Inference
 * from Transformers via Speculative Decoding" (arXiv 2211.17192), as restated
 * in the paper-graph-ui teardown of that paper (§2.2 "Standardized Sampling",
 * §2.3 "Algorithm Walkthrough", Phases 3-4), the multigrid.ai explainer
 * "Speculative Decoding: Two Models, One Output" ("The algorithm"), the
 * fullstackaihub "Speculative Decoding Paper Breakdown" (§3 "The Algorithm at
 * Position i") and the interactiveml post on the correction distribution.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument except `workspace` of spec_workspace_size is a
 *    DEVICE pointer (cudaMalloc / torch CUDA memory) of the current device.
 *    The caller owns all buffers; the library allocates nothing and keeps no
 *    state between calls except what it leaves in the caller's workspace.
 *  - All arrays are dense row-major.  Logits are IEEE float32 (SPEC_F32) or
 *    bfloat16 (SPEC_BF16); the target holds gamma+1 rows of V per batch row b,
 *    the draft gamma rows of V.  gamma is the padded draft width.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on it.  The return value covers host-side
 *    argument checks and launch errors only.  What the device finds
 *    (non-finite logit rows, draft ids outside [0, V), uniforms outside
 *    [0, 1), draft_len outside [0, gamma]) marks the affected batch row
 *    invalid -- n_accepted[b] = -1 and emitted[b, :] = -1 -- and is recorded in
 *    the workspace's error word, read by spec_check_status.
 *  - The first kernel of a sampling call is launched as a programmatic
 *    dependent of the launch before it on `stream` (CUDA programmatic dependent
 *    launch): its thread blocks may become resident while that kernel drains,
 *    but they read no input and write no output or workspace slot before it
 *    has finished and its writes are visible, so stream order holds as for a
 *    plain launch.  The last kernel of a call allows the next launch on the
 *    stream to be scheduled early; a caller's kernel launched that way must
 *    itself wait (griddepcontrol.wait / cudaGridDependencySynchronize) before
 *    it reads this call's outputs, as programmatic launches require.
 *  - Tuning overrides read from the environment at every call (for
 *    measurements; results are the same up to float32 rounding order within
 *    the documented tolerances): SPECVERIFY_SLICE / SPECVERIFY_DSLICE (stream /
 *    draw slice, elements), SPECVERIFY_ROW_CLUSTER (CTAs per batch row of the
 *    early exit's one-launch kernel), SPECVERIFY_EARLY_FORM (see the early exit),
 *    SPECVERIFY_CLUSTER / SPECVERIFY_STATS_SLICE (statistics cluster size /
 *    slice), SPECVERIFY_DRAW_CLUSTER (0 / 1: a row's draw CTAs as a
 *    thread-block cluster), SPECVERIFY_PDL=0 (plain launch of a call's first
 *    kernel), SPECVERIFY_NUCLEUS_PATH=bounds / exact / weighted (how the
 *    nucleus threshold of a row over 128 KB is selected; the same threshold
 *    either way).
 *  - A row is invalid if any logit row it reads holds a NaN or +inf or is
 *    entirely -inf.  Ragged rows (draft_len[b] = gamma_b < gamma) never read
 *    target rows i > gamma_b, draft rows i >= gamma_b, ids i >= gamma_b, or
 *    uniforms gamma_b <= i < gamma.
 *  - Limits: B >= 0 (B = 0 is a no-op), 0 <= gamma <= SPEC_MAX_GAMMA,
 *    1 <= V <= SPEC_MAX_VOCAB.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_MAX_GAMMA 64
#define SPEC_MAX_VOCAB 262144

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_ARG = 1,          /* bad size, null pointer, temperature, draft_len or uniform */
  SPEC_ERR_DTYPE = 2,        /* unknown dtype */
  SPEC_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  SPEC_ERR_NONFINITE = 4,    /* a logit row read holds NaN / +inf or is all -inf */
  SPEC_ERR_TOKEN_RANGE = 5,  /* a draft id read lies outside [0, V) */
  SPEC_ERR_TIMEOUT = 6,      /* a bounded wait of the early exit's one-launch kernel ran out */
  SPEC_ERR_WORKSPACE = 7,    /* workspace too small or not 256-byte aligned */
  SPEC_ERR_BOUNDS = 8        /* an index check failed: only libspecverify_debug.so (built with
                                -DSPEC_DEBUG_BOUNDS) checks kernel indices and reports this */
} spec_status_t;

/* Bytes of device workspace the entry points need for (B, gamma, V): an error
 * word, per-row arrival counters, greedy argmax keys, per-slice softmax
 * normalisers, the logits at the draft tokens, and the chunk masses of the
 * drawn rows.  The workspace must be zero-filled once before its first
 * use (cudaMemset or spec_workspace_init); every call leaves the slots it used
 * at zero again, so one workspace serves any sequence of calls of any shape on
 * one stream.  Calls that overlap on the GPU must use different workspaces.
 * Returns 0 for invalid sizes.  No CUDA call is made. */
size_t spec_workspace_size(int B, int gamma, int V, int dtype);

/* Zero-fills `ws_bytes` of workspace on `stream` (cudaMemsetAsync). */
int spec_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* Speculative sampling verification, Algorithm 1 Phases 3-4 (paper-graph-ui
 * teardown §2.3; multigrid.ai "The algorithm"; fullstackaihub §3).
 *
 * For each batch row b with gamma_b = draft_len[b] (or gamma if draft_len is
 * NULL):  p_i = softmax(target[b,i,:] / T) for i <= gamma_b and q_i =
 * softmax(draft[b,i,:] / T) for i < gamma_b (temperature standardisation,
 * §2.2).  Guess x_i = draft_ids[b,i] is accepted iff p_i(x_i) > 0 and
 * uniforms[b,i] <= min(1, p_i(x_i)/q_i(x_i)); the walk stops at the first
 * rejection, n = n_accepted[b].  If n < gamma_b the emitted token is drawn from
 * norm(max(0, p_n - q_n)) (from p_n if that residual mass is <= 1e-15, the
 * interactiveml correction rule), else from p_{gamma_b} (bonus token).  The
 * draw is an inverse CDF driven by uniforms[b, gamma]: the smallest token k
 * whose running weight sum exceeds uniforms[b,gamma] * (total weight).
 *
 *   target_logits  [B, gamma+1, V]  dtype
 *   draft_logits   [B, gamma, V]    dtype (may be NULL when gamma == 0)
 *   draft_ids      [B, gamma]       int32 (may be NULL when gamma == 0)
 *   draft_len      [B]              int32 in [0, gamma], or NULL for all gamma
 *   uniforms       [B, gamma+1]     float32 in [0, 1)
 *   temperature    > 0, finite
 *   emitted        [B, gamma+1]     int32 out: x_0..x_{n-1}, the drawn token, then -1
 *   n_accepted     [B]              int32 out: n in [0, gamma_b], or -1 for an invalid row
 *   workspace      >= spec_workspace_size(B, gamma, V, dtype) bytes, 256-byte aligned
 */
int spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                       float temperature, int B, int gamma, int V,
                       int32_t* emitted, int32_t* n_accepted,
                       void* workspace, size_t ws_bytes, void* stream);

/* The two phases of spec_verify_sample, for callers that want to schedule them
 * separately (for instance, the draw phase next to other work on the GPU).
 * spec_verify_sample_stream reads every logit once and leaves per-slice
 * softmax normalisers and the logits at the draft tokens in the workspace;
 * spec_verify_sample_draw takes the accept decisions, draws, writes emitted
 * and n_accepted, and returns the workspace to its zero state.  Call them in
 * this order, on the same stream, with identical arguments and workspace, and
 * nothing else using that workspace in between; together they are exactly
 * spec_verify_sample.  Arguments, layouts and errors as spec_verify_sample. */
int spec_verify_sample_stream(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                              float temperature, int B, int gamma, int V,
                              int32_t* emitted, int32_t* n_accepted,
                              void* workspace, size_t ws_bytes, void* stream);
int spec_verify_sample_draw(const void* target_logits, const void* draft_logits, int dtype,
                            const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                            float temperature, int B, int gamma, int V,
                            int32_t* emitted, int32_t* n_accepted,
                            void* workspace, size_t ws_bytes, void* stream);

/* Byte-lean early exit: spec_verify_sample that takes position i + 1 of a batch
 * row into account only while the row has not stopped -- at its first
 * rejection, at an invalid position, or at the bonus position gamma_b.  A
 * logit row after the first rejection does not count, so a NaN / +inf or all
 * -inf row there does not make the batch row invalid as it does in
 * spec_verify_sample; ids and uniforms of every position are still checked.
 * Two forms, chosen per call by the batch's size:
 *  - one launch of a kernel with a thread-block cluster per batch row, which
 *    decides each position before streaming the next, so a row reads the n + 1
 *    target and n + 1 draft rows up to its first rejection n (n + 1 and n for a
 *    bonus draw) instead of 2 gamma_b + 1: about sum_k alpha^k rows when each
 *    guess is accepted with probability alpha (§3.1).  Taken when one position
 *    of the batch (2 B V logits) is at least 64 MB; it splits the vocabulary its
 *    own way, so its float32 sums round differently from spec_verify_sample's
 *    and a draw within about 1e-6 of a CDF edge may pick the neighbouring token;
 *  - otherwise spec_verify_sample's two kernels, with the decisions taken as
 *    above: exactly spec_verify_sample's outputs for valid inputs (smaller
 *    batches gain nothing from skipping rows: their per-position latency
 *    outweighs the bytes).
 * SPECVERIFY_EARLY_FORM=1 / 2 forces the one-launch / two-kernel form.  A
 * cluster slot that does not fill within about 0.1 s (which valid launches
 * never see) marks the row invalid with SPEC_ERR_TIMEOUT.  Arguments,
 * layouts, workspace and the other errors as spec_verify_sample. */
int spec_verify_sample_early_exit(const void* target_logits, const void* draft_logits, int dtype,
                                  const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                                  float temperature, int B, int gamma, int V,
                                  int32_t* emitted, int32_t* n_accepted,
                                  void* workspace, size_t ws_bytes, void* stream);

/* spec_verify_sample without a workspace argument, for callers that cannot
 * allocate device memory: for instance a plugin handed only its input and
 * output buffers by a host program that owns every allocator, or a serving loop
 * that must not call cudaMalloc once it is running (cudaMalloc can block on the
 * whole device and can fail under memory pressure).  The paper has no
 * counterpart to this entry point; it only changes where the scratch lives.
 *
 * The scratch is one fixed array of SPEC_NOALLOC_SCRATCH_BYTES inside this
 * library, held by every GPU that loads the library until the process exits.
 * Calls whose spec_workspace_size(B, gamma, V, dtype) exceeds it return
 * SPEC_ERR_WORKSPACE without touching the GPU (use spec_verify_sample with a
 * workspace of your own then); so does every other argument error
 * spec_verify_sample reports on the host (SPEC_ERR_ARG, SPEC_ERR_DTYPE): the
 * array is left as it was.  The first call on a device looks up the array's
 * device address on that device (cudaGetSymbolAddress) and keeps it; make that
 * first call before any stream capture, and do not call this entry point on a
 * device after cudaDeviceReset of that device in the same process (the kept
 * address would be stale).  Every call uses the same array, so calls that
 * overlap on the GPU (other streams, other threads) race and corrupt each
 * other's results: serialise them.  Each call clears the counters it needs at
 * zero on `stream` before its kernels (cudaMemsetAsync; nothing is allocated).
 * The input checks the device makes (non-finite or all -inf logit rows, draft
 * ids outside [0, V), uniforms outside [0, 1), draft_len outside [0, gamma])
 * show as n_accepted[b] = -1 and emitted[b, :] = -1 only, since the caller has
 * no workspace to read an error word from.  Arguments, layouts and results
 * otherwise as spec_verify_sample. */
#define SPEC_NOALLOC_SCRATCH_BYTES (16u << 20)
int spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits, int dtype,
                               const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                               float temperature, int B, int gamma, int V,
                               int32_t* emitted, int32_t* n_accepted, void* stream);

/* Draft-side sampler: the step before verification, Algorithm 1 Phase 1
 * (paper-graph-ui teardown §2.3 "Algorithm Walkthrough": each guess is drawn
 * from the approximation model's distribution, x ~ q).  For each row r of
 * `logits`, q = softmax(logits[r, :] / T) (temperature standardisation, §2.2)
 * and tokens[r] is the inverse-CDF draw driven by uniforms[r]: the smallest
 * token k whose running weight sum exceeds uniforms[r] * (total weight), the
 * same draw spec_verify_sample makes for its bonus token.
 *
 *   logits       [R, V]  dtype (the draft model's logits at one position, one row per sequence)
 *   uniforms     [R]     float32 in [0, 1)
 *   temperature  > 0, finite
 *   tokens       [R]     int32 out: the drawn token, or -1 for an invalid row
 *   workspace    >= spec_workspace_size(R, 0, V, dtype) bytes, 256-byte aligned, zero at rest
 *
 * Two kernel launches: the streaming pass of spec_verify_sample over the rows,
 * then one CTA per row that re-reads only the vocabulary slice holding the
 * draw.  A row holding NaN / +inf or only -inf, or whose uniform lies outside
 * [0, 1), gets -1 and is recorded in the workspace's error word. */
int spec_sample_rows(const void* logits, int dtype, const float* uniforms, float temperature,
                     int R, int V, int32_t* tokens,
                     void* workspace, size_t ws_bytes, void* stream);

/* Lenient verification (paper-graph-ui teardown §5 on Appendix A.5 "lenience"):
 * q is multiplied by the lenience l in (0, 1] before it is compared with p, so
 * guess x_i is accepted iff p_i(x_i) > 0 and u_i <= min(1, p_i(x_i) / (l q_i(x_i))),
 * and a rejection draws from norm(max(0, p_n - l q_n)).  The pages state the
 * scaled comparison and its guarantee -- no token is drawn with probability
 * above p(x)/l -- but not the residual; scaling q there too is the plainest
 * reading and keeps the guarantee.  l = 1 is spec_verify_sample exactly.  Other
 * arguments as spec_verify_sample; lenience outside (0, 1] returns SPEC_ERR_ARG. */
int spec_verify_sample_lenient(const void* target_logits, const void* draft_logits, int dtype,
                               const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                               float temperature, float lenience, int B, int gamma, int V,
                               int32_t* emitted, int32_t* n_accepted,
                               void* workspace, size_t ws_bytes, void* stream);

/* Top-k and nucleus (top-p) standardisation (paper-graph-ui teardown §2.2
 * "Standardized Sampling": keep the k largest probabilities, or the shortest
 * descending prefix whose mass reaches top_p, and renormalise).  Softmax is
 * increasing in the logit, so the kept set of a row is {x : l(x) >= tau}; these
 * write tau per row and the *_masked entry points below apply it.
 *   spec_topk_threshold: tau = the k-th largest logit of the row (k >= 1); ties
 *     at tau are all kept; tau = -inf when fewer than k logits are finite.
 *   spec_topp_threshold: tau = the logit of the token at which the descending
 *     running probability of softmax(l / T) first reaches top_p (0 < top_p <= 1;
 *     ties at tau kept; -inf for top_p = 1).  Masses are summed in 2^-40 fixed
 *     point, so a running mass within about 1e-6 of top_p may stop one token
 *     earlier or later than an exact sum would.
 *   logits [R, V] dtype (device), thr [R] float32 (device, out).  A row holding
 *   NaN or +inf (or, for top-p, no finite logit) gets tau = NaN, which the masked
 *   entry points treat as an invalid row.  One kernel launch, no workspace.
 *   Returns SPEC_ERR_ARG / SPEC_ERR_DTYPE for bad host arguments. */
int spec_topk_threshold(const void* logits, int dtype, int R, int V, int k, float* thr, void* stream);
int spec_topp_threshold(const void* logits, int dtype, float temperature, float top_p, int R, int V, float* thr,
                        void* stream);

/* spec_verify_sample on standardised distributions: p_i and q_i are the
 * softmaxes of the logit rows with every logit below the row's threshold set to
 * -inf (renormalised over the kept tokens), for the accept tests, the residual
 * and the bonus draw alike.  target_thr [B, gamma+1] and draft_thr [B, gamma]
 * are float32 device arrays (either may be NULL: no truncation on that side;
 * -inf in an entry: none for that row).  Other arguments as spec_verify_sample. */
int spec_verify_sample_masked(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_ids, const int32_t* draft_len, const float* uniforms,
                              const float* target_thr, const float* draft_thr, float temperature,
                              int B, int gamma, int V, int32_t* emitted, int32_t* n_accepted,
                              void* workspace, size_t ws_bytes, void* stream);

/* spec_sample_rows on standardised distributions: thr [R] float32 (device, may be
 * NULL) as above. */
int spec_sample_rows_masked(const void* logits, int dtype, const float* uniforms, const float* thr,
                            float temperature, int R, int V, int32_t* tokens,
                            void* workspace, size_t ws_bytes, void* stream);

/* Greedy verification: argmax standardisation (paper-graph-ui teardown §2.2;
 * multigrid.ai on sampling temperature).  a_i = argmax_k target[b,i,k], lowest
 * index on ties; guesses are accepted while a_i == draft_ids[b,i]; the emitted
 * token at n is a_n (n < gamma_b) or a_{gamma_b}.  Reads the target logits
 * only; draft_logits is accepted for symmetry and never read (may be NULL).
 * Outputs and errors as spec_verify_sample. */
int spec_verify_greedy(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_ids, const int32_t* draft_len,
                       int B, int gamma, int V,
                       int32_t* emitted, int32_t* n_accepted,
                       void* workspace, size_t ws_bytes, void* stream);

/* Per-position acceptance statistics (paper-graph-ui teardown Definition 3.2,
 * Lemma 3.3, Theorem 3.5): for i < gamma_b,
 *   beta[b,i]        = sum_x min(p_i(x), q_i(x))     (acceptance rate, 1 - DLK)
 *   p_draft[b,i]     = p_i(x_i),  q_draft[b,i] = q_i(x_i)
 *   accept_prob[b,i] = min(1, p_i(x_i)/q_i(x_i)), 0 if p_i(x_i) = 0
 *   resid_mass[b,i]  = sum_x max(0, p_i(x) - q_i(x))  (residual normaliser)
 * Each output is [B, gamma] float32 and may be NULL.  Positions i >= gamma_b
 * and invalid positions get NaN. */
int spec_accept_stats(const void* target_logits, const void* draft_logits, int dtype,
                      const int32_t* draft_ids, const int32_t* draft_len, float temperature,
                      int B, int gamma, int V,
                      float* beta, float* p_draft, float* q_draft, float* accept_prob,
                      float* resid_mass,
                      void* workspace, size_t ws_bytes, void* stream);

/* Planning helpers (paper-graph-ui teardown §3.1-§3.5).  Host functions, no CUDA call.
 *   spec_expected_tokens:      E[# tokens per step] = (1 - alpha^(gamma+1)) / (1 - alpha)   (Eq. 1;
 *                              gamma + 1 at alpha = 1).  NaN for alpha outside [0, 1] or gamma < 0.
 *   spec_walltime_improvement: Theorem 3.8, E[# tokens] / (gamma c + 1), c = cost of M_q / cost of M_p.
 *   spec_operations_factor:    Theorem 3.11, (gamma c_hat + gamma + 1) / E[# tokens].
 *   spec_optimal_gamma:        gamma* = argmax over gamma in [1, max_gamma] of Theorem 3.8 (§3.5: every
 *                              gamma is evaluated; ties go to the smaller gamma); writes the improvement at
 *                              gamma* to *improvement if not NULL.  -1 for invalid arguments. */
double spec_expected_tokens(double alpha, int gamma);
double spec_walltime_improvement(double alpha, int gamma, double c);
double spec_operations_factor(double alpha, int gamma, double c_hat);
int spec_optimal_gamma(double alpha, double c, int max_gamma, double* improvement);

/* Corpus acceptance rate alpha = E[beta] (Corollary 3.6): the mean of the finite entries of the device
 * array beta[0, n) (for instance the beta output of spec_accept_stats, where NaN marks positions that
 * were not verified), accumulated in double in a fixed order.  out is a device pointer to two doubles:
 * out[0] = alpha (NaN if there is no finite entry), out[1] = the number of finite entries.  One kernel
 * launch on `stream`; returns SPEC_ERR_ARG for n < 0 or NULL pointers. */
int spec_alpha_mean(const float* beta, long long n, double* out, void* stream);

/* Synchronises `stream`, reads and clears the workspace's error word, and
 * returns the lowest-numbered spec_status_t it records (SPEC_OK if none). */
int spec_check_status(void* workspace, void* stream);

/* Launch plan the sampling / statistics kernel would use for (B, gamma, V,
 * dtype) on the current device: thread-block cluster size (CTAs per
 * vocabulary row), slice length per CTA, dynamic shared memory per CTA, CTAs
 * per row for the greedy kernel.  Any output pointer may be NULL.  Host
 * pointers. */
int spec_verify_plan(int B, int gamma, int V, int dtype, int* cluster_size, int* slice_len,
                     int* smem_bytes, int* greedy_ctas_per_row);

/* Static text for a spec_status_t. */
const char* spec_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
