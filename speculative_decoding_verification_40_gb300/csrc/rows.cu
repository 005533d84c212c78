// The early exit's one-launch kernel on sm_103a: one thread-block cluster per batch row, which reads a
// row's logits only up to its first rejection.
//
// Speculative sampling, Algorithm 1 Phases 3-4 (Leviathan, Kalman & Matias, "Fast Inference from
// Transformers via Speculative Decoding"; paper-graph-ui teardown §2.3 "Algorithm Walkthrough",
// multigrid.ai "The algorithm", fullstackaihub §3 "The Algorithm at Position i"), with temperature
// standardisation p = softmax(l / T) (§2.2); the expected number of positions read is about
// sum_k alpha^k (§3.1 Eq. 1) instead of gamma.
//
// The CS CTAs of batch row b's cluster split the vocabulary: CTA r owns the slice [r L, r L + L) of
// every logit row of b.  Position by position (i = 0 .. gamma_b) each CTA streams its slice of target
// row (b, i) and of draft row (b, i) once from HBM (16-byte loads that do not allocate in L1) into
// online softmax normalisers (running max m and S = sum 2^((l - m) log2(e)/T), one hardware exp2 per
// element), reads the logits at the draft token x_i if its slice holds it, and pushes (m_p, S_p, m_q,
// S_q) -- and those logits -- into slot i of the shared memory of every CTA of the cluster
// (st.shared::cluster), followed by a remote arrival on that CTA's mbarrier of slot i.  Slot i is
// complete once every CTA of the row has pushed position i.  Warp 0 then waits (bounded) for it,
// combines the CS partials in rank order (every CTA gets the same bits) and takes the accept decision
// u_i <= min(1, p_i(x_i) / q_i(x_i)) with p_i(x_i) > 0.  The row goes on to position i + 1 only if the
// guess was accepted.
//
// At the first rejection n -- or at gamma_b when every guess is accepted -- the whole CTA reads its slice
// of the drawn row(s) again, just after streaming it, so from L2, as chunk masses of the draw weights
// w = max(0, p_n - q_n) (p_{gamma_b} for the bonus) and of p_n.  The slice masses then meet in every CTA
// at a cluster barrier, each CTA finds the slice holding u_final * Z (Z the total; p_n's when the
// residual mass is <= 1e-15), and the CTA owning that slice picks the chunk from its chunk masses and the
// token by warp scans over the recomputed weights of that one chunk.  No workspace round trip and no
// second launch.
//
// Every wait is bounded: a slot that does not complete within about 0.1 s marks the row invalid with
// SPEC_ERR_TIMEOUT.  The CTAs of a row always end at one cluster barrier, which every one of them
// reaches, so no CTA leaves while another may still write into its shared memory.
#include <atomic>
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"
#include "softmax.cuh"
#include "verify_common.cuh"

namespace specv {

namespace {

constexpr uint32_t kWaitPolls = 1u << 20;  // bounded waits: about 0.1 s of polls

struct RowsSmem {
  float2 sw[kMaxCluster];            // slice masses (w, p_n) of the drawn row, one per CTA
  float2 cs[kMaxChunksPerSlice];     // chunk masses (w, p_n) of this CTA's slice of the drawn row
  float red[2][5][kSW];              // block merge of the normalisers, by position parity
  int x[kMaxGamma];                  // draft ids of the row
  float u[kMaxGamma];                // accept uniforms of the row
  uint32_t err;                      // what makes the row invalid (error-word bits)
  int n;                             // drawn position: the first rejection, or gamma_b; -1 until known
  int draw;                          // 1 while the chunk masses of position n are to be computed
  int resid;                         // the draw is a residual draw
  float cp, cq, tt, dt;              // weights of the drawn row (see RowState)
  float2 mass;                       // this CTA's slice masses (w, p_n) of the drawn row
};

// Exchange slots in dynamic shared memory, one per position: the CS partials (m_p, S_p, m_q, S_q), the
// logits at the draft token, and an mbarrier that completes once every CTA of the row has pushed.
struct Slots {
  float4* part;               // [G + 1][CS]
  float2* xl;                 // [G + 1]
  unsigned long long* mbar;   // [G + 1]
};

__host__ __device__ inline size_t slots_bytes(int G1, int CS) {
  return align_up((size_t)G1 * CS * 16, 16) + align_up((size_t)G1 * 8, 16) + align_up((size_t)G1 * 8, 16);
}

__device__ __forceinline__ Slots carve_slots(unsigned char* base, int G1, int CS) {
  Slots s;
  s.part = reinterpret_cast<float4*>(base);
  base += align_up((size_t)G1 * CS * 16, 16);
  s.xl = reinterpret_cast<float2*>(base);
  base += align_up((size_t)G1 * 8, 16);
  s.mbar = reinterpret_cast<unsigned long long*>(base);
  return s;
}

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}

// Remote arrival (release at cluster scope: this thread's earlier stores into that CTA come first).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Non-blocking test of phase `parity`, with acquire at cluster scope.
__device__ __forceinline__ bool mbar_done_cluster(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Warp-uniform test: true once every lane has observed slot i complete.
__device__ __forceinline__ bool slot_ready(const Slots& sl, int i) {
  return __all_sync(0xffffffffu, mbar_done_cluster(smem_addr(&sl.mbar[i]), 0u));
}

// Warp-uniform bounded wait for slot i; false if it did not complete within kWaitPolls polls.
__device__ __forceinline__ bool slot_wait(const Slots& sl, int i) {
  for (uint32_t k = 0; k < kWaitPolls; ++k) {
    if (slot_ready(sl, i)) return true;
    __nanosleep(64);
  }
  return false;
}

// Per-thread online normalisers of this CTA's slice of target row (b, i) and, for i < gamma_b, of draft
// row (b, i), read from global memory, folded over each warp into red[par] (see fold_warp).
template <typename T, bool kMask>
__device__ __forceinline__ void thread_partials(const T* tp, const T* dp, bool has_q, int n, bool vec, float sc,
                                                float tt, float dt, float (&v)[6]) {
  v[0] = -INFINITY, v[1] = 0.f, v[2] = -INFINITY, v[3] = -INFINITY, v[4] = 0.f, v[5] = -INFINITY;
  if (n > 0) slice_normalisers<T, kMask>(tp, dp, has_q, n, vec, sc, tt, dt, v[0], v[1], v[2], v[3], v[4], v[5]);
}

// Butterfly of the threads' (m_p, S_p, raw_p, m_q, S_q, raw_q) over each warp; lane 0 of each consumer
// warp writes the warp's values to red[par].  The caller's block barrier makes them visible to warp 0.
__device__ __forceinline__ void fold_warp(float (&v)[6], RowsSmem& sm, int par, float sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float mp = v[0], sp = v[1], mq = v[3], sq = v[4];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mp, o), os = __shfl_xor_sync(0xffffffffu, sp, o);
    const float qm = __shfl_xor_sync(0xffffffffu, mq, o), qs = __shfl_xor_sync(0xffffffffu, sq, o);
    merge(mp, sp, om, os, sc);
    merge(mq, sq, qm, qs, sc);
  }
  const float rp = warp_max_nan(max_nan(v[2], v[5]));
  if (lane == 0) {
    sm.red[par][0][warp] = mp;
    sm.red[par][1][warp] = sp;
    sm.red[par][2][warp] = mq;
    sm.red[par][3][warp] = sq;
    sm.red[par][4][warp] = rp;
  }
}

// Warp 0, after the block barrier: the CTA's partial from the warps' values in red[par], merged over
// lanes 0..7 (a fixed butterfly), with NaN maxima if the slice holds a NaN or +inf.  Every lane returns it.
__device__ __forceinline__ float4 cta_partial(const RowsSmem& sm, int par, float sc) {
  const int lane = threadIdx.x & 31;
  float Mp = lane < kSW ? sm.red[par][0][lane] : -INFINITY, Sp = lane < kSW ? sm.red[par][1][lane] : 0.f;
  float Mq = lane < kSW ? sm.red[par][2][lane] : -INFINITY, Sq = lane < kSW ? sm.red[par][3][lane] : 0.f;
  float raw = lane < kSW ? sm.red[par][4][lane] : -INFINITY;
#pragma unroll
  for (int o = kSW / 2; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, Mp, o), os = __shfl_xor_sync(0xffffffffu, Sp, o);
    const float qm = __shfl_xor_sync(0xffffffffu, Mq, o), qs = __shfl_xor_sync(0xffffffffu, Sq, o);
    merge(Mp, Sp, om, os, sc);
    merge(Mq, Sq, qm, qs, sc);
    raw = max_nan(raw, __shfl_xor_sync(0xffffffffu, raw, o));
  }
  Mp = __shfl_sync(0xffffffffu, Mp, 0);
  Sp = __shfl_sync(0xffffffffu, Sp, 0);
  Mq = __shfl_sync(0xffffffffu, Mq, 0);
  Sq = __shfl_sync(0xffffffffu, Sq, 0);
  raw = __shfl_sync(0xffffffffu, raw, 0);
  const bool bad = !(raw < INFINITY);  // NaN or +inf in this slice
  return make_float4(bad ? NAN : Mp, Sp, bad ? NAN : Mq, Sq);
}

// Warp 0: this CTA's partial of position i (and the logits at x_i if it owns them) into slot i of every
// CTA of the cluster, lane r serving CTA r: its stores, then its release arrival on that CTA's slot.
__device__ __forceinline__ void push_partial(float4 nm, bool owner, float2 xl, int CS, uint32_t rank, const Slots& sl,
                                             int i) {
  const int lane = threadIdx.x & 31;
  if (lane < CS) {
    const uint32_t r = static_cast<uint32_t>(lane);
    const float4* dst = sl.part + (size_t)i * CS + rank;
    dsmem_st_v4(dsmem_map(smem_addr(dst), r), nm.x, nm.y, nm.z, nm.w);
    if (owner) dsmem_st_v2(dsmem_map(smem_addr(&sl.xl[i]), r), xl.x, xl.y);
    mbar_arrive_remote(dsmem_map(smem_addr(&sl.mbar[i]), r));
  }
}

// Chunk masses of this CTA's slice of the drawn row -- (w, p) with w = max(0, p - q) for a residual draw,
// w = p otherwise -- one warp per chunk of kR x 32 lanes x 16 bytes, into sm.cs; then warp 0 sums them in
// order into sm.mass.  The p masses are the fallback's when the residual mass is degenerate.  The token
// scan recomputes the same weights (weights_of) for the chunk it picks.
template <typename T>
__device__ void chunk_masses(const T* tr, const T* dr, bool resid, int n, bool vec, const RowState& st, float sc,
                             RowsSmem& sm) {
  constexpr int kV = Elems<T>::kVec;
  constexpr int seg = 32 * kV;
  constexpr int cpc = kR * seg;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = (n + cpc - 1) / cpc;
  for (int c = warp; c < nch; c += kSW) {
    float lw = 0.f, lp = 0.f;
    if (vec && (c + 1) * cpc <= n) {
      uint4 rt[kR], rd[kR];
#pragma unroll
      for (int r = 0; r < kR; ++r) {  // every load of the chunk in flight at once
        rt[r] = ldg_stream(tr + c * cpc + r * seg + lane * kV);
        if (resid) rd[r] = ldg_stream(dr + c * cpc + r * seg + lane * kV);
      }
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        float lt[kV], ld[kV], pv[kV], wv[kV];
        Elems<T>::widen(rt[r], lt);
        if (resid) Elems<T>::widen(rd[r], ld);
        weights_of<kV>(lt, ld, resid, st, sc, pv, wv);
        lw += lane_sum<kV>(wv);
        lp += lane_sum<kV>(pv);
      }
    } else {
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        float pv[kV], wv[kV];
        seg_weights<T>(tr, dr, resid, n, vec, c * cpc + r * seg + lane * kV, st, sc, pv, wv);
        lw += lane_sum<kV>(wv);
        lp += lane_sum<kV>(pv);
      }
    }
    lw = warp_sum(lw);
    lp = warp_sum(lp);
    if (lane == 0) sm.cs[c] = make_float2(lw, lp);
  }
  __syncthreads();
  if (warp == 0) {
    float w = 0.f, q = 0.f;
    for (int c = lane; c < nch; c += 32) {
      w += sm.cs[c].x;
      q += sm.cs[c].y;
    }
    w = warp_sum(w);
    q = warp_sum(q);
    if (lane == 0) sm.mass = make_float2(w, q);
  }
  __syncthreads();
}

// Warp 0 of the CTA owning the drawn slice: the chunk holding t (slice-relative, t - pre) from the chunk
// masses, then the token inside it by warp scans over its recomputed weights.  fb: t lies beyond the
// row's mass (rounding), so the draw is the last token of positive weight.  Returns the token's index in
// the slice, or -1 if the slice has no positive weight.
template <typename T>
__device__ int token_in_slice(const T* tr, const T* dr, bool resid, int n, bool vec, const RowState& st, float sc,
                              float t, bool fb, const RowsSmem& sm) {
  // resid: the residual weights (chunk masses .x); otherwise p (chunk masses .y)
  constexpr int kV = Elems<T>::kVec;
  constexpr int seg = 32 * kV;
  constexpr int cpc = kR * seg;
  const int lane = threadIdx.x & 31;
  const int nch = (n + cpc - 1) / cpc;
  // chunk: lane l takes a run of consecutive chunks, a warp scan gives the mass before each run, and the
  // first chunk whose running mass passes t is the pick (the last chunk of positive mass otherwise)
  const int m = (nch + 31) / 32;
  const int r0 = lane * m, r1 = min(r0 + m, nch);
  float ls = 0.f;
  int lpos = -1;
  for (int c = r0; c < r1; ++c) {
    const float v = resid ? sm.cs[c].x : sm.cs[c].y;
    ls += v;
    if (v > 0.f) lpos = c;
  }
  const float inc = warp_inclusive_scan(ls, lane);
  float cum = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) cum = 0.f;
  int hitc = -1;
  float hpre = 0.f;
  if (!fb) {
    for (int c = r0; c < r1; ++c) {
      const float v = resid ? sm.cs[c].x : sm.cs[c].y;
      if (v > 0.f && cum + v > t) {
        hitc = c;
        hpre = cum;
        break;
      }
      cum += v;
    }
  }
  const unsigned hit = __ballot_sync(0xffffffffu, hitc >= 0);
  const unsigned pos = __ballot_sync(0xffffffffu, lpos >= 0);
  int pc = -1;
  float tt = 0.f;
  bool fallback = fb;
  if (hit) {
    const int l = __ffs(hit) - 1;
    pc = __shfl_sync(0xffffffffu, hitc, l);
    tt = t - __shfl_sync(0xffffffffu, hpre, l);
  } else if (pos) {
    pc = __shfl_sync(0xffffffffu, lpos, 31 - __clz(pos));
    fallback = true;
  }
  if (pc < 0) return -1;
  // the token inside chunk pc: every segment's loads issued at once for a whole aligned chunk, then the scan
  const bool vchunk = vec && (pc + 1) * cpc <= n;
  uint4 rt[kR], rd[kR];
  if (vchunk) {
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      rt[r] = ldg_stream(tr + pc * cpc + r * seg + lane * kV);
      rd[r] = resid ? ldg_stream(dr + pc * cpc + r * seg + lane * kV) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  int tok = -1, lasttok = -1;
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    if (tok >= 0) continue;  // warp-uniform
    const int base = pc * cpc + r * seg + lane * kV;
    float pv[kV], wv[kV];
    if (vchunk) {
      float lt[kV], ld[kV];
      Elems<T>::widen(rt[r], lt);
      Elems<T>::widen(rd[r], ld);
      weights_of<kV>(lt, ld, resid, st, sc, pv, wv);
    } else {
      seg_weights<T>(tr, dr, resid, n, vec, base, st, sc, pv, wv);
    }
    const float lsum = lane_sum<kV>(wv);
    const float incl = warp_inclusive_scan(lsum, lane);
    float exc = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) exc = 0.f;
    int lastj = -1;
#pragma unroll
    for (int j = 0; j < kV; ++j)
      if (wv[j] > 0.f) lastj = j;
    const unsigned nz = __ballot_sync(0xffffffffu, lsum > 0.f);
    if (nz) {  // last positive weight so far: the fallback when rounding leaves t past the total
      const int l = 31 - __clz(nz);
      lasttok = __shfl_sync(0xffffffffu, base + lastj, l);
    }
    const unsigned h = fallback ? 0u : __ballot_sync(0xffffffffu, lsum > 0.f && incl > tt);
    if (h) {
      const int l = __ffs(h) - 1;
      int k = -1;
      if (lane == l) {
        float c = exc;
        for (int j = 0; j < kV; ++j) {
          c += wv[j];
          if (wv[j] > 0.f && c > tt) {
            k = base + j;
            break;
          }
        }
        if (k < 0) k = base + lastj;
      }
      tok = __shfl_sync(0xffffffffu, k, l);
    } else {
      tt -= __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  return tok >= 0 ? tok : lasttok;
}

// Row state of the drawn position n for the weight helpers.
__device__ __forceinline__ RowState drawn_state(const RowsSmem& sm) {
  RowState st = {};
  st.cp = sm.cp;
  st.cq = sm.cq;
  st.tt = sm.tt;
  st.dt = sm.dt;
  return st;
}

}  // namespace

template <typename T, bool kMask>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_rows_kernel(const SampleParams a) {
  __shared__ __align__(16) RowsSmem sm;
  extern __shared__ __align__(128) unsigned char dyn[];
  // A programmatic dependent of whatever precedes it on the stream: read nothing before that grid has
  // finished and its writes are visible.  The next launch may be scheduled from here on (it waits too).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int kV = Elems<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CS = a.rcs;
  const uint32_t rank = cluster_ctarank();
  const int b = static_cast<int>(blockIdx.x) / CS;
  const int G1 = a.G + 1;
  const int lo = static_cast<int>(rank) * a.rslice;
  const int nel = max(0, min(a.V, lo + a.rslice) - lo);  // this CTA's slice length
  const float sc = a.scale;
  const bool vec = a.vec != 0;
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  int32_t* e = a.emitted + (size_t)b * G1;
  // uniform over the cluster (host-checked sizes); a failed check gives an invalid row
  const bool sizes_ok = bounds_ok(b < a.B && CS <= kMaxCluster && (int)rank < CS &&
                                      (a.rslice + kR * 32 * kV - 1) / (kR * 32 * kV) <= kMaxChunksPerSlice,
                                  a.ws.err);
  if (gb < 0 || gb > a.G || !sizes_ok) {  // invalid draft length: nothing of the row is read, no slot used
    if (rank == 0 && tid == 0) {
      for (int j = 0; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = -1;
      atomicOr(a.ws.err, sizes_ok ? kErrArg : kErrBounds);
    }
    return;
  }
  const Slots sl = carve_slots(dyn, G1, CS);
  if (tid == 0) {
    for (int i = 0; i <= gb; ++i) mbar_init(smem_addr(&sl.mbar[i]), static_cast<uint32_t>(CS));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sm.err = 0u;
    sm.n = -1;
    sm.draw = 0;
  }
  if (tid < gb) {  // the row's draft ids and accept uniforms
    sm.x[tid] = __ldg(a.ids + (size_t)b * a.G + tid);
    sm.u[tid] = __ldg(a.uniforms + (size_t)b * G1 + tid);
  }
  cluster_arrive_relaxed();  // this CTA has started and its slots are initialised
  __syncthreads();

  const T* trow = reinterpret_cast<const T*>(a.target) + (size_t)b * G1 * a.V + lo;
  const T* drow = reinterpret_cast<const T*>(a.draft) + (size_t)b * a.G * a.V + lo;
  // Warp 0: the decision on position i from slot i (complete): validity, the accept test, and whether it
  // is the row's drawn position (its weights then go to sm for the chunk masses).
  auto decide = [&](int i) {
    const float4 pr = lane < CS ? sl.part[(size_t)i * CS + lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    const float4 nm = combine_partials(pr, CS, sc);
    if (lane == 0) {
      uint32_t err = 0;
      int code = 1;
      if (i < gb) {
        code = accept_test(a, nm, sm.x[i], sm.u[i], sl.xl[i], err);
      } else if (!(nm.x > -INFINITY && nm.x < INFINITY)) {
        err |= kErrNonfinite;
      }
      if (err) {
        sm.err |= err;
      } else if (sm.n < 0 && sm.err == 0u && (code == 0 || i == gb)) {
        sm.n = i;
        sm.draw = 1;
        sm.resid = i < gb ? 1 : 0;
        sm.cp = -nm.x * sc - log2f(nm.y);
        sm.cq = i < gb ? -nm.z * sc - log2f(nm.w) + log2f(a.lq) : 0.f;  // the residual's q is l q
        sm.tt = kMask && a.tthr ? __ldg(a.tthr + (size_t)b * G1 + i) : -INFINITY;
        sm.dt = kMask && i < gb && a.dthr ? __ldg(a.dthr + (size_t)b * a.G + i) : -INFINITY;
      }
    }
    __syncwarp();
  };
  // All threads: the chunk masses of this CTA's slice of the drawn row, once warp 0 has found it.
  auto masses_if_drawn = [&]() {
    if (sm.draw) {
      const int n = sm.n;
      chunk_masses<T>(trow + (size_t)n * a.V, drow + (size_t)n * a.V, sm.resid != 0, nel, vec, drawn_state(sm), sc,
                      sm);
      if (tid == 0) sm.draw = 0;
      __syncthreads();
    }
  };

  int stop = gb;  // the last position streamed
  for (int i = 0; i <= gb; ++i) {
    const bool has_q = i < gb;
    const T* tp = trow + (size_t)i * a.V;
    const T* dp = has_q ? drow + (size_t)i * a.V : tp;
    const float tt = kMask && a.tthr ? __ldg(a.tthr + (size_t)b * G1 + i) : -INFINITY;
    const float dt = kMask && has_q && a.dthr ? __ldg(a.dthr + (size_t)b * a.G + i) : -INFINITY;
    bool owner = false;
    float2 xl = make_float2(0.f, 0.f);
    if (has_q && warp == 0) {  // issued before the slice, consumed after it
      const int xo = sm.x[i] - lo;
      owner = xo >= 0 && xo < nel;
      if (owner && lane == 0) xl = make_float2(masked(Elems<T>::one(tp, xo), tt), masked(Elems<T>::one(dp, xo), dt));
    }
    float v[6];
    thread_partials<T, kMask>(tp, dp, has_q, nel, vec, sc, tt, dt, v);
    fold_warp(v, sm, i & 1, sc);
    __syncthreads();
    if (i == 0) cluster_wait_acquire();  // every CTA of the cluster has started: its slots may be written
    if (warp == 0) {
      const float4 nm = cta_partial(sm, i & 1, sc);
      xl.x = __shfl_sync(0xffffffffu, xl.x, 0);
      xl.y = __shfl_sync(0xffffffffu, xl.y, 0);
      push_partial(nm, owner, xl, CS, rank, sl, i);
    }
    // the decision on position i before the next is streamed: warp 0 waits (bounded) for its slot
    if (warp == 0) {
      if (slot_wait(sl, i))
        decide(i);
      else if (lane == 0)
        sm.err |= kErrTimeout;
    }
    __syncthreads();
    masses_if_drawn();
    if (sm.n >= 0 || sm.err != 0u) {  // stopped at a rejection or an invalid position
      stop = i;
      break;
    }
  }
  // Ids and uniforms of the positions after the stop are still checked, as in the all-positions path; the
  // final uniform always.
  if (stop < gb && tid > stop && tid < gb) {
    uint32_t err = 0;
    if (sm.x[tid] < 0 || sm.x[tid] >= a.V) err |= kErrToken;
    if (!(sm.u[tid] >= 0.f && sm.u[tid] < 1.f)) err |= kErrArg;
    if (err) atomicOr(&sm.err, err);
  }
  const float uf = __ldg(a.uniforms + (size_t)b * G1 + a.G);
  if (tid == 0 && !(uf >= 0.f && uf < 1.f)) atomicOr(&sm.err, kErrArg);
  __syncthreads();
  // The slice masses of the drawn row meet in every CTA at the row's one cluster barrier, which every CTA
  // of the row reaches: each has pushed and arrived on every slot before it, so after it no CTA writes
  // into another's shared memory.
  const bool valid = sm.err == 0u && sm.n >= 0;  // the same in every CTA, barring a timed-out wait
  if (warp == 0 && lane < CS)
    dsmem_st_v2(dsmem_map(smem_addr(&sm.sw[rank]), static_cast<uint32_t>(lane)), valid ? sm.mass.x : 0.f,
                valid ? sm.mass.y : 0.f);
  cluster_arrive_release();
  cluster_wait_acquire();
  if (!valid) {
    if (rank == 0 && tid == 0) {
      for (int j = 0; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = -1;
      atomicOr(a.ws.err, sm.err != 0u ? sm.err : kErrNonfinite);
    }
    return;
  }
  const int n = sm.n;
  float Z = 0.f, P = 0.f;
  for (int r = 0; r < CS; ++r) {  // rank order: the same totals in every CTA
    Z += sm.sw[r].x;
    P += sm.sw[r].y;
  }
  // a residual whose mass is degenerate (<= 1e-15) draws from p_n instead (rare: a rejection implies a
  // positive residual in exact arithmetic)
  const bool resid = sm.resid != 0 && Z > kZFloor;
  const float tot = resid ? Z : P;
  // No CTA touches another's shared memory from here on.  The slice holding t = u_final * total: the
  // first with positive mass whose running mass passes t, else (rounding) the last one of positive mass.
  const float t = uf * tot;
  int sd = -1, lastd = -1;
  float cum = 0.f, pre = 0.f, lastpre = 0.f;
  for (int r = 0; r < CS; ++r) {
    const float v = resid ? sm.sw[r].x : sm.sw[r].y;
    if (v > 0.f) {
      if (sd < 0 && cum + v > t) {
        sd = r;
        pre = cum;
      }
      lastd = r;
      lastpre = cum;
    }
    cum += v;
  }
  const bool fb = sd < 0;
  if (fb) {
    sd = lastd;
    pre = lastpre;
  }
  if (sd != static_cast<int>(rank) || warp != 0) return;
  const T* tr = trow + (size_t)n * a.V;
  const T* dr = resid ? drow + (size_t)n * a.V : tr;
  int tok = token_in_slice<T>(tr, dr, resid, nel, vec, drawn_state(sm), sc, t - pre, fb, sm);
  if (tok >= 0) tok += lo;
  if (!bounds_ok(tok < a.V, a.ws.err)) tok = -1;
  // the outputs, one lane per slot: the accepted drafts, the drawn token, then -1
  for (int j = lane; j < G1; j += 32) e[j] = tok < 0 ? -1 : j < n ? sm.x[j] : j == n ? tok : -1;
  if (lane == 0) {
    a.n_acc[b] = tok >= 0 ? n : -1;
    if (tok < 0) atomicOr(a.ws.err, kErrNonfinite);  // no weight anywhere (cannot happen for a valid row)
  }
}

namespace {

// Dynamic shared memory of a launch: the exchange slots.
size_t rows_dyn_smem(int G, int CS) { return slots_bytes(G + 1, CS); }

template <typename T, bool kMask>
cudaError_t launch_rows_t(const SampleParams& p, cudaStream_t stream, bool pdl) {
  auto kernel = verify_rows_kernel<T, kMask>;
  // clusters of more than 8 CTAs need the non-portable size allowed, and the slots of the largest sizes
  // more than 48 KB of dynamic shared memory: once per device and kernel
  static std::atomic<unsigned long long> prepared{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(prepared.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(rows_dyn_smem(kMaxGamma, kMaxCluster)));
    if (e != cudaSuccess) return e;
    prepared.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.B * p.rcs));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = rows_dyn_smem(p.G, p.rcs);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.rcs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <typename T>
cudaError_t max_clusters_t(int G, int cs, int* out) {
  auto kernel = verify_rows_kernel<T, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(rows_dyn_smem(kMaxGamma, kMaxCluster)));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs * 1024));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = rows_dyn_smem(G, cs);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, kernel, &cfg);
}

}  // namespace

cudaError_t rows_launch(const SampleParams& p, int dtype, cudaStream_t stream, bool pdl) {
  const bool mask = p.tthr != nullptr || p.dthr != nullptr;
  if (dtype == 0) return mask ? launch_rows_t<float, true>(p, stream, pdl) : launch_rows_t<float, false>(p, stream, pdl);
  return mask ? launch_rows_t<__nv_bfloat16, true>(p, stream, pdl) : launch_rows_t<__nv_bfloat16, false>(p, stream, pdl);
}

cudaError_t rows_max_active_clusters(int dtype, int G, int cs, int* out) {
  return dtype == 0 ? max_clusters_t<float>(G, cs, out) : max_clusters_t<__nv_bfloat16>(G, cs, out);
}

}  // namespace specv
