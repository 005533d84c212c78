// Sampling verification on sm_103a: a streaming pass over the logits, then a
// draw pass over the rows the draws need.
//
// Speculative sampling, Algorithm 1 Phases 3-4 (Leviathan, Kalman & Matias,
// "Fast Inference from Transformers via Speculative Decoding"; paper-graph-ui
// teardown §2.3 "Algorithm Walkthrough", multigrid.ai "The algorithm",
// fullstackaihub §3 "The Algorithm at Position i"), with temperature
// standardisation p = softmax(l / T) (§2.2).
//
// Stream kernel, one CTA per (batch row b, position i, vocabulary slice s):
//   reads slice s of target row (b, i) and, for i < gamma_b, of draft row
//   (b, i) once, with 16-byte loads that do not allocate in L1, keeping online
//   softmax normalisers -- the running max m and S = sum 2^((l - m) log2(e)/T),
//   rescaled when m grows, one hardware exp2 per element -- and writes (m, S)
//   for p and q; the CTA holding the draft token x_i records l_p(x_i),
//   l_q(x_i).  No CTA waits for or signals another.
// Draw kernel, one CTA per (batch row b, draw slice d), rows in reverse order
//   so the rows the stream kernel read last are still in L2:
//   every CTA of row b combines the slice normalisers, takes the accept
//   decisions u_i <= min(1, p_i(x_i)/q_i(x_i)) (with p(x) > 0) and finds the
//   first rejection n -- the same arithmetic in every CTA, so they agree bit
//   for bit -- then, over slice d of target row n (and of draft row n for a
//   residual draw), writes the mass of w = max(0, p_n - q_n) and of p_n per
//   chunk.  A draw from p_n over a row of several stream slices takes its
//   slice from the stream pass's slice normalisers first, and only that
//   slice's chunks are summed.  The last CTA of row b (atomic arrival counter) picks, from
//   u_final * (total mass), the slice, then the chunk from the stored chunk
//   masses, then the token by warp scans over that chunk's recomputed
//   weights: the residual draw, the draw from p_n when the residual mass is
//   <= 1e-15, or the bonus draw from p_{gamma_b} when nothing was rejected.
//   It writes the row's outputs and returns every slot the row used to zero.
// p and q are never written to memory; HBM traffic is the logits read once
// plus, per batch row, at most the two drawn rows (a residual draw) or one
// stream slice of the drawn row (a draw from p), where they have left L2.
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"
#include "softmax.cuh"
#include "verify_common.cuh"

namespace specv {

namespace {

constexpr int kShortRowBytes = 8192;  // rows up to this size take the one-launch path

struct DrawSmem {
  float mp[kMaxGamma + 1], sp[kMaxGamma + 1], mq[kMaxGamma + 1], sq[kMaxGamma + 1];
  int acc[kMaxGamma + 1];
  uint32_t perr[kMaxGamma + 1];  // error bits per position (early-exit validity)
  float2 xl[kMaxGamma];  // logits at the draft tokens (short-row path)
  float2 cs[kMaxRowChunks];  // chunk masses of the drawn row (w, p), gathered by the resolving CTA
  float2 ds[kMaxSlices];     // slice masses of the drawn row (w, p)
  uint32_t err;
  int last, pick, mode, c0, c1;
  float t, pre;
  // a draw from p over several stream slices: the chunks [pcl, pch) of the slice the partials place u_final
  // in and the mass to find inside it (pcl = -1: the whole row's chunks)
  int pcl, pch;
  float ptp;
};

// Inputs of the row's decisions that the stream kernel does not write, loaded by the draw kernel before
// it waits for the stream kernel: thread i <= gamma_b holds x_i and u_i, thread 0 also u_final.
struct RowInputs {
  int x;
  float u, uf;
};

__device__ __forceinline__ RowInputs load_row_inputs(const SampleParams& a, int b, int gb) {
  const int tid = threadIdx.x;
  RowInputs in = {0, 0.f, 0.f};
  if (tid < gb) in.x = __ldg(a.ids + (size_t)b * a.G + tid);
  if (tid < gb) in.u = __ldg(a.uniforms + (size_t)b * (a.G + 1) + tid);
  if (tid == 0) in.uf = __ldg(a.uniforms + (size_t)b * (a.G + 1) + a.G);
  return in;
}

// A draw from p_n over a row of NS > 1 stream slices, by warp 0: the slice masses p(slice s) =
// S_s 2^((m_s - M) log2(e)/T) / S from the stream pass's partials of position n, summed in the order that
// made S (so that they total exactly 1); the slice holding u_final -- the first of positive mass whose
// running total passes it -- into sm as its chunk range [pcl, pch) (cpc elements per chunk; stream slices
// are whole chunks), with the mass u_final - (the slices before it) left to find inside it (pcl = -1 if
// no slice has mass).  uf is read from lane 0.  Only the chosen slice's chunks are then read again.
__device__ __noinline__ void partial_pick(const SampleParams& a, int b, int n, float uf, int cpc, DrawSmem& sm) {
  const int lane = threadIdx.x & 31;
  const int NS = a.nslices;
  const float4 pr = load_partial(reinterpret_cast<const float4*>(a.ws.part) + ((size_t)b * (a.G + 1) + n) * NS, NS);
  const float M = sm.mp[n], S = sm.sp[n];
  // the same terms, summed in the same order, as combine_partials
  const float P = (pr.x > -INFINITY && M < INFINITY) ? pr.y * fast_exp2((pr.x - M) * a.scale) : 0.f;
  float pre = 0.f, run = 0.f;
  for (int r = 0; r < NS; ++r) {
    if (r == lane) pre = run;
    run += __shfl_sync(0xffffffffu, P, r);
  }
  const float u = __shfl_sync(0xffffffffu, uf, 0);
  const float cum = (pre + P) / S;  // pre + P: the running sum after this slice, the float combine saw
  // u < 1 and the last slice of positive mass ends at S / S = 1, so a slice of positive mass is found
  const unsigned hit = __ballot_sync(0xffffffffu, lane < NS && P > 0.f && cum > u);
  const unsigned pos = __ballot_sync(0xffffffffu, lane < NS && P > 0.f);
  const int sl = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  const float pre_s = __shfl_sync(0xffffffffu, pre, sl < 0 ? 0 : sl);
  if (lane == 0) {
    if (sl < 0) {
      sm.pcl = -1;
    } else {
      const int per = a.slice / cpc;
      const int nc = (a.V + cpc - 1) / cpc;
      sm.pcl = sl * per;
      sm.pch = min(sl * per + per, nc);
      sm.ptp = fmaxf(u - pre_s / S, 0.f);
    }
  }
}

// staged: the caller already put the row normalisers in sm.mp .. sm.sq and the logits at the draft
// tokens in sm.xl (the short-row path); otherwise they are combined from the workspace here.
__device__ RowState decide_row(const SampleParams& a, int b, int gb, const RowInputs& in, DrawSmem& sm,
                               bool staged = false) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = a.G + 1;
  const int NS = a.nslices;
  const float sc = a.scale;
  float2 xl = make_float2(0.f, 0.f);
  if (staged) {
    if (tid < gb) xl = sm.xl[tid];
  } else {
    const float4* part = reinterpret_cast<const float4*>(a.ws.part) + (size_t)b * G1 * NS;
    // the logits at the draft tokens, loaded while the warps combine the slice normalisers
    if (tid < gb) xl = __ldcg(reinterpret_cast<const float2*>(a.ws.xl) + (size_t)b * a.G + tid);
    // per-position normalisers from the slice partials (fixed combination order); each warp loads the
    // partials of its first two positions before combining them, one round trip for gamma_b < 2 x warps
    const int i0 = warp, i1 = warp + kSW;
    const float4 pr0 = i0 <= gb ? load_partial(part + (size_t)i0 * NS, NS) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 pr1 = i1 <= gb ? load_partial(part + (size_t)i1 * NS, NS) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = warp; i <= gb; i += kSW) {
      const float4 nm = i == i0 ? combine_partials(pr0, NS, sc)
                      : i == i1 ? combine_partials(pr1, NS, sc)
                                : position_norm(part + (size_t)i * NS, NS, sc);
      if (lane == 0) {
        sm.mp[i] = nm.x;
        sm.sp[i] = nm.y;
        sm.mq[i] = nm.z;
        sm.sq[i] = nm.w;
      }
    }
  }
  if (tid == 0) sm.err = 0;
  __syncthreads();
  // validity and accept decisions, one thread per position
  uint32_t err = 0;
  if (tid <= gb) {
    const int i = tid;
    int code = 1;
    if (i < gb) {
      code = accept_test(a, make_float4(sm.mp[i], sm.sp[i], sm.mq[i], sm.sq[i]), in.x, in.u, xl, err);
    } else if (!(sm.mp[i] > -INFINITY && sm.mp[i] < INFINITY)) {
      err |= kErrNonfinite;
    }
    sm.acc[i] = err ? -1 : code;
    // early-exit validity (a.lazy): a logit row after the first rejection counts as never read, so only the
    // id and uniform checks of those positions stand; the stop position is found after the barrier
    if (a.lazy) sm.perr[i] = err;
  }
  if (tid == 0 && !(in.uf >= 0.f && in.uf < 1.f)) {
    if (a.lazy)
      atomicOr(&sm.err, kErrArg);
    else
      err |= kErrArg;
  }
  if (err && !a.lazy) atomicOr(&sm.err, err);
  __syncthreads();
  if (a.lazy) {
    if (tid == 0) {
      int s = gb;  // the first position not accepted: a rejection, an invalid position, or the bonus
      for (int i = 0; i < gb; ++i) {
        if (sm.acc[i] != 1) {
          s = i;
          break;
        }
      }
      uint32_t e = 0;
      for (int i = 0; i <= gb; ++i) e |= i <= s ? sm.perr[i] : (sm.perr[i] & (kErrToken | kErrArg));
      sm.err |= e;
    }
    __syncthreads();
  }
  RowState st = {};
  int n = gb;
  for (int i = 0; i < gb; ++i) {
    if (sm.acc[i] == 0) {
      n = i;
      break;
    }
  }
  st.n = n;
  st.err = sm.err;
  st.uf = in.uf;
  st.x = in.x;
  if (st.err) {
    st.flags = kRowInvalid;
  } else {
    st.flags = n < gb ? kRowResid : 0;
    st.cp = -sm.mp[n] * a.scale - log2f(sm.sp[n]);
    st.tt = a.tthr ? __ldg(a.tthr + (size_t)b * G1 + n) : -INFINITY;
    st.dt = -INFINITY;
    if (n < gb) {
      st.cq = -sm.mq[n] * a.scale - log2f(sm.sq[n]) + log2f(a.lq);  // the residual's q is l q
      if (a.dthr) st.dt = __ldg(a.dthr + (size_t)b * a.G + n);
    }
  }
  return st;
}

// Slice masses of the drawn row from its chunk masses in shared memory, one warp per slice: lane l sums
// chunks l, l + 32, ... of the slice, then a fixed butterfly over the lanes.  which: 1 = w, 2 = p, 3 = both.
__device__ __forceinline__ void slice_sums(DrawSmem& sm, int ND, int cps, int nc, int which) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int d = warp; d < ND; d += kSW) {
    const int lo = d * cps, hi = min(lo + cps, nc);
    float W = 0.f, P = 0.f;
    for (int c = lo + lane; c < hi; c += 32) {
      W += sm.cs[c].x;
      P += sm.cs[c].y;
    }
    W = warp_sum(W);
    P = warp_sum(P);
    if (lane == 0) {
      if (which & 1) sm.ds[d].x = W;
      if (which & 2) sm.ds[d].y = P;
    }
  }
}

// Last CTA of row b: slice, chunk and token of the draw; the row's outputs; every slot back to zero.
// kPick: the row has several stream slices, and a draw from p may take its slice from the partials
// (partial_pick); without it every draw scans the whole row's chunks.
template <typename T, bool kPick>
__device__ void resolve_row(const SampleParams& a, int b, int gb, const RowState& st, DrawSmem& sm) {
  constexpr int kV = Elems<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31;
  const int G1 = a.G + 1;
  const int ND = a.ndslices;
  const int seg = 32 * kV;
  const int cpc = kR * seg;
  const int cps = a.dslice / cpc;
  const int nc = (a.V + cpc - 1) / cpc;
  float2* dch = reinterpret_cast<float2*>(a.ws.dch) + (size_t)b * ND * cps;
  int32_t* e = a.emitted + (size_t)b * G1;
  const bool resid = st.flags & kRowResid;
  const bool failed = st.flags & kRowInvalid;
  // a draw from p whose stream slice the partials picked (sm.pcl >= 0): only that slice's chunks count
  bool pmode = kPick && !failed && sm.pcl >= 0;
  // the chunk masses of the whole row in shared memory: already there when the row has one draw CTA,
  // else one round trip for all of them
  const bool staged = ND == 1 || a.cluster != 0;
  if (!failed && !staged)
    for (int c = tid; c < ND * cps; c += kST) sm.cs[c] = __ldcg(dch + c);
  __syncthreads();
  // slice masses: one warp per slice, a fixed-order reduction of its chunk masses
  if (!failed && !pmode) slice_sums(sm, ND, cps, nc, 3);
  __syncthreads();
  if (!failed && resid) {
    // a residual whose mass is degenerate (<= 1e-15) draws from p instead; the draw CTAs summed only the
    // residual, so this CTA sums the p masses of the chunks now -- of the slice the partials pick when the
    // row has several stream slices, else of the whole row (rare: a rejection implies a positive residual
    // in exact arithmetic)
    float Z = 0.f;
    for (int d = 0; d < ND; ++d) Z += sm.ds[d].x;
    if (!(Z > kZFloor)) {
      const int warp = tid >> 5;
      const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + st.n) * a.V;
      int pc0 = 0, pc1 = nc;
      if (kPick) {
        if (tid < 32) partial_pick(a, b, st.n, st.uf, cpc, sm);
        __syncthreads();
        pmode = sm.pcl >= 0;
        if (pmode) {
          pc0 = sm.pcl;
          pc1 = sm.pch;
        }
      }
      for (int c = pc0 + warp; c < pc1; c += kSW) {
        float lp = 0.f;
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          float pv[kV], wv[kV];
          seg_weights<T>(tr, tr, false, a.V, a.vec != 0, c * cpc + r * seg + lane * kV, st, a.scale, pv, wv);
          lp += lane_sum<kV>(pv);
        }
        lp = warp_sum(lp);
        if (lane == 0) sm.cs[c].y = lp;
      }
      __syncthreads();
      if (!pmode) {
        slice_sums(sm, ND, cps, nc, 2);
        __syncthreads();
      }
    }
  }
  if (pmode && tid == 0) {  // the chunks of the partials' slice, the target mass inside it
    sm.c0 = sm.pcl;
    sm.c1 = sm.pch;
    sm.t = sm.ptp;
    sm.pre = 0.f;
    sm.mode = 1;
    sm.pick = 0;
  }
  if (!failed && !pmode && tid == 0) {
    // total mass in slice order; the residual, or p when the residual mass is degenerate
    const float uf = st.uf;
    float Z = 0.f, P = 0.f;
    for (int d = 0; d < ND; ++d) {
      Z += sm.ds[d].x;
      P += sm.ds[d].y;
    }
    const bool use_p = !resid || !(Z > kZFloor);
    const float tot = use_p ? P : Z;
    const float t = uf * tot;
    int sd = -1, lastd = -1;
    float cum = 0.f, pre = 0.f, lastpre = 0.f;
    for (int d = 0; d < ND; ++d) {
      const float v = use_p ? sm.ds[d].y : sm.ds[d].x;
      if (v > 0.f) {
        if (sd < 0 && cum + v > t) {
          sd = d;
          pre = cum;
        }
        lastd = d;
        lastpre = cum;
      }
      cum += v;
    }
    const bool fallback = sd < 0;
    if (fallback) {
      sd = lastd;
      pre = lastpre;
    }
    sm.pick = sd;
    sm.mode = (use_p ? 1 : 0) | (fallback ? 2 : 0);
    sm.t = t;
    sm.pre = pre;
    sm.c0 = sd * cps;
    sm.c1 = min(sd * cps + cps, nc);
  }
  if (failed && tid == 0) sm.pick = -1;
  __syncthreads();
  // chunk within the chosen slice, by warp 0: each lane takes a run of consecutive chunks, a warp scan
  // gives the mass before each run, and the first chunk whose running mass passes t is the pick (the
  // last chunk of positive mass if rounding leaves t beyond the slice, or if the slice pick fell back)
  const int sd = sm.pick;
  if (sd >= 0) {
    if (tid < 32) {
      const int c0 = sm.c0, c1 = sm.c1;
      const bool use_p = sm.mode & 1;
      const bool fb = sm.mode & 2;
      const float t = sm.t;
      const int m = (c1 - c0 + 31) / 32;
      const int r0 = c0 + lane * m, r1 = min(r0 + m, c1);
      float ls = 0.f;
      int lpos = -1;
      for (int c = r0; c < r1; ++c) {
        const float v = use_p ? sm.cs[c].y : sm.cs[c].x;
        ls += v;
        if (v > 0.f) lpos = c;
      }
      const float inc = warp_inclusive_scan(ls, lane);
      float cum = __shfl_up_sync(0xffffffffu, inc, 1);
      cum = sm.pre + (lane == 0 ? 0.f : cum);
      int hitc = -1;
      float hpre = 0.f;
      if (!fb) {
        for (int c = r0; c < r1; ++c) {
          const float v = use_p ? sm.cs[c].y : sm.cs[c].x;
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
      float cpre = 0.f;
      if (hit) {
        const int l = __ffs(hit) - 1;
        pc = __shfl_sync(0xffffffffu, hitc, l);
        cpre = __shfl_sync(0xffffffffu, hpre, l);
      } else if (pos) {
        pc = __shfl_sync(0xffffffffu, lpos, 31 - __clz(pos));
      }
      if (lane == 0) {
        sm.pick = pc;
        sm.mode = (use_p ? 1 : 0) | (hit ? 0 : 2);
        sm.pre = cpre;
      }
    }
    __syncthreads();
  }
  const int pc = sd >= 0 ? sm.pick : -1;
  if (pc >= 0 && tid < 32) {  // warp 0: the token inside the chunk, segment by segment
    const bool use_p = sm.mode & 1;
    const bool fallback = sm.mode & 2;
    const bool res = resid && !use_p;
    const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + st.n) * a.V;
    const T* dr = resid ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + st.n) * a.V : tr;
    // a whole chunk of aligned rows: every segment's loads issued at once (one round trip), then the scan
    const bool vchunk = a.vec != 0 && (pc + 1) * cpc <= a.V;
    uint4 rt[kR], rd[kR];
    if (vchunk) {
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        rt[r] = ldg_stream(tr + pc * cpc + r * seg + lane * kV);
        rd[r] = res ? ldg_stream(dr + pc * cpc + r * seg + lane * kV) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float tt = sm.t - sm.pre;
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
        weights_of<kV>(lt, ld, res, st, a.scale, pv, wv);
      } else {
        seg_weights<T>(tr, dr, res, a.V, a.vec != 0, base, st, a.scale, pv, wv);
      }
      const float ls = lane_sum<kV>(wv);
      const float inc = warp_inclusive_scan(ls, lane);
      float exc = __shfl_up_sync(0xffffffffu, inc, 1);
      if (lane == 0) exc = 0.f;
      int lastj = -1;
#pragma unroll
      for (int j = 0; j < kV; ++j)
        if (wv[j] > 0.f) lastj = j;
      const unsigned nz = __ballot_sync(0xffffffffu, ls > 0.f);
      if (nz) {  // last positive weight so far: the fallback when rounding leaves t past the total
        const int l = 31 - __clz(nz);
        lasttok = __shfl_sync(0xffffffffu, base + lastj, l);
      }
      const unsigned hit = fallback ? 0u : __ballot_sync(0xffffffffu, ls > 0.f && inc > tt);
      if (hit) {
        const int l = __ffs(hit) - 1;
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
        tt -= __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    if (tok < 0) tok = lasttok;
    if (!bounds_ok(tok < a.V, a.ws.err)) tok = -1;
    // the outputs, one lane per slot: the accepted drafts, the drawn token, then -1
    for (int j = lane; j < G1; j += 32)
      e[j] = tok < 0 ? -1 : j < st.n ? (j < 32 ? st.x : __ldg(a.ids + (size_t)b * a.G + j)) : j == st.n ? tok : -1;
    if (lane == 0) {
      a.n_acc[b] = tok >= 0 ? st.n : -1;
      if (tok < 0) atomicOr(a.ws.err, kErrNonfinite);  // no weight anywhere (cannot happen for a valid row)
    }
  } else if (tid == 0) {
    for (int j = 0; j < G1; ++j) e[j] = -1;
    a.n_acc[b] = -1;
    atomicOr(a.ws.err, failed ? st.err : kErrNonfinite);
  }
  // every slot of this row back to zero for the next call
  const int NS = a.nslices;
  float4* part = reinterpret_cast<float4*>(a.ws.part) + (size_t)b * G1 * NS;
  for (int k = tid; k < (gb + 1) * NS; k += kST) part[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = tid; k < gb; k += kST) reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + k] = make_float2(0.f, 0.f);
  if (!staged)
    for (int k = tid; k < ND * cps; k += kST) dch[k] = make_float2(0.f, 0.f);
  if (tid == 0) {
    a.ws.ticket[b] = 0u;
  }
}

}  // namespace

// ----------------------------------------------------------------------------- stream kernel


// Block merge of the threads' normalisers in a fixed order (identical for p and q): warp shuffles, then
// thread 0 over the warps.  Thread 0 returns the block's (m_p, S_p, m_q, S_q) and raw maximum.
__device__ __forceinline__ void block_normalisers(float mp, float sp, float rp, float mq, float sq, float rq,
                                                  float sc, float (*red)[kSW], float* rawr, float4& out,
                                                  float& raw) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mp, o), os = __shfl_xor_sync(0xffffffffu, sp, o);
    const float qm = __shfl_xor_sync(0xffffffffu, mq, o), qs = __shfl_xor_sync(0xffffffffu, sq, o);
    merge(mp, sp, om, os, sc);
    merge(mq, sq, qm, qs, sc);
  }
  rp = warp_max_nan(max_nan(rp, rq));
  if (lane == 0) {
    red[0][warp] = mp;
    red[1][warp] = sp;
    red[2][warp] = mq;
    red[3][warp] = sq;
    rawr[warp] = rp;
  }
  __syncthreads();
  if (tid == 0) {
    float Mp = red[0][0], Sp = red[1][0], Mq = red[2][0], Sq = red[3][0], r = rawr[0];
    for (int w = 1; w < kSW; ++w) {
      merge(Mp, Sp, red[0][w], red[1][w], sc);
      merge(Mq, Sq, red[2][w], red[3][w], sc);
      r = max_nan(r, rawr[w]);
    }
    out = make_float4(Mp, Sp, Mq, Sq);
    raw = r;
  }
}

template <typename T, bool kMask>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_stream_kernel(const SampleParams a) {
  __shared__ float red[4][kSW];
  __shared__ float rawr[kSW];
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent of whatever precedes it on the stream (the previous call's
  // draw kernel, or the caller's kernel that wrote the logits): its CTAs may be resident early, and read
  // nothing until that grid has finished and its writes are visible.  Only then may the draw kernel be
  // scheduled (it reads the row inputs before its own wait).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int NS = a.nslices;
  const int s = blockIdx.x % NS;
  const int G1 = a.G + 1;
  const int pos = blockIdx.x / NS;
  const int b = pos / G1;
  const int i = pos - b * G1;
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  if (gb < 0 || gb > a.G || i > gb) return;  // invalid length (the draw kernel reports it) or padding
  const bool has_q = i < gb;
  const float sc = a.scale;
  const int lo = s * a.slice;
  const int n = min(a.V, lo + a.slice) - lo;
  if (!bounds_ok(b < a.B && i <= a.G && s < NS && NS <= kMaxSlices && n > 0 && lo + n <= a.V, a.ws.err)) return;
  const T* tp = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + i) * a.V + lo;
  const T* dp = has_q ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + i) * a.V + lo : tp;

  float mp = -INFINITY, sp = 0.f, rp = -INFINITY;
  float mq = -INFINITY, sq = 0.f, rq = -INFINITY;
  const float tt = kMask && a.tthr ? __ldg(a.tthr + pos) : -INFINITY;
  const float dt = kMask && has_q && a.dthr ? __ldg(a.dthr + (size_t)b * a.G + i) : -INFINITY;
  slice_normalisers<T, kMask>(tp, dp, has_q, n, a.vec != 0, sc, tt, dt, mp, sp, rp, mq, sq, rq);
  float4 nrm;
  float raw;
  block_normalisers(mp, sp, rp, mq, sq, rq, sc, red, rawr, nrm, raw);
  if (tid == 32 && has_q) {  // the logits at the draft token, if this slice holds it
    const int x = __ldg(a.ids + (size_t)b * a.G + i);
    if (x >= lo && x < lo + n)
      reinterpret_cast<float2*>(a.ws.xl)[(size_t)b * a.G + i] =
          make_float2(masked(Elems<T>::one(tp, x - lo), tt), masked(Elems<T>::one(dp, x - lo), dt));
  }
  if (tid == 0) {
    const bool bad = !(raw < INFINITY);  // NaN or +inf in this slice
    reinterpret_cast<float4*>(a.ws.part)[(size_t)pos * NS + s] =
        make_float4(bad ? NAN : nrm.x, nrm.y, bad ? NAN : nrm.z, nrm.w);
  }
}

// ----------------------------------------------------------------------------- draw kernel

// Draw slice d of batch row b once the row's slice normalisers are in the workspace: decisions, chunk
// masses of the drawn row(s) in this slice, and the row's resolution in its last draw CTA.
template <typename T, bool kPick>
__device__ __forceinline__ void draw_slice_of_row(const SampleParams& a, int b, int d, int gb, const RowInputs& in,
                                                  DrawSmem& sm, bool staged = false) {
  constexpr int kV = Elems<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ND = a.ndslices;
  const int G1 = a.G + 1;
  if (gb < 0 || gb > a.G) {  // invalid draft length: nothing was streamed for this row
    if (d == 0 && tid == 0) {
      int32_t* e = a.emitted + (size_t)b * G1;
      for (int j = 0; j < G1; ++j) e[j] = -1;
      a.n_acc[b] = -1;
      atomicOr(a.ws.err, kErrArg);
    }
    return;
  }
  const RowState st = decide_row(a, b, gb, in, sm, staged);
  // a draw from p over several stream slices: only the slice the partials place u_final in is read again
  if (kPick) {
    if (tid == 0) sm.pcl = -1;
    __syncthreads();
    if (!(st.flags & (kRowInvalid | kRowResid))) {
      if (tid < 32) partial_pick(a, b, st.n, in.uf, kR * 32 * kV, sm);
      __syncthreads();
    }
  }
  // a clustered row (a.cluster): every CTA stores its chunk masses straight into the shared memory of
  // rank 0, which resolves the row; every CTA has started once the start-of-kernel arrivals are met
  const bool clustered = a.cluster != 0;
  uint32_t root_cs = 0;
  if (clustered) {
    cluster_wait();
    root_cs = dsmem_map(smem_addr(&sm.cs[0]), 0u);
  }
  if (!(st.flags & kRowInvalid)) {
    const bool resid = st.flags & kRowResid;
    const bool vec = a.vec != 0;
    const T* tr = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + st.n) * a.V;
    const T* dr = resid ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + st.n) * a.V : tr;
    const int seg = 32 * kV;                     // elements per segment
    const int cpc = kR * seg;                    // elements per chunk
    const int cps = a.dslice / cpc;              // chunks per slice
    int c0 = d * cps;
    int c1 = min(c0 + cps, (a.V + cpc - 1) / cpc);
    if (kPick && sm.pcl >= 0) {
      c0 = max(c0, sm.pcl);
      c1 = min(c1, sm.pch);
    }
    float2* dch = reinterpret_cast<float2*>(a.ws.dch) + (size_t)b * ND * cps;
    if (!bounds_ok(cps <= kMaxChunksPerSlice && ND * cps <= kMaxRowChunks &&
                       (size_t)ND * cps <= chunks_per_row(a.V) && st.n <= gb,
                   a.ws.err))
      return;
    const float sc = a.scale;
    for (int c = c0 + warp; c < c1; c += kSW) {
      float lw = 0.f;
      if (vec && (c + 1) * cpc <= a.V) {
        uint4 rt[kR], rd[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) {  // every load of the chunk in flight at once
          rt[r] = ldg_stream(tr + c * cpc + r * seg + lane * kV);
          if (resid) rd[r] = ldg_stream(dr + c * cpc + r * seg + lane * kV);
        }
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          float lt[kV], ld[kV];
          Elems<T>::widen(rt[r], lt);
          if (resid) Elems<T>::widen(rd[r], ld);
          float sw = 0.f;
          if (!resid) {
            // bonus or p draw: the weights are p (pairs through the packed f32x2 FMA for bfloat16)
            if constexpr (sizeof(T) == 2) {
              const unsigned long long sc2 = pack2(sc, sc), c2 = pack2(st.cp, st.cp);
#pragma unroll
              for (int j = 0; j < kV; j += 2) {
                float e0, e1;
                unpack2(fma2(pack2(masked(lt[j], st.tt), masked(lt[j + 1], st.tt)), sc2, c2), e0, e1);
                sw += fast_exp2(e0) + fast_exp2(e1);
              }
            } else {
#pragma unroll
              for (int j = 0; j < kV; ++j) sw += fast_exp2(fmaf(masked(lt[j], st.tt), sc, st.cp));
            }
          } else if constexpr (sizeof(T) == 2) {
            // residual: (p, q) pairs through the packed FMA -- per lane the same operations as
            // seg_weights, so the chunk masses and the final scan see identical weights
            const unsigned long long sc2 = pack2(sc, sc), c2 = pack2(st.cp, st.cq);
#pragma unroll
            for (int j = 0; j < kV; ++j) {
              float ep, eq;
              unpack2(fma2(pack2(masked(lt[j], st.tt), masked(ld[j], st.dt)), sc2, c2), ep, eq);
              sw += fmaxf(fast_exp2(ep) - fast_exp2(eq), 0.f);
            }
          } else {
#pragma unroll
            for (int j = 0; j < kV; ++j)
              sw += fmaxf(fast_exp2(fmaf(masked(lt[j], st.tt), sc, st.cp)) -
                              fast_exp2(fmaf(masked(ld[j], st.dt), sc, st.cq)),
                          0.f);
          }
          lw += sw;
        }
      } else {
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          float pv[kV], wv[kV];
          seg_weights<T>(tr, dr, resid, a.V, vec, c * cpc + r * seg + lane * kV, st, sc, pv, wv);
          lw += lane_sum<kV>(wv);
        }
      }
      // the chunk's weight mass (the residual, or p); the p masses of a residual row are only needed
      // when its residual mass is degenerate, and the resolving CTA computes them then.  A row with one
      // draw CTA keeps them in shared memory for its resolution; otherwise they go to the workspace.
      const float cw = warp_sum(lw);
      if (lane == 0) {
        const float2 v = make_float2(cw, resid ? 0.f : cw);
        if (clustered)
          dsmem_st_v2(root_cs + static_cast<uint32_t>(c * sizeof(float2)), v.x, v.y);
        else if (ND > 1)
          dch[c] = v;
        else
          sm.cs[c] = v;
      }
    }
    if (ND > 1 && !clustered && lane == 0) __threadfence();  // the chunk masses before the arrival count
  }
  if (clustered) {
    cluster_sync();  // every CTA's chunk masses are in rank 0's shared memory
    if (cluster_ctarank() == 0) resolve_row<T, kPick>(a, b, gb, st, sm);
    return;
  }
  __syncthreads();  // every warp's chunk masses written (and fenced) before the arrival
  if (tid == 0) {
    if (ND > 1) {
      __threadfence();
      sm.last = atomicAdd(a.ws.ticket + b, 1u) == static_cast<unsigned>(ND - 1);
    } else {
      sm.last = 1;
    }
  }
  __syncthreads();
  if (sm.last) {
    if (ND > 1) __threadfence();
    resolve_row<T, kPick>(a, b, gb, st, sm);
  }
}

template <typename T, bool kPick>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_draw_kernel(const SampleParams a) {
  __shared__ DrawSmem sm;
  if (a.cluster) cluster_arrive_relaxed();  // this CTA has started (its shared memory may be written)
  // the next call's stream kernel may be scheduled now; it waits for this grid before reading anything
  asm volatile("griddepcontrol.launch_dependents;");
  const int ND = a.ndslices;
  const int b = a.B - 1 - static_cast<int>(blockIdx.x / ND);  // last-streamed rows first: still in L2
  const int d = static_cast<int>(blockIdx.x % ND);
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  // the row's draft ids and uniforms are inputs: load them while the stream kernel drains
  const RowInputs in = (gb >= 0 && gb <= a.G) ? load_row_inputs(a, b, gb) : RowInputs{0, 0.f, 0.f};
  // launched as a programmatic dependent of the stream kernel: wait for all of it (and its writes)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  draw_slice_of_row<T, kPick>(a, b, d, gb, in, sm);
}

// ----------------------------------------------------------------------------- short rows, one launch

// Rows of at most kShortRowBytes (one stream slice and one draw slice per row): the whole step in one
// CTA per batch row and one launch.  Warp w computes the normalisers of positions w, w + 8, ... over
// the whole row (16-byte loads, four per lane and row in flight, the online softmax of the
// stream pass, then a butterfly merge over the lanes) into shared memory; after a barrier the CTA runs
// the draw code above on them (one draw slice: decisions, chunk masses, resolution, all from shared
// memory).  For short rows the step is latency-bound, and one launch and one CTA per row
// remove the second launch and the round trip between the two kernels.
template <typename T, bool kMask>
__global__ void __launch_bounds__(kStreamThreads, 4) verify_short_kernel(const SampleParams a) {
  // a programmatic dependent of the previous launch on the stream: read nothing before it has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ DrawSmem sm;
  constexpr int kV = Elems<T>::kVec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int G1 = a.G + 1;
  const int gb = a.draft_len ? __ldg(a.draft_len + b) : a.G;
  const bool valid = gb >= 0 && gb <= a.G;
  const RowInputs in = valid ? load_row_inputs(a, b, gb) : RowInputs{0, 0.f, 0.f};
  const float sc = a.scale;
  const int nv = a.V / kV;  // whole vectors of the row (rows are 16-byte aligned here)
  if (valid && bounds_ok(a.nslices == 1 && a.ndslices == 1, a.ws.err)) {
    for (int i = warp; i <= gb; i += kSW) {
      const bool has_q = i < gb;
      const T* tp = reinterpret_cast<const T*>(a.target) + ((size_t)b * G1 + i) * a.V;
      const T* dp = has_q ? reinterpret_cast<const T*>(a.draft) + ((size_t)b * a.G + i) * a.V : tp;
      const float tt = kMask && a.tthr ? __ldg(a.tthr + (size_t)b * G1 + i) : -INFINITY;
      const float dt = kMask && has_q && a.dthr ? __ldg(a.dthr + (size_t)b * a.G + i) : -INFINITY;
      float mp = -INFINITY, sp = 0.f, rp = -INFINITY, mq = -INFINITY, sq = 0.f, rq = -INFINITY;
      for (int v0 = 0; v0 < nv; v0 += 4 * 32) {  // four vectors per lane and row in flight
        uint4 rt[4], rd[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + lane + 32 * u;
          if (v < nv) {
            rt[u] = ldg_stream(reinterpret_cast<const uint4*>(tp) + v);
            if (has_q) rd[u] = ldg_stream(reinterpret_cast<const uint4*>(dp) + v);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (v0 + lane + 32 * u < nv) {
            const uint4 r1[1] = {rt[u]};
            online_group<T, 1, kMask>(mp, sp, rp, r1, sc, tt);
            if (has_q) {
              const uint4 q1[1] = {rd[u]};
              online_group<T, 1, kMask>(mq, sq, rq, q1, sc, dt);
            }
          }
        }
      }
      for (int k = nv * kV + lane; k < a.V; k += 32) {  // elements past the last whole vector
        float f[1] = {Elems<T>::one(tp, k)};
        online<1, kMask>(mp, sp, rp, f, sc, tt);
        if (has_q) {
          f[0] = Elems<T>::one(dp, k);
          online<1, kMask>(mq, sq, rq, f, sc, dt);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mp, o), os = __shfl_xor_sync(0xffffffffu, sp, o);
        const float qm = __shfl_xor_sync(0xffffffffu, mq, o), qs = __shfl_xor_sync(0xffffffffu, sq, o);
        merge(mp, sp, om, os, sc);
        merge(mq, sq, qm, qs, sc);
      }
      rp = warp_max_nan(max_nan(rp, rq));
      if (lane == 0) {
        const bool bad = !(rp < INFINITY);  // NaN or +inf in the row
        sm.mp[i] = bad ? NAN : mp;
        sm.sp[i] = sp;
        sm.mq[i] = bad ? NAN : mq;
        sm.sq[i] = sq;
        if (has_q) {  // the logits at the draft token (an id outside [0, V) is reported by the accept test)
          const int x = __ldg(a.ids + (size_t)b * a.G + i);
          sm.xl[i] = (x >= 0 && x < a.V) ? make_float2(masked(Elems<T>::one(tp, x), tt), masked(Elems<T>::one(dp, x), dt))
                                         : make_float2(0.f, 0.f);
        }
      }
    }
  }
  __syncthreads();  // the normalisers in shared memory
  draw_slice_of_row<T, false>(a, b, 0, gb, in, sm, true);
}

// The one-launch path applies to 16-byte aligned rows of at most kShortRowBytes with one stream slice and
// one draw slice per row.
static bool short_rows(const SampleParams& p, size_t esz) {
  return p.vec != 0 && static_cast<size_t>(p.V) * esz <= static_cast<size_t>(kShortRowBytes) &&
         p.nslices == 1 && p.ndslices == 1;
}

// The first kernel of a sampling call is launched as a programmatic dependent of the launch before it on
// the stream (its CTAs wait in griddepcontrol.wait before reading anything), so back-to-back calls do
// not pay a launch gap.  SPECVERIFY_PDL=0 launches it plainly.
static bool pdl_first() {
  const char* env = std::getenv("SPECVERIFY_PDL");
  return !(env && std::atoi(env) == 0);
}

// The early exit's form from the environment: 1 = the one-launch kernel, 2 = the two-kernel path, 0 = unset.
static int form_env(const char* name) {
  const char* env = std::getenv(name);
  if (!env) return 0;
  const int v = std::atoi(env);
  return v == 1 || v == 2 ? v : 0;
}

// A row's draw CTAs form one cluster when there are 2 to 8 of them (the portable cluster size) and the
// whole draw grid is resident at once (at most 4 CTAs per SM): their chunk masses meet in rank 0's
// shared memory at a cluster barrier instead of going through the workspace behind an arrival counter,
// which shortens the draw's chain of round trips (c1: 16.7 vs 18.8 us per call; c2, back to back: 60.3
// vs 62.1 us).  A draw grid of more than one wave keeps the counter: its CTAs take SM slots one by one
// as the stream kernel drains, where a cluster waits for ndslices free slots in one GPC.
// SPECVERIFY_DRAW_CLUSTER=0 / 1 forces the counter / the cluster for 2 to 8 draw CTAs per row.
static bool draw_clusters(const SampleParams& p) {
  if (p.ndslices < 2 || p.ndslices > 8) return false;
  if (const char* env = std::getenv("SPECVERIFY_DRAW_CLUSTER")) return std::atoi(env) != 0;
  return static_cast<long long>(p.B) * p.ndslices <= 4LL * (p.sms > 0 ? p.sms : 152);
}

template <typename T>
static cudaError_t launch_draw(const SampleParams& p, cudaStream_t stream) {
  SampleParams q = p;
  q.cluster = draw_clusters(p) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.B * p.ndslices));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(q.cluster ? p.ndslices : 1);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = q.cluster ? 2 : 1;
  return p.nslices > 1 ? cudaLaunchKernelEx(&cfg, verify_draw_kernel<T, true>, q)
                       : cudaLaunchKernelEx(&cfg, verify_draw_kernel<T, false>, q);
}

// The early exit runs the one-launch kernel, which streams a row's positions one after the other and
// stops at the first rejection, when one position of the whole batch is large enough for the bytes it
// skips to outweigh its per-position latency: at least 64 MB over the batch's target and draft rows
// (c3: 256 x 2 rows of 608 KB, 193 vs 285 us for all positions; c4: 131 MB, 127 vs 134 us).  Smaller
// batches (c2: 33 MB, 76 vs 61 us) take the two-kernel all-positions path, whose draw then takes the
// decisions with early-exit validity (logit rows after the first rejection do not count).  Both give
// the early exit's results.  SPECVERIFY_EARLY_FORM=1 / 2 forces the one-launch / two-kernel form.
static bool early_one_launch(const SampleParams& p, int dtype) {
  if (p.rcs <= 0) return false;  // no cluster plan for this shape on this device
  const int f = form_env("SPECVERIFY_EARLY_FORM");
  if (f) return f == 1;
  const long long position_bytes = 2LL * p.B * p.V * (dtype == 0 ? 4 : 2);
  return position_bytes >= (64LL << 20);
}

cudaError_t sample_early_exit_launch(SampleParams p, int dtype, cudaStream_t stream) {
  if (early_one_launch(p, dtype)) return rows_launch(p, dtype, stream, pdl_first());
  p.lazy = 1;
  return sample_launch(p, dtype, 3, stream);
}

// ----------------------------------------------------------------------------- row sampler

// One CTA per row b of logits [R, V] (launched after the stream kernel with gamma = 0, which left the
// row's slice normalisers in the workspace): x ~ softmax(l / T) by the inverse CDF with uniforms[b].
// The slice holding the draw is picked from the slice masses S_s 2^((m_s - M) log2(e)/T) of the stream
// pass, so only that slice is read again; inside it the weights w = 2^(l log2(e)/T - M log2(e)/T) give
// chunk masses, then warp scans find the token.  If rounding leaves the target beyond the slice's
// recomputed mass, the draw is the slice's last token of positive weight.
namespace {

template <typename T>
__device__ __forceinline__ void row_weights(const T* row, bool vec, int base, int n, float sc, float nm, float thr,
                                            float (&w)[Elems<T>::kVec]) {
  constexpr int kV = Elems<T>::kVec;
  float f[kV];
  if (vec && base + kV <= n) {
    Elems<T>::widen(__ldg(reinterpret_cast<const uint4*>(row + base)), f);
  } else {
#pragma unroll
    for (int j = 0; j < kV; ++j) f[j] = base + j < n ? Elems<T>::one(row, base + j) : -INFINITY;
  }
#pragma unroll
  for (int j = 0; j < kV; ++j) w[j] = fast_exp2(fmaf(masked(f[j], thr), sc, nm));
}

}  // namespace

// Inverse-CDF draw inside one slice of n logits (the whole CTA calls it): chunk masses of the weights
// w = 2^(l sc + nm) into cm, then warp 0 finds the chunk and the token whose running sum first exceeds t.
// If rounding leaves t beyond the slice's mass the draw is the slice's last token of positive weight.
// Returns the token's index in the slice in warp 0 (-1 elsewhere, or if the slice has no positive weight).
template <typename T>
__device__ int draw_in_slice(const T* srow, int n, bool vec, float sc, float nm, float thr, float t, float* cm) {
  constexpr int kV = Elems<T>::kVec;
  constexpr int kCpc = kR * 32 * kV;  // elements per chunk: kR vectors per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = (n + kCpc - 1) / kCpc;
  for (int c = warp; c < nch; c += kSW) {
    float acc = 0.f;
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      float w[kV];
      row_weights<T>(srow, vec, c * kCpc + (r * 32 + lane) * kV, n, sc, nm, thr, w);
#pragma unroll
      for (int j = 0; j < kV; ++j) acc += w[j];
    }
    acc = warp_sum(acc);
    if (lane == 0) cm[c] = acc;
  }
  __syncthreads();
  if (warp != 0) return -1;

  int chunk = -1, lastc = -1;
  float carry = 0.f;
  for (int g = 0; g * 32 < nch; ++g) {
    const int c = g * 32 + lane;
    const float v = c < nch ? cm[c] : 0.f;
    const float incl = carry + warp_inclusive_scan(v, lane);
    const unsigned hit = __ballot_sync(0xffffffffu, incl > t);
    const unsigned pos = __ballot_sync(0xffffffffu, v > 0.f);
    if (pos) lastc = g * 32 + 31 - __clz(pos);
    if (hit && chunk < 0) {
      const int l0 = __ffs(hit) - 1;
      chunk = g * 32 + l0;
      t -= __shfl_sync(0xffffffffu, incl - v, l0);
    }
    carry = __shfl_sync(0xffffffffu, incl, 31);
  }
  const bool fallback = chunk < 0;
  if (fallback) chunk = lastc;  // t beyond the slice's mass: the last chunk of positive mass
  int token = -1, lastk = -1;
  if (chunk >= 0) {
    float cc = 0.f;
    for (int r = 0; r < kR && token < 0; ++r) {
      const int base = chunk * kCpc + (r * 32 + lane) * kV;
      float w[kV];
      row_weights<T>(srow, vec, base, n, sc, nm, thr, w);
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < kV; ++j) ls += w[j];
      const float incl = cc + warp_inclusive_scan(ls, lane);
      int lpos = -1;  // this lane's last element of positive weight
#pragma unroll
      for (int j = 0; j < kV; ++j)
        if (w[j] > 0.f) lpos = j;
      const unsigned pos = __ballot_sync(0xffffffffu, lpos >= 0);
      if (pos) {
        const int l1 = 31 - __clz(pos);
        lastk = __shfl_sync(0xffffffffu, base + lpos, l1);
      }
      const unsigned hit = fallback ? 0u : __ballot_sync(0xffffffffu, incl > t);
      if (hit) {
        const int l0 = __ffs(hit) - 1;
        int k = -1;
        if (lane == l0) {  // walk this lane's elements in order
          float run = incl - ls;
#pragma unroll
          for (int j = 0; j < kV; ++j) {
            run += w[j];
            if (k < 0 && run > t) k = base + j;
          }
          if (k < 0) k = base + lpos;  // rounding inside the lane: its last positive weight
        }
        token = __shfl_sync(0xffffffffu, k, l0);
      }
      cc = __shfl_sync(0xffffffffu, incl, 31);
    }
    if (token < 0) token = lastk;  // rounding inside the chunk: its last positive weight
  }
  return token;
}

// Online normaliser (m, S) of a contiguous segment of n logits, merged over the warp (every lane gets
// it), and the NaN-propagating raw maximum.  16-byte loads when vec, four in flight per lane.
template <typename T, bool kMask>
__device__ __forceinline__ void warp_segment(const T* __restrict__ seg, int n, bool vec, float sc, float thr,
                                             float& m, float& sm, float& raw) {
  constexpr int kV = Elems<T>::kVec;
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  m = -INFINITY;
  sm = 0.f;
  raw = -INFINITY;
  if (n > 0) {
    if (vec) {
      const uint4* v4 = reinterpret_cast<const uint4*>(seg);
      const int nv = n / kV;
      int j = lane;
      for (; j + (U - 1) * 32 < nv; j += U * 32) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = ldg_stream(v4 + j + u * 32);
        online_group<T, U, kMask>(m, sm, raw, r, sc, thr);
      }
      for (; j < nv; j += 32) {
        const uint4 r[1] = {ldg_stream(v4 + j)};
        online_group<T, 1, kMask>(m, sm, raw, r, sc, thr);
      }
    } else {
      for (int k = lane; k < n; k += 32) {
        float f[1] = {Elems<T>::one(seg, k)};
        online<1, kMask>(m, sm, raw, f, sc, thr);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, sm, o);
    merge(m, sm, om, os, sc);
  }
  raw = warp_max_nan(raw);
}

// Elements per warp segment of a slice of L elements (eight segments, whole warp-loads each).
template <typename T>
__host__ __device__ __forceinline__ int segment_len(int L) {
  return static_cast<int>(align_up((L + kSW - 1) / kSW, 32 * Elems<T>::kVec));
}

// Rows that fit one slice: one CTA per row, one launch.  Warp w streams the contiguous segment w of
// the row once for its online normalisers (m_w, S_w); thread 0 combines the eight segments in order,
// picks the segment holding u * Z from their masses S_w 2^((m_w - M) log2(e)/T), and the CTA draws
// inside that segment only (its second read, an eighth of the row, hits L2).
template <typename T, bool kMask>
__global__ void __launch_bounds__(kST) sample_rows_fused_kernel(const SampleParams a) {
  __shared__ float segm[kSW], segs[kSW], segr[kSW];
  __shared__ float cm[kMaxChunksPerSlice];
  __shared__ float sh_t, sh_m;
  __shared__ int sh_w, sh_err;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const float sc = a.scale;
  const int V = a.V;
  const T* row = reinterpret_cast<const T*>(a.target) + (size_t)b * V;
  const bool vec = a.vec != 0;
  const int segE = segment_len<T>(V);
  const float thr = kMask && a.tthr ? __ldg(a.tthr + b) : -INFINITY;
  {
    const int lo = warp * segE;
    float m, sm, raw;
    warp_segment<T, kMask>(row + lo, min(V, lo + segE) - lo, vec, sc, thr, m, sm, raw);
    if (lane == 0) {
      segm[warp] = m;
      segs[warp] = sm;
      segr[warp] = raw;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float M = segm[0], raw = segr[0];
    for (int w = 1; w < kSW; ++w) {
      M = max_nan(M, segm[w]);
      raw = max_nan(raw, segr[w]);
    }
    const float u = __ldg(a.uniforms + b);
    uint32_t err = 0;
    if (!(raw < INFINITY) || !(M > -INFINITY)) err |= kErrNonfinite;
    if (!(u >= 0.f && u < 1.f)) err |= kErrArg;
    float e[kSW], Z = 0.f;
    for (int w = 0; w < kSW; ++w) {
      e[w] = (!err && segm[w] > -INFINITY) ? segs[w] * fast_exp2((segm[w] - M) * sc) : 0.f;
      Z += e[w];
    }
    const float t = u * Z;
    int sel = -1, last = 0;
    float before = 0.f, acc = 0.f;
    for (int w = 0; w < kSW; ++w) {
      if (e[w] > 0.f) last = w;
      if (sel < 0 && acc + e[w] > t) {
        sel = w;
        before = acc;
      }
      acc += e[w];
    }
    sh_err = static_cast<int>(err);
    sh_m = M;
    sh_w = sel >= 0 ? sel : last;
    sh_t = sel >= 0 ? t - before : INFINITY;  // beyond every segment: take the last positive weight
  }
  __syncthreads();
  if (sh_err) {
    if (tid == 0) {
      a.emitted[b] = -1;
      atomicOr(a.ws.err, static_cast<uint32_t>(sh_err));
    }
    return;
  }
  const int lo = sh_w * segE;
  const int n = min(V, lo + segE) - lo;
  const int tok = draw_in_slice<T>(row + lo, n, vec, sc, -sh_m * sc, thr, sh_t, cm);
  if (tid == 0) a.emitted[b] = (tok >= 0 && bounds_ok(lo + tok < V, a.ws.err)) ? lo + tok : -1;
}

// Rows longer than one slice, pass 1: one CTA per (row b, slice s); warp w writes the normaliser of
// its segment of the slice, (m, S) with m = NaN if the segment holds NaN or +inf, to the workspace's
// per-row segment list [b][s * 8 + w].
template <typename T, bool kMask>
__global__ void __launch_bounds__(kST, 4) sample_stream_kernel(const SampleParams a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  asm volatile("griddepcontrol.launch_dependents;");
  const int NS = a.nslices;
  const int s = blockIdx.x % NS;
  const int b = blockIdx.x / NS;
  const int segE = segment_len<T>(a.slice);
  const int lo = s * a.slice + warp * segE;
  const int hi = min(a.V, min(s * a.slice + a.slice, lo + segE));
  if (!bounds_ok(b < a.B && (size_t)NS * kSW <= chunks_per_row(a.V), a.ws.err)) return;
  float m, sm, raw;
  const float thr = kMask && a.tthr ? __ldg(a.tthr + b) : -INFINITY;
  warp_segment<T, kMask>(reinterpret_cast<const T*>(a.target) + (size_t)b * a.V + lo, hi - lo, a.vec != 0, a.scale,
                         thr, m, sm, raw);
  if (lane == 0)
    reinterpret_cast<float2*>(a.ws.dch)[(size_t)b * chunks_per_row(a.V) + s * kSW + warp] =
        make_float2(raw < INFINITY ? m : NAN, sm);
}

// Pass 2: one CTA per row.  The row's NS * 8 segment normalisers (in order) give the segment masses;
// the segment holding u * Z is read again (an eighth of a slice) for the draw.
template <typename T>
__global__ void __launch_bounds__(kST) sample_rows_kernel(const SampleParams a) {
  __shared__ float cm[kMaxChunksPerSlice];
  __shared__ float wsum[kSW], wmax[kSW];
  __shared__ float sh_t;
  __shared__ int sh_sel;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int NG = a.nslices * kSW;  // segments of the row, at most 256
  const float sc = a.scale;
  // launched as a programmatic dependent of the stream kernel: wait for all of it (and its writes)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float2* segp = reinterpret_cast<float2*>(a.ws.dch) + (size_t)b * chunks_per_row(a.V);
  float2 sg = make_float2(-INFINITY, 0.f);
  if (tid < NG) {
    sg = __ldcg(segp + tid);
    segp[tid] = make_float2(0.f, 0.f);  // the workspace goes back to zero
  }
  // row max (NaN-propagating), then the masses' inclusive scan in segment order
  float mx = warp_max_nan(sg.x);
  if (lane == 0) wmax[warp] = mx;
  if (tid == 0) sh_sel = -1;
  __syncthreads();
  float M = wmax[0];
  for (int w = 1; w < kSW; ++w) M = max_nan(M, wmax[w]);
  const float u = __ldg(a.uniforms + b);
  uint32_t err = 0;
  if (!(M > -INFINITY && M < INFINITY)) err |= kErrNonfinite;
  if (!(u >= 0.f && u < 1.f)) err |= kErrArg;
  const float e = (!err && sg.x > -INFINITY) ? sg.y * fast_exp2((sg.x - M) * sc) : 0.f;
  const float incl_w = warp_inclusive_scan(e, lane);
  if (lane == 31) wsum[warp] = incl_w;
  __syncthreads();
  float before_w = 0.f, Z = 0.f;
  for (int w = 0; w < kSW; ++w) {
    if (w < warp) before_w += wsum[w];
    Z += wsum[w];
  }
  const float t = u * Z;
  const float incl = before_w + incl_w;  // running mass through segment tid (nondecreasing in tid)
  // the first segment whose running mass exceeds t is the number of segments whose running mass does not
  const int first = __syncthreads_count(tid < NG && incl <= t);
  if (first < NG && tid == first) sh_t = t - (incl - e);
  if (e > 0.f) atomicMax(&sh_sel, tid);  // the last segment of positive mass (sh_sel started at -1)
  __syncthreads();
  if (err) {
    if (tid == 0) {
      a.emitted[b] = -1;
      atomicOr(a.ws.err, err);
    }
    return;
  }
  // beyond the last segment (rounding at u * Z near Z): the draw is the last positive weight
  const bool beyond = first >= NG;
  const int g = beyond ? sh_sel : first;
  const int s = g / kSW, w = g % kSW;
  const int segE = segment_len<T>(a.slice);
  const int lo = s * a.slice + w * segE;
  const int n = min(a.V, min(s * a.slice + a.slice, lo + segE)) - lo;
  if (!bounds_ok(g >= 0 && g < NG && n > 0 && segE <= kMaxChunksPerSlice * kR * 32 * Elems<T>::kVec, a.ws.err)) {
    if (tid == 0) a.emitted[b] = -1;
    return;
  }
  const T* srow = reinterpret_cast<const T*>(a.target) + (size_t)b * a.V + lo;
  const float thr = a.tthr ? __ldg(a.tthr + b) : -INFINITY;
  const int tok = draw_in_slice<T>(srow, n, a.vec != 0, sc, -M * sc, thr, beyond ? INFINITY : sh_t, cm);
  if (tid == 0) a.emitted[b] = (tok >= 0 && bounds_ok(lo + tok < a.V, a.ws.err)) ? lo + tok : -1;
}

template <typename T>
static cudaError_t launch_rows(const SampleParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_rows_kernel<T>, p);
}

template <typename T, bool kMask>
static cudaError_t rows_sample_launch_t(const SampleParams& p, cudaStream_t stream) {
  const dim3 block(kStreamThreads);
  if (p.nslices == 1) {
    sample_rows_fused_kernel<T, kMask><<<dim3(static_cast<unsigned>(p.B)), block, 0, stream>>>(p);
    return cudaGetLastError();
  }
  sample_stream_kernel<T, kMask><<<dim3(static_cast<unsigned>((long long)p.B * p.nslices)), block, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_rows<T>(p, stream);
}

cudaError_t rows_sample_launch(const SampleParams& p, int dtype, cudaStream_t stream) {
  const bool mask = p.tthr != nullptr;
  if (dtype == 0) return mask ? rows_sample_launch_t<float, true>(p, stream) : rows_sample_launch_t<float, false>(p, stream);
  return mask ? rows_sample_launch_t<__nv_bfloat16, true>(p, stream)
              : rows_sample_launch_t<__nv_bfloat16, false>(p, stream);
}

template <typename K>
static cudaError_t launch_first(K kernel, dim3 grid, const SampleParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kStreamThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_first() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <typename T, bool kMask>
static cudaError_t sample_launch_t(const SampleParams& p, int phases, cudaStream_t stream) {
  if (phases == 3 && !p.lazy && short_rows(p, sizeof(T)))
    return launch_first(verify_short_kernel<T, kMask>, dim3(static_cast<unsigned>(p.B)), p, stream);
  const dim3 g1(static_cast<unsigned>((long long)p.B * (p.G + 1) * p.nslices));
  if (phases & 1) {
    const cudaError_t e = launch_first(verify_stream_kernel<T, kMask>, g1, p, stream);
    if (e != cudaSuccess) return e;
  }
  return (phases & 2) ? launch_draw<T>(p, stream) : cudaSuccess;
}

cudaError_t sample_launch(const SampleParams& p, int dtype, int phases, cudaStream_t stream) {
  const bool mask = p.tthr != nullptr || p.dthr != nullptr;
  if (dtype == 0) return mask ? sample_launch_t<float, true>(p, phases, stream) : sample_launch_t<float, false>(p, phases, stream);
  return mask ? sample_launch_t<__nv_bfloat16, true>(p, phases, stream)
              : sample_launch_t<__nv_bfloat16, false>(p, phases, stream);
}

}  // namespace specv
