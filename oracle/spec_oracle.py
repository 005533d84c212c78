"""Float64 CPU oracle for the batched verification step of speculative sampling.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import this module.  It shares no code with the CUDA path
and never runs on the product path.

Source: Leviathan, Kalman & Matias, "Fast Inference from Transformers via
Speculative Decoding" (arXiv 2211.17192), as restated by the four pages read
for this build:
  [p1] paper-graph-ui teardown: §2.2 "Standardized Sampling", §2.3 "Algorithm
       Walkthrough" (Phases 1-4), Appendix A.1 proof, §3.1 Eq. 1, Def. 3.2,
       Lemma 3.3, Thm 3.5, Cor. 3.6;
  [p2] multigrid.ai "Speculative Decoding: Two Models, One Output", "The
       algorithm" and "What the speedup depends on";
  [p3] fullstackaihub "Speculative Decoding Paper Breakdown", §3 "The
       Algorithm at Position i" and the verification sketch;
  [p4] interactiveml "The exact decoding shortcut ...", the correction
       distribution with its degenerate-mass rule.

Everything is a plain loop over rows b and positions i with whole-vocabulary
numpy float64 vector ops; nothing is blocked, fused or reordered.  Inputs are
widened exactly: float32 logits by value, bfloat16 logits from their bit
patterns (uint16), uniforms from float32.

Readings taken where the pages are silent or disagree (each is also listed in
the design notes):
  R1  the final draw (residual or bonus) uses one extra uniform, column gamma of
      the [B, gamma+1] uniform array; column i < gamma is the accept test of
      position i.
  R2  residual and bonus tokens are sampled by inverse CDF: the smallest k with
      C_k > u * Z, C the running sum of the weights; if rounding leaves no such
      k, the largest k with a positive weight.
  R3  a draft with p(x) = 0 is never accepted (the ratio test is taken as
      "p(x) > 0 and u <= min(1, p(x)/q(x))"); q(x) = 0 < p(x) gives ratio 1.
  R4  if the residual mass Z = sum max(0, p - q) is <= 1e-15 the draw falls back
      to p [p4].
  R5  greedy mode: argmax of the target logits, lowest index on ties; accept
      while the argmax equals the draft; emit the argmax at the first mismatch
      or the bonus position.  Temperature does not enter.
  R6  ragged rows: row b verifies draft_len[b] = gamma_b positions; target rows
      i > gamma_b, draft rows i >= gamma_b, ids i >= gamma_b and uniforms
      gamma_b <= i < gamma are never read.
  R7  a row is invalid (n_accepted = -1, emitted all -1) if any logit row it
      reads holds NaN or +inf or is entirely -inf, if a draft id it reads lies
      outside [0, V), if a uniform it reads lies outside [0, 1), or if
      draft_len[b] lies outside [0, gamma].
  R8  boundary draws: a row is flagged when a tested uniform lies within 1e-5
      of its acceptance threshold, or the final uniform lies within 1e-5 of a
      CDF edge of the chosen token (both on the normalised scale).
  R9  top-k keeps every token whose logit is >= the k-th largest logit (ties at
      the boundary are all kept); fewer than k finite logits keep everything.
  R11 lenience l in (0, 1] multiplies q wherever it meets p: the accept test is
      u <= min(1, p(x) / (l q(x))) and the residual is norm(max(0, p - l q)).
      The pages state the scaling of q in the comparison and the resulting
      guarantee (no token drawn with probability above p(x)/l), not the
      residual; this residual is the plainest reading and meets the guarantee.
      PARITY UNPINNED for the lenient residual (verify_row with lenience < 1):
      the pages fix the bound and the acceptance rate sum min(q, p/l), which
      are pinned, but nothing they print fixes the residual itself.
  R10 nucleus (top-p) keeps every token whose logit is >= that of the token at
      which the descending running probability first reaches top_p (ties kept);
      top_p >= 1 keeps everything.  A standardised row is the logit row with
      the dropped tokens set to -inf, so p is renormalised over the kept set.
"""
from __future__ import annotations

import numpy as np

BOUNDARY_EPS = 1e-5     # R8
Z_FLOOR = 1e-15         # R4, [p4] correction distribution


# ----------------------------------------------------------------------------- inputs

def widen(logits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of float32 logits, or of bfloat16 bit patterns (uint16)."""
    if dtype == "bf16":
        bits = np.asarray(logits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        with np.errstate(invalid="ignore"):   # NaN payloads widen to NaN
            return bits.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(logits, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def row_is_valid(logits: np.ndarray) -> bool:
    """R7: no NaN, no +inf, at least one finite entry."""
    return not (np.isnan(logits).any() or np.isposinf(logits).any() or np.isneginf(logits).all())


def softmax_t(logits: np.ndarray, T: float) -> np.ndarray:
    """Temperature standardisation [p1 §2.2]: p = softmax(logits / T).

    The max is subtracted before exp (a shift that leaves softmax unchanged);
    -inf logits get probability 0.
    """
    z = logits / T
    m = np.max(z)
    e = np.exp(z - m)
    return e / np.sum(e)


# ----------------------------------------------------------------------------- top-k / nucleus (R9, R10)

def topk_threshold(logits: np.ndarray, k: int) -> float:
    """Top-k standardisation [p1 §2.2]: keep the k largest probabilities, zero the rest, renormalise.

    Softmax is increasing in the logit, so the k largest probabilities are the k largest logits.  R9:
    the kept set is every token whose logit is >= tau, the k-th largest logit (ties at tau are all
    kept); tau = -inf (keep everything) when fewer than k logits are finite.
    """
    fin = np.sort(logits[np.isfinite(logits)])[::-1]
    if k > fin.size:
        return float("-inf")
    return float(fin[k - 1])


def topp_threshold(logits: np.ndarray, T: float, top_p: float):
    """Nucleus standardisation [p1 §2.2]: sort the probabilities descending, keep the shortest prefix
    whose cumulative mass reaches top_p, zero the rest, renormalise.

    R10: tau is the logit of the token at which the running mass first reaches top_p (ties at tau are
    all kept); tau = -inf when top_p >= 1.  Returns (tau, flagged): flagged when the running mass at
    that token or at the one before lies within 1e-5 of top_p, where float32 and float64 sums may pick
    different tokens (counted, like R8's boundary draws).
    """
    if top_p >= 1.0:
        return float("-inf"), False
    p = softmax_t(logits, T)
    order = np.argsort(-p, kind="stable")
    c = np.cumsum(p[order])
    j = int(np.searchsorted(c, top_p, side="left"))      # first running mass >= top_p
    j = min(j, p.size - 1)
    flagged = abs(c[j] - top_p) < BOUNDARY_EPS or (j > 0 and abs(c[j - 1] - top_p) < BOUNDARY_EPS)
    return float(logits[order[j]]), bool(flagged)


def apply_threshold(logits: np.ndarray, tau: float) -> np.ndarray:
    """Logits below tau become -inf (probability 0 after the softmax); NaN stays NaN."""
    out = np.array(logits, dtype=np.float64, copy=True)
    out[out < tau] = -np.inf
    return out


# ----------------------------------------------------------------------------- one row

def inverse_cdf(w: np.ndarray, u: float):
    """R2: token k = min{k : C_k > u*Z} over the running sum C of weights w, Z = sum(w).

    Returns (k, flagged) where flagged is R8's test on the normalised CDF edges.
    """
    Z = float(np.sum(w))
    C = np.cumsum(w)
    t = u * Z
    k = int(np.searchsorted(C, t, side="right"))
    if k >= w.shape[0]:
        k = int(np.nonzero(w > 0)[0][-1])
    lo = C[k - 1] if k > 0 else 0.0
    hi = C[k]
    flagged = abs(t - lo) / Z < BOUNDARY_EPS or abs(t - hi) / Z < BOUNDARY_EPS
    return k, bool(flagged)


def draw_boundary_probability(w: np.ndarray) -> float:
    """Probability, over a final uniform u ~ U[0, 1), that R8 flags the draw from weights w.

    The draw lands in cell k (normalised width c_k = w_k / Z) and is flagged when u lies within 1e-5 of
    one of that cell's two edges; both strips lie inside the cell, so cell k contributes min(c_k, 2e-5).
    """
    Z = float(np.sum(w))
    c = np.asarray(w, dtype=np.float64)[np.asarray(w) > 0] / Z
    return float(np.minimum(c, 2.0 * BOUNDARY_EPS).sum())


def accept_boundary_probability(r: float) -> float:
    """Probability, over u ~ U[0, 1), that an accept test with threshold r is flagged by R8: the length of
    [0, 1) within 1e-5 of r."""
    return max(0.0, min(1.0, r + BOUNDARY_EPS) - max(0.0, r - BOUNDARY_EPS))


def draw_candidates(w: np.ndarray, u: float) -> list[int]:
    """Tokens whose normalised CDF cell [C_{k-1}/Z, C_k/Z] (w_k > 0) lies within 1e-5 of u (R8).

    A draw flagged by R8 may land on any of these once the CDF is perturbed by
    less than 1e-5 of its total; the chosen token of inverse_cdf is always one.
    """
    Z = float(np.sum(w))
    C = np.cumsum(w) / Z
    lo = np.concatenate([[0.0], C[:-1]])
    ok = (w > 0) & (lo - BOUNDARY_EPS <= u) & (u <= C + BOUNDARY_EPS)
    return [int(k) for k in np.nonzero(ok)[0]]


def verify_row(tl: np.ndarray, dl: np.ndarray, ids: np.ndarray, gb: int, u: np.ndarray, T: float,
               lenience: float = 1.0):
    """Algorithm 1 Phases 3-4 for one row [p1 §2.3; p2 "The algorithm"; p3 §3].

    tl [gamma+1, V] and dl [gamma, V] float64 logits, ids [gamma], u [gamma+1]
    (column gamma is the final-draw uniform, R1), gb = draft_len of this row.
    Returns dict(emitted list of gamma+1 ints, n, boundary, valid).
    """
    gamma = dl.shape[0]
    V = tl.shape[1]
    bad = dict(emitted=[-1] * (gamma + 1), n=-1, boundary=False, valid=False, accept_boundary=False,
               candidates=[], flag_prob=0.0)
    if not (0 <= gb <= gamma):
        return bad
    for i in range(gb + 1):
        if not row_is_valid(tl[i]):
            return bad
    for i in range(gb):
        if not row_is_valid(dl[i]):
            return bad
        if not (0 <= int(ids[i]) < V):
            return bad
        if not (0.0 <= u[i] < 1.0):
            return bad
    if not (0.0 <= u[gamma] < 1.0):
        return bad

    p = [softmax_t(tl[i], T) for i in range(gb + 1)]
    q = [softmax_t(dl[i], T) for i in range(gb)]

    # Phase 3: walk the guesses left to right, stop at the first rejection.
    n = gb
    boundary = False
    flag_prob = 0.0       # expected R8 flags of this row had its tested uniforms been fresh draws
    for i in range(gb):
        x = int(ids[i])
        px, qx = p[i][x], q[i][x]
        lq = lenience * qx                         # R11: lenience scales q [p1 §5, Appendix A.5]
        r = 1.0 if px >= lq else px / lq          # min(1, p/q) [p1 §2.3 Phase 3]
        flag_prob += accept_boundary_probability(r)
        if abs(u[i] - r) < BOUNDARY_EPS:
            boundary = True
        if not (px > 0.0 and u[i] <= r):          # R3
            n = i
            break

    # Phase 4: residual on rejection, bonus from p_{gamma_b+1} otherwise.
    if n < gb:
        w = np.maximum(0.0, p[n] - lenience * q[n])  # norm(max(0, p - q)) [p1 Phase 4; p3 §3]; R11
        if np.sum(w) <= Z_FLOOR:                  # R4 [p4]
            w = p[n]
    else:
        w = p[gb]                                  # bonus t ~ p_{gamma+1} [p1 Phase 4]
    tok, flag = inverse_cdf(w, float(u[gamma]))
    flag_prob += draw_boundary_probability(w)
    accept_boundary = boundary
    boundary = boundary or flag
    emitted = [int(ids[i]) for i in range(n)] + [tok] + [-1] * (gamma - n)
    cands = draw_candidates(w, float(u[gamma])) if flag else [tok]
    return dict(emitted=emitted, n=n, boundary=boundary, valid=True, accept_boundary=accept_boundary,
                candidates=cands, flag_prob=flag_prob)


def greedy_row(tl: np.ndarray, ids: np.ndarray, gb: int, gamma: int):
    """Argmax standardisation [p1 §2.2; p2 "sampling temperature"]: R5."""
    V = tl.shape[1]
    bad = dict(emitted=[-1] * (gamma + 1), n=-1, valid=False)
    if not (0 <= gb <= gamma):
        return bad
    for i in range(gb + 1):
        if not row_is_valid(tl[i]):
            return bad
    for i in range(gb):
        if not (0 <= int(ids[i]) < V):
            return bad
    a = [int(np.argmax(tl[i])) for i in range(gb + 1)]   # np.argmax: first maximum
    n = gb
    for i in range(gb):
        if a[i] != int(ids[i]):
            n = i
            break
    emitted = [int(ids[i]) for i in range(n)] + [a[n]] + [-1] * (gamma - n)
    return dict(emitted=emitted, n=n, valid=True)


def stats_position(tl_i: np.ndarray, dl_i: np.ndarray, x: int, T: float):
    """Per-position diagnostics [p1 Def. 3.2, Lemma 3.3, Thm 3.5; p3 §3 proof].

    beta = sum_x min(p, q) (acceptance rate), resid = sum_x max(0, p - q),
    p(x), q(x) at the draft and accept_prob = min(1, p(x)/q(x)) (0 if p(x) = 0).
    Returns None when the position is invalid (R7).
    """
    V = tl_i.shape[0]
    if not (row_is_valid(tl_i) and row_is_valid(dl_i) and 0 <= x < V):
        return None
    p = softmax_t(tl_i, T)
    q = softmax_t(dl_i, T)
    px, qx = float(p[x]), float(q[x])
    if px <= 0.0:
        ap = 0.0
    else:
        ap = 1.0 if px >= qx else px / qx
    return dict(beta=float(np.sum(np.minimum(p, q))), resid=float(np.sum(np.maximum(0.0, p - q))),
                p_x=px, q_x=qx, accept_prob=ap)


# ----------------------------------------------------------------------------- batched

def _draft_len(draft_len, B, gamma):
    if draft_len is None:
        return np.full(B, gamma, dtype=np.int64)
    return np.asarray(draft_len, dtype=np.int64)


def verify_sample(target, draft, dtype, ids, draft_len, uniforms, T, rows=None, tthr=None, dthr=None,
                  lenience=1.0):
    """spec_verify_sample's contract, row by row.  target [B,gamma+1,V], draft [B,gamma,V].

    tthr [B,gamma+1] / dthr [B,gamma] (float32, optional) standardise each logit row first: logits
    below the row's threshold are dropped (top-k / nucleus, R9 / R10), as spec_verify_sample_masked.

    `rows` restricts the work to a subset of b (the outputs still have B rows;
    rows not computed hold -2).  Returns dict of numpy arrays: emitted
    [B,gamma+1] int64, n_accepted [B], boundary [B] bool, valid [B] bool, and
    flag_prob [B], the probability that R8 would flag the row if each tested
    uniform and the final one were fresh U[0, 1) draws (the expected boundary
    count of a batch is its sum).
    """
    B, G1, V = target.shape
    gamma = G1 - 1
    gl = _draft_len(draft_len, B, gamma)
    u = np.asarray(uniforms, dtype=np.float32).astype(np.float64)
    ids = np.asarray(ids)
    emitted = np.full((B, G1), -2, dtype=np.int64)
    n_acc = np.full(B, -2, dtype=np.int64)
    boundary = np.zeros(B, dtype=bool)
    accept_boundary = np.zeros(B, dtype=bool)
    valid = np.zeros(B, dtype=bool)
    flag_prob = np.zeros(B)
    candidates = {}
    for b in (range(B) if rows is None else rows):
        gb = int(gl[b])
        tb = widen(target[b], dtype)
        db = widen(draft[b], dtype) if gamma > 0 else np.zeros((0, V))
        if tthr is not None:
            tb = np.stack([apply_threshold(tb[i], float(np.float32(tthr[b][i]))) for i in range(G1)])
        if dthr is not None and gamma > 0:
            db = np.stack([apply_threshold(db[i], float(np.float32(dthr[b][i]))) for i in range(gamma)])
        res = verify_row(tb, db, ids[b], gb, u[b], float(np.float32(T)), float(np.float32(lenience)))
        emitted[b] = res["emitted"]
        n_acc[b] = res["n"]
        boundary[b] = res["boundary"]
        accept_boundary[b] = res["accept_boundary"]
        valid[b] = res["valid"]
        flag_prob[b] = res["flag_prob"]
        candidates[b] = res["candidates"]
    return dict(emitted=emitted, n_accepted=n_acc, boundary=boundary, accept_boundary=accept_boundary,
                valid=valid, candidates=candidates, flag_prob=flag_prob)


def sample_rows(logits, dtype, uniforms, T, rows=None, thr=None):
    """spec_sample_rows's contract: x ~ softmax(l / T) per row by R2's inverse CDF [p1 §2.3 Phase 1, §2.2].

    logits [R, V] (float32, or bfloat16 bits as uint16), uniforms [R].  Rows with an invalid logit row
    (R7) or a uniform outside [0, 1) get -1.  Returns tokens, boundary (R8) and candidates per row.
    """
    logits = np.asarray(logits)
    uniforms = np.asarray(uniforms)
    R = logits.shape[0]
    idx = range(R) if rows is None else rows
    out = {"tokens": np.full(R, -1, np.int64), "boundary": np.zeros(R, bool), "valid": np.zeros(R, bool),
           "candidates": {}}
    for r in idx:
        l = widen(logits[r], dtype)
        if thr is not None:
            l = apply_threshold(l, float(np.float32(thr[r])))
        u = float(uniforms[r])
        if not (row_is_valid(l) and 0.0 <= u < 1.0):
            continue
        w = softmax_t(l, T)
        k, flagged = inverse_cdf(w, u)
        out["tokens"][r] = k
        out["boundary"][r] = flagged
        out["valid"][r] = True
        if flagged:
            out["candidates"][r] = draw_candidates(w, u)
    return out


def verify_greedy(target, dtype, ids, draft_len, rows=None):
    """spec_verify_greedy's contract, row by row (R5)."""
    B, G1, V = target.shape
    gamma = G1 - 1
    gl = _draft_len(draft_len, B, gamma)
    ids = np.asarray(ids)
    emitted = np.full((B, G1), -2, dtype=np.int64)
    n_acc = np.full(B, -2, dtype=np.int64)
    valid = np.zeros(B, dtype=bool)
    for b in (range(B) if rows is None else rows):
        res = greedy_row(widen(target[b], dtype), ids[b], int(gl[b]), gamma)
        emitted[b] = res["emitted"]
        n_acc[b] = res["n"]
        valid[b] = res["valid"]
    return dict(emitted=emitted, n_accepted=n_acc, valid=valid)


STAT_KEYS = ("beta", "p_x", "q_x", "accept_prob", "resid")


def accept_stats(target, draft, dtype, ids, draft_len, T, rows=None):
    """spec_accept_stats's contract: per-position diagnostics [B, gamma]; NaN where not computed."""
    B, G1, V = target.shape
    gamma = G1 - 1
    gl = _draft_len(draft_len, B, gamma)
    ids = np.asarray(ids)
    out = {k: np.full((B, gamma), np.nan) for k in STAT_KEYS}
    valid = np.zeros((B, gamma), dtype=bool)
    for b in (range(B) if rows is None else rows):
        gb = int(gl[b])
        if not (0 <= gb <= gamma):
            continue
        for i in range(gb):
            s = stats_position(widen(target[b, i], dtype), widen(draft[b, i], dtype), int(ids[b, i]),
                               float(np.float32(T)))
            if s is None:
                continue
            valid[b, i] = True
            for k in STAT_KEYS:
                out[k][b, i] = s[k]
    out["valid"] = valid
    return out


# ----------------------------------------------------------------------------- closed forms

def exact_joint(p: np.ndarray, q: np.ndarray) -> dict:
    """Closed-form output law of one verification step with position-fixed distributions.

    p [gamma+1, V], q [gamma, V] probability rows.  From the A.1 argument [p1
    "Why This Procedure Preserves the Target Distribution"; p3 §3 proof]:
    accepting a_1..a_n has probability prod_j min(p_j(a_j), q_j(a_j)); after a
    rejection at n+1 the step emits c with probability max(0, p_{n+1}(c) -
    q_{n+1}(c)) (rejection mass times the normalised residual); after gamma
    acceptances the bonus c has probability p_{gamma+1}(c).  Keys are emitted
    token tuples.
    """
    gamma = q.shape[0]
    V = p.shape[1]
    out: dict = {}

    def rec(prefix, mass, i):
        if mass == 0.0:
            return
        if i == gamma:
            for c in range(V):
                if p[i][c] > 0:
                    out[tuple(prefix) + (c,)] = out.get(tuple(prefix) + (c,), 0.0) + mass * p[i][c]
            return
        for c in range(V):
            r = max(0.0, p[i][c] - q[i][c])
            if r > 0:
                out[tuple(prefix) + (c,)] = out.get(tuple(prefix) + (c,), 0.0) + mass * r
        for a in range(V):
            m = min(p[i][a], q[i][a])
            if m > 0:
                rec(prefix + [a], mass * m, i + 1)

    rec([], 1.0, 0)
    return out


def expected_tokens(alpha: float, gamma: int) -> float:
    """E[# tokens per step] = (1 - alpha^(gamma+1)) / (1 - alpha) [p1 §3.1 Eq. 1; p2]."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def walltime_improvement(alpha: float, gamma: int, c: float) -> float:
    """Thm 3.8 [p1 "Walltime Improvement Analysis"; p2; p3 §4]."""
    return expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def operations_factor(alpha: float, gamma: int, c_hat: float) -> float:
    """Thm 3.11 [p1 "Number of Arithmetic Operations"]."""
    return (gamma * c_hat + gamma + 1.0) / expected_tokens(alpha, gamma)


def optimal_gamma(alpha: float, c: float, max_gamma: int) -> int:
    """gamma* = argmax over gamma in 1..max_gamma of Thm 3.8's improvement [p1 §3.5 "Choosing gamma"],
    by evaluating every gamma as that section prescribes; ties go to the smaller gamma."""
    best, best_v = 1, walltime_improvement(alpha, 1, c)
    for g in range(2, max_gamma + 1):
        v = walltime_improvement(alpha, g, c)
        if v > best_v:
            best, best_v = g, v
    return best


def alpha_from_beta(beta) -> tuple[float, int]:
    """alpha = E[beta] over a corpus of positions [p1 Corollary 3.6]: the mean of the finite beta values
    (NaN marks positions that were not verified), and how many there were."""
    b = np.asarray(beta, dtype=np.float64).reshape(-1)
    b = b[np.isfinite(b)]
    return (float(b.mean()) if b.size else float("nan")), int(b.size)
