"""Pins of the float64 oracle to what the pages and the mathematics fix (CPU only).

Each test ties the oracle to something other than itself: numbers printed on
the pages (tests/golden/), closed forms proved there, library routines, or a
black-box measurement of the oracle's own output law (tests/law.py) compared
with the closed-form law of the A.1 argument.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O
from law import all_small_cases, first_token_marginal, measure_law

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


def _run_row(tl, dl, ids, u):
    return O.verify_row(tl, dl, ids, dl.shape[0], u, 1.0)


# ----------------------------------------------------------------------------- exactness (A.1)

@pytest.mark.parametrize("case", list(all_small_cases()), ids=lambda c: f"V{c[0]}g{c[1]}")
def test_measured_law_equals_closed_form_joint(case):
    """Brute force over V <= 4, gamma <= 2: the oracle's law equals the A.1 closed form."""
    V, gamma, p, q = case
    law = measure_law(_run_row, p, q)
    exact = O.exact_joint(p, q)
    keys = set(law) | set(exact)
    err = max(abs(law.get(k, 0.0) - exact.get(k, 0.0)) for k in keys)
    assert err < 1e-12, (err, law, exact)
    assert abs(sum(law.values()) - 1.0) < 1e-12


@pytest.mark.parametrize("case", list(all_small_cases(seed=11)), ids=lambda c: f"V{c[0]}g{c[1]}")
def test_first_emitted_token_is_distributed_as_p1(case):
    """The theorem the pages prove: the first emitted token has law p_1, whatever q is."""
    V, gamma, p, q = case
    law = measure_law(_run_row, p, q)
    assert np.max(np.abs(first_token_marginal(law, V) - p[0])) < 1e-12


def test_disjoint_support_draft_still_gives_p():
    """Disjoint supports: nothing is ever accepted, beta = 0, and the emitted token still has law p."""
    p = np.array([[0.5, 0.5, 0.0, 0.0], [0.25, 0.25, 0.25, 0.25]])
    q = np.array([[0.0, 0.0, 0.3, 0.7]])
    law = measure_law(_run_row, p, q)
    assert all(len(k) == 1 for k in law)
    assert np.max(np.abs(first_token_marginal(law, 4) - p[0])) < 1e-14
    with np.errstate(divide="ignore"):
        s = O.stats_position(np.log(p[0]), np.log(q[0]), 2, 1.0)
    assert s["beta"] == 0.0 and abs(s["resid"] - 1.0) < 1e-15 and s["accept_prob"] == 0.0


def test_identical_distributions_accept_everything():
    """p == q: DLK = 0, beta = 1, every guess is accepted and the bonus comes from p_{gamma+1}."""
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(3), size=3)
    law = measure_law(_run_row, p, p[:2].copy())
    assert all(len(k) == 3 for k in law)
    s = O.stats_position(np.log(p[0]), np.log(p[0]), 1, 1.0)
    assert s["beta"] == pytest.approx(1.0, abs=1e-15) and s["resid"] == 0.0 and s["accept_prob"] == 1.0


# ----------------------------------------------------------------------------- acceptance rate (Thm 3.5)

def test_acceptance_rate_is_overlap_and_one_minus_tv():
    """Measured P(accept first guess) = sum min(p, q) = 1 - DLK = 1 - (1/2) sum |p - q|."""
    rng = np.random.default_rng(5)
    for V in (2, 3, 4):
        for _ in range(5):
            p = rng.dirichlet(np.ones(V), size=2)
            q = rng.dirichlet(np.ones(V), size=1)
            law = measure_law(_run_row, p, q)
            accept = sum(v for k, v in law.items() if len(k) == 2)
            s = O.stats_position(np.log(p[0]), np.log(q[0]), 0, 1.0)
            tv = 0.5 * np.sum(np.abs(p[0] - q[0]))
            mid = 0.5 * (p[0] + q[0])
            dlk = np.sum(np.abs(p[0] - mid))          # Definition 3.2
            assert accept == pytest.approx(s["beta"], abs=1e-12)
            assert s["beta"] == pytest.approx(1.0 - tv, abs=1e-14)
            assert s["beta"] == pytest.approx(1.0 - dlk, abs=1e-14)
            assert s["resid"] == pytest.approx(tv, abs=1e-14)


def test_per_position_accept_probability_is_min_one_ratio():
    """Measured acceptance threshold of one draft = min(1, p(x)/q(x)) (Phase 3)."""
    p = np.array([[0.1, 0.2, 0.3, 0.4], [0.25] * 4])
    q = np.array([[0.4, 0.1, 0.3, 0.2]])
    with np.errstate(divide="ignore"):
        tl, dl = np.log(p), np.log(q)
    for x in range(4):
        lo, hi = 0.0, 1.0
        for _ in range(60):
            mid = 0.5 * (lo + hi)
            n = O.verify_row(tl, dl, np.array([x]), 1, np.array([mid, 0.5]), 1.0)["n"]
            lo, hi = (mid, hi) if n == 1 else (lo, mid)
        assert lo == pytest.approx(min(1.0, p[0, x] / q[0, x]), abs=1e-12)


def test_two_token_example():
    rows = {r[0]: r[1:] for r in _rows("two_token_example.txt")}
    p = np.array([[float(rows["A"][0]), float(rows["B"][0])], [0.5, 0.5]])
    q = np.array([[float(rows["A"][1]), float(rows["B"][1])]])
    law = measure_law(_run_row, p, q)
    accept = sum(v for k, v in law.items() if len(k) == 2)
    assert accept == pytest.approx(float(rows["acceptance"][0]), abs=1e-12)
    corrected = {k: v for k, v in law.items() if len(k) == 1}
    assert set(corrected) == {(0,)}                 # every rejection is corrected to A
    assert np.max(np.abs(first_token_marginal(law, 2) - p[0])) < 1e-12


# ----------------------------------------------------------------------------- E[# tokens] (Eq. 1)

def _measured_expected_tokens(alpha, gamma):
    """p_i = (alpha, 1 - alpha), q_i = one-hot(0): every guess is accepted with probability alpha."""
    p = np.tile([alpha, 1.0 - alpha], (gamma + 1, 1))
    q = np.tile([1.0, 0.0], (gamma, 1))
    law = measure_law(_run_row, p, q)
    return sum(len(k) * v for k, v in law.items())


@pytest.mark.parametrize("row", _rows("expected_tokens.txt"), ids=lambda r: f"a{r[0]}g{r[1]}")
def test_expected_tokens_match_pages(row):
    alpha, gamma, printed = float(row[0]), int(row[1]), float(row[2])
    e = _measured_expected_tokens(alpha, gamma)
    assert e == pytest.approx(O.expected_tokens(alpha, gamma), abs=1e-12)
    assert abs(e - printed) <= 0.005 + 1e-12


def test_expected_tokens_alpha_08_gamma_4_is_33616():
    assert _measured_expected_tokens(0.8, 4) == pytest.approx(3.3616, abs=1e-12)


@pytest.mark.parametrize("row", _rows("table1_speed_ops.txt"), ids=lambda r: f"a{r[0]}g{r[1]}")
def test_table1_speed_and_operations(row):
    alpha, gamma, speed, ops = float(row[0]), int(row[1]), float(row[2]), float(row[3])
    assert abs(O.walltime_improvement(alpha, gamma, 0.0) - speed) <= 0.005 + 1e-12
    assert abs(O.operations_factor(alpha, gamma, 0.0) - ops) <= 0.005 + 1e-12
    assert O.walltime_improvement(alpha, gamma, 0.0) == pytest.approx(_measured_expected_tokens(alpha, gamma),
                                                                      abs=1e-12)


@pytest.mark.parametrize("row", _rows("speedup_examples.txt"), ids=lambda r: f"a{r[0]}g{r[1]}c{r[2]}")
def test_speedup_examples(row):
    alpha, gamma, c, printed, dec = float(row[0]), int(row[1]), float(row[2]), float(row[3]), int(row[4])
    assert abs(O.walltime_improvement(alpha, gamma, c) - printed) <= 0.5 * 10 ** -dec + 1e-12


# ----------------------------------------------------------------------------- standardisation

def test_softmax_matches_scipy():
    rng = np.random.default_rng(0)
    for T in (0.3, 0.7, 1.0, 2.5):
        l = rng.normal(0, 4, size=1000)
        l[::17] = -np.inf
        np.testing.assert_allclose(O.softmax_t(l, T), scipy.special.softmax(l / T), rtol=1e-13, atol=0)


def test_bf16_widening_matches_torch_on_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ours = O.widen(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_greedy_is_sampling_with_one_hot_standardisation():
    """Argmax standardisation: greedy verification equals sampling with one-hot p and q."""
    rng = np.random.default_rng(9)
    for trial in range(200):
        V, gamma = int(rng.integers(2, 9)), int(rng.integers(0, 5))
        tl = np.round(rng.normal(0, 1, size=(gamma + 1, V)), 1)   # rounding makes ties common
        dl = np.where(rng.random((gamma, V)) < 0.5, tl[:gamma], rng.normal(0, 1, size=(gamma, V)))
        ids = np.array([int(np.argmax(d)) for d in dl], dtype=np.int64)
        g = O.greedy_row(tl, ids, gamma, gamma)
        with np.errstate(divide="ignore"):
            tp = np.log(np.eye(V)[[int(np.argmax(t)) for t in tl]])
            dq = np.log(np.eye(V)[ids]) if gamma else np.zeros((0, V))
        u = rng.random(gamma + 1) * 0.999
        s = O.verify_row(tp, dq, ids, gamma, u, 1.0)
        assert s["emitted"] == g["emitted"] and s["n"] == g["n"]


def test_greedy_lowest_index_tie_break():
    tl = np.array([[1.0, 3.0, 3.0, 0.0], [5.0, 5.0, -np.inf, 5.0]])
    g = O.greedy_row(tl, np.array([2]), 1, 1)
    assert g["n"] == 0 and g["emitted"] == [1, -1]
    g = O.greedy_row(tl, np.array([1]), 1, 1)
    assert g["n"] == 1 and g["emitted"] == [1, 0]


def test_temperature_zero_limit_of_sampling_is_greedy():
    """As T -> 0 the temperature softmax tends to the argmax one-hot, so sampling tends to greedy."""
    rng = np.random.default_rng(2)
    for _ in range(50):
        V, gamma = 6, 3
        tl = rng.normal(0, 1, size=(gamma + 1, V))
        dl = tl[:gamma] + rng.normal(0, 0.3, size=(gamma, V))
        ids = np.argmax(dl, axis=1)
        g = O.greedy_row(tl, ids, gamma, gamma)
        s = O.verify_row(tl, dl, ids, gamma, np.full(gamma + 1, 0.5), 1e-3)
        assert s["emitted"] == g["emitted"]


# ----------------------------------------------------------------------------- inverse CDF, readings

def test_inverse_cdf_gamma_zero_is_plain_sampling_from_p():
    """gamma = 0 degenerates to one inverse-CDF draw from p_1: the measured law is p_1."""
    p = np.array([[0.1, 0.0, 0.45, 0.45]])
    law = measure_law(_run_row, p, np.zeros((0, 4)))
    m = first_token_marginal(law, 4)
    np.testing.assert_allclose(m, p[0], atol=1e-14)


def test_inverse_cdf_picks_smallest_index_with_cdf_above_target():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    assert O.inverse_cdf(w, 0.0)[0] == 1
    assert O.inverse_cdf(w, 0.3)[0] == 3
    assert O.inverse_cdf(w, 0.9)[0] == 4
    assert O.inverse_cdf(w, 0.999999999)[0] == 4
    k, flag = O.inverse_cdf(w, 0.25)       # exactly on an edge: lands right of it, and is flagged
    assert k == 3 and flag


def test_boundary_flags():
    p = np.array([[0.3, 0.7], [0.5, 0.5]])
    q = np.array([[0.6, 0.4]])
    tl, dl = np.log(p), np.log(q)
    r = 0.5   # min(1, 0.3/0.6)
    near = O.verify_row(tl, dl, np.array([0]), 1, np.array([r + 5e-6, 0.3]), 1.0)
    far = O.verify_row(tl, dl, np.array([0]), 1, np.array([r + 5e-3, 0.3]), 1.0)
    assert near["boundary"] and not far["boundary"]
    # residual is (0, 0.3) normalised to (0, 1): u_f anywhere leads to token 1; edges at 0 and 1
    assert far["emitted"] == [1, -1]
    edge = O.verify_row(tl, dl, np.array([0]), 1, np.array([r + 5e-3, 2e-6]), 1.0)
    assert edge["boundary"]


def test_degenerate_residual_falls_back_to_p():
    """R4: residual mass <= 1e-15 -> draw from p [interactiveml correction distribution]."""
    tl = np.log(np.array([[0.5, 0.5], [0.5, 0.5]]))
    dl = tl[:1] + np.array([[1e-15, 0.0]])     # q(0) exceeds p(0) by ~2.5e-16: Z ~ 2.5e-16
    s = O.stats_position(tl[0], dl[0], 0, 1.0)
    assert 0.0 < s["resid"] <= O.Z_FLOOR and s["accept_prob"] < 1.0
    u_reject = float(np.nextafter(1.0, 0.0))
    # the residual alone would put all its mass on token 1; the fallback to p sends u_f = 0.25 to token 0
    s = O.verify_row(tl, dl, np.array([0]), 1, np.array([u_reject, 0.25]), 1.0)
    assert s["n"] == 0 and s["emitted"] == [0, -1]


def test_zero_probability_draft_never_accepted():
    tl = np.log(np.array([[0.0, 1.0], [0.5, 0.5]]))
    dl = np.log(np.array([[0.0, 1.0]]))
    s = O.verify_row(tl, dl, np.array([0]), 1, np.array([0.0, 0.5]), 1.0)
    assert s["n"] == 0 and s["emitted"] == [1, -1]


def test_invalid_rows_and_ignored_padding():
    V, gamma = 5, 3
    rng = np.random.default_rng(1)
    tl = rng.normal(size=(gamma + 1, V))
    dl = rng.normal(size=(gamma, V))
    ids = np.array([1, 2, 3])
    u = np.array([0.1, 0.2, 0.3, 0.4])
    assert O.verify_row(tl, dl, ids, gamma, u, 1.0)["valid"]
    for mutate in ("nan", "posinf", "allneg", "id", "u", "ulast", "len"):
        t, d, x, uu, gb = tl.copy(), dl.copy(), ids.copy(), u.copy(), gamma
        if mutate == "nan":
            t[1, 2] = np.nan
        elif mutate == "posinf":
            d[0, 0] = np.inf
        elif mutate == "allneg":
            t[3] = -np.inf
        elif mutate == "id":
            x[1] = V
        elif mutate == "u":
            uu[0] = 1.0
        elif mutate == "ulast":
            uu[gamma] = -0.1
        elif mutate == "len":
            gb = gamma + 1
        r = O.verify_row(t, d, x, gb, uu, 1.0)
        assert not r["valid"] and r["n"] == -1 and r["emitted"] == [-1] * (gamma + 1), mutate
    # ragged row of length 1: padded rows, ids and uniforms are never read
    t, d, x, uu = tl.copy(), dl.copy(), ids.copy(), u.copy()
    t[2:] = np.nan
    d[1:] = np.nan
    x[1:] = -1
    uu[1:gamma] = np.nan
    r = O.verify_row(t, d, x, 1, uu, 1.0)
    assert r["valid"] and 0 <= r["n"] <= 1 and r["emitted"][r["n"] + 1:] == [-1] * (gamma - r["n"])


def test_batched_wrappers_match_rows():
    rng = np.random.default_rng(4)
    B, gamma, V = 6, 3, 17
    t = rng.normal(size=(B, gamma + 1, V)).astype(np.float32)
    d = (t[:, :gamma] + rng.normal(size=(B, gamma, V))).astype(np.float32)
    ids = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    gl = np.array([3, 0, 1, 2, 3, 3], dtype=np.int32)
    u = rng.random((B, gamma + 1)).astype(np.float32)
    out = O.verify_sample(t, d, "f32", ids, gl, u, 0.9)
    for b in range(B):
        r = O.verify_row(t[b].astype(np.float64), d[b].astype(np.float64), ids[b], int(gl[b]),
                         u[b].astype(np.float64), float(np.float32(0.9)))
        assert list(out["emitted"][b]) == r["emitted"] and out["n_accepted"][b] == r["n"]
    g = O.verify_greedy(t, "f32", ids, gl)
    st = O.accept_stats(t, d, "f32", ids, gl, 0.9)
    for b in range(B):
        r = O.greedy_row(t[b].astype(np.float64), ids[b], int(gl[b]), gamma)
        assert list(g["emitted"][b]) == r["emitted"]
        for i in range(gamma):
            if i < gl[b]:
                assert np.isfinite(st["beta"][b, i])
            else:
                assert np.isnan(st["beta"][b, i])


def test_draw_candidates_cover_the_near_edge_tokens():
    w = np.array([0.5, 1e-7, 0.0, 0.4999999, 1e-6])
    Z = w.sum()
    u = 0.5 / Z                       # exactly the upper edge of token 0
    c = O.draw_candidates(w, u)
    assert 0 in c and 1 in c and 3 in c and 2 not in c
    k, flag = O.inverse_cdf(w, u)
    assert flag and k in c
    assert O.draw_candidates(w, 0.25) == [0]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_boundary_probability_is_the_flagged_fraction_of_uniforms(seed):
    """R8's expected flag rate, checked by brute force: over a fine stratified grid of final uniforms, the
    fraction that inverse_cdf flags equals draw_boundary_probability (cells wider and narrower than the
    2e-5 band, zero weights, a dominant token), and over accept uniforms the fraction within 1e-5 of r
    equals accept_boundary_probability (r inside, at 1, near 0)."""
    rng = np.random.default_rng(seed)
    w = np.concatenate([rng.random(6), rng.random(40) * 1e-6, [0.0, 0.0], [3.0]])
    rng.shuffle(w)
    N = 400_000
    u = (np.arange(N) + 0.5) / N
    Z = w.sum()
    C = np.cumsum(w)
    k = np.searchsorted(C, u * Z, side="right")
    lo = np.where(k > 0, C[np.maximum(k - 1, 0)], 0.0)
    hi = C[np.minimum(k, w.size - 1)]
    flagged = (np.abs(u * Z - lo) / Z < O.BOUNDARY_EPS) | (np.abs(u * Z - hi) / Z < O.BOUNDARY_EPS)
    # the vectorised test above is inverse_cdf's own flag; spot-check that on a few uniforms
    for j in range(0, N, N // 50):
        assert O.inverse_cdf(w, float(u[j]))[1] == bool(flagged[j])
    assert flagged.mean() == pytest.approx(O.draw_boundary_probability(w), abs=3.0 / N)
    for r in (0.5, 1.0, 3e-6, 0.0, 0.99999):
        frac = (np.abs(u - r) < O.BOUNDARY_EPS).mean()
        assert frac == pytest.approx(O.accept_boundary_probability(r), abs=3.0 / N)


def test_boundary_probability_of_a_row_sums_its_tested_positions():
    """verify_row's flag_prob: one accept band per tested position (up to and including the first
    rejection) plus the final draw's band mass."""
    p = np.array([[0.3, 0.7], [0.5, 0.5]])
    q = np.array([[0.6, 0.4]])
    tl, dl = np.log(p), np.log(q)
    rej = O.verify_row(tl, dl, np.array([0]), 1, np.array([0.9, 0.3]), 1.0)     # rejected: residual (0, 1)
    assert rej["n"] == 0
    assert rej["flag_prob"] == pytest.approx(2e-5 + min(1.0, 2e-5))
    acc = O.verify_row(tl, dl, np.array([0]), 1, np.array([0.1, 0.3]), 1.0)     # accepted: bonus (0.5, 0.5)
    assert acc["n"] == 1
    assert acc["flag_prob"] == pytest.approx(2e-5 + 4e-5)


# ----------------------------------------------------------------------------- draft-side sampler

def _stratified(N):
    return ((np.arange(N) + 0.5) / N).astype(np.float64)


@pytest.mark.parametrize("T", [1.0, 2.0, 0.5])
def test_sample_rows_stratified_uniforms_reproduce_the_softmax(T):
    """Inverse CDF over a stratified grid u_j = (j + 1/2)/N hits token k floor- or ceil(N p_k) times,
    with p_k = w_k^(1/T) / sum w^(1/T) for logits log w (closed form, not the oracle's softmax)."""
    wts = np.array([1.0, 4.0, 0.5, 2.5, 0.0, 8.0, 1e-3])
    with np.errstate(divide="ignore"):
        l = np.log(wts).astype(np.float32)
    N = 20000
    R = N
    logits = np.tile(l, (R, 1))
    out = O.sample_rows(logits, "f32", _stratified(N), T)
    counts = np.bincount(out["tokens"], minlength=wts.size)
    pw = wts ** (1.0 / T)
    p = pw / pw.sum()
    assert counts[4] == 0                                # zero weight is never drawn
    assert np.all(np.abs(counts - N * p) <= 1.0 + 1e-6 * N), (counts, N * p)


def test_sample_rows_edges():
    l = np.array([[0.0, 0.0, -np.inf, 0.0],              # u = 0 draws the first positive weight
                  [0.0, 0.0, -np.inf, 0.0],              # u just below 1 draws the last positive weight
                  [np.nan, 0.0, 0.0, 0.0],               # invalid row
                  [-np.inf] * 4,                         # all -inf: invalid
                  [0.0, 1.0, 2.0, 3.0]], dtype=np.float32)
    u = np.array([0.0, np.nextafter(np.float32(1), np.float32(0)), 0.5, 0.5, 1.0], dtype=np.float32)
    out = O.sample_rows(l, "f32", u, 1.0)
    assert list(out["tokens"]) == [0, 3, -1, -1, -1]     # u = 1 is outside [0, 1)


def test_sample_rows_is_the_bonus_draw_of_verification():
    """gamma = 0 verification emits exactly the sampler's draw (same inverse CDF, same uniform)."""
    rng = np.random.default_rng(7)
    l = rng.normal(0, 2, size=(6, 50)).astype(np.float32)
    u = rng.random(6).astype(np.float32)
    out = O.sample_rows(l, "f32", u, 0.8)
    ver = O.verify_sample(l[:, None, :], np.zeros((6, 0, 50), np.float32), "f32", np.zeros((6, 0), np.int64),
                          None, u[:, None], 0.8)
    assert list(out["tokens"]) == [int(e[0]) for e in ver["emitted"]]


# ----------------------------------------------------------------------------- gamma* (§3.5) and alpha (Cor. 3.6)

@pytest.mark.parametrize("row", _rows("gamma_star.txt"), ids=lambda r: f"a{r[0]}c{r[1]}")
def test_optimal_gamma_matches_pages(row):
    alpha, c, g = float(row[0]), float(row[1]), int(row[2])
    assert O.optimal_gamma(alpha, c, 200) == g


def test_gamma_one_improvement_is_corollary_39():
    """Cor. 3.9: at gamma = 1 the improvement factor is (1 + alpha)/(1 + c)."""
    rng = np.random.default_rng(4)
    for alpha, c in rng.random((50, 2)):
        assert O.walltime_improvement(alpha, 1, c) == pytest.approx((1 + alpha) / (1 + c), rel=1e-13)


def test_optimal_gamma_without_draft_cost_is_the_cap():
    """c = 0: the factor grows with gamma for alpha < 1, so the search returns its upper end."""
    for alpha in (0.3, 0.8, 0.95):
        assert O.optimal_gamma(alpha, 0.0, 17) == 17


def test_alpha_is_the_mean_of_finite_beta():
    b = np.array([[0.5, 0.7, np.nan], [0.9, np.nan, np.nan]])
    a, n = O.alpha_from_beta(b)
    assert n == 3 and a == pytest.approx(0.7, abs=1e-15)
    a, n = O.alpha_from_beta(np.full(4, np.nan))
    assert n == 0 and np.isnan(a)


# ----------------------------------------------------------------------------- top-k / nucleus (R9, R10)

def test_topk_threshold_brute_force_and_ties():
    l = np.array([3.0, 1.0, 3.0, 2.0, -np.inf])
    assert O.topk_threshold(l, 1) == 3.0 and O.topk_threshold(l, 2) == 3.0      # the tie at 3 is kept
    assert O.topk_threshold(l, 3) == 2.0 and O.topk_threshold(l, 4) == 1.0
    assert O.topk_threshold(l, 5) == -np.inf                                       # fewer finite logits
    rng = np.random.default_rng(8)
    for _ in range(200):
        v = rng.normal(0, 3, rng.integers(1, 60))
        k = int(rng.integers(1, v.size + 2))
        tau = O.topk_threshold(v, k)
        kept = np.count_nonzero(v >= tau)
        assert kept == min(k, v.size)                                # no ties in continuous draws
        assert np.all(np.sort(v)[::-1][:min(k, v.size)] >= tau)


def test_topp_threshold_worked_values():
    p = np.array([0.5, 0.3, 0.15, 0.05])
    l = np.log(p)
    assert O.topp_threshold(l, 1.0, 0.7) == (pytest.approx(np.log(0.3)), False)   # keep {0.5, 0.3}
    assert O.topp_threshold(l, 1.0, 0.81)[0] == pytest.approx(np.log(0.15))        # keep three
    assert O.topp_threshold(l, 1.0, 0.5)[0] == pytest.approx(np.log(0.5))          # the top token reaches it
    tau, flagged = O.topp_threshold(l, 1.0, 0.8)                                   # 0.5 + 0.3 hits 0.8
    assert flagged
    assert O.topp_threshold(l, 1.0, 1.0) == (-np.inf, False)


def test_topp_threshold_invariants():
    rng = np.random.default_rng(9)
    for _ in range(200):
        l = rng.normal(0, 2, 40)
        T, top_p = float(rng.uniform(0.5, 2)), float(rng.uniform(0.05, 0.99))
        tau, flagged = O.topp_threshold(l, T, top_p)
        p = O.softmax_t(l, T)
        kept = p[l >= tau].sum()
        assert kept >= top_p - 1e-12                                 # the kept mass reaches top_p
        assert kept - p[l == tau].sum() < top_p + 1e-12              # without the boundary token it does not


def test_top1_standardised_sampling_is_greedy_verification():
    """Top-k with k = 1 on both sides turns p and q into one-hot argmax distributions [p1 §2.2], so
    speculative sampling accepts exactly the guesses greedy verification accepts."""
    rng = np.random.default_rng(10)
    B, gamma, V = 40, 4, 30
    t = rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
    d = (t[:, :gamma] + rng.normal(0, 1.5, (B, gamma, V))).astype(np.float32)
    ids = np.argmax(d, axis=2)
    tthr = np.array([[O.topk_threshold(t[b, i].astype(np.float64), 1) for i in range(gamma + 1)]
                     for b in range(B)], dtype=np.float32)
    dthr = np.array([[O.topk_threshold(d[b, i].astype(np.float64), 1) for i in range(gamma)]
                     for b in range(B)], dtype=np.float32)
    u = rng.random((B, gamma + 1)).astype(np.float32)
    s = O.verify_sample(t, d, "f32", ids, None, u, 1.0, tthr=tthr, dthr=dthr)
    g = O.verify_greedy(t, "f32", ids, None)
    assert np.array_equal(s["emitted"], g["emitted"]) and np.array_equal(s["n_accepted"], g["n_accepted"])


def test_thresholded_sampler_draws_from_the_truncated_softmax():
    wts = np.array([1.0, 4.0, 0.5, 2.5, 8.0, 0.2])
    l = np.log(wts)
    tau = O.topk_threshold(l, 3)                                    # keeps 8, 4, 2.5
    N = 14500
    out = O.sample_rows(np.tile(l.astype(np.float32), (N, 1)), "f32", _stratified(N), 1.0,
                        thr=np.full(N, tau, np.float32))
    counts = np.bincount(out["tokens"], minlength=wts.size)
    keep = wts >= 2.5
    p = np.where(keep, wts, 0) / wts[keep].sum()
    assert np.all(np.abs(counts - N * p) <= 1.0 + 1e-9)


# ----------------------------------------------------------------------------- lenience (R11)

def _lenient_run(l):
    def run(tl, dl, ids, u):
        return O.verify_row(tl, dl, ids, dl.shape[0], u, 1.0, lenience=l)
    return run


@pytest.mark.parametrize("l", [0.1, 0.5, 0.9])
@pytest.mark.parametrize("case", list(all_small_cases(seed=13))[::2], ids=lambda c: f"V{c[0]}g{c[1]}")
def test_lenience_keeps_the_pages_bound(case, l):
    """[p1] Appendix A.5 as restated in §5: with lenience l no token is drawn with probability above
    p(x)/l; the first guess is accepted with probability sum_x min(q(x), p(x)/l) (q multiplied by l
    before the comparison)."""
    V, gamma, p, q = case
    law = measure_law(_lenient_run(l), p, q)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    first = first_token_marginal(law, V)
    assert np.all(first <= p[0] / l + 1e-12), (first, p[0] / l)
    if gamma >= 1:
        accept = sum(v for k, v in law.items() if len(k) >= 2)
        assert accept == pytest.approx(np.minimum(q[0], p[0] / l).sum(), abs=1e-12)


@pytest.mark.parametrize("l", [0.1, 0.5, 0.9])
@pytest.mark.parametrize("case", list(all_small_cases(seed=13))[::2], ids=lambda c: f"V{c[0]}g{c[1]}")
def test_lenient_residual_consistency_not_a_pin(case, l):
    """Consistency check, not a pin: the pages state the scaled comparison and the p(x)/l bound but
    not the residual drawn after a lenient rejection, so R11's norm(max(0, p - l q)) rests on a
    reading.  This only checks that the oracle's measured first-token law is the one that reading
    implies (accepted mass min(q, p/l), the rejection mass spread over the normalised residual);
    it restates the reading's formula and cannot show the reading itself is the pages'."""
    V, gamma, p, q = case
    if gamma < 1:
        return
    first = first_token_marginal(measure_law(_lenient_run(l), p, q), V)
    acc = np.minimum(q[0], p[0] / l)
    resid = np.maximum(0.0, p[0] - l * q[0])
    R = 1.0 - acc.sum()
    expect = acc + (R * resid / resid.sum() if resid.sum() > 0 else 0.0)
    assert np.max(np.abs(first - expect)) < 1e-12


def test_lenience_one_is_the_exact_method():
    for V, gamma, p, q in list(all_small_cases(seed=17))[:6]:
        assert measure_law(_lenient_run(1.0), p, q) == measure_law(_run_row, p, q)
