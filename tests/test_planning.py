"""Planning helpers of the C ABI: Eq. 1, Theorems 3.8 / 3.11, gamma* (§3.5) against the oracle and the
values the pages print (host functions: CPU); alpha = E[beta] (Corollary 3.6) as a device reduction (GPU)."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle as O
import speculative_decoding_verification_40_gb300 as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.split("#", 1)[0].strip()
            if ln:
                rows.append(ln.split())
    return rows


def test_expected_tokens_and_factors_match_the_oracle():
    rng = np.random.default_rng(11)
    for alpha, c in rng.random((200, 2)):
        for g in (0, 1, 3, 7, 20):
            assert S.expected_tokens(alpha, g) == pytest.approx(O.expected_tokens(alpha, g), rel=1e-14)
            assert S.walltime_improvement(alpha, g, c) == pytest.approx(O.walltime_improvement(alpha, g, c),
                                                                         rel=1e-14)
            assert S.operations_factor(alpha, g, c) == pytest.approx(O.operations_factor(alpha, g, c), rel=1e-14)
    assert S.expected_tokens(1.0, 5) == 6.0
    assert math.isnan(S.expected_tokens(1.5, 2)) and math.isnan(S.expected_tokens(0.5, -1))


@pytest.mark.parametrize("row", _rows("expected_tokens.txt"), ids=lambda r: f"a{r[0]}g{r[1]}")
def test_expected_tokens_match_pages(row):
    assert abs(S.expected_tokens(float(row[0]), int(row[1])) - float(row[2])) <= 0.005 + 1e-12


@pytest.mark.parametrize("row", _rows("table1_speed_ops.txt"), ids=lambda r: f"a{r[0]}g{r[1]}")
def test_table1(row):
    alpha, gamma = float(row[0]), int(row[1])
    assert abs(S.walltime_improvement(alpha, gamma, 0.0) - float(row[2])) <= 0.005 + 1e-12
    assert abs(S.operations_factor(alpha, gamma, 0.0) - float(row[3])) <= 0.005 + 1e-12


@pytest.mark.parametrize("row", _rows("speedup_examples.txt"), ids=lambda r: f"a{r[0]}g{r[1]}c{r[2]}")
def test_speedup_examples(row):
    alpha, gamma, c, printed, dec = float(row[0]), int(row[1]), float(row[2]), float(row[3]), int(row[4])
    assert abs(S.walltime_improvement(alpha, gamma, c) - printed) <= 0.5 * 10 ** -dec + 1e-12


@pytest.mark.parametrize("row", _rows("gamma_star.txt"), ids=lambda r: f"a{r[0]}c{r[1]}")
def test_optimal_gamma_matches_pages(row):
    g, v = S.optimal_gamma(float(row[0]), float(row[1]), 200)
    assert g == int(row[2])
    assert v == pytest.approx(O.walltime_improvement(float(row[0]), g, float(row[1])), rel=1e-14)


def test_optimal_gamma_matches_the_oracle_search():
    rng = np.random.default_rng(12)
    for alpha, c in rng.random((300, 2)):
        c *= 0.3
        assert S.optimal_gamma(alpha, c, 64)[0] == O.optimal_gamma(alpha, c, 64)
    with pytest.raises(ValueError):
        S.optimal_gamma(0.5, -0.1, 8)


@pytest.mark.gpu
def test_alpha_mean_on_the_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import workloads as W
    w = W.make(4, device="cuda")                    # ragged: NaN beta at padded positions
    st = S.accept_stats(w.target, w.draft, w.ids, w.T, w.draft_len)
    assert S.check_status() == 0
    a, n = S.alpha_mean(st["beta"])
    ra, rn = O.alpha_from_beta(st["beta"].cpu().numpy())
    assert n == rn == int(w.draft_len.sum())
    assert a == pytest.approx(ra, rel=1e-12)
    a, n = S.alpha_mean(torch.full((5,), float("nan"), device="cuda"))
    assert n == 0 and math.isnan(a)
    a, n = S.alpha_mean(torch.empty(0, device="cuda"))
    assert n == 0
