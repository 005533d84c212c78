"""Distributional tests of the CUDA path over 10^6 seeded draws (GPU).

The output law of one verification step is fixed by the pages: the first
emitted token has law p_1 for any draft distribution (the A.1 argument), the
number of emitted tokens has mean (1 - alpha^(gamma+1)) / (1 - alpha) when each
guess is accepted with probability alpha (Eq. 1), and the whole emitted tuple
follows the closed-form joint (oracle.exact_joint).  Every row of a call is an
independent step with its own uniforms.
"""
from __future__ import annotations

import numpy as np
import pytest
import scipy.stats
import torch

import oracle as O
from workloads.philox import uniform_f32

pytestmark = pytest.mark.gpu
N = 1_000_000
P_MIN = 1e-3


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


def _draws(S, p, q, seed, dtype=torch.float32):
    """N independent verification steps with position-fixed p [gamma+1, V], q [gamma, V]."""
    gamma, V = q.shape[0], p.shape[1]
    with np.errstate(divide="ignore"):
        lp, lq = np.log(p), np.log(q)
    t = torch.tensor(lp, dtype=torch.float32).to(dtype).cuda().unsqueeze(0).expand(N, gamma + 1, V).contiguous()
    d = torch.tensor(lq, dtype=torch.float32).to(dtype).cuda().unsqueeze(0).expand(N, gamma, V).contiguous()
    # drafts x_i ~ q_i by inverse CDF of independent uniforms (input generation, float64)
    ux = uniform_f32((N, gamma), seed, 11, "cuda").double()
    cq = torch.tensor(np.cumsum(q, axis=1), dtype=torch.float64, device="cuda")
    ids = torch.stack([torch.searchsorted(cq[i].contiguous(), ux[:, i].contiguous(), right=True)
                       for i in range(gamma)], 1).clamp_(max=V - 1).to(torch.int32) if gamma else \
        torch.zeros(N, 0, dtype=torch.int32, device="cuda")
    u = uniform_f32((N, gamma + 1), seed, 12, "cuda")
    em, na = S.verify_sample(t, d, ids.contiguous(), u, 1.0)
    assert S.check_status() == 0
    return em.cpu().numpy(), na.cpu().numpy()


def _chisq(counts, probs):
    """Chi-square p-value, merging cells with expected count < 5 into one."""
    counts = np.asarray(counts, dtype=np.float64)
    exp = np.asarray(probs, dtype=np.float64) * counts.sum()
    small = exp < 5
    if small.any():
        counts = np.append(counts[~small], counts[small].sum())
        exp = np.append(exp[~small], exp[small].sum())
        if exp[-1] == 0:
            assert counts[-1] == 0
            counts, exp = counts[:-1], exp[:-1]
    return scipy.stats.chisquare(counts, exp * counts.sum() / exp.sum()).pvalue


def test_first_token_law_is_p1(S):
    rng = np.random.default_rng(21)
    V, gamma = 16, 3
    p = rng.dirichlet(np.ones(V) * 0.7, size=gamma + 1)
    q = rng.dirichlet(np.ones(V) * 0.7, size=gamma)
    em, na = _draws(S, p, q, 1)
    counts = np.bincount(em[:, 0], minlength=V)
    assert _chisq(counts, p[0]) > P_MIN


def test_first_token_law_is_p1_for_disjoint_draft(S):
    V, gamma = 12, 2
    p = np.zeros((gamma + 1, V))
    q = np.zeros((gamma, V))
    p[:, :6] = np.array([0.3, 0.25, 0.2, 0.1, 0.1, 0.05])
    q[:, 6:] = 1.0 / 6
    em, na = _draws(S, p, q, 2)
    assert (na == 0).all()
    assert _chisq(np.bincount(em[:, 0], minlength=V), p[0]) > P_MIN


def test_expected_tokens_alpha_08_gamma_4(S):
    alpha, gamma = 0.8, 4
    p = np.tile([alpha, 1 - alpha], (gamma + 1, 1))
    q = np.tile([1.0, 0.0], (gamma, 1))
    em, na = _draws(S, p, q, 3)
    tokens = na.astype(np.float64) + 1.0
    exact = O.expected_tokens(alpha, gamma)       # 3.3616
    assert abs(exact - 3.3616) < 1e-12
    se = tokens.std() / np.sqrt(N)
    assert abs(tokens.mean() - exact) < 5 * se, (tokens.mean(), exact, se)
    # the number accepted is a geometric law truncated at gamma
    law = [alpha ** n * (1 - alpha) for n in range(gamma)] + [alpha ** gamma]
    assert _chisq(np.bincount(na, minlength=gamma + 1), law) > P_MIN


@pytest.mark.parametrize("V,gamma", [(2, 1), (3, 2), (4, 2), (4, 1)])
def test_joint_law_matches_closed_form(S, V, gamma):
    rng = np.random.default_rng(100 + 10 * V + gamma)
    p = rng.dirichlet(np.ones(V), size=gamma + 1)
    q = rng.dirichlet(np.ones(V), size=gamma)
    exact = O.exact_joint(p, q)
    keys = sorted(exact)
    em, na = _draws(S, p, q, 4 + V + gamma)
    index = {k: j for j, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for row_n, cnt in zip(*np.unique(np.concatenate([na[:, None], em], axis=1), axis=0, return_counts=True)):
        n = int(row_n[0])
        key = tuple(int(x) for x in row_n[1:n + 2])
        assert key in index, key
        counts[index[key]] += cnt
    assert _chisq(counts, [exact[k] for k in keys]) > P_MIN


def test_bf16_logits_law(S):
    """bf16 logits: the law is that of the bf16-rounded distributions."""
    rng = np.random.default_rng(5)
    V, gamma = 8, 2
    p = rng.dirichlet(np.ones(V), size=gamma + 1)
    q = rng.dirichlet(np.ones(V), size=gamma)
    pb = torch.softmax(torch.tensor(np.log(p), dtype=torch.float32).to(torch.bfloat16).double(), -1).numpy()
    em, na = _draws(S, p, q, 6, dtype=torch.bfloat16)
    assert _chisq(np.bincount(em[:, 0], minlength=V), pb[0]) > P_MIN
