"""Draft-side sampler (spec_sample_rows) vs the float64 oracle, and its output law (GPU).

x ~ softmax(l / T) per row by the inverse CDF of one uniform: token-exact
against the oracle outside counted boundary draws (a draw within 1e-5 of a CDF
edge must be one of the oracle's candidates), and over 10^6 rows the drawn
tokens follow q (chi-square).
"""
from __future__ import annotations

import numpy as np
import pytest
import scipy.stats
import torch

import oracle as O
import workloads as W
from workloads.philox import normal_f32, uniform_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


def _compare(logits, u, T, tokens, rows=None):
    """(compared, boundary rows, mismatches) of the GPU tokens against the oracle."""
    dt = "bf16" if logits.dtype == torch.bfloat16 else "f32"
    ref = O.sample_rows(W.logits_as_numpy(logits), dt, u.cpu().numpy(), T, rows=rows)
    tok = tokens.cpu().numpy()
    mism, flagged, n = [], [], 0
    for r in (range(logits.shape[0]) if rows is None else rows):
        n += 1
        if ref["boundary"][r]:
            flagged.append(r)
            if int(tok[r]) not in ref["candidates"][r]:
                mism.append((r, int(tok[r]), ref["candidates"][r]))
            continue
        if int(tok[r]) != int(ref["tokens"][r]):
            mism.append((r, int(tok[r]), int(ref["tokens"][r])))
    return n, flagged, mism


@pytest.mark.parametrize("k", [0, 1, 2, 3, 4])
def test_sampler_parity_on_the_draft_rows(S, k):
    w = W.make(k, device="cuda", with_ids=False)
    logits, u = W.sampler_rows(w)
    tok = S.sample_rows(logits, u, w.T)
    assert S.check_status() == 0
    R = logits.shape[0]
    rows = None if R <= 64 else sorted(set(np.random.default_rng(k).choice(R, 96, replace=False).tolist()) |
                                       {0, R - 1})
    n, flagged, mism = _compare(logits, u, w.T, tok, rows)
    print(f"{w.name}: {n} rows compared, {len(flagged)} boundary draws")
    assert not mism, mism[:5]
    assert len(flagged) <= n // 4 + 1
    t = tok.cpu().numpy()
    assert t.min() >= 0 and t.max() < w.V


@pytest.mark.parametrize("R,V,dtype,offset", [
    (7, 1, "f32", 0),
    (9, 130, "bf16", 0),
    (5, 50001, "f32", 0),           # V*4 not a multiple of 16: scalar loads
    (5, 50001, "bf16", 1),          # rows off a 16-byte boundary
    (6, 77777, "bf16", 0),
    (3, 262144, "f32", 0),          # largest vocabulary: 16 slices
    (3, 262144, "bf16", 0),
    (300, 4096, "f32", 0),
])
def test_sampler_odd_sizes(S, R, V, dtype, offset):
    g = 3.0 * normal_f32((R * V + offset,), 77, R + V, "cuda")
    if dtype == "bf16":
        g = g.to(torch.bfloat16)
    logits = g[offset:].view(R, V)
    if offset:
        assert logits.data_ptr() % 16 != 0      # rows start off the 16-byte boundary
    u = uniform_f32((R,), 5, V, "cuda")
    tok = S.sample_rows(logits, u, 0.9)
    assert S.check_status() == 0
    n, flagged, mism = _compare(logits, u, 0.9, tok)
    assert not mism, mism[:5]


def test_sampler_invalid_rows_and_edges(S):
    V = 1000
    l = normal_f32((6, V), 3, 1, "cuda") * 2.0
    l[1, 17] = float("nan")
    l[2, :] = float("-inf")
    l[3, 5] = float("inf")
    u = torch.tensor([0.3, 0.3, 0.3, 0.3, 0.0, 1.0], device="cuda")
    tok = S.sample_rows(l.contiguous(), u, 1.0).cpu().tolist()
    code = S.check_status(raise_on_error=False)
    assert tok[1] == tok[2] == tok[3] == tok[5] == -1
    assert code == 1                          # lowest status recorded: a uniform outside [0, 1)
    ref = O.sample_rows(l.cpu().numpy(), "f32", u.cpu().numpy(), 1.0)
    assert tok[0] == ref["tokens"][0] and tok[4] == ref["tokens"][4]
    # only NaN / inf rows now: the recorded status is the non-finite one
    S.sample_rows(l[1:4].contiguous(), u[:3].contiguous(), 1.0)
    assert S.check_status(raise_on_error=False) == 4


def test_sampler_leaves_the_workspace_at_zero(S):
    w = W.make(2, device="cuda", B=8)
    logits, u = W.sampler_rows(w)
    ws = torch.zeros(S.workspace_size(logits.shape[0], 0, w.V, logits.dtype) +
                     S.workspace_size(w.B, w.gamma, w.V, logits.dtype), dtype=torch.uint8, device="cuda")
    S.sample_rows(logits, u, w.T, workspace=ws)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0
    # the same workspace then serves a verification call
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, workspace=ws)
    from parity import compare_sample
    _, _, mism = compare_sample(w, em, na)
    assert not mism


def test_sampler_law_is_q(S):
    """10^6 rows with the same logits: token counts follow softmax(l / T) (chi-square)."""
    N, V, T = 1_000_000, 40, 0.7
    rng = np.random.default_rng(3)
    lq = rng.normal(0, 2.0, V)
    lq[7] = -np.inf
    q = np.exp((lq - lq.max()) / T)
    q /= q.sum()
    for dtype in (torch.float32, torch.bfloat16):
        row = torch.tensor(lq, dtype=torch.float32).to(dtype)
        qd = np.exp((row.float().double().numpy() - lq.max()) / T)   # law of the rounded logits
        qd /= qd.sum()
        logits = row.cuda().unsqueeze(0).expand(N, V).contiguous()
        u = uniform_f32((N,), 9, 1 if dtype == torch.float32 else 2, "cuda")
        tok = S.sample_rows(logits, u, T).cpu().numpy()
        assert S.check_status() == 0
        counts = np.bincount(tok, minlength=V)
        assert counts[7] == 0
        keep = qd > 0
        exp = qd[keep] * N
        assert scipy.stats.chisquare(counts[keep], exp * counts[keep].sum() / exp.sum()).pvalue > 1e-3
