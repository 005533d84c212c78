"""Byte-lean early exit (spec_verify_sample_early_exit) gives exactly spec_verify_sample's outputs (GPU).

Positions are streamed one after the other and a row stops at its first
rejection; the accept tests and the draw use the same arithmetic as the
all-positions path, so emitted tokens and n_accepted agree bit for bit, and
both agree with the float64 oracle outside counted boundary draws.
"""
from __future__ import annotations

import pytest
import torch

import workloads as W
from parity import compare_sample

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


def _both(S, w, **kw):
    em0, na0 = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, **kw)
    em1, na1 = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, phase="early_exit", **kw)
    return em0, na0, em1, na1


@pytest.mark.parametrize("k", [0, 1, 2, 3, 4])
def test_early_exit_equals_the_all_positions_path(S, k):
    w = W.make(k, device="cuda")
    em0, na0, em1, na1 = _both(S, w)
    assert S.check_status() == 0
    assert torch.equal(em0, em1) and torch.equal(na0, na1)
    rows = None if w.B <= 64 else list(range(0, w.B, max(1, w.B // 96)))
    n, flagged, mism = compare_sample(w, em1, na1, rows=rows)
    assert not mism, mism[:5]


@pytest.mark.parametrize("B,gamma,V,dtype,ragged,offset", [
    (5, 3, 50001, "f32", True, 0),
    (6, 2, 20000, "bf16", True, 3),
    (3, 0, 3000, "f32", False, 0),
    (4, 5, 1, "f32", False, 0),
    (64, 8, 4096, "bf16", True, 0),
    (2, 1, 262144, "f32", False, 0),
])
def test_early_exit_odd_sizes(S, B, gamma, V, dtype, ragged, offset):
    from test_gpu_edge import make_case
    w = make_case(B, gamma, V, dtype, T=0.9, ragged=ragged, storage_offset=offset)
    em0, na0, em1, na1 = _both(S, w)
    assert S.check_status() == 0
    assert torch.equal(em0, em1) and torch.equal(na0, na1)
    _, _, mism = compare_sample(w, em1, na1)
    assert not mism, mism[:3]


def test_early_exit_reads_nothing_after_the_first_rejection(S):
    """A NaN logit row after the first rejection invalidates the row for spec_verify_sample (it reads every
    position) but not for the early exit, which never reads it."""
    w = W.make(2, device="cuda", B=16)
    em0, na0 = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T)
    assert S.check_status() == 0
    na = na0.cpu().numpy()
    rows = [b for b in range(w.B) if na[b] < w.gamma - 1]
    assert rows
    t = w.target.clone()
    for b in rows:
        t[b, int(na[b]) + 2, 7] = float("nan")        # a position the early exit never reaches
    em1, na1 = S.verify_sample(t, w.draft, w.ids, w.uniforms, w.T, phase="early_exit")
    assert S.check_status() == 0
    assert torch.equal(em0, em1) and torch.equal(na0, na1)
    em2, na2 = S.verify_sample(t, w.draft, w.ids, w.uniforms, w.T)
    assert S.check_status(raise_on_error=False) == 4
    assert all(int(na2[b]) == -1 for b in rows)


def test_early_exit_invalid_rows_match(S):
    w = W.make(1, device="cuda")
    t = w.target.clone()
    t[0, 0, 3] = float("nan")                           # read by both paths
    ids = w.ids.clone()
    ids[1, 0] = w.V + 5                                 # id out of range at position 0
    em0, na0 = S.verify_sample(t, w.draft, ids, w.uniforms, w.T)
    c0 = S.check_status(raise_on_error=False)
    em1, na1 = S.verify_sample(t, w.draft, ids, w.uniforms, w.T, phase="early_exit")
    c1 = S.check_status(raise_on_error=False)
    assert c0 == c1 == 4
    assert torch.equal(em0, em1) and torch.equal(na0, na1)
    assert int(na1[0]) == -1 and int(na1[1]) == -1


def test_early_exit_leaves_the_workspace_at_zero(S):
    w = W.make(4, device="cuda", B=64)
    ws = torch.zeros(S.workspace_size(w.B, w.gamma, w.V, w.target.dtype), dtype=torch.uint8, device="cuda")
    for phase in ("early_exit", "both", "early_exit"):
        S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, workspace=ws, phase=phase)
        assert S.check_status(ws) == 0
        assert int(torch.count_nonzero(ws)) == 0
