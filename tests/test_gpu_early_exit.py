"""Byte-lean early exit (spec_verify_sample_early_exit) (GPU).

A row's positions are read only up to its first rejection.  Two forms give it: the one-launch kernel (a
thread-block cluster per batch row that decides each position before streaming the next), chosen for
batches whose positions are large, and the two-kernel all-positions path with early-exit validity (a
logit row after the first rejection does not count), chosen for small ones; SPECVERIFY_EARLY_FORM=1 / 2
forces one.  The two-kernel form takes exactly spec_verify_sample's arithmetic, so its outputs are
identical to spec_verify_sample's.  The one-launch form splits the vocabulary its own way, so its float32
sums round differently: its tokens equal spec_verify_sample's on every row that is not a boundary draw,
and both match the float64 oracle outside counted boundary draws.
"""
from __future__ import annotations

import pytest
import torch

import workloads as W
from parity import compare_sample, host_inputs
import oracle as O

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


def _agree(w, em0, na0, em1, na1, exact, rows=None):
    """The early exit against spec_verify_sample and the oracle, on `rows` (all by default)."""
    rows = list(range(w.B)) if rows is None else list(rows)
    if exact:
        assert torch.equal(em0, em1) and torch.equal(na0, na1)
    h = host_inputs(w)
    ref = O.verify_sample(h["target"], h["draft"], h["dtype"], h["ids"], h["draft_len"], h["uniforms"], h["T"],
                          rows=rows)
    same = [b for b in rows if not ref["boundary"][b]]
    assert torch.equal(em0[same], em1[same]) and torch.equal(na0[same], na1[same])
    _, _, mism = compare_sample(w, em1, na1, h, rows=rows)
    assert not mism, mism[:5]


@pytest.mark.parametrize("form", ["auto", "1", "2"])
@pytest.mark.parametrize("k", [0, 1, 2, 3, 4])
def test_early_exit_equals_the_all_positions_path(S, monkeypatch, k, form):
    if form != "auto":
        monkeypatch.setenv("SPECVERIFY_EARLY_FORM", form)
    w = W.make(k, device="cuda")
    em0, na0, em1, na1 = _both(S, w)
    assert S.check_status() == 0
    rows = None if w.B <= 64 else list(range(0, w.B, max(1, w.B // 96)))
    exact = form == "2" or (form == "auto" and k in (0, 1, 2))
    _agree(w, em0, na0, em1, na1, exact, rows)


@pytest.mark.parametrize("form", ["1", "2"])
@pytest.mark.parametrize("B,gamma,V,dtype,ragged,offset", [
    (5, 3, 50001, "f32", True, 0),
    (6, 2, 20000, "bf16", True, 3),
    (3, 0, 3000, "f32", False, 0),
    (4, 5, 1, "f32", False, 0),
    (64, 8, 4096, "bf16", True, 0),
    (2, 1, 262144, "f32", False, 0),
])
def test_early_exit_odd_sizes(S, monkeypatch, B, gamma, V, dtype, ragged, offset, form):
    from test_gpu_edge import make_case
    monkeypatch.setenv("SPECVERIFY_EARLY_FORM", form)
    w = make_case(B, gamma, V, dtype, T=0.9, ragged=ragged, storage_offset=offset)
    em0, na0, em1, na1 = _both(S, w)
    assert S.check_status() == 0
    _agree(w, em0, na0, em1, na1, exact=form == "2")


@pytest.mark.parametrize("form", ["1", "2"])
def test_early_exit_reads_nothing_after_the_first_rejection(S, monkeypatch, form):
    """A NaN logit row after the first rejection invalidates the row for spec_verify_sample (it reads every
    position) but not for the early exit, for which that row is never read (one-launch form) or does not
    count (two-kernel form)."""
    monkeypatch.setenv("SPECVERIFY_EARLY_FORM", form)
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
    _agree(w, em0, na0, em1, na1, exact=form == "2")
    em2, na2 = S.verify_sample(t, w.draft, w.ids, w.uniforms, w.T)
    assert S.check_status(raise_on_error=False) == 4
    assert all(int(na2[b]) == -1 for b in rows)


@pytest.mark.parametrize("form", ["1", "2"])
def test_early_exit_invalid_rows_match(S, monkeypatch, form):
    monkeypatch.setenv("SPECVERIFY_EARLY_FORM", form)
    w = W.make(1, device="cuda")
    t = w.target.clone()
    t[0, 0, 3] = float("nan")                           # read by both paths
    ids = w.ids.clone()
    ids[1, 0] = w.V + 5                                 # id out of range at position 0
    ids[2, 3] = w.V + 7                                 # id out of range at the last position: checked by both
    em0, na0 = S.verify_sample(t, w.draft, ids, w.uniforms, w.T)
    c0 = S.check_status(raise_on_error=False)
    em1, na1 = S.verify_sample(t, w.draft, ids, w.uniforms, w.T, phase="early_exit")
    c1 = S.check_status(raise_on_error=False)
    assert c0 == c1 == 4
    assert torch.equal(na0[:3], na1[:3]) and torch.equal(em0[:3], em1[:3])
    assert int(na1[0]) == -1 and int(na1[1]) == -1 and int(na1[2]) == -1


@pytest.mark.parametrize("form", ["1", "2"])
def test_early_exit_leaves_the_workspace_at_zero(S, monkeypatch, form):
    monkeypatch.setenv("SPECVERIFY_EARLY_FORM", form)
    w = W.make(4, device="cuda", B=64)
    ws = torch.zeros(S.workspace_size(w.B, w.gamma, w.V, w.target.dtype), dtype=torch.uint8, device="cuda")
    for phase in ("early_exit", "both", "early_exit"):
        S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, workspace=ws, phase=phase)
        assert S.check_status(ws) == 0
        assert int(torch.count_nonzero(ws)) == 0
