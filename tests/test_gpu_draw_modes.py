"""The draw kernel's two ways of meeting a row's chunk masses agree (GPU).

A row drawn by 2 to 8 CTAs either sends their chunk masses to the row's rank-0 CTA of a thread-block
cluster (the default for small batches, whose draw grid is at most one CTA per SM) or writes them to the
workspace behind an arrival counter (larger batches).  Both compute the same masses and resolve them the
same way, so the emitted tokens must be identical, both must match the float64 oracle outside counted
boundary draws, and both must leave the workspace at zero.  SPECVERIFY_DRAW_CLUSTER forces one or the
other.
"""
from __future__ import annotations

import pytest
import torch

from parity import compare_sample
from test_gpu_edge import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


@pytest.mark.parametrize("B,gamma,V,dtype,ragged", [
    (8, 4, 32128, "bf16", False),     # the c1 shape: 8 draw CTAs of 4096 elements per row
    (24, 6, 20000, "f32", True),      # 5 draw CTAs per row, ragged draft lengths, a partial last chunk
    (3, 2, 9000, "bf16", False),      # V not a whole number of chunks
])
def test_cluster_and_counter_draws_agree(S, monkeypatch, B, gamma, V, dtype, ragged):
    w = make_case(B, gamma, V, dtype, T=0.9, ragged=ragged)
    outs = []
    for mode in ("1", "0"):
        monkeypatch.setenv("SPECVERIFY_DRAW_CLUSTER", mode)
        ws = torch.zeros(S.workspace_size(B, gamma, V, w.target.dtype), dtype=torch.uint8, device="cuda")
        for phase in ("both", "early_exit"):
            em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, workspace=ws,
                                     phase=phase)
            assert S.check_status(ws) == 0
            assert int(torch.count_nonzero(ws)) == 0
            outs.append((em.cpu(), na.cpu()))
    for em, na in outs[1:]:
        assert torch.equal(em, outs[0][0]) and torch.equal(na, outs[0][1])
    n, flagged, mism = compare_sample(w, outs[0][0].cuda(), outs[0][1].cuda())
    assert not mism, mism[:3]
    assert len(flagged) <= n // 4 + 1
