"""The two forms of sampling verification and the draw kernel's two ways of meeting a row's chunk masses
(GPU).

spec_verify_sample (and the early exit) run the one-launch kernel: a thread-block cluster per batch row.
spec_verify_sample_stream then spec_verify_sample_draw are the two-kernel form, whose draw kernel meets a
row's chunk masses either in the rank-0 CTA of a thread-block cluster (small batches) or in the workspace
behind an arrival counter (larger batches); SPECVERIFY_DRAW_CLUSTER forces one or the other.  Both ways
of the two-kernel form compute the same masses, so their tokens must be identical; the one-launch form
and its early exit must be identical to each other; all of them must match the float64 oracle outside
counted boundary draws, and leave the workspace at zero.
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
    ws = torch.zeros(S.workspace_size(B, gamma, V, w.target.dtype), dtype=torch.uint8, device="cuda")

    def run(phase):
        if phase == "split":
            em = torch.full((B, gamma + 1), 7, dtype=torch.int32, device="cuda")
            na = torch.full((B,), 7, dtype=torch.int32, device="cuda")
            for ph in ("stream", "draw"):
                S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, workspace=ws, phase=ph,
                                emitted=em, n_accepted=na)
        else:
            em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, workspace=ws,
                                     phase=phase)
        assert S.check_status(ws) == 0
        assert int(torch.count_nonzero(ws)) == 0
        return em.cpu(), na.cpu()

    split = []
    for mode in ("1", "0"):
        monkeypatch.setenv("SPECVERIFY_DRAW_CLUSTER", mode)
        split.append(run("split"))
    assert torch.equal(split[0][0], split[1][0]) and torch.equal(split[0][1], split[1][1])
    one = [run("both"), run("early_exit")]
    assert torch.equal(one[0][0], one[1][0]) and torch.equal(one[0][1], one[1][1])
    for em, na in (split[0], one[0]):
        n, flagged, mism = compare_sample(w, em.cuda(), na.cuda())
        assert not mism, mism[:3]
        assert len(flagged) <= n // 4 + 1
