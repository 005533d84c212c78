"""The one-launch path for short rows (spec_verify_sample with rows of at most 8 KB) against the oracle (GPU).

Rows of at most 8 KB that start on 16-byte boundaries take one CTA per batch row and one launch (the
normalisers by a warp per position, then the draw code of the two-kernel path).  The results must
match the float64 oracle token for token outside counted boundary draws, invalid rows must be
reported as in the two-kernel path, and the workspace must come back to zero.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from parity import compare_sample, host_inputs
from test_gpu_edge import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


@pytest.mark.parametrize("B,gamma,V,dtype,ragged", [
    (1, 4, 1024, "f32", False),      # the c0 shape
    (33, 7, 2048, "f32", True),      # 8 KB rows, ragged draft lengths
    (200, 3, 4096, "bf16", True),
    (5, 0, 1024, "f32", False),      # gamma = 0: one draw from p_1
    (4, 64, 256, "f32", False),      # the largest gamma: eight positions per warp
    (9, 12, 512, "bf16", False),     # more positions than warps
])
def test_short_rows_match_oracle(S, B, gamma, V, dtype, ragged):
    w = make_case(B, gamma, V, dtype, T=0.8, ragged=ragged)
    ws = torch.zeros(S.workspace_size(B, gamma, V, w.target.dtype), dtype=torch.uint8, device="cuda")
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, workspace=ws)
    assert S.check_status(ws) == 0
    assert int(torch.count_nonzero(ws)) == 0
    n, flagged, mism = compare_sample(w, em, na)
    assert not mism, mism[:3]
    assert len(flagged) <= n // 4 + 1


def test_short_rows_standardised(S):
    w = make_case(40, 5, 2048, "f32", T=1.0, ragged=True)
    tthr = S.topk_threshold(w.target, 20)
    dthr = S.topk_threshold(w.draft, 20)
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, target_thr=tthr,
                             draft_thr=dthr)
    assert S.check_status() == 0
    h = host_inputs(w)
    ref = O.verify_sample(h["target"], h["draft"], h["dtype"], h["ids"], h["draft_len"], h["uniforms"], h["T"],
                          tthr=tthr.cpu().numpy(), dthr=dthr.cpu().numpy())
    emc, nac = em.cpu().numpy(), na.cpu().numpy()
    for b in range(w.B):
        if ref["boundary"][b]:
            continue
        assert int(nac[b]) == int(ref["n_accepted"][b]) and list(emc[b]) == list(ref["emitted"][b]), b


def test_short_rows_invalid_rows(S):
    w = make_case(6, 3, 1024, "f32", T=1.0)
    gl = torch.full((6,), 3, dtype=torch.int32, device="cuda")
    gl[1] = 4                                 # draft length out of range
    w.target[3, 2, 100] = float("nan")        # a NaN in a target row that is read
    w.draft_len = gl
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, gl)
    code = S.check_status(raise_on_error=False)
    assert code == 1                          # the lowest status recorded: the bad draft length
    assert int(na[1]) == -1 and (em[1] == -1).all()
    assert int(na[3]) == -1 and (em[3] == -1).all()
    _, _, mism = compare_sample(w, em, na)
    assert not mism
