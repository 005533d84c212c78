"""spec_verify_sample_noalloc, the entry point for callers that cannot allocate device memory (GPU).

It runs the same kernels as spec_verify_sample with their scratch in a fixed array inside the library,
so on the same inputs it must give exactly the tokens of spec_verify_sample with a caller workspace.
This file is collected last so that a run stopping at the first failure has run every other test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    fn = S.lib.spec_verify_sample_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, i32, vp, vp, vp, f32, i32, i32, i32, vp, vp, vp]
    fn.restype = i32
    return S


def _noalloc(S, w):
    em = torch.full((w.B, w.gamma + 1), 123, dtype=torch.int32, device="cuda")
    na = torch.full((w.B,), 123, dtype=torch.int32, device="cuda")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    code = S.lib.spec_verify_sample_noalloc(
        p(w.target), p(w.draft), 1 if w.dtype == "bf16" else 0, p(w.ids), p(w.draft_len), p(w.uniforms), w.T,
        w.B, w.gamma, w.V, p(em), p(na), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return code, em, na


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row(S):
    # two different shapes in a row: the shared scratch must come back clean between calls
    for w in (W.make(4, device="cuda", B=96), W.make(1, device="cuda")):
        ref_em, ref_na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len)
        assert S.check_status() == 0
        code, em, na = _noalloc(S, w)
        torch.cuda.synchronize()
        assert code == 0
        assert torch.equal(em, ref_em) and torch.equal(na, ref_na)
        assert (na >= 0).all()


def test_noalloc_rejects_sizes_beyond_its_scratch(S):
    limit = 16 << 20
    B, gamma, V = 4096, 8, 32000
    assert S.lib.spec_workspace_size(B, gamma, V, 1) > limit
    dummy = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    code = S.lib.spec_verify_sample_noalloc(dummy, dummy, 1, dummy, None, dummy, 1.0, B, gamma, V, dummy, dummy,
                                            None)
    assert code == 7  # SPEC_ERR_WORKSPACE
