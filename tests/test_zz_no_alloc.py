"""spec_verify_sample_noalloc, the entry point for callers that cannot allocate device memory (GPU).

Some callers are handed their input and output buffers by a host program that owns every allocator (a
plugin), or must not call cudaMalloc once serving has started (it can block the whole device and fail
under memory pressure).  This entry point runs the same kernels as spec_verify_sample with their scratch
in a fixed array inside the library, so on the same inputs it must give exactly the tokens of
spec_verify_sample with a caller workspace, and the oracle's tokens outside boundary draws.
This file is collected last so that a run stopping at the first failure has run every other test.
"""
from __future__ import annotations

import ctypes

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
    fn = S.lib.spec_verify_sample_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, i32, vp, vp, vp, f32, i32, i32, i32, vp, vp, vp]
    fn.restype = i32
    return S


def _noalloc(S, w, draft_len="w", ids=None, T=None):
    em = torch.full((w.B, w.gamma + 1), 123, dtype=torch.int32, device="cuda")
    na = torch.full((w.B,), 123, dtype=torch.int32, device="cuda")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dl = w.draft_len if draft_len == "w" else draft_len
    code = S.lib.spec_verify_sample_noalloc(
        p(w.target), p(w.draft), 1 if w.dtype == "bf16" else 0, p(w.ids if ids is None else ids), p(dl),
        p(w.uniforms), w.T if T is None else T, w.B, w.gamma, w.V, p(em), p(na),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return code, em, na


def _check_against_both(S, w, oracle_rows=None):
    ref_em, ref_na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len)
    assert S.check_status() == 0
    code, em, na = _noalloc(S, w)
    torch.cuda.synchronize()
    assert code == 0
    assert torch.equal(em, ref_em) and torch.equal(na, ref_na)
    assert (na >= 0).all()
    _, _, mism = compare_sample(w, em, na, rows=oracle_rows)
    assert not mism, mism[:3]


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row(S):
    # two different shapes in a row: the shared scratch must come back clean between calls
    for w in (W.make(4, device="cuda", B=96), W.make(1, device="cuda")):
        _check_against_both(S, w)


@pytest.mark.parametrize("k", [3, 4])
def test_noalloc_full_size_workloads(S, k):
    """c3 (B=256, gamma=5, V=152064, fp32) and c4 (B=1024, ragged gamma <= 8, V=32000, bf16), the largest
    scratch needs, at full size; the oracle checks every eighth row."""
    w = W.make(k, device="cuda")
    assert S.lib.spec_workspace_size(w.B, w.gamma, w.V, 1 if w.dtype == "bf16" else 0) <= 16 << 20
    _check_against_both(S, w, oracle_rows=range(0, w.B, 8))


def test_noalloc_after_invalid_rows_and_rejected_calls(S):
    """Calls with invalid rows (a draft length of -1, a draft id past V) and a call rejected on the host
    (temperature 0) leave nothing behind that changes the next valid call."""
    w = W.make(1, device="cuda")
    bad_len = torch.full((w.B,), w.gamma, dtype=torch.int32, device="cuda")
    bad_len[0] = -1
    bad_ids = w.ids.clone()
    bad_ids[1, 0] = w.V + 5
    code, em, na = _noalloc(S, w, draft_len=bad_len, ids=bad_ids)
    torch.cuda.synchronize()
    assert code == 0
    assert int(na[0]) == -1 and int(na[1]) == -1 and (em[:2] == -1).all()
    assert (na[2:] >= 0).all()
    assert _noalloc(S, w, T=0.0)[0] == 1  # SPEC_ERR_ARG, before the scratch is touched
    for _ in range(2):
        _check_against_both(S, w)


def test_noalloc_rejects_sizes_beyond_its_scratch(S):
    limit = 16 << 20
    B, gamma, V = 4096, 8, 32000
    assert S.lib.spec_workspace_size(B, gamma, V, 1) > limit
    dummy = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    code = S.lib.spec_verify_sample_noalloc(dummy, dummy, 1, dummy, None, dummy, 1.0, B, gamma, V, dummy, dummy,
                                            None)
    assert code == 7  # SPEC_ERR_WORKSPACE
