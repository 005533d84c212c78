"""Lenient verification (spec_verify_sample_lenient) vs the float64 oracle, and its output law (GPU)."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import scipy.stats
import torch

import oracle as O
import workloads as W
from parity import host_inputs
from workloads.philox import uniform_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


@pytest.mark.parametrize("l", [0.5, 0.2])
@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_lenient_parity(S, k, l):
    w = W.make(k, device="cuda")
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, lenience=l)
    assert S.check_status() == 0
    h = host_inputs(w)
    rows = None if w.B <= 64 else list(range(0, w.B, max(1, w.B // 80)))
    ref = O.verify_sample(h["target"], h["draft"], h["dtype"], h["ids"], h["draft_len"], h["uniforms"], h["T"],
                          rows=rows, lenience=l)
    emc, nac = em.cpu().numpy(), na.cpu().numpy()
    mism = []
    for b in (range(w.B) if rows is None else rows):
        if ref["boundary"][b]:
            continue
        if int(nac[b]) != int(ref["n_accepted"][b]) or list(emc[b]) != list(ref["emitted"][b]):
            mism.append((b, int(nac[b]), list(emc[b]), int(ref["n_accepted"][b]), list(ref["emitted"][b])))
    assert not mism, mism[:4]
    # lenience accepts at least as many guesses as the exact test on the same uniforms
    em1, na1 = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len)
    assert bool((na >= na1).all())


def test_lenience_one_is_spec_verify_sample(S):
    w = W.make(2, device="cuda")
    em0, na0 = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T)
    em1 = torch.empty_like(em0)
    na1 = torch.empty_like(na0)
    ws = S.workspace_for(w.target.device, S.workspace_size(w.B, w.gamma, w.V, w.target.dtype))
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = S.lib.spec_verify_sample_lenient(p(w.target), p(w.draft), 1, p(w.ids), None, p(w.uniforms), w.T, 1.0,
                                            w.B, w.gamma, w.V, p(em1), p(na1), p(ws), ws.numel(),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0 and S.check_status() == 0
    assert torch.equal(em0, em1) and torch.equal(na0, na1)


def test_lenient_first_token_law(S):
    """10^6 steps with fixed p, q: the first emitted token follows R11's law min(q, p/l) + R * residual,
    which never exceeds p/l (chi-square)."""
    N, V, gamma, l = 1_000_000, 12, 2, 0.4
    rng = np.random.default_rng(31)
    p = rng.dirichlet(np.ones(V) * 0.8, size=gamma + 1)
    q = rng.dirichlet(np.ones(V) * 0.8, size=gamma)
    lp, lq = np.log(p), np.log(q)
    t = torch.tensor(lp, dtype=torch.float32).cuda().unsqueeze(0).expand(N, gamma + 1, V).contiguous()
    d = torch.tensor(lq, dtype=torch.float32).cuda().unsqueeze(0).expand(N, gamma, V).contiguous()
    ux = uniform_f32((N, gamma), 41, 1, "cuda").double()
    cq = torch.tensor(np.cumsum(q, axis=1), dtype=torch.float64, device="cuda")
    ids = torch.stack([torch.searchsorted(cq[i].contiguous(), ux[:, i].contiguous(), right=True)
                       for i in range(gamma)], 1).clamp_(max=V - 1).to(torch.int32).contiguous()
    u = uniform_f32((N, gamma + 1), 41, 2, "cuda")
    em, na = S.verify_sample(t, d, ids, u, 1.0, lenience=l)
    assert S.check_status() == 0
    first = np.bincount(em[:, 0].cpu().numpy(), minlength=V)
    pf, qf = p[0], q[0]
    acc = np.minimum(qf, pf / l)
    resid = np.maximum(0.0, pf - l * qf)
    law = acc + (1.0 - acc.sum()) * resid / resid.sum()
    assert np.all(law <= pf / l + 1e-12)
    assert scipy.stats.chisquare(first, law * N).pvalue > 1e-3
