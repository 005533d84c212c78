"""Top-k / nucleus standardisation on the GPU against the float64 oracle (GPU).

Thresholds: top-k is exact (a selection over the logits), nucleus is exact
except where the running mass lies within 1e-5 of top_p (the oracle flags those
rows; the GPU may then stop one token earlier or later).  Verification and
sampling on standardised rows take the thresholds as inputs, so they are
token-exact against the oracle given the same thresholds, outside counted
boundary draws.
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


def _rows_np(x):
    dt = "bf16" if x.dtype == torch.bfloat16 else "f32"
    return W.logits_as_numpy(x.reshape(-1, x.shape[-1])), dt


def _random_rows(R, V, dtype, seed, offset=0):
    g = 2.5 * normal_f32((R * V + offset,), seed, V, "cuda")
    if dtype == "bf16":
        g = g.to(torch.bfloat16)
    return g[offset:].view(R, V)


@pytest.mark.parametrize("R,V,dtype,offset", [(6, 1000, "f32", 0), (5, 50001, "bf16", 0), (4, 77777, "f32", 1),
                                              (3, 262144, "bf16", 0), (9, 1, "f32", 0), (7, 130, "bf16", 3)])
@pytest.mark.parametrize("k", [1, 2, 50, 129, 100000])
def test_topk_threshold_is_exact(S, R, V, dtype, offset, k):
    l = _random_rows(R, V, dtype, 30 + k, offset)
    if V >= 8:
        l[0, 3] = float("-inf")
        l[1, 5] = l[1, 6]                        # a tie
    thr = S.topk_threshold(l, k).cpu().numpy()
    h, dt = _rows_np(l)
    for r in range(R):
        assert np.float32(thr[r]) == np.float32(O.topk_threshold(O.widen(h[r], dt), k)), (r, thr[r])


def test_topk_threshold_invalid_and_degenerate_rows(S):
    l = normal_f32((4, 300), 3, 3, "cuda")
    l[0, 7] = float("nan")
    l[1, 9] = float("inf")
    l[2, :] = float("-inf")
    l[3, :] = 1.5                                # every logit tied
    thr = S.topk_threshold(l, 10).cpu().numpy()
    assert np.isnan(thr[0]) and np.isnan(thr[1]) and thr[2] == -np.inf and thr[3] == np.float32(1.5)


def _long_rows(V, dtype, offset):
    """Rows of V logits that steer the threshold kernel down each of its paths.  The kernel bins the row
    against the max R of its first sixteenth (at least 4096 logits) and sets aside the logits above R;
    it falls back to binning against the true max when more than 2048 lie above R, or (nucleus) when the
    max lies 10 or more log2 units above R."""
    R = 12
    l = _random_rows(R, V, dtype, 77, offset)
    pre = max(4096, V // 16)
    l[1, V - 3] = float("nan")                                   # NaN late in the row
    l[2, V // 2 + 1] = float("inf")                              # +inf late in the row
    l[3, :] = float("-inf")                                      # nothing finite
    l[4, :] = 1.5                                                # all tied: a bin past the sort buffer
    l[5, :] = float("-inf")                                      # 40 finite logits, all after the prefix
    l[5, V - 40:] = 0.25 * torch.arange(40, device="cuda", dtype=l.dtype)
    l[6, :] = float("-inf")                                      # a single finite logit
    l[6, V - 1] = -2.0
    l[7] = (l[7].float() + W.zipf_log_prior(V, 1.1, "cuda")).to(l.dtype)  # the max inside the prefix
    l[8] = torch.linspace(-8.0, 8.0, V, device="cuda").to(l.dtype)         # increasing: overflow past 2048
    l[9, pre:pre + 30] = 14.0 + torch.arange(30, device="cuda", dtype=l.dtype) * 0.125  # a peak after the
    l[10, :pre] -= 30.0                                          # prefix 30 below the rest: nucleus fallback
    l[11, :pre] = float("-inf")                                  # empty prefix
    return l


@pytest.mark.parametrize("V,dtype,offset", [(150001, "bf16", 0), (100000, "f32", 0), (70001, "f32", 1),
                                           (262144, "f32", 0), (9000, "bf16", 0)])
def test_thresholds_on_every_selection_path(S, V, dtype, offset):
    """Top-k exact and nucleus exact outside flagged rows against the oracle on rows that end the selection
    inside the logits above the provisional max, inside the histogram, in the radix selection, and in both
    fallbacks; NaN / +inf rows give NaN, rows with nothing finite -inf (top-k) or NaN (nucleus)."""
    l = _long_rows(V, dtype, offset)
    h, dt = _rows_np(l)
    for k in (1, 50, 9000):
        thr = S.topk_threshold(l, k).cpu().numpy()
        assert np.isnan(thr[1]) and np.isnan(thr[2]) and thr[3] == -np.inf
        for r in [0] + list(range(4, l.shape[0])):
            assert np.float32(thr[r]) == np.float32(O.topk_threshold(O.widen(h[r], dt), k)), (k, r, thr[r])
    for top_p, T in ((0.5, 1.0), (0.9, 0.7), (0.999, 1.3), (1.0, 1.0)):
        thr = S.topp_threshold(l, T, top_p).cpu().numpy()
        assert np.isnan(thr[1]) and np.isnan(thr[2]) and np.isnan(thr[3])
        for r in [0] + list(range(4, l.shape[0])):
            tau, flag = O.topp_threshold(O.widen(h[r], dt), float(np.float32(T)), float(np.float32(top_p)))
            if not flag:
                assert np.float32(thr[r]) == np.float32(tau), (top_p, r, thr[r], tau)


@pytest.mark.parametrize("V,dtype", [(152064, "f32"), (128256, "bf16"), (200003, "f32")])
def test_nucleus_selection_paths_agree(S, monkeypatch, V, dtype):
    """Rows over 128 KB select the nucleus threshold from float sums whose error bounds must leave a single
    candidate, else from an exact fixed-point pass; a bracket too wide takes the weighted histogram.  The
    three (SPECVERIFY_NUCLEUS_PATH = bounds / exact / weighted) must give the same bits, and match the
    oracle outside flagged rows.  V = 200003 fp32 rows are not 16-byte aligned (scalar loads)."""
    R = 16
    l = _random_rows(R, V, dtype, 91, 0)
    l = (l.float() + W.zipf_log_prior(V, 1.0, "cuda")[None, :]).to(l.dtype)
    h, dt = _rows_np(l)
    for top_p, T in ((0.5, 1.0), (0.9, 0.7), (0.99, 1.3)):
        outs = []
        for path in ("bounds", "exact", "weighted"):
            monkeypatch.setenv("SPECVERIFY_NUCLEUS_PATH", path)
            outs.append(S.topp_threshold(l, T, top_p).view(torch.int32).cpu())
        monkeypatch.delenv("SPECVERIFY_NUCLEUS_PATH")
        assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2]), (top_p, outs)
        thr = outs[0].view(torch.float32).numpy()
        for r in range(R):
            tau, flag = O.topp_threshold(O.widen(h[r], dt), float(np.float32(T)), float(np.float32(top_p)))
            if not flag:
                assert np.float32(thr[r]) == np.float32(tau), (top_p, r, thr[r], tau)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("top_p,T", [(0.5, 1.0), (0.9, 0.7), (0.99, 1.3), (0.05, 1.0), (1.0, 1.0)])
def test_topp_threshold_matches_oracle(S, dtype, top_p, T):
    R, V = 48, 32000
    l = _random_rows(R, V, dtype, 40, 0).float()
    l = (l + W.zipf_log_prior(V, 1.1, "cuda")[None, :]).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    thr = S.topp_threshold(l.contiguous(), T, top_p).cpu().numpy()
    h, dt = _rows_np(l)
    flagged = 0
    for r in range(R):
        lr = O.widen(h[r], dt)
        tau, flag = O.topp_threshold(lr, float(np.float32(T)), float(np.float32(top_p)))
        if flag:
            # the stopping token may be any whose running mass (before or at it) lies within 1e-5 of top_p
            flagged += 1
            p = O.softmax_t(lr, float(np.float32(T)))
            order = np.argsort(-p, kind="stable")
            c = np.cumsum(p[order])
            c0 = np.concatenate([[0.0], c[:-1]])
            near = (np.abs(c - top_p) < 1e-5) | (np.abs(c0 - top_p) < 1e-5) | (lr[order] == tau)
            cands = {np.float32(v) for v in lr[order][near]}
            assert np.float32(thr[r]) in cands, (r, thr[r], tau)
        else:
            assert np.float32(thr[r]) == np.float32(tau), (r, thr[r], tau)
    if top_p <= 0.9:
        assert flagged <= R // 8


@pytest.mark.parametrize("k_or_p", [("k", 50), ("p", 0.9), ("k", 1)])
@pytest.mark.parametrize("wk", [1, 2, 4])
def test_standardised_verification_parity(S, k_or_p, wk):
    """Thresholds from the GPU, drafts resampled from the standardised q by the masked sampler, then
    masked verification against the oracle on the same thresholds."""
    w = W.make(wk, device="cuda", B=None if wk != 4 else 256)
    kind, val = k_or_p
    if kind == "k":
        tthr, dthr = S.topk_threshold(w.target, val), S.topk_threshold(w.draft, val)
    else:
        tthr, dthr = S.topp_threshold(w.target, w.T, val), S.topp_threshold(w.draft, w.T, val)
    R = w.B * w.gamma
    ud = uniform_f32((R,), 77, wk, "cuda")
    ids = S.sample_rows(w.draft.reshape(R, w.V), ud, w.T, thr=dthr.reshape(R).contiguous()).view(w.B, w.gamma)
    if w.draft_len is not None:        # padded draft rows hold NaN: no draw there (recorded), a dummy id
        S.check_status(raise_on_error=False)
        pad = torch.arange(w.gamma, device="cuda")[None, :] >= w.draft_len[:, None]
        ids = torch.where(pad, torch.zeros_like(ids), ids)
    else:
        assert S.check_status() == 0
    assert int(ids.min()) >= 0
    w.ids = ids.contiguous()
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, target_thr=tthr,
                             draft_thr=dthr)
    assert S.check_status() == 0
    h = {"target": W.logits_as_numpy(w.target), "draft": W.logits_as_numpy(w.draft),
         "dtype": "bf16" if w.target.dtype == torch.bfloat16 else "f32", "ids": w.ids.cpu().numpy(),
         "draft_len": None if w.draft_len is None else w.draft_len.cpu().numpy(),
         "uniforms": w.uniforms.cpu().numpy(), "T": w.T}
    rows = None if w.B <= 64 else list(range(0, w.B, 3))
    ref = O.verify_sample(h["target"], h["draft"], h["dtype"], h["ids"], h["draft_len"], h["uniforms"], h["T"],
                          rows=rows, tthr=tthr.cpu().numpy(), dthr=dthr.cpu().numpy())
    emc, nac = em.cpu().numpy(), na.cpu().numpy()
    mism, flagged = [], 0
    for b in (range(w.B) if rows is None else rows):
        if ref["boundary"][b]:
            flagged += 1
            continue
        if int(nac[b]) != int(ref["n_accepted"][b]) or list(emc[b]) != list(ref["emitted"][b]):
            mism.append((b, int(nac[b]), list(emc[b]), int(ref["n_accepted"][b]), list(ref["emitted"][b])))
    assert not mism, mism[:4]
    if kind == "k" and val == 1:       # one-hot p: exactly greedy verification where the target max is unique
        gem, gna = S.verify_greedy(w.target, w.ids, w.draft_len)
        t = w.target.float()
        uniq = ((t == t.amax(dim=2, keepdim=True)).sum(dim=2) == 1)
        gl = w.draft_len if w.draft_len is not None else torch.full((w.B,), w.gamma, device="cuda")
        used = torch.arange(w.gamma + 1, device="cuda")[None, :] <= gl[:, None]
        ok = (uniq | ~used).all(dim=1)
        assert int(ok.sum()) > w.B // 2
        assert torch.equal(gem[ok], em[ok]) and torch.equal(gna[ok], na[ok])


def test_masked_sampler_parity_and_law(S):
    R, V, T = 64, 50001, 0.8
    l = (_random_rows(R, V, "f32", 50, 0) + W.zipf_log_prior(V, 1.0, "cuda")[None, :]).contiguous()
    thr = S.topp_threshold(l, T, 0.8)
    u = uniform_f32((R,), 51, 1, "cuda")
    tok = S.sample_rows(l, u, T, thr=thr)
    assert S.check_status() == 0
    ref = O.sample_rows(l.cpu().numpy(), "f32", u.cpu().numpy(), T, thr=thr.cpu().numpy())
    t = tok.cpu().numpy()
    for r in range(R):
        if ref["boundary"][r]:
            assert int(t[r]) in ref["candidates"][r]
        else:
            assert int(t[r]) == int(ref["tokens"][r])
    # law: 10^6 draws from one row with top-k = 7 follow the truncated softmax
    N, V2 = 1_000_000, 64
    rng = np.random.default_rng(5)
    lr = rng.normal(0, 1.5, V2).astype(np.float32)
    rows = torch.tensor(lr, device="cuda").unsqueeze(0).expand(N, V2).contiguous()
    thr2 = S.topk_threshold(rows[:1].contiguous(), 7).expand(N).contiguous()
    tok = S.sample_rows(rows, uniform_f32((N,), 52, 2, "cuda"), 1.0, thr=thr2).cpu().numpy()
    assert S.check_status() == 0
    keep = lr >= np.sort(lr)[::-1][6]
    assert keep.sum() == 7
    counts = np.bincount(tok, minlength=V2)
    assert counts[~keep].sum() == 0
    p = np.exp(lr[keep].astype(np.float64) - lr.max())
    p /= p.sum()
    assert scipy.stats.chisquare(counts[keep], p * N).pvalue > 1e-3
