"""CUDA path vs the float64 oracle on the five seeded workloads at their full sizes (GPU).

Every call goes through the C ABI (via the ctypes binding) in the launch
configuration the bench times.  Sampling is token-exact outside counted
boundary draws, greedy is bit-exact, statistics agree within tests/parity.py's
tolerances.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from parity import (compare_greedy, compare_sample, compare_stats, flag_cap, host_inputs, record, report_entry,
                    sample_report)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


def _report(name, n, flagged, mism):
    print(f"{name}: compared {n} rows, boundary draws {len(flagged)}, mismatches {len(mism)}")


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_sample_parity_full_config(S, k):
    w = W.make(k, device="cuda")
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len)
    assert S.check_status() == 0
    rep = sample_report(w, em, na)
    _report(w.name, rep["compared"], rep["flagged"], rep["mism"])
    record(report_entry("sample_parity_full_config", w, rep))
    assert not rep["mism"], rep["mism"][:5]
    # boundary rows (low-probability tokens make some draws boundary draws by definition) stay within what
    # the oracle's flag bands explain
    assert len(rep["flagged"]) <= rep["cap"], (len(rep["flagged"]), rep["expected_flags"])


def test_sample_parity_c0_many_calls(S):
    """c0 is 1000 independent verify calls (B=1, gamma=4, V=1024): every one is compared with the oracle."""
    total = {"compared": 0, "flagged": [], "accept_boundary": 0, "draw_boundary": 0, "expected_flags": 0.0,
             "mism": []}
    for call in range(1000):
        w = W.make(0, device="cuda", call=call)
        em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T)
        rep = sample_report(w, em, na)
        assert not rep["mism"], (call, rep["mism"])
        total["compared"] += rep["compared"]
        total["flagged"] += [call for _ in rep["flagged"]]
        total["accept_boundary"] += rep["accept_boundary"]
        total["draw_boundary"] += rep["draw_boundary"]
        total["expected_flags"] += rep["expected_flags"]
    assert S.check_status() == 0
    total["cap"] = flag_cap(total["expected_flags"])
    record(report_entry("sample_parity_c0_1000_calls", w, total, calls=1000))
    assert total["compared"] == 1000
    assert len(total["flagged"]) <= total["cap"], (len(total["flagged"]), total["expected_flags"])


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_greedy_parity_full_config(S, k):
    w = W.make(k, device="cuda")
    em, na = S.verify_greedy(w.target, w.greedy_ids, w.draft_len)
    assert S.check_status() == 0
    mism = compare_greedy(w, w.greedy_ids, em, na)
    # sampled drafts as guesses too: mostly early mismatches
    em2, na2 = S.verify_greedy(w.target, w.ids, w.draft_len)
    mism2 = compare_greedy(w, w.ids, em2, na2)
    record({"test": "greedy_parity_full_config", "workload": w.name, "rows_compared": 2 * w.B,
            "mismatches": len(mism) + len(mism2), "exemptions": 0})
    assert not mism, mism[:5]
    assert not mism2, mism2[:5]


@pytest.mark.parametrize("k", [0, 1, 2, 3, 4])
def test_stats_parity_full_config(S, k):
    w = W.make(k, device="cuda")
    st = S.accept_stats(w.target, w.draft, w.ids, w.T, w.draft_len)
    assert S.check_status() == 0
    rel = {}
    worst, n = compare_stats(w, st, rel=rel)
    print(w.name, n, worst)
    record({"test": "stats_parity_full_config", "workload": w.name, "positions_compared": n,
            "worst_normalised_error": worst, "worst_relative_error": {k: v for k, v in rel.items()
                                                                      if not k.endswith("_abs")},
            "worst_absolute_error": {k[:-4]: v for k, v in rel.items() if k.endswith("_abs")}})
    assert n > 0
    for key, v in worst.items():
        assert v <= 1.0, (key, v)


def test_c2_acceptance_rate_is_near_08(S):
    """The c2 recipe promises mean beta ~ 0.8 per row (sigma calibrated by the oracle)."""
    w = W.make(2, device="cuda")
    st = S.accept_stats(w.target, w.draft, w.ids, w.T)
    beta = st["beta"].mean(dim=1).cpu().numpy()
    assert np.all(np.abs(beta - 0.8) < 0.02), beta


def test_c4_special_rows(S):
    """p == q rows accept everything; disjoint rows accept nothing; one-hot targets emit the hot token."""
    w = W.make(4, device="cuda")
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len)
    em, na = em.cpu(), na.cpu()
    gl = w.draft_len.cpu()
    kind = w.row_kind.cpu()
    hot = w.meta["hot"]
    oh_rows = (kind == W.ROW_ONE_HOT).nonzero().flatten().tolist()
    for b in range(w.B):
        gb = int(gl[b])
        if kind[b] == W.ROW_P_EQ_Q:
            assert int(na[b]) == gb
        elif kind[b] == W.ROW_DISJOINT:
            assert int(na[b]) == 0
        elif kind[b] == W.ROW_ONE_HOT:
            n = int(na[b])
            assert int(em[b, n]) == int(hot[oh_rows.index(b), n])
    st = S.accept_stats(w.target, w.draft, w.ids, w.T, w.draft_len)
    beta = st["beta"].cpu()
    for b in range(w.B):
        gb = int(gl[b])
        if kind[b] == W.ROW_P_EQ_Q:
            assert (beta[b, :gb] == 1.0).all() or torch.allclose(beta[b, :gb], torch.ones(gb), atol=1e-6)
            assert (st["resid"].cpu()[b, :gb] == 0).all()
            assert (st["accept_prob"].cpu()[b, :gb] == 1.0).all()
        elif kind[b] == W.ROW_DISJOINT:
            assert (beta[b, :gb] == 0).all()


def test_repeated_calls_are_identical_and_workspace_resets(S):
    w = W.make(1, device="cuda")
    a = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T)
    g = S.verify_greedy(w.target, w.greedy_ids)
    b = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T)
    g2 = S.verify_greedy(w.target, w.greedy_ids)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(g[0], g2[0]) and torch.equal(g[1], g2[1])
    ws = S.workspace_for(torch.device("cuda"), 0)
    # every counter, record slot and key the calls used is zero again (error word included)
    nbytes = S.workspace_size(w.B, w.gamma, w.V)
    head = ws[:256].cpu()
    assert int(head[:4].view(torch.int32).item()) == 0
    tickets = ws[256:256 + 4 * w.B].cpu().view(torch.int32)
    assert int(tickets.abs().sum()) == 0
    assert nbytes > 0


def test_cluster_sizes_agree(S, monkeypatch):
    """Every cluster size (vocabulary split) gives the oracle's tokens on the same inputs."""
    w = W.make(1, device="cuda", B=16)
    h = host_inputs(w)
    outs = []
    for cs in (1, 2, 4, 8, 16):
        if cs == 1 and w.V * 8 > 220 * 1024:
            continue
        monkeypatch.setenv("SPECVERIFY_CLUSTER", str(cs))
        em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T)
        st = S.accept_stats(w.target, w.draft, w.ids, w.T)
        n, flagged, mism = compare_sample(w, em, na, h)
        assert not mism, (cs, mism[:3])
        worst, _ = compare_stats(w, st, h)
        assert max(worst.values()) <= 1.0, (cs, worst)
        outs.append(em.cpu())
    assert S.check_status() == 0


@pytest.mark.parametrize("k", [1, 4])
def test_split_phases_agree_with_the_whole_call(S, k):
    """spec_verify_sample_stream then spec_verify_sample_draw (the two-kernel form) and spec_verify_sample
    (one launch) split the vocabulary differently, so their float32 sums round differently: both match the
    oracle, and their tokens are identical on every row that is not a boundary draw."""
    w = W.make(k, device="cuda", B=64 if k == 4 else None)
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len)
    em2 = torch.full_like(em, 7)
    na2 = torch.full_like(na, 7)
    S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, emitted=em2, n_accepted=na2,
                    phase="stream")
    S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, emitted=em2, n_accepted=na2,
                    phase="draw")
    assert S.check_status() == 0
    h = host_inputs(w)
    n, flagged, mism = compare_sample(w, em, na, h)
    assert not mism, mism[:3]
    n2, flagged2, mism2 = compare_sample(w, em2, na2, h)
    assert not mism2, mism2[:3]
    assert flagged == flagged2
    same = [b for b in range(w.B) if b not in set(flagged)]
    assert torch.equal(em[same], em2[same]) and torch.equal(na[same], na2[same])
