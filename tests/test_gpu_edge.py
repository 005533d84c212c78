"""Edge cases of the CUDA path against the oracle (GPU): ragged tails, unaligned rows, degenerate sizes,
invalid inputs reported through the device error word, ties in greedy mode."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity import compare_greedy, compare_sample, compare_stats, host_inputs
from workloads.philox import normal_f32, uniform_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_40_gb300 as S
    return S


def make_case(B, gamma, V, dtype="f32", T=1.0, sigma=1.0, seed=5, ragged=False, storage_offset=0):
    """Random logits of the c-workload kind at arbitrary sizes; optionally unaligned rows."""
    dev = "cuda"
    t = 2.0 * normal_f32((B, gamma + 1, V), seed, 1, dev) + W.zipf_log_prior(V, 1.1, dev)
    d = t[:, :gamma] + sigma * normal_f32((B, gamma, V), seed, 2, dev)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t, d = t.to(tdt), d.to(tdt)
    if storage_offset:
        tt = torch.empty(t.numel() + storage_offset, dtype=tdt, device=dev)[storage_offset:].view(t.shape)
        tt.copy_(t)
        dd = torch.empty(d.numel() + storage_offset, dtype=tdt, device=dev)[storage_offset:].view(d.shape)
        dd.copy_(d)
        t, d = tt, dd
    ids = W._gumbel_drafts(d, T, seed, 3) if gamma else torch.zeros(B, 0, dtype=torch.int32, device=dev)
    u = uniform_f32((B, gamma + 1), seed, 4, dev)
    gl = None
    if ragged:
        gl = torch.floor((gamma + 1) * uniform_f32((B,), seed, 5, dev)).to(torch.int32)  # 0..gamma
    return W.Workload(name=f"B{B}g{gamma}V{V}{dtype}", B=B, gamma=gamma, V=V, dtype=dtype, T=T, target=t,
                      draft=d, ids=ids, uniforms=u, draft_len=gl,
                      greedy_ids=torch.argmax(d.float(), dim=2).to(torch.int32) if gamma else ids)


@pytest.mark.parametrize("B,gamma,V,dtype,ragged,offset", [
    (3, 2, 5000, "f32", False, 0),        # one CTA, 40 chunks, ragged last chunk
    (5, 3, 50001, "f32", True, 0),        # V*4 not a multiple of 16: scalar load path
    (5, 3, 50001, "bf16", True, 0),
    (4, 4, 77777, "bf16", False, 0),
    (6, 2, 20000, "f32", False, 1),       # rows start off a 16-byte boundary
    (6, 2, 20000, "bf16", True, 3),
    (2, 1, 262144, "bf16", False, 0),     # largest vocabulary
    (2, 1, 262144, "f32", False, 0),
    (3, 0, 3000, "f32", False, 0),        # gamma = 0: one inverse-CDF draw from p_1
    (4, 5, 1, "f32", False, 0),           # V = 1
    (7, 6, 130, "bf16", True, 0),
    (64, 8, 4096, "bf16", True, 0),       # many rows, ragged draft lengths including 0
])
def test_odd_sizes_match_oracle(S, B, gamma, V, dtype, ragged, offset):
    w = make_case(B, gamma, V, dtype, T=0.9, ragged=ragged, storage_offset=offset)
    h = host_inputs(w)
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len)
    assert S.check_status() == 0
    n, flagged, mism = compare_sample(w, em, na, h)
    assert not mism, mism[:3]
    gem, gna = S.verify_greedy(w.target, w.greedy_ids, w.draft_len)
    assert not compare_greedy(w, w.greedy_ids, gem, gna, h)
    if gamma:
        st = S.accept_stats(w.target, w.draft, w.ids, w.T, w.draft_len)
        worst, _ = compare_stats(w, st, h)
        assert max(worst.values()) <= 1.0, worst
    assert S.check_status() == 0


def test_empty_batch(S):
    t = torch.empty(0, 5, 100, device="cuda")
    em, na = S.verify_sample(t, torch.empty(0, 4, 100, device="cuda"), torch.empty(0, 4, dtype=torch.int32,
                             device="cuda"), torch.empty(0, 5, device="cuda"), 1.0)
    assert em.shape == (0, 5) and na.shape == (0,)


def _invalid_case():
    w = make_case(8, 3, 3000, "f32", T=1.0)
    return w


@pytest.mark.parametrize("what,code", [("nan_target", 4), ("posinf_draft", 4), ("allneg_target", 4),
                                       ("id_range", 5), ("u_range", 1), ("u_final", 1), ("len_range", 1)])
def test_invalid_rows_are_reported_and_isolated(S, what, code):
    w = _invalid_case()
    bad = 3
    gl = torch.full((w.B,), w.gamma, dtype=torch.int32, device="cuda")
    if what == "nan_target":
        w.target[bad, 3, 17] = float("nan")        # the bonus row: invalid even if never drawn from
    elif what == "posinf_draft":
        w.draft[bad, 1, 5] = float("inf")
    elif what == "allneg_target":
        w.target[bad, 0] = float("-inf")
    elif what == "id_range":
        w.ids[bad, 2] = w.V
    elif what == "u_range":
        w.uniforms[bad, 1] = 1.0
    elif what == "u_final":
        w.uniforms[bad, w.gamma] = -0.25
    elif what == "len_range":
        gl[bad] = w.gamma + 1
    w.draft_len = gl
    h = host_inputs(w)
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, gl)
    assert S.check_status(raise_on_error=False) == code
    assert S.check_status(raise_on_error=False) == 0        # reading clears the word
    assert int(na[bad]) == -1 and (em[bad] == -1).all()
    n, flagged, mism = compare_sample(w, em, na, h)
    assert not mism
    ref = O.verify_sample(h["target"], h["draft"], "f32", h["ids"], h["draft_len"], h["uniforms"], w.T)
    assert not ref["valid"][bad] and ref["valid"].sum() == w.B - 1
    gem, gna = S.verify_greedy(w.target, w.ids, gl)
    gcode = S.check_status(raise_on_error=False)
    if what in ("nan_target", "allneg_target", "id_range", "len_range"):   # greedy reads target rows and ids only
        assert int(gna[bad]) == -1 and gcode == code
    else:
        assert int(gna[bad]) >= 0 and gcode == 0
    assert not compare_greedy(w, w.ids, gem, gna, h)


def test_padding_is_never_read(S):
    """NaN logits, ids of -1 and NaN uniforms beyond draft_len do not invalidate a row."""
    w = make_case(16, 6, 2048, "bf16", ragged=True)
    gl = w.draft_len
    for b in range(w.B):
        gb = int(gl[b])
        w.target[b, gb + 1:] = float("nan")
        w.draft[b, gb:] = float("nan")
        w.ids[b, gb:] = -1
        w.uniforms[b, gb:w.gamma] = float("nan")
    h = host_inputs(w)
    em, na = S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, gl)
    assert S.check_status() == 0
    n, flagged, mism = compare_sample(w, em, na, h)
    assert not mism and (na.cpu() >= 0).all()


def test_greedy_ties_and_signed_zero(S):
    V = 64
    t = torch.full((4, 3, V), -5.0, device="cuda")
    t[0, 0, [7, 9, 40]] = 3.0          # three-way tie: lowest index 7
    t[0, 1, [2, 3]] = 1.5
    t[1, 0] = -1.0
    t[1, 0, 10] = -0.0                  # -0 and +0 tie: lowest index wins
    t[1, 0, 20] = 0.0
    t[1, 0, 5] = 0.0
    t[2, :, :] = 0.0                    # all equal: index 0 everywhere
    t[3, 0, 63] = 1.0
    t[3, 1, 0] = 1.0
    ids = torch.tensor([[7, 2], [5, 0], [0, 0], [63, 1]], dtype=torch.int32, device="cuda")
    for dt in (torch.float32, torch.bfloat16):
        tt = t.to(dt)
        em, na = S.verify_greedy(tt, ids)
        assert S.check_status() == 0
        ref = O.verify_greedy(W.logits_as_numpy(tt), "bf16" if dt == torch.bfloat16 else "f32", ids.cpu().numpy(),
                              None)
        assert np.array_equal(em.cpu().numpy(), ref["emitted"]), (em, ref["emitted"])
        assert np.array_equal(na.cpu().numpy(), ref["n_accepted"])
    assert em[0].tolist() == [7, 2, 0] and em[1].tolist() == [5, 0, 0] and em[3].tolist() == [63, 0, -1]


def test_one_hot_and_identical_rows_without_boundary_exemption(S):
    V, gamma, B = 1000, 4, 32
    base = normal_f32((B, gamma + 1, V), 9, 1, "cuda")
    hot = torch.randint(0, V, (B, gamma + 1), generator=torch.Generator().manual_seed(1)).cuda()
    onehot = torch.full_like(base, float("-inf")).scatter_(2, hot.unsqueeze(2), 0.0)
    d = base[:, :gamma].contiguous()
    ids = W._gumbel_drafts(d, 1.0, 3, 3)
    u = uniform_f32((B, gamma + 1), 9, 4, "cuda")
    em, na = S.verify_sample(onehot, d, ids, u, 1.0)
    em, na = em.cpu(), na.cpu()
    for b in range(B):
        n = int(na[b])
        assert int(em[b, n]) == int(hot[b, n])
        for i in range(n):
            assert int(ids[b, i]) == int(hot[b, i])
    same = base.contiguous()
    em, na = S.verify_sample(same, same[:, :gamma].contiguous(), ids, u, 1.0)
    assert (na == gamma).all()
    assert S.check_status() == 0


@pytest.mark.parametrize("dtype,V", [("f32", 5000), ("f32", 70000), ("bf16", 40000)])
def test_degenerate_residual_draws_from_p(S, dtype, V):
    """R4 on the GPU: the draft token has p(x) = 0 (always rejected) and q(x) ~ 1e-17, every other logit
    equal, so the residual max(0, p - q) has mass ~1e-17 <= 1e-15 and the draw falls back to p."""
    B, gamma = 16, 1
    base = 2.0 * normal_f32((B, 1, V), 71, V, "cuda")
    t = torch.cat([base, base], dim=1).clone()
    d = base.clone()
    ids = torch.randint(0, V, (B, 1), generator=torch.Generator("cuda").manual_seed(3), device="cuda",
                        dtype=torch.int32)
    rows = torch.arange(B, device="cuda")
    mx = base.amax(dim=2)[:, 0]
    t[rows, 0, ids[:, 0].long()] = float("-inf")           # p(x) = 0
    d[rows, 0, ids[:, 0].long()] = mx - 40.0               # q(x) about e^-40 of the top token
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t, d = t.to(tdt).contiguous(), d.to(tdt).contiguous()
    u = uniform_f32((B, gamma + 1), 72, V, "cuda")
    w = W.Workload(name="degenerate", B=B, gamma=gamma, V=V, dtype=dtype, T=1.0, target=t, draft=d, ids=ids,
                   uniforms=u)
    em, na = S.verify_sample(t, d, ids, u, 1.0)
    assert S.check_status() == 0
    assert bool((na == 0).all())
    n, flagged, mism = compare_sample(w, em, na)
    assert not mism, mism[:3]
