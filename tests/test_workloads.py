"""Seeded input generators: determinism, shapes and the structure each workload promises (CPU)."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from workloads.philox import normal_f32, random_words, uniform_f32


def test_philox_is_deterministic_and_offset_consistent():
    a = random_words(1000, 5, 9)
    b = random_words(600, 5, 9, offset=400)
    assert torch.equal(a[400:], b)
    assert not torch.equal(random_words(100, 5, 9), random_words(100, 5, 10))
    assert int(a.min()) >= 0 and int(a.max()) < 2 ** 32


def test_uniform_and_normal_moments():
    u = uniform_f32((400000,), 3, 1).double()
    assert abs(u.mean().item() - 0.5) < 3e-3 and abs(u.var().item() - 1 / 12) < 2e-3
    assert u.min().item() >= 0.0 and u.max().item() < 1.0
    z = normal_f32((400000,), 3, 2).double()
    assert abs(z.mean().item()) < 1e-2 and abs(z.var().item() - 1.0) < 1e-2


def test_c0_c1_shapes_and_draft_law():
    w0 = W.make(0)
    assert w0.target.shape == (1, 5, 1024) and w0.target.dtype == torch.float32
    assert w0.uniforms.shape == (1, 5) and w0.ids.shape == (1, 4)
    w1 = W.make(1)
    assert w1.target.dtype == torch.bfloat16 and w1.draft.shape == (8, 4, 32128)
    assert torch.equal(W.make(1).ids, w1.ids)            # seeded
    assert not torch.equal(W.make(0, call=1).target, w0.target)
    # greedy drafts are the argmax of the draft logits
    assert torch.equal(w1.greedy_ids, torch.argmax(w1.draft.float(), dim=2).to(torch.int32))


def test_gumbel_drafts_follow_q():
    """x ~ softmax(l/T) by Gumbel-max: empirical frequencies match the softmax."""
    V, n, T = 5, 200000, 0.7
    logits = torch.tensor([0.0, 1.0, -0.5, 2.0, float("-inf")])
    d = logits.view(1, 1, V).expand(n, 1, V).contiguous()
    ids = W._gumbel_drafts(d, T, 77, 3).flatten()
    freq = torch.bincount(ids.long(), minlength=V).double() / n
    q = torch.softmax(logits.double() / T, 0)
    assert freq[4] == 0
    assert torch.max(torch.abs(freq - q)).item() < 5e-3


def test_c4_row_mix_and_padding():
    B, g, V = 120, 8, 32000          # the c4 recipe on fewer rows
    w = W.make(4, B=B)
    gl = w.draft_len
    assert gl.min().item() >= 1 and gl.max().item() <= 8
    kinds = w.row_kind
    assert [(kinds == c).sum().item() for c in range(4)] == [84, 12, 12, 12]
    t, d = w.target.float(), w.draft.float()
    for b in range(B):
        gb = int(gl[b])
        assert torch.isnan(t[b, gb + 1:]).all() and torch.isnan(d[b, gb:]).all()
        assert (w.ids[b, gb:] == -1).all() and torch.isnan(w.uniforms[b, gb:g]).all()
        assert torch.isfinite(w.uniforms[b, g])
        k = int(kinds[b])
        if k == W.ROW_P_EQ_Q:
            assert torch.equal(w.target[b, :gb].view(torch.int16), w.draft[b, :gb].view(torch.int16))
        elif k == W.ROW_DISJOINT:
            tf = torch.isfinite(t[b, :gb])
            df = torch.isfinite(d[b, :gb])
            assert not (tf & df).any() and tf.any(dim=1).all() and df.any(dim=1).all()
        elif k == W.ROW_ONE_HOT:
            assert (torch.isfinite(t[b, :gb + 1]).sum(dim=1) == 1).all()


def test_c2_sigma_table():
    sig = W.load_c2_sigma()
    assert sig is not None and len(sig) == 64 and all(0.0 < s < 10.0 for s in sig)


def test_logits_as_numpy_round_trips_bf16_bits():
    x = torch.tensor([1.0, -2.5, float("inf"), float("-inf")], dtype=torch.bfloat16)
    a = W.logits_as_numpy(x)
    assert a.dtype == np.uint16 and list(a) == [0x3F80, 0xC020, 0x7F80, 0xFF80]
