"""The C-ABI library loads, exports every declared symbol, and rejects bad arguments on the host (CPU only).

No call here reaches a CUDA compute path: every rejected call fails validation
before the library touches the device.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import speculative_decoding_verification_40_gb300 as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "spec_verify_sample" in names and "spec_verify_greedy" in names and "spec_accept_stats" in names
    lib = ctypes.CDLL(S.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size():
    assert S.lib.spec_workspace_size(64, 8, 128256, 1) >= 256 + 64 * 4 + 64 * 9 * 16
    assert S.lib.spec_workspace_size(-1, 8, 100, 0) == 0
    assert S.lib.spec_workspace_size(1, 65, 100, 0) == 0
    assert S.lib.spec_workspace_size(1, 4, 0, 0) == 0
    assert S.lib.spec_workspace_size(1, 4, 100, 7) == 0


FAKE_WS = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: validation fails first
BIG = 1 << 40


def sample(**kw):
    a = dict(t=ctypes.c_void_p(4096), d=ctypes.c_void_p(8192), dtype=0, ids=ctypes.c_void_p(12288), gl=None,
             u=ctypes.c_void_p(16384), T=1.0, B=2, G=3, V=100, em=ctypes.c_void_p(20480),
             na=ctypes.c_void_p(24576), ws=FAKE_WS, wsb=BIG, st=None)
    a.update(kw)
    return S.lib.spec_verify_sample(a["t"], a["d"], a["dtype"], a["ids"], a["gl"], a["u"], a["T"], a["B"], a["G"],
                                    a["V"], a["em"], a["na"], a["ws"], a["wsb"], a["st"])


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=3), 2),
    (dict(B=-1), 1),
    (dict(G=65), 1),
    (dict(G=-1), 1),
    (dict(V=0), 1),
    (dict(V=262145), 1),
    (dict(ws=None), 7),
    (dict(ws=ctypes.c_void_p((1 << 20) + 8)), 7),
    (dict(wsb=16), 7),
    (dict(T=0.0), 1),
    (dict(T=-1.0), 1),
    (dict(T=float("nan")), 1),
    (dict(T=float("inf")), 1),
    (dict(t=None), 1),
    (dict(d=None), 1),
    (dict(ids=None), 1),
    (dict(u=None), 1),
    (dict(em=None), 1),
    (dict(na=None), 1),
])
def test_sample_rejects_bad_arguments_on_the_host(kw, code):
    assert sample(**kw) == code


def test_empty_batch_is_a_no_op():
    assert sample(B=0, t=None, d=None, ids=None, u=None, em=None, na=None, ws=None) == 0


def test_greedy_and_stats_reject_bad_arguments():
    L = S.lib
    assert L.spec_verify_greedy(None, None, 0, ctypes.c_void_p(64), None, 1, 2, 10, ctypes.c_void_p(64),
                                ctypes.c_void_p(64), FAKE_WS, BIG, None) == 1
    assert L.spec_verify_greedy(ctypes.c_void_p(64), None, 9, None, None, 1, 2, 10, None, None, FAKE_WS, BIG,
                                None) == 2
    assert L.spec_accept_stats(ctypes.c_void_p(64), ctypes.c_void_p(64), 0, ctypes.c_void_p(64), None, 0.0, 1, 2,
                               10, None, None, None, None, None, FAKE_WS, BIG, None) == 1
    assert L.spec_accept_stats(None, None, 1, None, None, 1.0, 0, 2, 10, None, None, None, None, None, None, 0,
                               None) == 0


def test_status_strings():
    for code in range(9):
        assert S.lib.spec_status_string(code).decode() == S.STATUS[code]


@pytest.mark.parametrize("B,G,V,bf16,cs", [(1, 4, 1024, 0, 1), (8, 4, 32128, 1, 1), (64, 8, 128256, 1, 4),
                                           (256, 5, 152064, 0, 10), (1024, 8, 32000, 1, 1)])
def test_launch_plans_for_the_five_workloads(B, G, V, bf16, cs, monkeypatch):
    monkeypatch.delenv("SPECVERIFY_CLUSTER", raising=False)
    import torch
    p = S.plan(B, G, V, torch.bfloat16 if bf16 else torch.float32)
    assert p["cluster_size"] == cs
    assert p["slice_len"] * cs >= V and p["slice_len"] % 8 == 0
    assert p["smem_bytes"] <= 227 * 1024


@pytest.mark.parametrize("B,G,V,ctas", [
    (8, 4, 32128, 8),       # c1: 40 positions x 4 slices of 8192 < 2 x 152 SMs -> slices of 4096
    (1, 4, 1024, 1),        # c0: one slice whatever its size
    (2, 1, 16384, 8),       # 4 positions: halved down to the 2048-element floor
    (64, 8, 128256, 16),    # c2: 576 positions fill the GPU at 8192
    (256, 5, 152064, 19),   # c3
])
def test_greedy_slices_fill_the_gpu_for_small_batches(B, G, V, ctas):
    # without a device the rule assumes 152 SMs: slices of 8192 target elements, halved (to 2048 at
    # least) while the batch gives fewer than two CTAs per SM
    import torch
    assert S.plan(B, G, V, torch.bfloat16)["greedy_ctas_per_row"] == ctas


def test_sample_rows_rejects_bad_arguments_on_the_host():
    L = S.lib
    p = ctypes.c_void_p(4096)

    def call(logits=p, dtype=0, u=p, T=1.0, R=3, V=100, tok=p, ws=FAKE_WS, wsb=BIG):
        return L.spec_sample_rows(logits, dtype, u, T, R, V, tok, ws, wsb, None)

    assert call(dtype=5) == 2
    assert call(R=-1) == 1
    assert call(V=0) == 1
    assert call(V=262145) == 1
    assert call(T=0.0) == 1
    assert call(T=float("nan")) == 1
    assert call(logits=None) == 1
    assert call(u=None) == 1
    assert call(tok=None) == 1
    assert call(ws=None) == 7
    assert call(wsb=16) == 7
    assert call(R=0, logits=None, u=None, tok=None, ws=None, wsb=0) == 0


def test_lenient_rejects_lenience_outside_unit_interval():
    L = S.lib
    p = ctypes.c_void_p(4096)
    for l in (0.0, -0.5, 1.5, float("nan")):
        assert L.spec_verify_sample_lenient(p, p, 0, p, None, p, 1.0, l, 2, 3, 100, p, p, FAKE_WS, BIG, None) == 1
