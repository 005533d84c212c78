"""Comparison of the CUDA path with the float64 oracle on the same seeded inputs.

Tolerances (also derived in the design notes):
  - tokens and n_accepted: bit-exact, except rows the oracle flags as boundary
    draws (a tested uniform within 1e-5 of its acceptance threshold, or the
    final uniform within 1e-5 of a CDF edge); those are counted, and the GPU
    output of such a row must still be well formed;
  - greedy: bit-exact, no exemption;
  - statistics p(x), q(x), min(1, p/q): relative 1e-5 (float32 logits) or 2e-3
    (bfloat16 logits), plus 1e-37 absolute for values in float32's subnormal
    range; beta and the residual mass: the same relative bound plus 1e-6
    absolute, the float32 rounding of sums over V terms of p and q
    (sum of |p - q| errors <= a few ulp x sum(p + q) = 2).  The absolute term is
    a departure from a purely relative 1e-5: a residual mass near 0 (beta near 1)
    cannot be summed to 1e-5 relative in float32.  The worst errors measured per
    statistic are written to the parity record.

The number of boundary rows is itself checked: it must stay below a cap derived
from the oracle's expected flag count E (the sum over rows of flag_prob, the
chance that fresh uniforms land in a flagged band), E + 4 sqrt(E) + 3.  A flag
rule that exempted many more rows than the bands' mass explains fails it.

With SPECVERIFY_PARITY_RECORD set to a path, each comparison appends one JSON
line (test, workload, rows compared, boundary rows by kind, expected flags, cap,
mismatches, worst statistic errors) to that file.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle as O
import workloads as W

RTOL = {"f32": 1e-5, "bf16": 2e-3}
ATOL_POINT = 1e-37
ATOL_SUM = 1e-6


def flag_cap(expected: float) -> float:
    """Largest boundary-row count accepted for an expected count E: E + 4 sqrt(E) + 3."""
    return expected + 4.0 * math.sqrt(expected) + 3.0


def record(entry: dict) -> None:
    """Appends one JSON line to the file SPECVERIFY_PARITY_RECORD names (nothing if it is unset)."""
    path = os.environ.get("SPECVERIFY_PARITY_RECORD")
    if not path:
        return
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "a") as f:
        f.write(json.dumps(entry, default=float) + "\n")


def host_inputs(w: W.Workload):
    return dict(target=W.logits_as_numpy(w.target), draft=W.logits_as_numpy(w.draft), dtype=w.dtype,
                ids=w.ids.cpu().numpy(), draft_len=None if w.draft_len is None else w.draft_len.cpu().numpy(),
                uniforms=w.uniforms.cpu().numpy(), T=w.T)


def check_well_formed(em_row, n, ids_row, gb, V):
    assert 0 <= n <= gb
    assert list(em_row[:n]) == list(ids_row[:n])
    assert 0 <= em_row[n] < V
    assert (em_row[n + 1:] == -1).all()


def sample_report(w: W.Workload, emitted: torch.Tensor, n_acc: torch.Tensor, h=None, rows=None, ref=None):
    """Token comparison with the oracle.  Returns a dict: compared, flagged (boundary rows), accept_boundary
    and draw_boundary counts, expected_flags (sum of the oracle's flag_prob over the rows), cap, mism."""
    h = h or host_inputs(w)
    if ref is None:
        ref = O.verify_sample(h["target"], h["draft"], h["dtype"], h["ids"], h["draft_len"], h["uniforms"],
                              h["T"], rows=rows)
    n, flagged, mism = _compare_rows(w, emitted, n_acc, h, rows, ref)
    sel = list(range(w.B) if rows is None else rows)
    acc_b = int(sum(bool(ref["accept_boundary"][b]) for b in flagged))
    expected = float(sum(ref["flag_prob"][b] for b in sel))
    return {"compared": n, "flagged": flagged, "accept_boundary": acc_b, "draw_boundary": len(flagged) - acc_b,
            "expected_flags": expected, "cap": flag_cap(expected), "mism": mism}


def report_entry(test: str, w: W.Workload, rep: dict, **extra) -> dict:
    """The parity record's line for one sampling comparison."""
    return {"test": test, "workload": w.name, "B": w.B, "gamma": w.gamma, "V": w.V, "dtype": w.dtype,
            "rows_compared": rep["compared"], "boundary_rows": len(rep["flagged"]),
            "accept_boundary_rows": rep["accept_boundary"], "draw_boundary_rows": rep["draw_boundary"],
            "expected_boundary_rows": round(rep["expected_flags"], 3), "boundary_cap": round(rep["cap"], 3),
            "mismatches": len(rep["mism"]), **extra}


def compare_sample(w: W.Workload, emitted: torch.Tensor, n_acc: torch.Tensor, h=None, rows=None):
    """Returns (number compared, boundary rows, mismatched rows)."""
    h = h or host_inputs(w)
    ref = O.verify_sample(h["target"], h["draft"], h["dtype"], h["ids"], h["draft_len"], h["uniforms"], h["T"],
                          rows=rows)
    return _compare_rows(w, emitted, n_acc, h, rows, ref)


def _compare_rows(w, emitted, n_acc, h, rows, ref):
    em = emitted.cpu().numpy()
    na = n_acc.cpu().numpy()
    gl = h["draft_len"] if h["draft_len"] is not None else np.full(w.B, w.gamma)
    mism, flagged, n = [], [], 0
    for b in (range(w.B) if rows is None else rows):
        n += 1
        if ref["boundary"][b]:
            flagged.append(b)
            if ref["valid"][b]:
                check_well_formed(em[b], int(na[b]), h["ids"][b], int(gl[b]), w.V)
                if not ref["accept_boundary"][b]:
                    # only the final draw is near a CDF edge: same walk, and a token within 1e-5 of the edge
                    nb = int(ref["n_accepted"][b])
                    if int(na[b]) != nb or list(em[b][:nb]) != list(ref["emitted"][b][:nb]) or \
                            int(em[b][nb]) not in ref["candidates"][b]:
                        mism.append((b, "boundary draw outside the 1e-5 candidates", int(na[b]), list(em[b]),
                                     nb, ref["candidates"][b]))
            continue
        if int(na[b]) != int(ref["n_accepted"][b]) or list(em[b]) != list(ref["emitted"][b]):
            mism.append((b, int(na[b]), list(em[b]), int(ref["n_accepted"][b]), list(ref["emitted"][b])))
    return n, flagged, mism


def compare_greedy(w: W.Workload, ids: torch.Tensor, emitted, n_acc, h=None, rows=None):
    h = h or host_inputs(w)
    ref = O.verify_greedy(h["target"], h["dtype"], ids.cpu().numpy(), h["draft_len"], rows=rows)
    em = emitted.cpu().numpy()
    na = n_acc.cpu().numpy()
    mism = []
    for b in (range(w.B) if rows is None else rows):
        if int(na[b]) != int(ref["n_accepted"][b]) or list(em[b]) != list(ref["emitted"][b]):
            mism.append((b, int(na[b]), list(em[b]), int(ref["n_accepted"][b]), list(ref["emitted"][b])))
    return mism


def compare_stats(w: W.Workload, st: dict, h=None, rows=None, rel=None):
    """Max normalised error per statistic (<= 1 passes) and the number of positions compared.  With a dict
    `rel`, also the worst plain relative error |gpu - oracle| / |oracle| per statistic (over nonzero
    oracle values) and the worst absolute error go into it, for the parity record."""
    h = h or host_inputs(w)
    ref = O.accept_stats(h["target"], h["draft"], h["dtype"], h["ids"], h["draft_len"], h["T"], rows=rows)
    rtol = RTOL[w.dtype]
    names = {"beta": "beta", "p_x": "p_x", "q_x": "q_x", "accept_prob": "accept_prob", "resid": "resid"}
    sel = np.zeros((w.B, w.gamma), dtype=bool)
    for b in (range(w.B) if rows is None else rows):
        sel[b] = True
    worst = {}
    for k, rk in names.items():
        g = st[k].cpu().numpy().astype(np.float64)
        o = ref[rk]
        valid = ref["valid"] & sel
        atol = ATOL_SUM if k in ("beta", "resid") else ATOL_POINT
        err = np.abs(g[valid] - o[valid]) / (rtol * np.abs(o[valid]) + atol)
        worst[k] = float(err.max()) if err.size else 0.0
        if rel is not None:
            nz = valid & (o != 0)
            r = np.abs(g[nz] - o[nz]) / np.abs(o[nz])
            rel[k] = float(r.max()) if r.size else 0.0
            rel[k + "_abs"] = float(np.abs(g[valid] - o[valid]).max()) if valid.any() else 0.0
        # positions the oracle does not compute are NaN on both sides
        inval = sel & ~ref["valid"]
        assert np.isnan(g[inval]).all(), k
    return worst, int((ref["valid"] & sel).sum())
