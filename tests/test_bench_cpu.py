"""bench.py's host-side contract, without a GPU: the reference arm's JSON line, the CPU-baseline parity count,
the rule that the recorded DRAM traffic is only reported for the kernel sources it was taken on, and the
logit copies the timed steps take in turn."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np

import bench
import oracle as O
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "c1", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["warmup"] >= 3 and d["value"] > 0 and d["higher_is_better"] is True
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"]["workload"].startswith("c1") and d["config"]["B"] == 8
    # whole batches: the claimed time is the timed steps' own wall time
    assert d["steps"] == 2 and d["ms_per_step"] > 0
    assert abs(d["value"] - d["config"]["positions_per_step"] / (d["ms_per_step"] * 1e-3)) < 1e-6 * d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_counts_parity_against_given_outputs():
    w = W.make(0, device="cpu")
    h = {"target": W.logits_as_numpy(w.target), "draft": W.logits_as_numpy(w.draft)}
    ref = O.verify_sample(h["target"], h["draft"], w.dtype, w.ids.numpy(), None, w.uniforms.numpy(), w.T)
    import torch
    em = torch.tensor(np.asarray(ref["emitted"], dtype=np.int32))
    na = torch.tensor(np.asarray(ref["n_accepted"], dtype=np.int32))
    out = bench.cpu_oracle_rate(w, 4, 1, gpu=(em, na))
    assert out["parity"]["rows_compared"] == 1 and out["parity"]["mismatches"] == 0
    assert out["cores"] == 1 and out["value"] > 0
    bad = em.clone()
    bad[0, int(na[0])] = (int(bad[0, int(na[0])]) + 1) % w.V      # a different drawn token
    out = bench.cpu_oracle_rate(w, 1, 1, gpu=(bad, na))
    assert out["parity"]["mismatches"] + out["parity"]["boundary_rows"] == 1


def test_recorded_traffic_follows_the_sources_digest(tmp_path, monkeypatch):
    digest = bench.kernel_sources_digest()
    assert len(digest) == 16 and digest == bench.kernel_sources_digest()
    f = tmp_path / "traffic.txt"
    f.write_text(f"# comment: ignored\nsources_digest: {digest}\nc3_bytes_per_launch: 1234\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("c3") == 1234.0
    assert bench.recorded_traffic("c2") is None
    f.write_text("sources_digest: 0000000000000000\nc3_bytes_per_launch: 1234\n")
    assert bench.recorded_traffic("c3") is None


def test_rotation_gives_distinct_copies_of_the_same_logits():
    w = W.make(0, device="cpu")
    copies = bench.rotation(w)
    assert len(copies) == 3
    assert copies[0][0] is w.target and copies[0][1] is w.draft
    ptrs = {t.data_ptr() for t, _ in copies} | {d.data_ptr() for _, d in copies}
    assert len(ptrs) == 6                       # six separate buffers: no step re-reads another's memory
    for t, d in copies[1:]:
        assert t.equal(w.target) and d.equal(w.draft)
