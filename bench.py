"""Throughput of the batched speculative-sampling verification step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload c3]

A step is one spec_verify_sample call (accept test, first rejection, residual
/ bonus inverse-CDF draw; every row of the hot path) over one batch of the
seeded synthetic workload, inputs resident in HBM.  The default workload is c3
(B=256, gamma=5, V=152064, fp32 logits, T=0.7): 1.71 GB of logits per call,
13x the L2; three copies of the logits are used in turn, so no call reads
logits an earlier call left in L2.  Prints one JSON line.

--impl reference times the float64 CPU oracle (the only reference
implementation of the method: the pages it follows publish no code) on the
same workload, batch and metric: every step verifies the whole batch on all
host cores.  Under torchrun each rank runs its own replica of the
workload on its own GPU (no data-path collective); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
METRIC = "verified draft positions/sec"
UNIT = "positions/s"


# ----------------------------------------------------------------------------- ranks

def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dist.init_process_group(backend=backend)
    return dist.get_rank(), ws, dist


def combine_ranks(elapsed_s: float, units: float, dist, device=None):
    """Max elapsed time and total units over ranks (the whole-job aggregate)."""
    if dist is None:
        return elapsed_s, units
    t = torch.tensor([elapsed_s, units], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[1])


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock, power and throttle reasons while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict | None:
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[5].lower() == "active", hwt=f[6].lower() == "active",
                                 swt=f[7].lower() == "active", pcap=f[8].lower() == "active"))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            if r["hw"]:
                reasons.add("hw_slowdown")
            if r["hwt"]:
                reasons.add("hw_thermal_slowdown")
            if r["swt"]:
                reasons.add("sw_thermal_slowdown")
            if r["pcap"]:
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "power_w_max": max(r["power"] for r in rows), "reasons": sorted(reasons), "samples": len(rows),
                "window": "timed region plus about 1 s of untimed calls before it"}


# ----------------------------------------------------------------------------- helpers

def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources the stream kernel (verify_stream_kernel, the roofline's kernel) is built from.
STREAM_KERNEL_SOURCES = ("common.cuh", "kernels.h", "sample.cu", "softmax.cuh", "verify_common.cuh")


def kernel_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_40_gb300", "csrc")
    for name in STREAM_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel sources."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for ln in f:
                if ":" in ln and not ln.startswith("#"):
                    k, v = ln.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("sources_digest") != kernel_sources_digest():
            return None
        return float(kv[f"{workload}_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None


def workload_desc(w: W.Workload) -> dict:
    return {"workload": f"{w.name}: {w.meta['desc']}", "B": w.B, "gamma": w.gamma, "V": w.V,
            "logits": "fp32" if w.dtype == "f32" else "bf16", "T": w.T, "positions_per_step": w.positions(),
            "read_once_bytes_per_step": w.read_once_bytes()}


def rotation(w: W.Workload, n: int = 3):
    """n copies of the workload's logits (the first is the workload's own), to be used in turn."""
    return [(w.target, w.draft)] + [(w.target.clone(), w.draft.clone()) for _ in range(n - 1)]


def time_device(fn, steps: int, warmup: int, stream):
    """Average device milliseconds per call: CUDA events on the launching stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


# ----------------------------------------------------------------------------- CPU oracle

def oracle_pool(procs: int):
    """Process pool for the oracle, started with spawn (safe after CUDA initialisation)."""
    import multiprocessing as mp
    return mp.get_context("spawn").Pool(procs)


def _oracle_rows(args):
    import oracle as O
    target, draft, dtype, ids, gl, u, T = args
    r = O.verify_sample(target, draft, dtype, ids, gl, u, T)
    return r["emitted"], r["n_accepted"], r["boundary"]


def cpu_oracle_rate(w: W.Workload, rows: int, procs: int, pool=None, gpu=None) -> dict:
    """Oracle positions/s over the first `rows` rows (repeated over the batch as needed), on `procs` processes.

    With gpu = (emitted, n_accepted) of the same batch, the oracle's outputs on the distinct rows of the
    sample are compared with the GPU's (token-exact outside the oracle's boundary rows) and counted."""
    h = {"target": W.logits_as_numpy(w.target), "draft": W.logits_as_numpy(w.draft),
         "ids": w.ids.cpu().numpy(), "gl": None if w.draft_len is None else w.draft_len.cpu().numpy(),
         "u": w.uniforms.cpu().numpy()}
    idx = [r % w.B for r in range(rows)]
    per = max(1, math.ceil(rows / max(1, procs)))
    chunks = [idx[s:s + per] for s in range(0, rows, per)]
    jobs = [(h["target"][c], h["draft"][c], w.dtype, h["ids"][c], None if h["gl"] is None else h["gl"][c],
             h["u"][c], w.T) for c in chunks]
    positions = sum(w.gamma if h["gl"] is None else int(h["gl"][r]) for r in idx)
    if procs <= 1:
        t0 = time.perf_counter()
        res = [_oracle_rows(j) for j in jobs]
        dt = time.perf_counter() - t0
    elif pool is not None:
        t0 = time.perf_counter()
        res = pool.map(_oracle_rows, jobs)
        dt = time.perf_counter() - t0
    else:
        with oracle_pool(procs) as pool:
            pool.map(_oracle_rows, jobs[:procs])       # start-up and imports outside the timing
            t0 = time.perf_counter()
            res = pool.map(_oracle_rows, jobs)
            dt = time.perf_counter() - t0
    out = {"value": positions / dt, "unit": UNIT, "cores": procs, "kind": "oracle",
           "sample": f"{rows} rows of {w.name} (float64 numpy oracle, {positions} positions) in {dt:.2f} s"}
    if gpu is not None:
        em, na = (t.cpu().numpy() for t in gpu)
        seen, checked, boundary, mism = set(), 0, 0, 0
        for c, (r_em, r_na, r_bd) in zip(chunks, res):
            for j, b in enumerate(c):
                if b in seen:
                    continue
                seen.add(b)
                checked += 1
                if r_bd[j]:
                    boundary += 1
                elif int(na[b]) != int(r_na[j]) or list(em[b]) != list(r_em[j]):
                    mism += 1
        out["parity"] = {"rows_compared": checked, "boundary_rows": boundary, "mismatches": mism}
    return out


# ----------------------------------------------------------------------------- arms

def gpu_local_cpus(index: int):
    """The host CPUs local to CUDA device `index` and their NUMA node, from the PCI device's sysfs entries
    (local_cpulist, numa_node), restricted to the CPUs this process may use; None if unknown."""
    try:
        p = torch.cuda.get_device_properties(index)
        dom, bus, devn = (getattr(p, k, None) for k in ("pci_domain_id", "pci_bus_id", "pci_device_id"))
        if None in (dom, bus, devn):
            return None
        base = f"/sys/bus/pci/devices/{dom:04x}:{bus:02x}:{devn:02x}.0"
        with open(base + "/local_cpulist") as f:
            spec = f.read().strip()
        with open(base + "/numa_node") as f:
            node = int(f.read().strip())
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        cpus &= os.sched_getaffinity(0)
        return {"cpus": cpus, "node": node} if cpus else None
    except (OSError, ValueError, AttributeError, RuntimeError):
        return None


def early_form(w: W.Workload) -> str:
    """Which form spec_verify_sample_early_exit takes for this batch (the library's rule: one launch when a
    position of the batch, 2 B V logits, is at least 64 MB)."""
    esz = 4 if w.dtype == "f32" else 2
    return "one-launch cluster kernel" if 2 * w.B * w.V * esz >= (64 << 20) else "two-kernel path, early-exit validity"


def c0_latency(S, dev, stream, ncalls: int = 50, reps: int = 20) -> dict:
    """c0 (B=1, gamma=4, V=1024): microseconds per call over independent calls, launched one by one and
    replayed from a captured CUDA graph (the library's calls are launches only, so they capture)."""
    calls = [W.make(0, device=dev, call=c) for c in range(ncalls)]
    ws = S.workspace_for(dev, S.workspace_size(1, 4, 1024, torch.float32))
    em = torch.empty(1, 5, dtype=torch.int32, device=dev)
    na = torch.empty(1, dtype=torch.int32, device=dev)

    def run_all():
        for w in calls:
            S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, emitted=em, n_accepted=na, workspace=ws)

    plain = time_device(run_all, reps, 3, stream) * 1e3 / ncalls
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        run_all()                                   # first calls (plan caches) outside the capture
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_all()
    graphed = time_device(graph.replay, reps, 3, stream) * 1e3 / ncalls
    assert S.check_status(ws) == 0
    return {"us_per_call": round(plain, 2), "us_per_call_cuda_graph": round(graphed, 2), "calls": ncalls}


def call_latency(fn, dev, stream, calls: int = 50, reps: int = 10):
    """Microseconds per call of fn: launched one by one, and replayed from a CUDA graph of `calls` calls."""
    def run_all():
        for _ in range(calls):
            fn()

    plain = time_device(run_all, reps, 3, stream) * 1e3 / calls
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        run_all()                                   # first calls (plan caches) outside the capture
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_all()
    graphed = time_device(graph.replay, reps, 3, stream) * 1e3 / calls
    return round(plain, 2), round(graphed, 2)


def run_ours(a, rank, world, dist):
    import speculative_decoding_verification_40_gb300 as S
    dev = torch.device("cuda", torch.cuda.current_device())
    k = int(a.workload.lstrip("c"))
    w = W.make(k, device=dev, B=a.batch or None)
    stream = torch.cuda.current_stream(dev)
    pos = w.positions()
    nbytes = w.read_once_bytes()
    ws = S.workspace_for(dev, S.workspace_size(w.B, w.gamma, w.V, w.target.dtype))
    em = torch.empty(w.B, w.gamma + 1, dtype=torch.int32, device=dev)
    na = torch.empty(w.B, dtype=torch.int32, device=dev)
    # Three copies of the logits, used in turn: a step never finds its logits in L2 from an earlier step
    # (with one copy, the rows the previous step's draw kernel read are still in L2 when the next step
    # streams them -- a reuse that fresh logits from a model never offer).
    copies = rotation(w)
    turn = [0]

    def logits():
        t, d = copies[turn[0] % len(copies)]
        turn[0] += 1
        return t, d

    def phase(ph, td=None):
        t, d = td or logits()
        S.verify_sample(t, d, w.ids, w.uniforms, w.T, w.draft_len, emitted=em, n_accepted=na,
                        workspace=ws, phase=ph)

    def step():
        phase("both")

    for _ in range(max(3, a.warmup)):
        step()
    torch.cuda.synchronize()
    assert S.check_status(ws) == 0

    # A step is one spec_verify_sample call: the stream kernel, then the draw kernel launched as its
    # programmatic dependent.  The timed steps are those calls; right after them the same steps run as
    # the two halves with events between them on the launching stream, which times the stream kernel
    # (the dominant one) live -- an event between the launches costs the draw kernel its early launch,
    # so the step time is not taken from that loop.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        # about 1 s of untimed calls so the clock samples see the GPU under this load
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
        barrier(dist, dev)
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(a.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(dist, dev)
        elapsed = start.elapsed_time(end) / 1e3
        for k in range(a.steps):
            td = logits()
            ev[k][0].record(stream)
            phase("stream", td)
            ev[k][1].record(stream)
            phase("draw", td)
        torch.cuda.synchronize()
    clocks = clk.summary()
    assert S.check_status(ws) == 0
    stream_ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / a.steps
    t_max, units = combine_ranks(elapsed, float(pos * a.steps), dist, dev)
    ms_per_step = elapsed * 1e3 / a.steps
    step_gbs = nbytes / (ms_per_step * 1e-3) / 1e9
    achieved = nbytes / (stream_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    traffic = recorded_traffic(w.name)

    # end to end through the public API: pinned host inputs -> device -> verify -> host results.  The
    # pinned buffers are allocated from the CPUs local to the GPU (so their pages sit on its host NUMA
    # node), unless --e2e-numa any.
    local = gpu_local_cpus(dev.index) if a.e2e_numa == "local" else None
    saved = os.sched_getaffinity(0) if local else None
    if local:
        os.sched_setaffinity(0, local["cpus"])
    try:
        host = {n: getattr(w, n).cpu().pin_memory() for n in ("target", "draft", "ids", "uniforms")}
        if w.draft_len is not None:
            host["draft_len"] = w.draft_len.cpu().pin_memory()
        out_em = torch.empty(w.B, w.gamma + 1, dtype=torch.int32).pin_memory()
        out_na = torch.empty(w.B, dtype=torch.int32).pin_memory()
    finally:
        if saved:
            os.sched_setaffinity(0, saved)
    dev_in = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_em.numel() * 4 + out_na.numel() * 4

    # Rows are independent, so the batch goes over in four row groups: group g is verified (one
    # spec_verify_sample call on its rows) while group g+1 is still being copied.  The host link, not
    # the GPU, bounds this number: pinned host memory reaches about 210 GB/s on this system.
    groups = [(g * w.B // 4, (g + 1) * w.B // 4) for g in range(4) if (g + 1) * w.B // 4 > g * w.B // 4]
    copy_stream = torch.cuda.Stream(dev)
    ws_g = S.workspace_for(dev, S.workspace_size(w.B, w.gamma, w.V, w.target.dtype))
    copied = [torch.cuda.Event() for _ in groups]

    def e2e_step():
        copy_stream.wait_stream(stream)
        with torch.cuda.stream(copy_stream):
            for gi, (lo, hi) in enumerate(groups):
                for n, t in host.items():
                    dev_in[n][lo:hi].copy_(t[lo:hi], non_blocking=True)
                copied[gi].record(copy_stream)
        for gi, (lo, hi) in enumerate(groups):
            stream.wait_event(copied[gi])
            S.verify_sample(dev_in["target"][lo:hi], dev_in["draft"][lo:hi], dev_in["ids"][lo:hi],
                            dev_in["uniforms"][lo:hi], w.T,
                            None if "draft_len" not in dev_in else dev_in["draft_len"][lo:hi],
                            emitted=em[lo:hi], n_accepted=na[lo:hi], workspace=ws_g)
        out_em.copy_(em, non_blocking=True)
        out_na.copy_(na, non_blocking=True)

    e2e_steps = max(3, min(a.steps, 20))
    e2e_ms = time_device(e2e_step, e2e_steps, 2, stream)
    assert S.check_status(ws_g) == 0
    _, e2e_units = combine_ranks(e2e_ms, float(pos), dist, dev)

    # the variants, one call each per step on the same batch (context for the line)
    greedy_ms = time_device(lambda: S.verify_greedy(logits()[0], w.greedy_ids, w.draft_len, workspace=ws),
                            max(10, a.steps), 3, stream)
    stats_ms = time_device(lambda: S.accept_stats(*logits(), w.ids, w.T, w.draft_len, workspace=ws),
                           max(10, a.steps), 3, stream)
    # the byte-lean early exit on the same batch: same outputs, logits read only up to each row's rejection
    early_ms = time_device(lambda: phase("early_exit"), max(10, a.steps), 3, stream)
    n_b = na.long()
    g_b = w.draft_len.long() if w.draft_len is not None else torch.full_like(n_b, w.gamma)
    early_rows = int(((n_b + 1) + torch.where(n_b < g_b, n_b + 1, g_b)).sum())
    # top-k / nucleus standardisation: per-row thresholds of the target and draft logits, then verification
    # on the standardised distributions (spec_verify_sample_masked)
    topk_ms = time_device(lambda: (S.topk_threshold(w.target, 50), S.topk_threshold(w.draft, 50)),
                          max(10, a.steps // 4), 3, stream)
    topp_ms = time_device(lambda: (S.topp_threshold(w.target, w.T, 0.9), S.topp_threshold(w.draft, w.T, 0.9)),
                          max(10, a.steps // 4), 3, stream)
    tthr, dthr = S.topp_threshold(w.target, w.T, 0.9), S.topp_threshold(w.draft, w.T, 0.9)
    masked_ms = time_device(lambda: S.verify_sample(*logits(), w.ids, w.uniforms, w.T, w.draft_len,
                                                    emitted=em, n_accepted=na, workspace=ws, target_thr=tthr,
                                                    draft_thr=dthr), max(10, a.steps), 3, stream)
    S.check_status(ws, raise_on_error=False)        # padded draft rows (NaN) have NaN thresholds: never read
    # lenient verification (q scaled by l = 0.5 in the accept test and the residual) on the same batch
    lenient_ms = time_device(lambda: S.verify_sample(*logits(), w.ids, w.uniforms, w.T, w.draft_len, emitted=em,
                                                     n_accepted=na, workspace=ws, lenience=0.5),
                             max(10, a.steps), 3, stream)
    S.check_status(ws)
    s_logits, s_u = W.sampler_rows(w)               # the draft-side sampler over every draft row
    sampler_ms = time_device(lambda: S.sample_rows(s_logits, s_u, w.T), max(10, a.steps), 3, stream)
    esz = 4 if w.dtype == "f32" else 2
    sampler_bytes = s_logits.shape[0] * w.V * esz   # every row once (the drawn slice again is on top)
    greedy_bytes = (w.B + pos) * w.V * esz          # target rows 0..gamma_b
    stats_bytes = 2 * pos * w.V * esz               # target and draft rows 0..gamma_b-1
    assert S.check_status(ws) == 0

    also = {}
    if not a.no_also:
        for kk in (2, 4):
            if kk == k:
                continue
            w2 = W.make(kk, device=dev)
            ws2 = S.workspace_for(dev, S.workspace_size(w2.B, w2.gamma, w2.V, w2.target.dtype))
            copies2 = rotation(w2)
            turn2 = [0]

            em2 = torch.empty(w2.B, w2.gamma + 1, dtype=torch.int32, device=dev)
            na2 = torch.empty(w2.B, dtype=torch.int32, device=dev)

            # output buffers passed in, so the loop times the library's launches, not the binding's allocations
            def call2():
                t, d = copies2[turn2[0] % len(copies2)]
                turn2[0] += 1
                S.verify_sample(t, d, w2.ids, w2.uniforms, w2.T, w2.draft_len, emitted=em2, n_accepted=na2,
                                workspace=ws2)

            ms = time_device(call2, max(20, a.steps), 5, stream)
            gbs = w2.read_once_bytes() / (ms * 1e-3) / 1e9

            def early2():
                t, d = copies2[turn2[0] % len(copies2)]
                turn2[0] += 1
                S.verify_sample(t, d, w2.ids, w2.uniforms, w2.T, w2.draft_len, emitted=em2, n_accepted=na2,
                                workspace=ws2, phase="early_exit")

            ems = time_device(early2, max(20, a.steps), 5, stream)
            also[w2.name] = {"ms_per_call": round(ms, 5), "positions_per_s": w2.positions() / (ms * 1e-3),
                             "rows_per_s": w2.B / (ms * 1e-3), "GB_per_s": round(gbs, 1),
                             "frac_of_measured_hbm": round(gbs / peak, 4),
                             "early_exit_ms_per_call": round(ems, 5),
                             "early_exit_form": early_form(w2),
                             "l2": "three copies of the logits used in turn"}
            del w2, copies2
        assert S.check_status(ws2) == 0

    if not a.no_also and k != 1:
        # c1 (B=8, gamma=4, V=32128, bf16): sampling and greedy verification per call; its 4.6 MB of logits
        # stay in L2 between calls, so these are latency figures, not HBM-bound ones
        w1 = W.make(1, device=dev)
        ws1 = S.workspace_for(dev, S.workspace_size(w1.B, w1.gamma, w1.V, w1.target.dtype))
        em1 = torch.empty(w1.B, w1.gamma + 1, dtype=torch.int32, device=dev)
        na1 = torch.empty(w1.B, dtype=torch.int32, device=dev)
        # output buffers passed in, so the timed loop is the library's launches, not the binding's allocations
        us_s, us_sg = call_latency(lambda: S.verify_sample(w1.target, w1.draft, w1.ids, w1.uniforms, w1.T,
                                                           emitted=em1, n_accepted=na1, workspace=ws1), dev, stream)
        us_g, us_gg = call_latency(lambda: S.verify_greedy(w1.target, w1.greedy_ids, emitted=em1, n_accepted=na1,
                                                           workspace=ws1), dev, stream)
        assert S.check_status(ws1) == 0
        also["c1"] = {"sampling_us_per_call": us_s, "sampling_us_per_call_cuda_graph": us_sg,
                      "greedy_us_per_call": us_g, "greedy_us_per_call_cuda_graph": us_gg,
                      "positions_per_s": w1.positions() / (us_s * 1e-6), "rows_per_s": w1.B / (us_s * 1e-6),
                      "GB_per_s": round(w1.read_once_bytes() / (us_s * 1e-6) / 1e9, 1),
                      "l2": "4.6 MB of logits, resident in L2 across calls"}
        del w1
    if not a.no_also:
        also["c0"] = c0_latency(S, dev, stream)
    line = {
        "metric": METRIC, "value": units / t_max, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded Philox workload, see workloads/)",
        "config": {**workload_desc(w), "l2": f"three copies of the logits used in turn ({len(copies)} x {nbytes / 1e9:.2f} GB "
                                             "read per step vs 129 MB of L2), so no step reads logits an earlier step "
                                             "left in L2; no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "rows_per_s": w.B * a.steps * world / t_max,
        "GB_per_s": step_gbs,
        "frac_of_measured_hbm_per_step": round(step_gbs / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": f"verify_stream_kernel<{'float' if w.dtype == 'f32' else 'bf16'}>",
                     "kernel_ms": stream_ms,
                     "algorithmic_bytes_per_launch": nbytes},
        "e2e": {"value": e2e_units / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "h2d_GB_per_s_upper_bound": round(h2d / (e2e_ms * 1e-3) / 1e9, 1),
                "pinned_buffers": (f"allocated from the GPU's local CPUs (host NUMA node {local['node']})" if local
                                   else "allocated without CPU placement")},
        "gpu_launches": 2 * a.steps,
        "clocks": clocks,
        "variants": {"greedy_ms_per_call": greedy_ms,
                     "greedy_GB_per_s": greedy_bytes / (greedy_ms * 1e-3) / 1e9,
                     "stats_ms_per_call": stats_ms,
                     "stats_GB_per_s": stats_bytes / (stats_ms * 1e-3) / 1e9,
                     "topk50_thresholds_ms": topk_ms, "topp09_thresholds_ms": topp_ms,
                     "thresholds_GB_per_s": (w.B * (2 * w.gamma + 1)) * w.V * esz / (topp_ms * 1e-3) / 1e9,
                     "masked_verify_ms_per_call": masked_ms,
                     "lenient_verify_ms_per_call": lenient_ms,
                     "early_exit_ms_per_call": early_ms, "early_exit_form": early_form(w),
                     "early_exit_rows_read": early_rows, "all_positions_rows_read": w.B + 2 * pos,
                     "early_exit_GB_per_s": early_rows * w.V * esz / (early_ms * 1e-3) / 1e9,
                     "sampler_rows": int(s_logits.shape[0]), "sampler_ms_per_call": sampler_ms,
                     "sampler_GB_per_s": sampler_bytes / (sampler_ms * 1e-3) / 1e9},
        "also": also,
    }
    if rank == 0 and not a.no_cpu_baseline:
        # the batch's plain outputs again (the variants above reused the output buffers)
        S.verify_sample(w.target, w.draft, w.ids, w.uniforms, w.T, w.draft_len, emitted=em, n_accepted=na,
                        workspace=ws)
        assert S.check_status(ws) == 0
        line["cpu_baseline"] = cpu_oracle_rate(w, a.cpu_rows, os.cpu_count() or 1, gpu=(em, na))
        one = cpu_oracle_rate(w, 16, 1)   # the same oracle on one core, a smaller sample
        line["cpu_baseline"]["single_core"] = {"value": one["value"], "unit": UNIT, "sample": one["sample"]}
    return line


_REF_INPUTS: dict = {}


def _ref_load(path):
    """The reference arm's inputs in a pool worker: memory-mapped from the files the parent wrote."""
    if _REF_INPUTS.get("path") != path:
        _REF_INPUTS.clear()
        _REF_INPUTS["path"] = path
        for n in ("target", "draft", "ids", "gl", "u"):
            f = os.path.join(path, n + ".npy")
            _REF_INPUTS[n] = np.load(f, mmap_mode="r") if os.path.exists(f) else None
    return _REF_INPUTS


def _ref_rows(args):
    import oracle as O
    path, lo, hi, dtype, T = args
    h = _ref_load(path)
    gl = None if h["gl"] is None else np.asarray(h["gl"][lo:hi])
    r = O.verify_sample(np.asarray(h["target"][lo:hi]), np.asarray(h["draft"][lo:hi]), dtype,
                        np.asarray(h["ids"][lo:hi]), gl, np.asarray(h["u"][lo:hi]), T)
    return int((r["n_accepted"] >= 0).sum())


def run_reference(a, rank, world):
    """The float64 CPU oracle as the reference arm: the same workload, metric and batch, every row of the
    batch in every step, over a spawn process pool on all host cores.  The inputs go to the workers once,
    as memory-mapped files; a step is the wall time of verifying the whole batch."""
    if rank != 0:
        return None
    import shutil
    import tempfile
    k = int(a.workload.lstrip("c"))
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = W.make(k, device=dev, B=a.batch or None)
    procs = os.cpu_count() or 1
    host = {"target": W.logits_as_numpy(w.target), "draft": W.logits_as_numpy(w.draft), "ids": w.ids.cpu().numpy(),
            "gl": None if w.draft_len is None else w.draft_len.cpu().numpy(), "u": w.uniforms.cpu().numpy()}
    need = sum(v.nbytes for v in host.values() if v is not None)
    shm = "/dev/shm" if os.path.isdir("/dev/shm") and shutil.disk_usage("/dev/shm").free > 2 * need else None
    path = tempfile.mkdtemp(prefix="specverify_ref_", dir=shm)
    try:
        for n, v in host.items():
            if v is not None:
                np.save(os.path.join(path, n + ".npy"), v)
        del host
        per = max(1, math.ceil(w.B / procs))
        jobs = [(path, lo, min(w.B, lo + per), w.dtype, w.T) for lo in range(0, w.B, per)]
        times = []
        with oracle_pool(procs) as pool:
            pool.map(_ref_rows, jobs)                  # start-up, imports and the first mapping
            for _ in range(a.warmup - 1):
                pool.map(_ref_rows, jobs)
            t_all = time.perf_counter()
            for _ in range(a.steps):
                t0 = time.perf_counter()
                pool.map(_ref_rows, jobs)
                times.append(time.perf_counter() - t0)
                if time.perf_counter() - t_all > 150:   # bounded: the whole run stays within a few minutes
                    break
    finally:
        shutil.rmtree(path, ignore_errors=True)
    total = sum(times)
    v = w.positions() * len(times) / total
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": len(times),
            "warmup": a.warmup, "ms_per_step": total * 1e3 / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Philox workload, see workloads/)",
            "config": {**workload_desc(w), "sample": f"every step verifies the whole batch of {w.B} rows"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": procs, "kind": "oracle",
                             "sample": f"the whole {w.name} batch ({w.B} rows, {w.positions()} positions) per "
                                       f"step, {len(times)} steps (float64 numpy oracle, spawn pool)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3", choices=["c1", "c2", "c3", "c4"])
    ap.add_argument("--cpu-rows", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", action="store_true")
    ap.add_argument("--e2e-numa", choices=["local", "any"], default="local",
                    help="where the e2e step's pinned host buffers are allocated from")
    ap.add_argument("--batch", type=int, default=0,
                    help="rows of the workload (same recipe; default: the workload's own B) -- for profiling "
                         "a smaller case of the same kernels")
    a = ap.parse_args()
    a.warmup = max(3, a.warmup)

    rank, world, dist = dist_init()
    if a.impl == "reference":
        line = run_reference(a, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    import __graft_entry__
    __graft_entry__.build()
    line = run_ours(a, rank, world, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
