"""Seeded synthetic inputs for the batched verification step.

Five workloads (c0..c4) with the shapes, dtypes, logit distributions and row
mixes of the verification step of speculative sampling (Leviathan, Kalman &
Matias, "Fast Inference from Transformers via Speculative Decoding", §2.3
Algorithm 1): target logits [B, gamma+1, V], draft logits [B, gamma, V], draft
ids [B, gamma] drawn from the draft distribution, caller-supplied uniforms
[B, gamma+1] and a temperature.

All randomness is Philox4x32-10 (workloads.philox), keyed by (seed, stream), so
a workload is the same on the CPU and on a GPU up to the last bit of the
float64 Box-Muller transform.  Drafts are drawn from softmax(draft/T) by the
Gumbel-max trick (argmax of logits/T plus Gumbel noise), which needs no
normalisation.  This module is shared by the tests, the bench and the oracle
harness; it holds none of the verification arithmetic.
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, field

import torch

from .philox import gumbel_f32, normal_f32, uniform_f32

# Stream ids inside one workload key.
S_TARGET, S_DRAFT, S_GUMBEL, S_SIGMA, S_GLEN, S_KIND, S_MASK, S_HOT = 1, 2, 3, 4, 5, 6, 7, 8
UNIFORM_SEED = 0  # the accept/draw uniforms come from Philox seed 0

SPECS = {
    0: dict(name="c0", B=1, gamma=4, V=1024, dtype="f32", T=1.0,
            desc="B=1, gamma=4, V=1024, fp32; target N(0,2^2), draft = target + N(0,0.5^2); T=1"),
    1: dict(name="c1", B=8, gamma=4, V=32128, dtype="bf16", T=1.0,
            desc="B=8, gamma=4, V=32128, bf16; target N(0,3^2) + Zipf(1.1) log-prior, draft = target + N(0,1); T=1"),
    2: dict(name="c2", B=64, gamma=8, V=128256, dtype="bf16", T=0.8,
            desc="B=64, gamma=8, V=128256, bf16; target Zipf(1.1) + N(0,2^2), per-row draft sigma for mean beta 0.8; T=0.8"),
    3: dict(name="c3", B=256, gamma=5, V=152064, dtype="f32", T=0.7,
            desc="B=256, gamma=5, V=152064, fp32; target N(0,2.5^2) + Zipf(1.0), draft sigma_b ~ U[0.1,2.0]; T=0.7"),
    4: dict(name="c4", B=1024, gamma=8, V=32000, dtype="bf16", T=1.0,
            desc="B=1024, ragged gamma_b ~ U{1..8} padded to 8, V=32000, bf16; 10% p==q, 10% disjoint, "
                 "10% one-hot target, rest Zipf(1.1)+N(0,2^2) with draft sigma 1; T=1"),
}

ROW_NORMAL, ROW_P_EQ_Q, ROW_DISJOINT, ROW_ONE_HOT = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
C2_SIGMA_FILE = os.path.join(_HERE, "c2_sigma.json")


@dataclass
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str            # "f32" or "bf16"
    T: float
    target: torch.Tensor  # [B, gamma+1, V] float32 or bfloat16
    draft: torch.Tensor   # [B, gamma, V]
    ids: torch.Tensor     # [B, gamma] int32 (padding -1 beyond draft_len)
    uniforms: torch.Tensor  # [B, gamma+1] float32
    draft_len: torch.Tensor | None = None  # [B] int32 or None (all gamma)
    greedy_ids: torch.Tensor | None = None  # [B, gamma] int32, argmax of the draft logits
    row_kind: torch.Tensor | None = None    # [B] int8 (ROW_* codes)
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "Workload":
        """The same workload with every tensor copied to `device` (one copy per tensor)."""
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return Workload(name=self.name, B=self.B, gamma=self.gamma, V=self.V, dtype=self.dtype, T=self.T,
                        target=mv(self.target), draft=mv(self.draft), ids=mv(self.ids), uniforms=mv(self.uniforms),
                        draft_len=mv(self.draft_len), greedy_ids=mv(self.greedy_ids), row_kind=mv(self.row_kind),
                        meta=self.meta)

    def positions(self) -> int:
        """Verified draft positions in one call: sum over rows of gamma_b."""
        if self.draft_len is None:
            return self.B * self.gamma
        return int(self.draft_len.sum().item())

    def read_once_bytes(self) -> int:
        """Bytes of logits a verification call must read once: (2*gamma_b + 1) rows of V per row b."""
        esz = 4 if self.dtype == "f32" else 2
        if self.draft_len is None:
            rows = self.B * (2 * self.gamma + 1)
        else:
            rows = int((2 * self.draft_len.to(torch.int64) + 1).sum().item())
        return rows * self.V * esz


def zipf_log_prior(V: int, s: float, device) -> torch.Tensor:
    """Zipf(s) log-prior over token ids, rank = id + 1: -s * ln(v + 1)."""
    v = torch.arange(V, dtype=torch.float64, device=device)
    return (-s * torch.log1p(v)).to(torch.float32)


def _to_dtype(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def _gumbel_drafts(draft: torch.Tensor, T: float, seed: int, stream: int) -> torch.Tensor:
    """x[b,i] ~ softmax(draft[b,i]/T) by Gumbel-max, computed row by row to bound memory."""
    B, G, V = draft.shape
    ids = torch.empty(B, G, dtype=torch.int32, device=draft.device)
    rows_per = max(1, (1 << 24) // max(1, V))
    flat = draft.reshape(B * G, V)
    out = ids.reshape(B * G)
    for s in range(0, B * G, rows_per):
        e = min(B * G, s + rows_per)
        g = gumbel_f32(((e - s) * V,), seed, stream * 4096 + s // rows_per, draft.device).reshape(e - s, V)
        z = flat[s:e].to(torch.float32) / T + g
        out[s:e] = torch.argmax(z, dim=1).to(torch.int32)
    return ids


def _uniforms(B: int, gamma: int, k: int, call: int, device) -> torch.Tensor:
    return uniform_f32((B, gamma + 1), UNIFORM_SEED, 100 + k + 16 * call, device)


def sampler_rows(w: "Workload", call: int = 0):
    """Inputs of the draft-side sampler on workload w: its draft logit rows (b, i) with i < gamma_b as an
    [R, V] tensor, and one uniform per row (Philox stream 200 + k + 16 * call)."""
    V = w.V
    if w.draft_len is None:
        rows = w.draft.reshape(-1, V)
    else:
        keep = (torch.arange(w.gamma, device=w.draft.device)[None, :] < w.draft_len[:, None]).reshape(-1)
        rows = w.draft.reshape(-1, V)[keep]
    k = int(w.name.lstrip("c"))
    u = uniform_f32((rows.shape[0],), UNIFORM_SEED, 200 + k + 16 * call, rows.device)
    return rows.contiguous(), u


def load_c2_sigma() -> list[float] | None:
    if not os.path.exists(C2_SIGMA_FILE):
        return None
    with open(C2_SIGMA_FILE) as f:
        return [float(x) for x in json.load(f)["sigma"]]


def c2_base(device="cpu", B=None):
    """Target logits and the fixed unit noise draw z of c2 (draft = target + sigma_b * z)."""
    sp = SPECS[2]
    B, g, V = B or sp["B"], sp["gamma"], sp["V"]
    seed = 1002
    prior = zipf_log_prior(V, 1.1, device)
    target = prior + 2.0 * normal_f32((B, g + 1, V), seed, S_TARGET, device)
    z = normal_f32((B, g, V), seed, S_DRAFT, device)
    return target, z


def make(k: int, device="cpu", call: int = 0, with_ids: bool = True, B: int | None = None) -> Workload:
    """Build workload c<k> on `device`.  `call` selects one of c0's independent calls.

    `B` overrides the batch size (same recipe, fewer or more rows) for quick tests.
    """
    sp = SPECS[k]
    B, gamma, V, dtype, T = B or sp["B"], sp["gamma"], sp["V"], sp["dtype"], sp["T"]
    seed = 1000 + k
    draft_len = None
    row_kind = None
    meta = {"desc": sp["desc"]}
    if k == 0:
        st = 16 * call
        target = 2.0 * normal_f32((B, gamma + 1, V), seed, S_TARGET + st, device)
        draft = target[:, :gamma] + 0.5 * normal_f32((B, gamma, V), seed, S_DRAFT + st, device)
        gseed_stream = S_GUMBEL + st
    elif k == 1:
        prior = zipf_log_prior(V, 1.1, device)
        target = 3.0 * normal_f32((B, gamma + 1, V), seed, S_TARGET, device) + prior
        draft = target[:, :gamma] + 1.0 * normal_f32((B, gamma, V), seed, S_DRAFT, device)
        gseed_stream = S_GUMBEL
    elif k == 2:
        target, z = c2_base(device, B)
        sig = load_c2_sigma()
        if sig is None:
            raise RuntimeError("workloads/c2_sigma.json is missing; run workloads/calibrate_c2.py")
        sig = [sig[b % len(sig)] for b in range(B)]
        sigma = torch.tensor(sig, dtype=torch.float32, device=device).view(B, 1, 1)
        draft = target[:, :gamma] + sigma * z
        del z
        meta["sigma"] = sig
        gseed_stream = S_GUMBEL
    elif k == 3:
        prior = zipf_log_prior(V, 1.0, device)
        target = 2.5 * normal_f32((B, gamma + 1, V), seed, S_TARGET, device) + prior
        sigma = 0.1 + 1.9 * uniform_f32((B,), seed, S_SIGMA, device)
        draft = target[:, :gamma] + sigma.view(B, 1, 1) * normal_f32((B, gamma, V), seed, S_DRAFT, device)
        meta["sigma"] = sigma.cpu().tolist()
        gseed_stream = S_GUMBEL
    elif k == 4:
        prior = zipf_log_prior(V, 1.1, device)
        base = prior + 2.0 * normal_f32((B, gamma + 1, V), seed, S_TARGET, device)
        draft = base[:, :gamma] + 1.0 * normal_f32((B, gamma, V), seed, S_DRAFT, device)
        target = base
        draft_len = (1 + torch.floor(8.0 * uniform_f32((B,), seed, S_GLEN, device))).to(torch.int32)
        perm = torch.argsort(uniform_f32((B,), seed, S_KIND, device))
        n10 = B // 10
        row_kind = torch.zeros(B, dtype=torch.int8, device=device)
        row_kind[perm[:n10]] = ROW_P_EQ_Q
        row_kind[perm[n10:2 * n10]] = ROW_DISJOINT
        row_kind[perm[2 * n10:3 * n10]] = ROW_ONE_HOT
        ninf = float("-inf")
        # p == q: draft logits are the target logits bit for bit
        eq = row_kind == ROW_P_EQ_Q
        draft[eq] = target[eq][:, :gamma]
        # disjoint support: a random half of the vocabulary is -inf in the target, the rest -inf in the draft
        dj = (row_kind == ROW_DISJOINT).nonzero().flatten()
        if dj.numel():
            mask = uniform_f32((dj.numel(), 1, V), seed, S_MASK, device) < 0.5
            t = target[dj]
            d = draft[dj]
            t = torch.where(mask, torch.full_like(t, ninf), t)
            d = torch.where(mask, d, torch.full_like(d, ninf))
            target[dj] = t
            draft[dj] = d
        # one-hot target: every logit -inf except one id per position
        oh = (row_kind == ROW_ONE_HOT).nonzero().flatten()
        if oh.numel():
            hot = torch.floor(V * uniform_f32((oh.numel(), gamma + 1), seed, S_HOT, device)).to(torch.int64)
            hot = hot.clamp_(max=V - 1)
            t = torch.full((oh.numel(), gamma + 1, V), ninf, dtype=torch.float32, device=device)
            t.scatter_(2, hot.unsqueeze(2), 0.0)
            target[oh] = t
            meta["hot"] = hot.cpu()
        gseed_stream = S_GUMBEL
        meta["row_kind_counts"] = {int(c): int((row_kind == c).sum()) for c in range(4)}
    else:
        raise ValueError(f"unknown workload {k}")

    target = _to_dtype(target, dtype)
    draft = _to_dtype(draft, dtype)
    if with_ids:
        ids = _gumbel_drafts(draft, T, seed, gseed_stream)
        greedy_ids = torch.argmax(draft.to(torch.float32), dim=2).to(torch.int32)
    else:
        ids = torch.zeros(B, gamma, dtype=torch.int32, device=device)
        greedy_ids = None
    uniforms = _uniforms(B, gamma, k, call, device)

    if draft_len is not None:
        # Padding beyond draft_len is never read: fill it with values a reader would trip on.
        pos = torch.arange(gamma + 1, device=device).view(1, gamma + 1)
        gl = draft_len.view(B, 1).to(torch.int64)
        nan = float("nan")
        tpad = (pos > gl)
        dpad = (pos[:, :gamma] >= gl)
        target[tpad] = nan
        draft[dpad] = nan
        ids[dpad] = -1
        if greedy_ids is not None:
            greedy_ids[dpad] = -1
        upad = torch.cat([dpad, torch.zeros(B, 1, dtype=torch.bool, device=device)], dim=1)
        uniforms[upad] = nan

    return Workload(name=sp["name"], B=B, gamma=gamma, V=V, dtype=dtype, T=T,
                    target=target.contiguous(), draft=draft.contiguous(), ids=ids.contiguous(),
                    uniforms=uniforms.contiguous(), draft_len=draft_len, greedy_ids=greedy_ids,
                    row_kind=row_kind, meta=meta)


def logits_as_numpy(x: torch.Tensor):
    """Host copy of a logit tensor for the oracle: float32 values, or bfloat16 bit patterns as uint16."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view("uint16")
    return x.to(torch.float32).numpy()
