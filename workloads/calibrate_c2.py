"""Writes workloads/c2_sigma.json: the per-row draft noise sigma_b of workload c2.

c2's draft logits are target + sigma_b * z with one fixed unit-normal draw z;
sigma_b is set by bisection on [0, 10] so that the mean over the 8 positions of
the acceptance rate beta_i = sum_x min(p_i(x), q_i(x)) at T = 0.8 is 0.8 +- 0.005.
beta comes from the float64 oracle (oracle.stats_position) on the bf16-rounded
logits the verifier sees.  Run once on the CPU:  python -m workloads.calibrate_c2
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from workloads import C2_SIGMA_FILE, SPECS, c2_base  # noqa: E402

TARGET_BETA = 0.8
TOL = 0.005


def _bf16_f64(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).to(torch.float64).numpy()


def mean_beta(t_rows: np.ndarray, target_f32: torch.Tensor, z: torch.Tensor, sigma: float, T: float) -> float:
    d = _bf16_f64(target_f32[:-1] + sigma * z)
    betas = [oracle.stats_position(t_rows[i], d[i], 0, T)["beta"] for i in range(d.shape[0])]
    return float(np.mean(betas))


def main():
    sp = SPECS[2]
    T = float(np.float32(sp["T"]))
    target, z = c2_base("cpu")
    sigmas, betas = [], []
    for b in range(sp["B"]):
        t_rows = _bf16_f64(target[b])
        lo, hi = 0.0, 10.0
        s, beta = 1.0, None
        for _ in range(40):
            s = 0.5 * (lo + hi)
            beta = mean_beta(t_rows, target[b], z[b], s, T)
            if abs(beta - TARGET_BETA) <= TOL:
                break
            if beta > TARGET_BETA:
                lo = s
            else:
                hi = s
        sigmas.append(round(s, 6))
        betas.append(beta)
        print(f"row {b:2d}: sigma {s:.6f} mean beta {beta:.5f}", flush=True)
    with open(C2_SIGMA_FILE, "w") as f:
        json.dump({"target_mean_beta": TARGET_BETA, "T": sp["T"], "sigma": sigmas,
                   "mean_beta": [round(x, 6) for x in betas]}, f, indent=1)
    print("wrote", C2_SIGMA_FILE)


if __name__ == "__main__":
    main()
