"""The kernels' index checks (debug-bounds build) stay silent on the GPU test cases (GPU).

compute-sanitizer is closed on this system; its stand-in is libspecverify_debug.so, built with
-DSPEC_DEBUG_BOUNDS, whose kernels check slice, chunk, segment and token indices and record
SPEC_ERR_BOUNDS in the error word (skipping the access) instead of reading or writing out of range.
This test builds it and reruns a set of the GPU parity tests against it in a child process: every one
checks the error word, so a failed index check fails the run.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_under_index_checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "specverify_build", os.path.join(ROOT, "speculative_decoding_verification_40_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    lib = mod.build(debug_bounds=True)
    assert lib.endswith("libspecverify_debug.so")
    env = dict(os.environ, SPECVERIFY_DEBUG_BOUNDS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_edge.py", "tests/test_gpu_sampler.py", "tests/test_gpu_early_exit.py",
           "tests/test_gpu_lenience.py", "-k", "not law and not parity_on_the_draft_rows[3]"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert "passed" in tail
