"""Builds libspecverify.so (the C-ABI verification library) in-tree with nvcc for sm_103a.

    python speculative_decoding_verification_40_gb300/build.py [--force] [--verbose] [--debug-bounds]

Each .cu file under csrc/ compiles to an object in _build/ (in parallel), and the
objects link into libspecverify.so next to this file with the CUDA runtime
linked statically.  Nothing is rebuilt when the library is newer than every source.
--debug-bounds builds libspecverify_debug.so instead (objects in _build_debug/), compiled with
-DSPEC_DEBUG_BOUNDS: the kernels check their indices and report SPEC_ERR_BOUNDS instead of accessing
out of range (the device-side stand-in for a memory checker).
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libspecverify.so")
DEBUG_BUILD = os.path.join(ROOT, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "libspecverify_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify.so")


def _sources():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + sorted(glob.glob(os.path.join(CSRC, "*.h")))
    deps.append(os.path.join(ROOT, "include", "spec_verify.h"))
    return srcs, deps


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    _, deps = _sources()
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug_bounds: bool = False) -> str:
    """Compile and link the library; returns its path.  Concurrent callers (one per rank) serialise on a lock."""
    lib, bdir = (DEBUG_LIB, DEBUG_BUILD) if debug_bounds else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    import fcntl
    with open(os.path.join(bdir, ".lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        if not force and up_to_date(lib):
            return lib
        flags = list(extra_flags or []) + (["-DSPEC_DEBUG_BOUNDS"] if debug_bounds else [])
        return _build_locked(verbose, flags, lib, bdir)


def _build_locked(verbose: bool, extra_flags: list[str] | None, lib: str = LIB, bdir: str = BUILD) -> str:
    cc = nvcc()
    srcs, _ = _sources()
    extra = list(extra_flags or [])
    if verbose:
        extra += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [cc, "-c", src, "-o", obj, *ARCH, *FLAGS, *extra]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = lib + ".tmp"
    cmd = [cc, "-shared", *ARCH, "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--debug-bounds", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug_bounds=a.debug_bounds))


if __name__ == "__main__":
    main()
