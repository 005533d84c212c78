"""Batched speculative-sampling verification on one GB300 (sm_103a).

Python binding of libspecverify.so, the C-ABI library declared in
include/spec_verify.h.  The functions here only marshal torch CUDA tensors
(device pointers, sizes, the current stream) into the C calls: every step of
the verification runs in the library's CUDA kernels.  Importing this package
fails if the library has not been built
(python speculative_decoding_verification_40_gb300/build.py).

Entry points (same names as the C ABI, without the spec_ prefix):
  verify_sample  -- accept test, first rejection, residual / bonus draw
  verify_greedy  -- argmax verification
  sample_rows    -- draft-side sampler: x ~ softmax(l / T) per row by the inverse CDF
  accept_stats   -- per-position beta, p(x), q(x), min(1, p/q), residual mass
  check_status   -- device-side error word of a workspace
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "SpecVerifyError", "verify_sample", "verify_greedy", "sample_rows", "accept_stats", "check_status", "workspace_size",
    "workspace_for", "plan", "LIB_PATH", "lib", "expected_tokens", "walltime_improvement", "operations_factor",
    "optimal_gamma", "alpha_mean", "topk_threshold", "topp_threshold",
]

# SPECVERIFY_DEBUG_BOUNDS=1 loads the debug-bounds build (kernel index checks that report SPEC_ERR_BOUNDS
# instead of accessing out of range; `build.py --debug-bounds`)
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libspecverify_debug.so" if os.environ.get("SPECVERIFY_DEBUG_BOUNDS") == "1"
                        else "libspecverify.so")

SPEC_F32, SPEC_BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unknown dtype", 3: "CUDA error", 4: "non-finite or all -inf logit row",
          5: "draft id outside [0, V)", 6: "timeout", 7: "workspace too small or misaligned", 8: "index check failed"}


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, 'unknown status')} (code {code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python speculative_decoding_verification_40_gb300/build.py`"
                          + (" --debug-bounds" if LIB_PATH.endswith("_debug.so") else ""))
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.spec_workspace_size.argtypes = [i32, i32, i32, i32]
    L.spec_workspace_size.restype = sz
    L.spec_workspace_init.argtypes = [vp, sz, vp]
    L.spec_workspace_init.restype = i32
    for name in ("spec_verify_sample", "spec_verify_sample_stream", "spec_verify_sample_draw",
                 "spec_verify_sample_early_exit"):
        fn = getattr(L, name)
        fn.argtypes = [vp, vp, i32, vp, vp, vp, f32, i32, i32, i32, vp, vp, vp, sz, vp]
        fn.restype = i32
    L.spec_sample_rows.argtypes = [vp, i32, vp, f32, i32, i32, vp, vp, sz, vp]
    L.spec_sample_rows.restype = i32
    L.spec_sample_rows_masked.argtypes = [vp, i32, vp, vp, f32, i32, i32, vp, vp, sz, vp]
    L.spec_sample_rows_masked.restype = i32
    L.spec_verify_sample_masked.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, f32, i32, i32, i32, vp, vp, vp, sz, vp]
    L.spec_verify_sample_masked.restype = i32
    L.spec_verify_sample_lenient.argtypes = [vp, vp, i32, vp, vp, vp, f32, f32, i32, i32, i32, vp, vp, vp, sz, vp]
    L.spec_verify_sample_lenient.restype = i32
    L.spec_topk_threshold.argtypes = [vp, i32, i32, i32, i32, vp, vp]
    L.spec_topk_threshold.restype = i32
    L.spec_topp_threshold.argtypes = [vp, i32, f32, f32, i32, i32, vp, vp]
    L.spec_topp_threshold.restype = i32
    L.spec_verify_greedy.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    L.spec_verify_greedy.restype = i32
    L.spec_accept_stats.argtypes = [vp, vp, i32, vp, vp, f32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_accept_stats.restype = i32
    dbl, i64 = ctypes.c_double, ctypes.c_longlong
    L.spec_expected_tokens.argtypes = [dbl, i32]
    L.spec_expected_tokens.restype = dbl
    L.spec_walltime_improvement.argtypes = [dbl, i32, dbl]
    L.spec_walltime_improvement.restype = dbl
    L.spec_operations_factor.argtypes = [dbl, i32, dbl]
    L.spec_operations_factor.restype = dbl
    L.spec_optimal_gamma.argtypes = [dbl, dbl, i32, ctypes.POINTER(dbl)]
    L.spec_optimal_gamma.restype = i32
    L.spec_alpha_mean.argtypes = [vp, i64, vp, vp]
    L.spec_alpha_mean.restype = i32
    L.spec_check_status.argtypes = [vp, vp]
    L.spec_check_status.restype = i32
    ip = ctypes.POINTER(ctypes.c_int)
    L.spec_verify_plan.argtypes = [i32, i32, i32, i32, ip, ip, ip, ip]
    L.spec_verify_plan.restype = i32
    L.spec_status_string.argtypes = [i32]
    L.spec_status_string.restype = ctypes.c_char_p
    return L


lib = _load()


# ----------------------------------------------------------------------------- helpers

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _raise(code: int, where: str):
    if code != 0:
        raise SpecVerifyError(code, where)


def workspace_size(B: int, gamma: int, V: int, dtype: torch.dtype = torch.float32) -> int:
    code = SPEC_BF16 if dtype == torch.bfloat16 else SPEC_F32
    return int(lib.spec_workspace_size(B, gamma, V, code))


_WS: dict = {}


def workspace_for(device: torch.device, nbytes: int) -> torch.Tensor:
    """Zero-filled per-device workspace of at least nbytes, grown on demand.

    The library leaves every counter it uses at zero after each call, so one
    workspace serves any sequence of calls on one stream; calls that may
    overlap on the GPU need workspaces of their own (pass `workspace=`).
    """
    device = torch.device(device)
    key = (device.type, device.index if device.index is not None else torch.cuda.current_device())
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=device)
        _WS[key] = ws
    return ws


def plan(B: int, gamma: int, V: int, dtype: torch.dtype = torch.float32) -> dict:
    """Launch plan of the sampling kernel: cluster size, slice length, shared memory, greedy CTAs per row."""
    cs, L, sm, g = (ctypes.c_int() for _ in range(4))
    code = SPEC_BF16 if dtype == torch.bfloat16 else SPEC_F32
    _raise(lib.spec_verify_plan(B, gamma, V, code, ctypes.byref(cs), ctypes.byref(L), ctypes.byref(sm),
                                ctypes.byref(g)), "spec_verify_plan")
    return {"cluster_size": cs.value, "slice_len": L.value, "smem_bytes": sm.value, "greedy_ctas_per_row": g.value}


def expected_tokens(alpha: float, gamma: int) -> float:
    """spec_expected_tokens: (1 - alpha^(gamma+1)) / (1 - alpha)."""
    return float(lib.spec_expected_tokens(alpha, gamma))


def walltime_improvement(alpha: float, gamma: int, c: float) -> float:
    """spec_walltime_improvement (Theorem 3.8)."""
    return float(lib.spec_walltime_improvement(alpha, gamma, c))


def operations_factor(alpha: float, gamma: int, c_hat: float) -> float:
    """spec_operations_factor (Theorem 3.11)."""
    return float(lib.spec_operations_factor(alpha, gamma, c_hat))


def optimal_gamma(alpha: float, c: float, max_gamma: int = 64) -> tuple[int, float]:
    """spec_optimal_gamma: (gamma*, improvement at gamma*)."""
    v = ctypes.c_double()
    g = int(lib.spec_optimal_gamma(alpha, c, max_gamma, ctypes.byref(v)))
    if g < 0:
        raise ValueError("alpha must lie in [0, 1], c >= 0, max_gamma >= 1")
    return g, v.value


def alpha_mean(beta: torch.Tensor) -> tuple[float, int]:
    """spec_alpha_mean: alpha = mean of the finite beta values (device reduction), and their count."""
    _cuda(beta, "beta", torch.float32)
    out = torch.empty(2, dtype=torch.float64, device=beta.device)
    _raise(lib.spec_alpha_mean(_p(beta), beta.numel(), _p(out), _stream(beta.device)), "spec_alpha_mean")
    o = out.cpu()
    return float(o[0]), int(o[1])


def check_status(workspace: torch.Tensor | None = None, device=None, raise_on_error: bool = True) -> int:
    """Synchronise the current stream, read and clear the workspace's device error word."""
    if workspace is None:
        device = torch.device(device or "cuda")
        workspace = workspace_for(device, 4096)
    code = int(lib.spec_check_status(_p(workspace), _stream(workspace.device)))
    if raise_on_error:
        _raise(code, "device")
    return code


def _shapes(target: torch.Tensor):
    if target.dim() != 3:
        raise ValueError("target logits must be [B, gamma+1, V]")
    B, G1, V = target.shape
    return B, G1 - 1, V


def _common(target, draft, ids, draft_len, gamma_needs_draft=True):
    B, G, V = _shapes(target)
    _cuda(target, "target_logits")
    if G > 0 and gamma_needs_draft:
        _cuda(draft, "draft_logits", target.dtype, (B, G, V))
    if G > 0:
        _cuda(ids, "draft_ids", torch.int32, (B, G))
    if draft_len is not None:
        _cuda(draft_len, "draft_len", torch.int32, (B,))
    return B, G, V


# ----------------------------------------------------------------------------- entry points

def verify_sample(target: torch.Tensor, draft: torch.Tensor, ids: torch.Tensor, uniforms: torch.Tensor,
                  temperature: float, draft_len: torch.Tensor | None = None, *, emitted=None, n_accepted=None,
                  workspace: torch.Tensor | None = None, check: bool = False, phase: str = "both",
                  target_thr: torch.Tensor | None = None, draft_thr: torch.Tensor | None = None,
                  lenience: float = 1.0):
    """spec_verify_sample: returns (emitted [B, gamma+1] int32, n_accepted [B] int32).

    phase="stream" / "draw" calls spec_verify_sample_stream / spec_verify_sample_draw: the two halves
    of the same computation, to be called in that order with the same arguments and workspace.
    phase="early_exit" calls spec_verify_sample_early_exit (same results, reads rows only up to the
    first rejection).
    """
    B, G, V = _common(target, draft, ids, draft_len)
    _cuda(uniforms, "uniforms", torch.float32, (B, G + 1))
    dev = target.device
    if emitted is None:
        emitted = torch.empty(B, G + 1, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    _cuda(emitted, "emitted", torch.int32, (B, G + 1))
    _cuda(n_accepted, "n_accepted", torch.int32, (B,))
    ws = workspace if workspace is not None else workspace_for(dev, workspace_size(B, G, V, target.dtype))
    if lenience != 1.0:  # spec_verify_sample_lenient
        if phase != "both" or target_thr is not None or draft_thr is not None:
            raise ValueError("lenience goes with phase='both' and no thresholds")
        code = lib.spec_verify_sample_lenient(_p(target), _p(draft) if G > 0 else None, _dtype_code(target),
                                              _p(ids) if G > 0 else None, _p(draft_len), _p(uniforms),
                                              float(temperature), float(lenience), B, G, V, _p(emitted),
                                              _p(n_accepted), _p(ws), ws.numel(), _stream(dev))
        _raise(code, "spec_verify_sample_lenient")
        if check:
            check_status(ws)
        return emitted, n_accepted
    if target_thr is not None or draft_thr is not None:  # spec_verify_sample_masked
        if phase != "both":
            raise ValueError("standardisation thresholds go with phase='both'")
        if target_thr is not None:
            _cuda(target_thr, "target_thr", torch.float32, (B, G + 1))
        if draft_thr is not None and G > 0:
            _cuda(draft_thr, "draft_thr", torch.float32, (B, G))
        code = lib.spec_verify_sample_masked(_p(target), _p(draft) if G > 0 else None, _dtype_code(target),
                                             _p(ids) if G > 0 else None, _p(draft_len), _p(uniforms),
                                             _p(target_thr), _p(draft_thr) if G > 0 else None, float(temperature),
                                             B, G, V, _p(emitted), _p(n_accepted), _p(ws), ws.numel(),
                                             _stream(dev))
        _raise(code, "spec_verify_sample_masked")
        if check:
            check_status(ws)
        return emitted, n_accepted
    fn = {"both": lib.spec_verify_sample, "stream": lib.spec_verify_sample_stream,
          "draw": lib.spec_verify_sample_draw, "early_exit": lib.spec_verify_sample_early_exit}[phase]
    code = fn(_p(target), _p(draft) if G > 0 else None, _dtype_code(target), _p(ids) if G > 0 else None,
              _p(draft_len), _p(uniforms), float(temperature), B, G, V, _p(emitted), _p(n_accepted), _p(ws),
              ws.numel(), _stream(dev))
    _raise(code, "spec_verify_sample" if phase == "both" else f"spec_verify_sample_{phase}")
    if check:
        check_status(ws)
    return emitted, n_accepted


def sample_rows(logits: torch.Tensor, uniforms: torch.Tensor, temperature: float, *, thr=None, tokens=None,
                workspace: torch.Tensor | None = None, check: bool = False) -> torch.Tensor:
    """spec_sample_rows (spec_sample_rows_masked with thr [R] float32): logits [R, V], uniforms [R]
    float32; returns tokens [R] int32."""
    if logits.dim() != 2:
        raise ValueError("logits must be [R, V]")
    R, V = logits.shape
    _cuda(logits, "logits")
    _cuda(uniforms, "uniforms", torch.float32, (R,))
    dev = logits.device
    if tokens is None:
        tokens = torch.empty(R, dtype=torch.int32, device=dev)
    _cuda(tokens, "tokens", torch.int32, (R,))
    ws = workspace if workspace is not None else workspace_for(dev, workspace_size(R, 0, V, logits.dtype))
    if thr is None:
        code = lib.spec_sample_rows(_p(logits), _dtype_code(logits), _p(uniforms), float(temperature), R, V,
                                    _p(tokens), _p(ws), ws.numel(), _stream(dev))
    else:
        _cuda(thr, "thr", torch.float32, (R,))
        code = lib.spec_sample_rows_masked(_p(logits), _dtype_code(logits), _p(uniforms), _p(thr),
                                           float(temperature), R, V, _p(tokens), _p(ws), ws.numel(), _stream(dev))
    _raise(code, "spec_sample_rows")
    if check:
        check_status(ws)
    return tokens


def topk_threshold(logits: torch.Tensor, k: int) -> torch.Tensor:
    """spec_topk_threshold: logits [..., V]; returns the per-row threshold (float32, shape [...])."""
    V = logits.shape[-1]
    _cuda(logits, "logits")
    R = logits.numel() // V
    thr = torch.empty(logits.shape[:-1], dtype=torch.float32, device=logits.device)
    _raise(lib.spec_topk_threshold(_p(logits), _dtype_code(logits), R, V, int(k), _p(thr), _stream(logits.device)),
           "spec_topk_threshold")
    return thr


def topp_threshold(logits: torch.Tensor, temperature: float, top_p: float) -> torch.Tensor:
    """spec_topp_threshold: logits [..., V]; returns the per-row threshold (float32, shape [...])."""
    V = logits.shape[-1]
    _cuda(logits, "logits")
    R = logits.numel() // V
    thr = torch.empty(logits.shape[:-1], dtype=torch.float32, device=logits.device)
    _raise(lib.spec_topp_threshold(_p(logits), _dtype_code(logits), float(temperature), float(top_p), R, V, _p(thr),
                                   _stream(logits.device)), "spec_topp_threshold")
    return thr


def verify_greedy(target: torch.Tensor, ids: torch.Tensor, draft_len: torch.Tensor | None = None,
                  draft: torch.Tensor | None = None, *, emitted=None, n_accepted=None,
                  workspace: torch.Tensor | None = None, check: bool = False):
    """spec_verify_greedy: returns (emitted [B, gamma+1] int32, n_accepted [B] int32)."""
    B, G, V = _common(target, draft, ids, draft_len, gamma_needs_draft=False)
    dev = target.device
    if emitted is None:
        emitted = torch.empty(B, G + 1, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    _cuda(emitted, "emitted", torch.int32, (B, G + 1))
    _cuda(n_accepted, "n_accepted", torch.int32, (B,))
    ws = workspace if workspace is not None else workspace_for(dev, workspace_size(B, G, V, target.dtype))
    code = lib.spec_verify_greedy(_p(target), _p(draft), _dtype_code(target), _p(ids) if G > 0 else None,
                                  _p(draft_len), B, G, V, _p(emitted), _p(n_accepted), _p(ws), ws.numel(),
                                  _stream(dev))
    _raise(code, "spec_verify_greedy")
    if check:
        check_status(ws)
    return emitted, n_accepted


def accept_stats(target: torch.Tensor, draft: torch.Tensor, ids: torch.Tensor, temperature: float,
                 draft_len: torch.Tensor | None = None, *, workspace: torch.Tensor | None = None,
                 check: bool = False) -> dict:
    """spec_accept_stats: dict of [B, gamma] float32 tensors beta, p_x, q_x, accept_prob, resid."""
    B, G, V = _common(target, draft, ids, draft_len)
    dev = target.device
    out = {k: torch.empty(B, G, dtype=torch.float32, device=dev) for k in ("beta", "p_x", "q_x", "accept_prob",
                                                                          "resid")}
    ws = workspace if workspace is not None else workspace_for(dev, workspace_size(B, G, V, target.dtype))
    code = lib.spec_accept_stats(_p(target), _p(draft) if G > 0 else None, _dtype_code(target),
                                 _p(ids) if G > 0 else None, _p(draft_len), float(temperature), B, G, V,
                                 _p(out["beta"]), _p(out["p_x"]), _p(out["q_x"]), _p(out["accept_prob"]),
                                 _p(out["resid"]), _p(ws), ws.numel(), _stream(dev))
    _raise(code, "spec_accept_stats")
    if check:
        check_status(ws)
    return out
