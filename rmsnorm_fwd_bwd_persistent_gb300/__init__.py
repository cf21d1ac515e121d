"""GB300 (sm_103a) RMSNorm: forward, fused dX+dW backward, and fused residual-add +
RMSNorm + E4M3 1x128 block quantization.

This module is a thin binding over the C ABI of ``librmsn_gb300.so`` (declared in
``include/rmsn.h``): it checks tensor dtypes/devices/contiguity, allocates outputs the
caller did not pass, and forwards raw device pointers and the current CUDA stream.
Every step of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback -- if the library is missing or was not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "RMSN_F32", "RMSN_BF16", "RMSN_MAX_H", "RmsnError", "library_path", "load_library",
    "rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes",
    "rmsnorm_fwd_residual", "rmsnorm_bwd_residual",
    "fused_add_rmsnorm_fp8_block_quant", "rmsn_status_string", "rmsn_plan", "rmsn_set_policy",
    "rmsn_device_status", "rmsn_set_small_t_max", "rmsn_small_t_max", "rmsn_selftest_wait_timeout",
    "OP_FWD", "OP_BWD", "OP_FUSED_QUANT", "OP_FWD_RESIDUAL", "OP_BWD_RESIDUAL",
]

RMSN_F32, RMSN_BF16 = 0, 1
RMSN_MAX_H = 16384
OP_FWD, OP_BWD, OP_FUSED_QUANT, OP_FWD_RESIDUAL, OP_BWD_RESIDUAL = 0, 1, 2, 3, 4

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "librmsn_gb300.so")
_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class RmsnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {rmsn_status_string(status)} (status {status})")


class _Plan(ctypes.Structure):
    _fields_ = [("vec_elems", ctypes.c_int), ("consumer_warps", ctypes.c_int),
                ("chunks_per_lane", ctypes.c_int), ("threads", ctypes.c_int),
                ("stages", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("grid", ctypes.c_int64), ("smem_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64)]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads ``librmsn_gb300.so`` (built by ``build.py``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m rmsnorm_fwd_bwd_persistent_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(_LIB_PATH)
        L.rmsn_status_string.restype = ctypes.c_char_p
        L.rmsn_status_string.argtypes = [ctypes.c_int]
        L.rmsnorm_fwd.restype = ctypes.c_int
        L.rmsnorm_fwd.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp, _i64, _i64,
                                  ctypes.c_float, _vp]
        L.rmsnorm_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.rmsnorm_bwd_workspace_bytes.argtypes = [_i64, _i64, ctypes.c_int, ctypes.c_int]
        L.rmsnorm_bwd.restype = ctypes.c_int
        L.rmsnorm_bwd.argtypes = [_vp, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp, _vp,
                                  _i64, _i64, ctypes.c_int, ctypes.c_int, _vp, ctypes.c_size_t,
                                  _vp]
        L.fused_add_rmsnorm_fp8_block_quant.restype = ctypes.c_int
        L.fused_add_rmsnorm_fp8_block_quant.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _vp,
                                                        _i64, _i64, ctypes.c_float, _vp]
        L.rmsn_plan.restype = ctypes.c_int
        L.rmsn_set_small_t_max.restype = ctypes.c_int
        L.rmsn_set_small_t_max.argtypes = [_i64]
        L.rmsn_small_t_max.restype = _i64
        L.rmsn_small_t_max.argtypes = []
        L.rmsn_selftest_wait_timeout.restype = ctypes.c_int
        L.rmsn_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _vp]
        L.rmsnorm_fwd_residual.restype = ctypes.c_int
        L.rmsnorm_fwd_residual.argtypes = [_vp, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp,
                                           _vp, _i64, _i64, ctypes.c_float, _vp]
        L.rmsnorm_bwd_residual.restype = ctypes.c_int
        L.rmsnorm_bwd_residual.argtypes = [_vp, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp,
                                           _vp, _vp, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                           _vp, ctypes.c_size_t, _vp]
        L.rmsn_plan.argtypes = [ctypes.c_int, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.POINTER(_Plan)]
        L.rmsn_set_policy.restype = ctypes.c_int
        L.rmsn_set_policy.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.rmsn_device_status.restype = ctypes.c_int
        L.rmsn_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint)]
        L.rmsnorm_bwd_noalloc.restype = ctypes.c_int
        L.rmsnorm_bwd_noalloc.argtypes = [_vp, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp,
                                          _vp, _i64, _i64, ctypes.c_int, _vp]
        _lib = L
        return _lib


def rmsn_status_string(status: int) -> str:
    return load_library().rmsn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise RmsnError(status, what)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return RMSN_F32
    if t.dtype == torch.bfloat16:
        return RMSN_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


# --------------------------------------------------------------------------- forward
def rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, y: torch.Tensor | None = None,
                rstd: torch.Tensor | None = None):
    """y = x * rstd * w, rstd = 1/sqrt(mean(x^2) + eps) per row.  Returns (y, rstd)."""
    _cuda(x, "x")
    _cuda(w, "w")
    if x.dim() != 2 or w.dim() != 1 or w.shape[0] != x.shape[1]:
        raise ValueError("x must be [T, H] and w [H]")
    T, H = x.shape
    if y is None:
        y = torch.empty_like(x)
    if rstd is None:
        rstd = torch.empty(T, device=x.device, dtype=torch.float32)
    _cuda(y, "y")
    _cuda(rstd, "rstd")
    if y.shape != x.shape or y.dtype != x.dtype or rstd.shape != (T,) or rstd.dtype != torch.float32:
        raise ValueError("y must match x; rstd must be float32 [T]")
    with torch.cuda.device(x.device):
        st = load_library().rmsnorm_fwd(_p(x), _dt(x), _p(w), _dt(w), _p(y), _p(rstd), T, H,
                                         float(eps), _stream(x))
    _check(st, "rmsnorm_fwd")
    return y, rstd


# -------------------------------------------------------------------------- backward
def rmsnorm_bwd_workspace_bytes(T: int, H: int, compensated: bool = False,
                                device: int | torch.device | None = None) -> int:
    if device is None:
        device = torch.cuda.current_device()
    if isinstance(device, torch.device):
        device = device.index if device.index is not None else torch.cuda.current_device()
    return int(load_library().rmsnorm_bwd_workspace_bytes(int(T), int(H), int(bool(compensated)),
                                                          int(device)))


def rmsnorm_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                deterministic: bool = True, compensated: bool = False,
                workspace: torch.Tensor | None = None, dx: torch.Tensor | None = None,
                dw: torch.Tensor | None = None):
    """Fused backward.  Returns (dx, dw); dw is float32 [H] (overwritten)."""
    for t, n in ((dy, "dy"), (x, "x"), (w, "w"), (rstd, "rstd")):
        _cuda(t, n)
    if x.dim() != 2 or dy.shape != x.shape or dy.dtype != x.dtype:
        raise ValueError("dy and x must be [T, H] of one dtype")
    T, H = x.shape
    if w.shape != (H,) or rstd.shape != (T,) or rstd.dtype != torch.float32:
        raise ValueError("w must be [H]; rstd float32 [T]")
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(H, device=x.device, dtype=torch.float32)
    _cuda(dx, "dx")
    _cuda(dw, "dw")
    if dx.shape != x.shape or dx.dtype != x.dtype or dw.shape != (H,) or dw.dtype != torch.float32:
        raise ValueError("dx must match x; dw must be float32 [H]")
    if workspace is None:
        n = rmsnorm_bwd_workspace_bytes(T, H, compensated, x.device)
        workspace = torch.empty(max(n, 16), device=x.device, dtype=torch.uint8)
    _cuda(workspace, "workspace")
    ws_ptr, ws_bytes = _p(workspace), workspace.numel() * workspace.element_size()
    with torch.cuda.device(x.device):
        st = load_library().rmsnorm_bwd(_p(dy), _p(x), _dt(x), _p(w), _dt(w), _p(rstd), _p(dx),
                                        _p(dw), T, H, int(bool(deterministic)),
                                        int(bool(compensated)), ws_ptr, ws_bytes, _stream(x))
    _check(st, "rmsnorm_bwd")
    return dx, dw


# --------------------------------------------------------------- residual variants
def rmsnorm_fwd_residual(x: torch.Tensor, residual: torch.Tensor, w: torch.Tensor,
                         eps: float = 1e-6, y: torch.Tensor | None = None,
                         h_new: torch.Tensor | None = None, rstd: torch.Tensor | None = None):
    """h_new = round(x + residual); y, rstd = the forward of h_new.  Returns (y, rstd, h_new).
    h_new may be `residual` itself (in-place update)."""
    for t, n in ((x, "x"), (residual, "residual"), (w, "w")):
        _cuda(t, n)
    if x.dim() != 2 or residual.shape != x.shape or residual.dtype != x.dtype:
        raise ValueError("x and residual must be [T, H] of one dtype")
    T, H = x.shape
    if w.shape != (H,):
        raise ValueError("w must be [H]")
    y = torch.empty_like(x) if y is None else y
    h_new = torch.empty_like(x) if h_new is None else h_new
    rstd = torch.empty(T, device=x.device, dtype=torch.float32) if rstd is None else rstd
    for t, n in ((y, "y"), (h_new, "h_new"), (rstd, "rstd")):
        _cuda(t, n)
    if y.shape != x.shape or y.dtype != x.dtype or h_new.shape != x.shape or \
            h_new.dtype != x.dtype or rstd.shape != (T,) or rstd.dtype != torch.float32:
        raise ValueError("y and h_new must match x; rstd must be float32 [T]")
    with torch.cuda.device(x.device):
        st = load_library().rmsnorm_fwd_residual(_p(x), _p(residual), _dt(x), _p(w), _dt(w), _p(y),
                                                 _p(h_new), _p(rstd), T, H, float(eps), _stream(x))
    _check(st, "rmsnorm_fwd_residual")
    return y, rstd, h_new


def rmsnorm_bwd_residual(dy: torch.Tensor, h: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                         g_residual: torch.Tensor, deterministic: bool = True,
                         compensated: bool = False, workspace: torch.Tensor | None = None,
                         dx_total: torch.Tensor | None = None, dw: torch.Tensor | None = None):
    """Backward of rmsnorm_fwd_residual at h = h_new: dx_total = dx + g_residual (FP32, one
    rounding), dw as rmsnorm_bwd.  Returns (dx_total, dw)."""
    for t, n in ((dy, "dy"), (h, "h"), (w, "w"), (rstd, "rstd"), (g_residual, "g_residual")):
        _cuda(t, n)
    if h.dim() != 2 or dy.shape != h.shape or dy.dtype != h.dtype or \
            g_residual.shape != h.shape or g_residual.dtype != h.dtype:
        raise ValueError("dy, h and g_residual must be [T, H] of one dtype")
    T, H = h.shape
    if w.shape != (H,) or rstd.shape != (T,) or rstd.dtype != torch.float32:
        raise ValueError("w must be [H]; rstd float32 [T]")
    dx_total = torch.empty_like(h) if dx_total is None else dx_total
    dw = torch.empty(H, device=h.device, dtype=torch.float32) if dw is None else dw
    _cuda(dx_total, "dx_total")
    _cuda(dw, "dw")
    if dx_total.shape != h.shape or dx_total.dtype != h.dtype or dw.shape != (H,) or \
            dw.dtype != torch.float32:
        raise ValueError("dx_total must match h; dw must be float32 [H]")
    if workspace is None:
        n = rmsnorm_bwd_workspace_bytes(T, H, compensated, h.device)
        workspace = torch.empty(max(n, 16), device=h.device, dtype=torch.uint8)
    _cuda(workspace, "workspace")
    ws_ptr, ws_bytes = _p(workspace), workspace.numel() * workspace.element_size()
    with torch.cuda.device(h.device):
        st = load_library().rmsnorm_bwd_residual(
            _p(dy), _p(h), _dt(h), _p(w), _dt(w), _p(rstd), _p(g_residual), _p(dx_total), _p(dw),
            T, H, int(bool(deterministic)), int(bool(compensated)), ws_ptr, ws_bytes, _stream(h))
    _check(st, "rmsnorm_bwd_residual")
    return dx_total, dw


# ------------------------------------------------------------- fused add+norm+quant
def fused_add_rmsnorm_fp8_block_quant(x: torch.Tensor, residual: torch.Tensor, w: torch.Tensor,
                                      eps: float = 1e-6, q: torch.Tensor | None = None,
                                      block_scale: torch.Tensor | None = None,
                                      normed: torch.Tensor | None = None):
    """residual <- bf16(x + residual) (in place); normed = bf16(h*rstd*w);
    per 1x128 block scale = amax/448 (buffer (H/128, round_up(T,4)), unit stride along rows);
    q = e4m3(normed/scale).  Returns (q [T,H] uint8 E4M3 codes, block_scale, normed)."""
    for t, n in ((x, "x"), (residual, "residual"), (w, "w")):
        _cuda(t, n)
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{n} must be bfloat16")
    if x.dim() != 2 or residual.shape != x.shape:
        raise ValueError("x and residual must be [T, H]")
    T, H = x.shape
    if w.shape != (H,):
        raise ValueError("w must be [H]")
    ld = (T + 3) // 4 * 4
    if q is None:
        q = torch.empty(T, H, device=x.device, dtype=torch.uint8)
    if block_scale is None:
        block_scale = torch.empty(H // 128, ld, device=x.device, dtype=torch.float32)
    if normed is None:
        normed = torch.empty_like(x)
    _cuda(normed, "normed")
    if q.dtype not in (torch.uint8, torch.float8_e4m3fn) or q.shape != (T, H) or not q.is_contiguous():
        raise ValueError("q must be a contiguous [T, H] uint8 / float8_e4m3fn tensor")
    if block_scale.dtype != torch.float32 or block_scale.dim() != 2 or \
            block_scale.shape[0] != H // 128 or not block_scale.is_contiguous():
        raise ValueError("block_scale must be a contiguous float32 (H/128, ld) tensor")
    if normed.shape != x.shape or normed.dtype != torch.bfloat16:
        raise ValueError("normed must be bfloat16 [T, H]")
    scale_ld = block_scale.shape[1]
    with torch.cuda.device(x.device):
        st = load_library().fused_add_rmsnorm_fp8_block_quant(
            _p(x), _p(residual), _p(w), _p(q), _p(block_scale), scale_ld, _p(normed), T, H,
            float(eps), _stream(x))
    _check(st, "fused_add_rmsnorm_fp8_block_quant")
    return q, block_scale, normed


# ---------------------------------------------------------------------- introspection
def rmsn_plan(op: int, T: int, H: int, x_dtype: int, w_dtype: int, compensated: bool = False,
              sm_count: int = 152) -> dict:
    p = _Plan()
    st = load_library().rmsn_plan(int(op), int(T), int(H), int(x_dtype), int(w_dtype),
                                  int(bool(compensated)), int(sm_count), ctypes.byref(p))
    _check(st, "rmsn_plan")
    return {f: getattr(p, f) for f, _ in _Plan._fields_}


def rmsn_set_policy(op: int, consumer_warps: int = 0, ctas_per_sm: int = 0, max_stages: int = 0):
    _check(load_library().rmsn_set_policy(int(op), int(consumer_warps), int(ctas_per_sm),
                                          int(max_stages)), "rmsn_set_policy")


def rmsn_set_small_t_max(t_max: int):
    """Deterministic backward calls with T <= t_max run the one-launch column-task kernel
    (0 disables).  Process-wide tuning hook."""
    _check(load_library().rmsn_set_small_t_max(int(t_max)), "rmsn_set_small_t_max")


def rmsn_small_t_max() -> int:
    return int(load_library().rmsn_small_t_max())


def rmsn_selftest_wait_timeout(limit_ns: int = 2_000_000):
    """Enqueues one CTA whose bounded wait runs out after limit_ns (no copy in flight);
    the next rmsn_device_status reports the timeout."""
    st = load_library().rmsn_selftest_wait_timeout(
        int(limit_ns), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _check(st, "rmsn_selftest_wait_timeout")


def rmsn_device_status(device: int | torch.device | None = None) -> int:
    """Synchronizes the current stream and returns (and clears) the device error word:
    0 if no kernel wait ran out since the last call."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    flags = ctypes.c_uint(0)
    with torch.cuda.device(dev):
        st = load_library().rmsn_device_status(
            ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream), ctypes.byref(flags))
    if st not in (0, 6):
        _check(st, "rmsn_device_status")
    return int(flags.value)
