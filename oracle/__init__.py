"""FP64 CPU oracle for the RMSNorm forward, the fused dX+dW backward and the fused
residual-add + RMSNorm + E4M3 1x128 block quantization.

TEST INFRASTRUCTURE ONLY.  The product package never imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs
do.  The arithmetic lives in ``rmsnorm_oracle.c`` (plain C99, binary64, compiled with
gcc, no fast-math, no FMA contraction); this file only builds it, marshals numpy arrays
and exposes it.  It shares no code with the CUDA path.

Every input array is one of:
  * ``np.float32``  -> stored as IEEE binary32,
  * ``np.uint16``   -> the bit patterns of bfloat16 values,
  * ``np.float64``  -> binary64 (used for finite-difference checks on tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` (gcc, seconds)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.or_bf16_round.restype = ctypes.c_uint16
            L.or_bf16_round.argtypes = [ctypes.c_double]
            L.or_bf16_round_n.restype = None
            L.or_bf16_round_n.argtypes = [_vp, _i64, _vp]
            L.or_e4m3_encode.restype = ctypes.c_uint8
            L.or_e4m3_encode.argtypes = [ctypes.c_float]
            L.or_e4m3_decode.restype = ctypes.c_float
            L.or_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.or_rmsnorm_fwd.restype = None
            L.or_rmsnorm_fwd.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _i64, _i64,
                                         ctypes.c_double, _vp, _vp, ctypes.c_int]
            L.or_rmsnorm_bwd.restype = None
            L.or_rmsnorm_bwd.argtypes = [_vp, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp,
                                         _i64, _i64, _vp, _vp, ctypes.c_int]
            L.or_fused_add_rmsnorm.restype = None
            L.or_fused_add_rmsnorm.argtypes = [_vp, _vp, _vp, _i64, _i64, ctypes.c_double,
                                               _vp, _vp, _vp, ctypes.c_int]
            L.or_block_quant_e4m3.restype = None
            L.or_block_quant_e4m3.argtypes = [_vp, _i64, _i64, _vp, _vp, _i64, ctypes.c_int]
            _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _fmt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported oracle input dtype {a.dtype}")


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------- forward
def rmsnorm_fwd(x: np.ndarray, w: np.ndarray, eps: float, nthreads: int | None = None,
                want_y: bool = True):
    """Forward in binary64.  x: [T, H]; w: [H].  Returns (y [T,H] f64 or None, rstd [T] f64)."""
    x, w = _c(x), _c(w)
    T, H = x.shape
    assert w.shape == (H,)
    y = np.empty((T, H), np.float64) if want_y else None
    rstd = np.empty((T,), np.float64)
    lib().or_rmsnorm_fwd(_ptr(x), _fmt(x), _ptr(w), _fmt(w), T, H, float(eps),
                         _ptr(y) if want_y else None, _ptr(rstd),
                         nthreads or default_threads())
    return y, rstd


# ---------------------------------------------------------------------------- backward
def rmsnorm_bwd(dy: np.ndarray, x: np.ndarray, w: np.ndarray, rstd: np.ndarray,
                nthreads: int | None = None, want_dx: bool = True, want_dw: bool = True):
    """Backward in binary64 at the given rstd (the forward's saved value).

    dy, x: [T, H] in the same storage format; w: [H]; rstd: [T] (converted exactly to
    binary64).  Returns (dx [T,H] f64 or None, dw [H] f64 or None)."""
    dy, x, w = _c(dy), _c(x), _c(w)
    r = np.ascontiguousarray(rstd, dtype=np.float64)
    T, H = x.shape
    assert dy.shape == (T, H) and w.shape == (H,) and r.shape == (T,)
    assert _fmt(dy) == _fmt(x)
    dx = np.empty((T, H), np.float64) if want_dx else None
    dw = np.empty((H,), np.float64) if want_dw else None
    lib().or_rmsnorm_bwd(_ptr(dy), _ptr(x), _fmt(x), _ptr(w), _fmt(w), _ptr(r), T, H,
                         _ptr(dx) if want_dx else None, _ptr(dw) if want_dw else None,
                         nthreads or default_threads())
    return dx, dw


# ------------------------------------------------------------- residual variants
def residual_add(x: np.ndarray, res: np.ndarray) -> np.ndarray:
    """h = x + res, rounded once to the storage format (FlashInfer PR #5741
    "cake_rmsnorm_train", Design/Forward: h_new = bf16(x + residual)).  The binary64 sum of
    two bf16 or two binary32 values is exact, so rounding it once (RNE) to the format is the
    correctly rounded sum.  Same storage format as the inputs (float64 stays float64)."""
    x, res = _c(x), _c(res)
    assert x.shape == res.shape and _fmt(x) == _fmt(res)
    if x.dtype == np.uint16:
        s = bf16_bits_to_f64(x) + bf16_bits_to_f64(res)
        return bf16_round(s).reshape(x.shape)
    s = x.astype(np.float64) + res.astype(np.float64)
    return s.astype(x.dtype)  # float32: RNE to binary32; float64: exact already


def rmsnorm_fwd_residual(x: np.ndarray, res: np.ndarray, w: np.ndarray, eps: float,
                         nthreads: int | None = None):
    """Forward fused with the residual add (PR #5741, Design/Forward and API: the forward
    with `residual=` returns y, rstd and h_new; h_new is what is normalized).
    Returns (y [T,H] f64, rstd [T] f64, h_new in the storage format)."""
    h = residual_add(x, res)
    y, rstd = rmsnorm_fwd(h, w, eps, nthreads)
    return y, rstd, h


def rmsnorm_bwd_residual(dy: np.ndarray, h: np.ndarray, w: np.ndarray, rstd: np.ndarray,
                         g_res: np.ndarray, nthreads: int | None = None,
                         want_dx: bool = True, want_dw: bool = True):
    """Backward of the residual forward at h = h_new (PR #5741, Design/Backward: the
    residual variant adds g_residual into the dx it returns, dx_total; dw is unchanged).
    Returns (dx_total [T,H] f64 or None, dw [H] f64 or None)."""
    dx, dw = rmsnorm_bwd(dy, h, w, rstd, nthreads, want_dx=want_dx, want_dw=want_dw)
    if want_dx:
        g = _c(g_res)
        gv = bf16_bits_to_f64(g) if g.dtype == np.uint16 else g.astype(np.float64)
        dx = dx + gv.reshape(dx.shape)
    return dx, dw


# ------------------------------------------------------------------ fused add + norm
def fused_add_rmsnorm(x_bits: np.ndarray, res_bits: np.ndarray, w_bits: np.ndarray,
                      eps: float, nthreads: int | None = None):
    """h = bf16(x + residual), rstd of h, normed = h*rstd*w (binary64, unrounded).

    All inputs are bf16 bit patterns (np.uint16).  Returns (h_bits [T,H] u16,
    n [T,H] f64, rstd [T] f64)."""
    x, r, w = _c(x_bits), _c(res_bits), _c(w_bits)
    for a in (x, r, w):
        assert a.dtype == np.uint16
    T, H = x.shape
    h = np.empty((T, H), np.uint16)
    n = np.empty((T, H), np.float64)
    rstd = np.empty((T,), np.float64)
    lib().or_fused_add_rmsnorm(_ptr(x), _ptr(r), _ptr(w), T, H, float(eps), _ptr(h), _ptr(n),
                               _ptr(rstd), nthreads or default_threads())
    return h, n, rstd


def block_quant_e4m3(n_bits: np.ndarray, ld: int, scale_init: np.ndarray | None = None,
                     nthreads: int | None = None):
    """1x128 block quantization of bf16 values (binary32 decisions).

    n_bits: [T, H] bf16 bits.  Returns (q [T,H] u8, scale [(H/128) * ld] f32); entries
    of ``scale`` that the definition does not write keep ``scale_init`` (NaN if None)."""
    n = _c(n_bits)
    assert n.dtype == np.uint16
    T, H = n.shape
    assert H % 128 == 0 and ld >= T
    q = np.empty((T, H), np.uint8)
    if scale_init is None:
        scale = np.full(((H // 128) * ld,), np.nan, np.float32)
    else:
        scale = np.array(scale_init, dtype=np.float32, copy=True).reshape(-1)
        assert scale.size == (H // 128) * ld
    lib().or_block_quant_e4m3(_ptr(n), T, H, _ptr(q), _ptr(scale), ld,
                              nthreads or default_threads())
    return q, scale


# -------------------------------------------------------------------- scalar codecs
def bf16_round(values) -> np.ndarray:
    """Round binary64 values to bf16 (nearest, ties to even); returns bit patterns."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64).reshape(-1))
    out = np.empty(v.shape, np.uint16)
    lib().or_bf16_round_n(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = np.asarray(values, dtype=np.float32).reshape(-1)
    L = lib()
    return np.array([L.or_e4m3_encode(float(a)) for a in v], dtype=np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).reshape(-1)
    L = lib()
    return np.array([L.or_e4m3_decode(int(a)) for a in c], dtype=np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> binary64 decode (a storage reinterpretation, no arithmetic)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
