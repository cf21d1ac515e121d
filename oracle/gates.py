"""Parity gates between a device result and the FP64 oracle.

TEST INFRASTRUCTURE ONLY (used by ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's sampled self-check).  Tolerances:

* fp32 outputs (``rstd``; ``y`` and ``dx`` of an fp32 input): relative 1e-5.  ``dx``
  cancels (``g - xhat*c``), so its elementwise bound is taken relative to the row:
  ``|d - ref| <= 1e-5*|ref| + 1e-5*rms_row(ref)``.
* bf16 outputs: within one bf16 ulp of the exact value: ``|d - ref| <= ulp_bf16(ref)``.
  Where the fp32 evaluation on the device can itself be off by more than half a bf16
  ulp (strong cancellation in ``dx``), the a-priori fp32 error bound ``B`` of that
  element is added: ``|d - ref| <= ulp_bf16(ref) + B``; such elements are counted.
* dW (fp32): ``|dw - ref| <= 1e-4 + 1e-4*|ref|`` against the FP64 sum at the saved rstd
  (miles-ext-kernels PR #15, Accuracy: the weight-gradient budget).
* fp8 codes and block scales: bit-exact, the oracle quantizing the device's own bf16
  normed output (FlashInfer PR #4480, Summary: the codes come from the normed values after
  their rounding to bf16, the same values that normed_out holds).
"""
from __future__ import annotations

import numpy as np

U32 = 2.0 ** -24  # unit roundoff of binary32


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |ref| (binade of |ref|; subnormal quantum below 2^-126)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126.0), -126.0)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_bf16(dev_bits: np.ndarray, ref: np.ndarray, extra: np.ndarray | None = None) -> dict:
    """Elementwise 1-ulp gate for bf16 outputs (optionally widened by ``extra``)."""
    d = bf16_to_f64(dev_bits)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(d - ref)
    ulp = ulp_bf16(ref)
    ok_plain = err <= ulp
    if extra is None:
        ok = ok_plain
        n_extra = 0
    else:
        ok = ok_plain | (err <= ulp + extra)
        n_extra = int(np.count_nonzero(ok & ~ok_plain))
    bad = ~ok | ~np.isfinite(d)
    return {"n": int(d.size), "n_fail": int(np.count_nonzero(bad)), "n_widened": n_extra,
            "max_err_in_ulp": float(np.max(err / ulp)) if d.size else 0.0,
            "first_fail": _first(bad)}


def check_f32_rel(dev: np.ndarray, ref: np.ndarray, rtol: float = 1e-5,
                  row_rms_term: bool = False) -> dict:
    d = np.asarray(dev, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = rtol * np.abs(ref)
    if row_rms_term:
        rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
        tol = tol + rtol * rms
    err = np.abs(d - ref)
    bad = ~(err <= tol) | ~np.isfinite(d)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / tol, np.where(err > 0, np.inf, 0.0))
    return {"n": int(d.size), "n_fail": int(np.count_nonzero(bad)),
            "worst_ratio": float(np.max(ratio)) if d.size else 0.0, "first_fail": _first(bad)}


def check_dw(dev: np.ndarray, ref: np.ndarray, atol: float = 1e-4, rtol: float = 1e-4) -> dict:
    """Weight-gradient budget: worst = max |dw - ref| / (atol + rtol*|ref|) must be <= 1."""
    d = np.asarray(dev, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ratio = np.abs(d - ref) / (atol + rtol * np.abs(ref))
    bad = ~(ratio <= 1.0) | ~np.isfinite(d)
    rel_l2 = float(np.linalg.norm(d - ref) / max(np.linalg.norm(ref), 1e-300))
    return {"n": int(d.size), "n_fail": int(np.count_nonzero(bad)),
            "worst": float(np.max(ratio)) if d.size else 0.0, "rel_l2": rel_l2,
            "first_fail": _first(bad)}


def dx_fp32_bound(dy: np.ndarray, x: np.ndarray, w: np.ndarray, rstd: np.ndarray,
                  dx_ref: np.ndarray) -> np.ndarray:
    """A-priori bound on the error of an fp32 evaluation of
    ``dx = rstd*(g - xhat*c)``, ``g = dy*w``, ``xhat = x*rstd``, ``c = mean(g*xhat)``
    before the final rounding to the output type (inputs exact in binary64).

    Each product and the final scaling carry one binary32 rounding; the row sum of
    ``H`` products carries at most ``(H-1)*u*sum|g*xhat|`` whatever its order.  The
    bound is doubled to cover second-order terms."""
    u = U32
    r = np.asarray(rstd, dtype=np.float64)[:, None]
    g = np.asarray(dy, np.float64) * np.asarray(w, np.float64)[None, :]
    xh = np.asarray(x, np.float64) * r
    H = g.shape[1]
    c = np.mean(g * xh, axis=1, keepdims=True)
    S = np.mean(np.abs(g * xh), axis=1, keepdims=True)
    dc = (H + 3) * u * S + u * np.abs(c)
    b = r * (2 * u * np.abs(g) + 3 * u * np.abs(xh * c) + np.abs(xh) * dc) + u * np.abs(dx_ref)
    return 2.0 * b


def _first(bad: np.ndarray):
    idx = np.argwhere(bad)
    return tuple(int(i) for i in idx[0]) if idx.size else None
