"""Parity gates between a device result and the FP64 oracle.

TEST INFRASTRUCTURE ONLY (used by ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's sampled self-check).  Tolerances:

* fp32 outputs (``rstd``; ``y`` and ``dx`` of an fp32 input): relative 1e-5.  ``dx``
  cancels (``g - xhat*c``), so its elementwise bound is taken relative to the row:
  ``|d - ref| <= 1e-5*|ref| + 1e-5*rms_row(ref)``.
* bf16 outputs: within one bf16 ulp of the exact value: ``|d - ref| <= ulp_bf16(ref)``.
  Where the fp32 evaluation on the device can itself be off by more than half a bf16
  ulp (strong cancellation in ``dx``), the a-priori fp32 error bound ``B`` of that
  element (``dx_fp32_bound``, for the summation tree the launch plan states) is added:
  ``|d - ref| <= ulp_bf16(ref) + B``.  Such "widened" elements are counted and reported,
  with their error in ulps of the row's own scale.
* dW (fp32): ``|dw - ref| <= 1e-4 + 1e-4*|ref|`` against the FP64 sum at the saved rstd
  (miles-ext-kernels PR #15, Accuracy: the weight-gradient budget).
* fp8 codes and block scales: bit-exact, the oracle quantizing the device's own bf16
  normed output (FlashInfer PR #4480, Summary: the codes come from the normed values after
  their rounding to bf16, the same values that normed_out holds).
"""
from __future__ import annotations

import numpy as np

U32 = 2.0 ** -24  # unit roundoff of binary32


def gamma(m: int, u: float = U32) -> float:
    """Higham's gamma_m = m*u / (1 - m*u): the relative error bound of m roundings."""
    return m * u / (1.0 - m * u)


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers in the binade of |ref| (2^(e-7) for |ref| in [2^e, 2^(e+1));
    the subnormal quantum 2^-133 below 2^-126).  The binade comes from frexp, which is
    exact (a logarithm would misplace values within rounding distance below a power of
    two)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    _, e = np.frexp(a)  # a = m * 2^e, m in [0.5, 1): the binade exponent is e - 1
    e = np.where(a > 0, np.maximum(e.astype(np.int64) - 1, -126), -126)
    return np.ldexp(1.0, e - 7)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to quiet NaNs
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_bf16(dev_bits: np.ndarray, ref: np.ndarray, extra: np.ndarray | None = None) -> dict:
    """Elementwise 1-ulp gate for bf16 outputs (optionally widened by ``extra``).

    Reports ``n_widened`` (elements that pass only thanks to ``extra``), ``frac_widened``,
    ``max_err_in_ulp`` over the elements that pass without widening, and, for 2-D inputs,
    ``max_widened_err_row_ulp``: the widened elements' largest error in bf16 ulps of their
    row's RMS (how large the widening is on the row's own scale)."""
    d = bf16_to_f64(dev_bits)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(d - ref)
    ulp = ulp_bf16(ref)
    ok_plain = err <= ulp
    if extra is None:
        ok = ok_plain
        widened = np.zeros_like(ok_plain)
    else:
        ok = ok_plain | (err <= ulp + extra)
        widened = ok & ~ok_plain
    n_extra = int(np.count_nonzero(widened))
    bad = ~ok | ~np.isfinite(d)
    plain_ratio = np.where(ok_plain, err / ulp, 0.0)
    out = {"n": int(d.size), "n_fail": int(np.count_nonzero(bad)), "n_widened": n_extra,
           "frac_widened": n_extra / d.size if d.size else 0.0,
           "max_err_in_ulp": float(np.max(plain_ratio)) if d.size else 0.0,
           "max_widened_err_row_ulp": 0.0, "first_fail": _first(bad)}
    if n_extra and ref.ndim == 2:
        rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
        row_ulp = np.broadcast_to(ulp_bf16(rms), ref.shape)
        out["max_widened_err_row_ulp"] = float(np.max(err[widened] / row_ulp[widened]))
    return out


def check_f32_rel(dev: np.ndarray, ref: np.ndarray, rtol: float = 1e-5,
                  row_rms_term: bool = False) -> dict:
    """``|d - ref| <= rtol*|ref|`` elementwise (plus ``rtol*rms_row(ref)`` if asked)."""
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
                  dx_ref: np.ndarray, depth: int) -> np.ndarray:
    """A-priori bound on the error of a binary32 evaluation of
    ``dx = rstd*(g - xhat*c)``, ``g = dy*w``, ``xhat = x*rstd``, ``c = mean(g*xhat)``,
    before the final rounding to the output type (inputs exact in binary64).

    The evaluation it covers: ``c' = rstd*c`` formed as a sum of the terms
    ``w_j*(dy_j*x_j)`` scaled by ``rstd^2/H``, in any tree in which no term passes through
    more than ``depth`` roundings (the product, the additions of the tree and the
    scaling, with the scale's own roundings, all counted); then
    ``dx = RN(rstd * RN(g^ - x*c'))`` with ``g^ = RN(dy*w)`` and the inner difference a
    fused multiply-add.  Standard error analysis (Higham, Accuracy and Stability of
    Numerical Algorithms, 2nd ed., Lemma 3.1 and section 4.2):

      |c'^ - c'|   <= gamma(depth) * rstd * mean_j |g_j * xhat_j|
      |dx^ - dx|   <= gamma(2)*|dx| + (1 + gamma(2)) * rstd * (u*|g| + |x| * |c'^ - c'|)

    where u = 2^-24 and gamma(m) = m*u / (1 - m*u).  ``depth`` comes from the launch plan
    (``row_dot_depth`` in the tests)."""
    u = U32
    r = np.asarray(rstd, dtype=np.float64)[:, None]
    g = np.asarray(dy, np.float64) * np.asarray(w, np.float64)[None, :]
    xh = np.asarray(x, np.float64) * r
    S = np.mean(np.abs(g * xh), axis=1, keepdims=True)
    dc = gamma(depth) * r * S  # bound on the error of c' = rstd * c
    g2 = gamma(2)
    return g2 * np.abs(dx_ref) + (1.0 + g2) * r * (u * np.abs(g) + np.abs(x) * dc)


def row_dot_depth(chain_terms: int, warps: int) -> int:
    """Largest number of roundings a term ``w_j*dy_j*x_j`` meets on its way into ``c'`` in
    the device's row-dot tree, as the library documents it: one for the product
    ``dy*x`` (exact for bf16 operands, counted anyway), ``chain_terms`` fused
    multiply-adds in a lane's sequential chain, one to add the lane's two chains, five
    for the 32-lane shuffle tree, one for the scaling by ``rstd^2/H`` and three for that
    factor's own roundings, and ``warps - 1`` for adding the warps' scaled parts in warp
    order: ``chain_terms + warps + 10``."""
    return int(chain_terms) + int(warps) + 10


def _first(bad: np.ndarray):
    idx = np.argwhere(bad)
    return tuple(int(i) for i in idx[0]) if idx.size else None
