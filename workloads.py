"""Seeded synthetic workloads for RMSNorm: shapes, dtypes and value distributions.

This module holds no part of the method's arithmetic: it only names the workloads and
draws their random inputs.  Both the device path (tests, benchmark) and the CPU oracle
legs take their inputs from here.

Distributions follow the workloads the pages measure on (FlashInfer PR #5741
"cake_rmsnorm_train", Performance / Accuracy: random BF16 activations and gradients,
FP32 or BF16 weights; FlashInfer PR #4480, Validation: random x and residual):
  x, dy ~ N(0, sigma) drawn in fp32 then rounded to the storage dtype (round to
  nearest even); w = 1 + 0.1 * N(0, 1); sigma is a standard deviation.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    x_dtype: torch.dtype
    w_dtype: torch.dtype
    eps: float = 1e-6
    x_std: float = 1.0
    dy_std: float = 1.0
    res_std: float = 2.0
    note: str = ""


# fwd + fused bwd, fp32 everything: the small case the oracle finishes instantly
SMALL_FP32 = Workload("rmsnorm_t64_h256_fp32", 64, 256, torch.float32, torch.float32)
# fwd + fused bwd at the headline shape
MAIN_BF16 = Workload("rmsnorm_t8192_h4096_bf16", 8192, 4096, torch.bfloat16, torch.bfloat16)
# fused residual add + RMSNorm + E4M3 1x128 block quant
FUSED_QUANT = Workload("fused_add_rmsnorm_fp8_t2048_h4096_bf16", 2048, 4096, torch.bfloat16,
                       torch.bfloat16, res_std=2.0)
# the same fused op at the headline shape (the step the benchmark times)
RESIDUAL_MAIN = Workload("rmsnorm_residual_t8192_h4096_bf16", 8192, 4096, torch.bfloat16,
                         torch.bfloat16, res_std=2.0)

FUSED_QUANT_MAIN = Workload("fused_add_rmsnorm_fp8_t8192_h4096_bf16", 8192, 4096,
                            torch.bfloat16, torch.bfloat16, res_std=2.0)
# deterministic backward sweep: bf16 x/dy, fp32 w
DET_SWEEP_H = (1536, 2048, 4096, 5120, 6144)
DET_SWEEP_T = (65, 4096, 65536, 131072)
DET_SWEEP = tuple(Workload(f"det_bwd_t{T}_h{H}", T, H, torch.bfloat16, torch.float32)
                  for H in DET_SWEEP_H for T in DET_SWEEP_T)
# large-T backward with the compensated weight gradient
TWOSUM_LARGE = Workload("twosum_bwd_t262144_h5120", 262144, 5120, torch.bfloat16,
                        torch.float32, x_std=3.0)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std: float, dtype: torch.dtype, g: torch.Generator, device) -> torch.Tensor:
    v = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v.to(dtype)


def weight(H: int, dtype: torch.dtype, g: torch.Generator, device) -> torch.Tensor:
    v = torch.randn(H, generator=g, device=device, dtype=torch.float32)
    return (1.0 + 0.1 * v).to(dtype)


def fwd_bwd_inputs(wl: Workload, device="cpu", seed: int = 0, T: int | None = None):
    """x, dy [T, H] (x_dtype) and w [H] (w_dtype), drawn in the order x, dy, w."""
    T = wl.T if T is None else T
    g = _gen(device, seed)
    x = _normal((T, wl.H), wl.x_std, wl.x_dtype, g, device)
    dy = _normal((T, wl.H), wl.dy_std, wl.x_dtype, g, device)
    w = weight(wl.H, wl.w_dtype, g, device)
    return x, dy, w


def fused_inputs(wl: Workload, device="cpu", seed: int = 0, T: int | None = None):
    """x, residual [T, H] bf16 and w [H] bf16, drawn in the order x, residual, w."""
    T = wl.T if T is None else T
    g = _gen(device, seed)
    x = _normal((T, wl.H), wl.x_std, torch.bfloat16, g, device)
    res = _normal((T, wl.H), wl.res_std, torch.bfloat16, g, device)
    w = weight(wl.H, torch.bfloat16, g, device)
    return x, res, w


def residual_inputs(wl: Workload, device="cpu", seed: int = 0, T: int | None = None):
    """Inputs of the residual training variant: x, residual, dy, g_residual [T, H] (x_dtype)
    and w [H] (w_dtype), drawn in the order x, residual, dy, g_residual, w; residual has
    standard deviation res_std, the others as in fwd_bwd_inputs."""
    T = wl.T if T is None else T
    g = _gen(device, seed)
    x = _normal((T, wl.H), wl.x_std, wl.x_dtype, g, device)
    res = _normal((T, wl.H), wl.res_std, wl.x_dtype, g, device)
    dy = _normal((T, wl.H), wl.dy_std, wl.x_dtype, g, device)
    g_res = _normal((T, wl.H), wl.dy_std, wl.x_dtype, g, device)
    w = weight(wl.H, wl.w_dtype, g, device)
    return x, res, dy, g_res, w


def round_up(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def to_oracle(t: torch.Tensor):
    """CPU numpy view of a tensor in the oracle's storage formats (bf16 -> uint16 bits)."""
    import numpy as np
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.float64):
        return t.numpy()
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


def _esize(dtype: torch.dtype) -> int:
    return torch.empty((), dtype=dtype).element_size()


def fwd_bytes(T: int, H: int, x_dtype: torch.dtype, w_dtype: torch.dtype) -> int:
    """Logical HBM bytes of one forward: read x, write y, read w once, write rstd
    (FlashInfer PR #5741, Performance: fwd 2TH x 2 + 4T for bf16)."""
    s, sw = _esize(x_dtype), _esize(w_dtype)
    return 2 * T * H * s + H * sw + 4 * T


def bwd_bytes(T: int, H: int, x_dtype: torch.dtype, w_dtype: torch.dtype) -> int:
    """Logical HBM bytes of one backward: read x and dy, write dx, read w and rstd,
    write dw (FlashInfer PR #5741, Performance: bwd 3 x 2TH + 4T + 4H for bf16)."""
    s, sw = _esize(x_dtype), _esize(w_dtype)
    return 3 * T * H * s + H * sw + 4 * T + 4 * H


def fwd_residual_bytes(T: int, H: int, x_dtype: torch.dtype, w_dtype: torch.dtype) -> int:
    """The forward's bytes plus reading residual and writing h_new (FlashInfer PR #5741,
    Performance: fwd ... [+ 2TH residual in, 2TH h_new out] for bf16)."""
    return fwd_bytes(T, H, x_dtype, w_dtype) + 2 * T * H * _esize(x_dtype)


def bwd_residual_bytes(T: int, H: int, x_dtype: torch.dtype, w_dtype: torch.dtype) -> int:
    """The backward's bytes plus reading g_residual (FlashInfer PR #5741, Performance:
    bwd ... [+ 2TH] for bf16)."""
    return bwd_bytes(T, H, x_dtype, w_dtype) + T * H * _esize(x_dtype)


def fused_quant_bytes(T: int, H: int) -> int:
    """Logical HBM bytes of the fused residual-add + RMSNorm + E4M3 1x128 block quant:
    read x and residual, write residual and normed (bf16), write q (1 B), write one fp32
    scale per 128 columns, read w once (FlashInfer PR #4480: ~9*M*H)."""
    return 9 * T * H + 4 * T * (H // 128) + 2 * H
