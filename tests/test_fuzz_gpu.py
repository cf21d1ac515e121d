"""GPU parity of every entry point on seeded random shapes against the FP64 oracle: T from
1 to ~20000 (log-uniform, most above the small-T route), H any multiple of the 16-byte
vector up to 16384 (log-uniform, most from 1024), random x/w dtypes, both dW settings and both reduction modes, so the launch planner's rules
(warps per CTA, vectors per lane, pairs or single rows, CTAs per SM, stages, the small-T
route) are crossed with ragged strips rather than only the listed shapes.
Forward and fused backward: FlashInfer PR #5741 "cake_rmsnorm_train", Design/Forward and
Design/Backward; residual variant: the same page, API; fused add + norm + E4M3 1x128 quant:
FlashInfer PR #4480 "Add FusedAddRMSNormFP8BlockQuant", Summary/Kernel."""
import dataclasses

import numpy as np
import pytest
import torch

import _parity as P
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF, F32 = torch.bfloat16, torch.float32
MAX_ELEMS = 6 << 20  # keeps every case to a few hundred milliseconds


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        xd = BF if rng.random() < 0.7 else F32
        wd = BF if rng.random() < 0.5 else F32
        vec = 8 if xd == BF else 4
        hlo = np.log(vec) if rng.random() < 0.2 else np.log(1024)  # most rows of 1-16 K
        H = int(round(np.exp(rng.uniform(hlo, np.log(16384))) / vec)) * vec
        H = min(max(H, vec), 16384)
        lo = 0.0 if rng.random() < 0.3 else np.log(257)  # most above the small-T route
        T = int(np.exp(rng.uniform(lo, np.log(20000))))
        if T * H > MAX_ELEMS:
            T = max(1, MAX_ELEMS // H)
        out.append((T, H, xd, wd, bool(rng.random() < 0.5), bool(rng.random() < 0.8)))
    return out


CASES = _cases(48, seed=20261203)
IDS = [f"T{c[0]}-H{c[1]}-{'bf16' if c[2] == BF else 'fp32'}x-{'bf16' if c[3] == BF else 'fp32'}w"
       f"-{'comp' if c[4] else 'blk'}-{'det' if c[5] else 'fast'}" for c in CASES]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fwd_bwd_random_shape(case):
    T, H, xd, wd, comp, det = case
    c = dataclasses.replace(wl.MAIN_BF16, T=T, H=H, x_dtype=xd, w_dtype=wd)
    x, dy, w = wl.fwd_bwd_inputs(c, DEV, seed=T * 7 + H)
    P.assert_ok(P.check_fwd(x, w, c.eps), f"fwd {case}")
    _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
    if xd == F32 and H > 8192:  # the fp32-x backward stops at H = 8192
        with pytest.raises(rmsn.RmsnError):
            rmsn.rmsnorm_bwd(dy, x, w, rstd)
        return
    P.assert_ok(P.check_bwd(dy, x, w, rstd, deterministic=det, compensated=comp), f"bwd {case}")


@pytest.mark.parametrize("case", CASES[::2], ids=IDS[::2])
def test_residual_random_shape(case):
    T, H, xd, wd, comp, det = case
    c = dataclasses.replace(wl.RESIDUAL_MAIN, T=T, H=H, x_dtype=xd, w_dtype=wd)
    x, res, dy, g, w = wl.residual_inputs(c, DEV, seed=T * 11 + H)
    rf = P.check_fwd_residual(x, res, w, c.eps)
    P.assert_ok(rf, f"fwd_residual {case}")
    if xd == F32 and H > 8192:
        return
    rb = P.check_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], g, deterministic=det,
                              compensated=comp)
    P.assert_ok(rb, f"bwd_residual {case}")


@pytest.mark.parametrize("case", CASES[1::2], ids=IDS[1::2])
def test_fused_random_shape(case):
    T, H = case[0], max(128, case[1] // 128 * 128)  # the quant wants H % 128 == 0, bf16
    c = dataclasses.replace(wl.FUSED_QUANT, T=T, H=H)
    x, res, w = wl.fused_inputs(c, DEV, seed=T * 5 + H)
    P.assert_ok(P.check_fused(x, res, w, c.eps, ld_pad=4 * (T % 3)), f"fused T={T} H={H}")
