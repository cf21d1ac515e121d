"""GPU parity of the strip backward in every class of launch geometry its plan picks (T
above the small-T route, so the deterministic calls run the strip kernel and the column
reduce):
4 CTAs of 4 warps, 5 of 3, 3 of 5 and 2 of 7 (rows that fill those warps at two vectors
per lane), narrow rows over short strips with twice the warps in half the CTAs, 2 CTAs of 8 warps with rows in pairs (two and three vectors per lane),
2 CTAs of 8 warps with rows one at a time (bf16, about three vectors per lane) and one CTA
of 16 warps (rows of at least 1024 vectors; bf16 rows of three vectors per lane one at a
time), each against the FP64 oracle, with plain and TwoSum-compensated dW, for rmsnorm_bwd and rmsnorm_bwd_residual (FlashInfer PR #5741
"cake_rmsnorm_train", Design/Backward; miles-ext-kernels PR #15, Changes #8848/#8849)."""
import dataclasses

import pytest
import torch

import _parity as P
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF, F32 = torch.bfloat16, torch.float32

# (T, H, x dtype, w dtype, consumer warps, vectors per lane, CTAs per SM)
GEOMETRIES = [
    (1000, 2048, BF, F32, 4, 2, 4),
    (16401, 1536, BF, F32, 3, 2, 5),   # long strips only
    (901, 2560, BF, BF, 5, 2, 3),
    (700, 2304, BF, F32, 5, 2, 3),     # last lanes' second vector empty
    (16390, 3584, BF, F32, 7, 2, 2),   # long strips only
    (900, 1280, F32, F32, 5, 2, 3),
    (777, 4096, BF, BF, 8, 2, 2),
    (600, 5120, BF, F32, 8, 3, 2),
    (13000, 5632, BF, BF, 8, 3, 2),  # rows one at a time (third vector 3/4 full)
    (12301, 6144, BF, F32, 8, 3, 2), # rows one at a time
    (600, 5632, BF, BF, 16, 2, 1),   # the same widths over a short strip: 16 warps
    (12288, 6144, BF, F32, 16, 2, 1),
    (1000, 8192, BF, BF, 16, 2, 1),
    (300, 16384, BF, F32, 16, 4, 1),
    (513, 4096, F32, F32, 16, 2, 1),
    (300, 8192, F32, BF, 16, 4, 1),
    (20000, 384, BF, F32, 1, 2, 16),
    (700, 384, BF, F32, 2, 1, 8),     # short strip: twice the warps, half the CTAs
    (500, 7168, BF, BF, 8, 4, 2),
    (400, 9216, BF, F32, 16, 3, 1),   # rows one at a time with 16 warps (third vector 1/4 full)
    (400, 12288, BF, F32, 16, 3, 1),  # rows one at a time with 16 warps
    (10000, 384, F32, F32, 2, 2, 8),
    (700, 384, F32, F32, 4, 1, 4),    # short strip
    (600, 2560, F32, BF, 8, 3, 2),    # fp32 rows of three vectors per lane: pairs kept in registers
    (300, 5120, F32, F32, 16, 3, 1),
    (450, 6144, F32, BF, 16, 3, 1),
    (600, 3584, F32, F32, 8, 4, 2),
]
IDS = [f"T{g[0]}-H{g[1]}-{'bf16' if g[2] == BF else 'fp32'}" for g in GEOMETRIES]


def _code(dt):
    return 1 if dt == BF else 0


@pytest.mark.parametrize("g", GEOMETRIES, ids=IDS)
def test_bwd_geometry(g):
    T, H, xd, wd, nw, nch, cps = g
    p = rmsn.rmsn_plan(rmsn.OP_BWD, T, H, _code(xd), _code(wd),
                       sm_count=torch.cuda.get_device_properties(0).multi_processor_count)
    assert (p["consumer_warps"], p["chunks_per_lane"], p["ctas_per_sm"]) == (nw, nch, cps)
    assert T > rmsn.rmsn_small_t_max()
    c = dataclasses.replace(wl.MAIN_BF16, T=T, H=H, x_dtype=xd, w_dtype=wd)
    x, dy, w = wl.fwd_bwd_inputs(c, DEV, seed=T + H)
    _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
    for comp in (False, True):
        P.assert_ok(P.check_bwd(dy, x, w, rstd, compensated=comp), f"bwd {T}x{H} comp={comp}")
    P.assert_ok(P.check_bwd(dy, x, w, rstd, deterministic=False), f"bwd fast {T}x{H}")


@pytest.mark.parametrize("g", GEOMETRIES, ids=IDS)
def test_bwd_residual_geometry(g):
    T, H, xd, wd, nw, nch, cps = g
    p = rmsn.rmsn_plan(rmsn.OP_BWD_RESIDUAL, T, H, _code(xd), _code(wd),
                       sm_count=torch.cuda.get_device_properties(0).multi_processor_count)
    assert (p["consumer_warps"], p["chunks_per_lane"], p["ctas_per_sm"]) == (nw, nch, cps)
    c = dataclasses.replace(wl.RESIDUAL_MAIN, T=T, H=H, x_dtype=xd, w_dtype=wd)
    x, res, dy, gr, w = wl.residual_inputs(c, DEV, seed=T * 3 + H)
    rf = P.check_fwd_residual(x, res, w, c.eps)
    P.assert_ok(rf, f"fwd_residual {T}x{H}")
    for comp in (False, True):
        rb = P.check_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], gr, compensated=comp)
        P.assert_ok(rb, f"bwd_residual {T}x{H} comp={comp}")
