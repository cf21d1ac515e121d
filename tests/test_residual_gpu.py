"""GPU parity of the residual training variant (rmsnorm_fwd_residual / rmsnorm_bwd_residual)
against the FP64 oracle, through the C ABI (FlashInfer PR #5741 "cake_rmsnorm_train",
Design and API: h_new = bf16(x + residual) is normalized; the backward returns
dx_total = dx + g_residual)."""
import dataclasses

import numpy as np
import pytest
import torch

import _parity as P
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = [(1, 256), (2, 8), (7, 136), (65, 1536), (129, 2048), (257, 4096), (33, 5120),
          (17, 6144), (5, 14400), (9, 16384), (300, 4104)]
DTYPES = [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
          (torch.float32, torch.float32), (torch.float32, torch.bfloat16)]


def _inputs(T, H, xd, wd, seed):
    c = dataclasses.replace(wl.RESIDUAL_MAIN, T=T, H=H, x_dtype=xd, w_dtype=wd)
    return wl.residual_inputs(c, DEV, seed=seed)


def _ok(H, xd):
    return H % (8 if xd == torch.bfloat16 else 4) == 0


@pytest.mark.parametrize("xd,wd", DTYPES)
@pytest.mark.parametrize("T,H", SHAPES)
def test_fwd_bwd_residual_parity(T, H, xd, wd):
    if not _ok(H, xd):
        pytest.skip("H not a multiple of the vector")
    x, res, dy, g, w = _inputs(T, H, xd, wd, seed=T * 13 + H)
    rf = P.check_fwd_residual(x, res, w, 1e-6)
    P.assert_ok(rf, f"fwd_residual T={T} H={H} {xd}/{wd}")
    # residual backward limit: fp32 x as the backward (H <= 8192)
    if xd == torch.float32 and H > 8192:
        with pytest.raises(rmsn.RmsnError):
            rmsn.rmsnorm_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], g)
        return
    for comp in (False, True):
        rb = P.check_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], g, compensated=comp)
        P.assert_ok(rb, f"bwd_residual T={T} H={H} {xd}/{wd} comp={comp}")


def test_residual_headline_shape():
    c = wl.RESIDUAL_MAIN
    x, res, dy, g, w = wl.residual_inputs(c, DEV, seed=0)
    rf = P.check_fwd_residual(x, res, w, c.eps)
    P.assert_ok(rf, c.name)
    P.assert_ok(P.check_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], g), c.name)


def test_fwd_residual_in_place():
    x, res, _, _, w = _inputs(129, 2048, torch.bfloat16, torch.bfloat16, seed=7)
    P.assert_ok(P.check_fwd_residual(x, res, w, 1e-6, inplace=True), "h_new over residual")


@pytest.mark.parametrize("alias", ["g", "dy"])
def test_bwd_residual_aliased_output(alias):
    x, res, dy, g, w = _inputs(257, 4096, torch.bfloat16, torch.bfloat16, seed=8)
    rf = P.check_fwd_residual(x, res, w, 1e-6)
    P.assert_ok(P.check_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], g, alias=alias),
                f"dx_total over {alias}")


def test_bwd_residual_nondeterministic_mode():
    x, res, dy, g, w = _inputs(129, 2048, torch.bfloat16, torch.float32, seed=9)
    rf = P.check_fwd_residual(x, res, w, 1e-6)
    P.assert_ok(P.check_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], g, deterministic=False),
                "atomic dw")


def test_bwd_residual_dw_bitwise_repeatable_and_equal_to_plain_dw():
    x, res, dy, g, w = _inputs(4096, 2048, torch.bfloat16, torch.float32, seed=10)
    _, rstd, h = rmsn.rmsnorm_fwd_residual(x, res, w, 1e-6)
    runs = []
    for _ in range(3):
        ws = torch.full((rmsn.rmsnorm_bwd_workspace_bytes(4096, 2048) // 4,), float("nan"), device=DEV)
        _, dw = rmsn.rmsnorm_bwd_residual(dy, h, w, rstd, g, workspace=ws)
        runs.append(dw.cpu().numpy().view(np.uint32).copy())
    assert all(np.array_equal(runs[0], r) for r in runs[1:])
    # g_residual enters dx only: dw has the bits of the plain backward at the same chunking
    # when both use the same CTAs per SM
    p1 = rmsn.rmsn_plan(rmsn.OP_BWD, 4096, 2048, 1, 0)
    p2 = rmsn.rmsn_plan(rmsn.OP_BWD_RESIDUAL, 4096, 2048, 1, 0)
    if p1["grid"] == p2["grid"]:
        _, dw_plain = rmsn.rmsnorm_bwd(dy, h, w, rstd)
        assert np.array_equal(dw_plain.cpu().numpy().view(np.uint32), runs[0])
    assert rmsn.rmsn_device_status() == 0


def test_residual_t0_and_errors():
    e = torch.empty(0, 512, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(512, device=DEV, dtype=torch.bfloat16)
    y, rstd, h = rmsn.rmsnorm_fwd_residual(e, e.clone(), w)
    assert y.shape == (0, 512) and h.shape == (0, 512)
    dw = torch.full((512,), float("nan"), device=DEV)
    rmsn.rmsnorm_bwd_residual(e, e, w, torch.empty(0, device=DEV), e, dw=dw)
    torch.cuda.synchronize()
    assert torch.all(dw == 0)  # the gradient of an empty batch
    x = torch.randn(4, 100, device=DEV).to(torch.bfloat16)  # H not a multiple of 8
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsnorm_fwd_residual(x, x.clone(), torch.ones(100, device=DEV, dtype=torch.bfloat16))
    assert rmsn.rmsn_device_status() == 0
