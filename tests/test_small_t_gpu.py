"""The small-T route of the deterministic backward (one launch: row tasks for dx, column
tasks for dw summed over the rows in a fixed order; miles-ext-kernels PR #15, Changes,
#8813) against the FP64 oracle, next to the strip route it replaces below the threshold."""
import dataclasses

import numpy as np
import pytest
import torch

import _parity as P
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture
def t_max():
    old = rmsn.rmsn_small_t_max()
    yield
    rmsn.rmsn_set_small_t_max(old)


def _inputs(T, H, xd, wd, seed):
    c = dataclasses.replace(wl.MAIN_BF16, T=T, H=H, x_dtype=xd, w_dtype=wd)
    x, dy, w = wl.fwd_bwd_inputs(c, DEV, seed=seed)
    _, rstd = rmsn.rmsnorm_fwd(x, w, 1e-6)
    return x, dy, w, rstd


@pytest.mark.parametrize("route", ["small", "strip"])
@pytest.mark.parametrize("comp", [False, True])
@pytest.mark.parametrize("xd,wd", [(torch.bfloat16, torch.float32), (torch.bfloat16, torch.bfloat16),
                                   (torch.float32, torch.float32)])
@pytest.mark.parametrize("T,H", [(1, 256), (3, 2048), (8, 8), (65, 1536), (65, 6144), (100, 4104),
                                 (128, 2048), (129, 5120), (256, 2048), (257, 1536)])
def test_small_t_parity(t_max, route, comp, xd, wd, T, H):
    if H % (8 if xd == torch.bfloat16 else 4):
        pytest.skip("H not a multiple of the vector")
    rmsn.rmsn_set_small_t_max(1024 if route == "small" else 0)
    x, dy, w, rstd = _inputs(T, H, xd, wd, seed=T + 7 * H)
    r = P.check_bwd(dy, x, w, rstd, deterministic=True, compensated=comp)
    P.assert_ok(r, f"{route} T={T} H={H} {xd}/{wd} comp={comp}")


def test_small_t_leaves_workspace_untouched_and_is_repeatable(t_max):
    assert rmsn.rmsn_small_t_max() == 256  # the default
    x, dy, w, rstd = _inputs(65, 2048, torch.bfloat16, torch.float32, seed=3)
    n = rmsn.rmsnorm_bwd_workspace_bytes(65, 2048)
    bits = []
    for _ in range(3):
        ws = torch.full((n // 4,), float("nan"), device=DEV)
        _, dw = rmsn.rmsnorm_bwd(dy, x, w, rstd, workspace=ws)
        torch.cuda.synchronize()
        assert torch.isnan(ws).all()
        bits.append(dw.cpu().numpy().view(np.uint32).copy())
    assert all(np.array_equal(bits[0], b) for b in bits[1:])
    assert rmsn.rmsn_device_status() == 0


def test_small_t_residual_variant(t_max):
    rmsn.rmsn_set_small_t_max(128)
    c = dataclasses.replace(wl.RESIDUAL_MAIN, T=65, H=2048)
    x, res, dy, g, w = wl.residual_inputs(c, DEV, seed=4)
    rf = P.check_fwd_residual(x, res, w, 1e-6)
    for comp in (False, True):
        P.assert_ok(P.check_bwd_residual(dy, rf["_h"], w, rf["_rstd_dev"], g, compensated=comp),
                    f"small-T residual comp={comp}")


def test_set_small_t_max_rejects_out_of_range(t_max):
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_small_t_max(-1)
