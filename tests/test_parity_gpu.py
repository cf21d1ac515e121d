"""GPU parity of the three operations against the FP64 oracle (through the C ABI).

Gates (the tolerances of the method's statement): fp32 outputs within relative 1e-5,
bf16 outputs within one bf16 ulp, dW within atol 1e-4 + rtol 1e-4 of the FP64 sum,
deterministic dW bit-identical run to run, fp8 bytes and scales bit-exact when the
oracle quantizes the device's own normed output.
"""
import dataclasses

import numpy as np
import pytest
import torch

import _parity as P
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"

# shapes that span several row groups / chunks, ragged T, and H not a multiple of a full
# warp's vector span (masked lanes)
SHAPES = [(1, 256), (2, 8), (7, 136), (63, 1024), (65, 1536), (129, 2048), (257, 4096),
          (33, 5120), (17, 6144), (9, 16384), (300, 4104)]


def _wl(base, T, H, x_dtype=None, w_dtype=None, **kw):
    return dataclasses.replace(base, T=T, H=H, x_dtype=x_dtype or base.x_dtype,
                               w_dtype=w_dtype or base.w_dtype, **kw)


DTYPES = [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
          (torch.float32, torch.float32), (torch.float32, torch.bfloat16)]


def _ok_shape(H, x_dtype):
    return H % (8 if x_dtype == torch.bfloat16 else 4) == 0


# ------------------------------------------------------------------------- forward
@pytest.mark.parametrize("xd,wd", DTYPES)
@pytest.mark.parametrize("T,H", SHAPES)
def test_fwd_parity_shapes(T, H, xd, wd):
    if not _ok_shape(H, xd):
        pytest.skip("H not a multiple of the vector")
    x, _, w = wl.fwd_bwd_inputs(_wl(wl.MAIN_BF16, T, H, xd, wd), DEV, seed=T * 31 + H)
    P.assert_ok(P.check_fwd(x, w, 1e-6), f"fwd T={T} H={H} {xd}/{wd}")


def test_fwd_small_fp32_config():
    c = wl.SMALL_FP32
    x, _, w = wl.fwd_bwd_inputs(c, DEV, seed=0)
    P.assert_ok(P.check_fwd(x, w, c.eps), c.name)


def test_fwd_main_bf16_config():
    c = wl.MAIN_BF16
    x, _, w = wl.fwd_bwd_inputs(c, DEV, seed=0)
    P.assert_ok(P.check_fwd(x, w, c.eps), c.name)


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_fwd_special_rows(scale):
    T, H = 70, 2048
    x, _, w = wl.fwd_bwd_inputs(_wl(wl.MAIN_BF16, T, H), DEV, seed=5)
    x = (x.float() * scale).to(torch.bfloat16)
    x[3] = 0                       # all-zero row: rstd = 1/sqrt(eps), y = 0
    x[4] = 1.5                     # constant row
    x[5] = 0
    x[5, 77] = -3.0                # one-hot row
    x[6] = (x[6].float() * 1e4).to(torch.bfloat16)  # a single extreme row
    r = P.check_fwd(x, w, 1e-6)
    P.assert_ok(r, f"special rows scale={scale}")
    rs = r["_rstd_dev"].cpu()
    assert rs[3].item() == pytest.approx(1000.0, rel=1e-6)


def test_fwd_t0_is_noop():
    x = torch.empty(0, 512, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(512, device=DEV, dtype=torch.bfloat16)
    y, r = rmsn.rmsnorm_fwd(x, w)
    assert y.shape == (0, 512) and r.shape == (0,)


# ------------------------------------------------------------------------ backward
@pytest.mark.parametrize("mode", ["det", "det_comp", "fast", "fast_comp"])
@pytest.mark.parametrize("xd,wd", DTYPES)
@pytest.mark.parametrize("T,H", SHAPES)
def test_bwd_parity_shapes(T, H, xd, wd, mode):
    if not _ok_shape(H, xd):
        pytest.skip("H not a multiple of the vector")
    x, dy, w = wl.fwd_bwd_inputs(_wl(wl.MAIN_BF16, T, H, xd, wd), DEV, seed=T * 7 + H)
    _, rstd = rmsn.rmsnorm_fwd(x, w, 1e-6)
    if xd == torch.float32 and H > 8192:  # the fp32 backward supports H <= 8192
        with pytest.raises(rmsn.RmsnError):
            rmsn.rmsnorm_bwd(dy, x, w, rstd)
        return
    r = P.check_bwd(dy, x, w, rstd, deterministic=mode.startswith("det"),
                    compensated=mode.endswith("comp"))
    P.assert_ok(r, f"bwd T={T} H={H} {xd}/{wd} {mode}")


def test_bwd_small_fp32_config():
    c = wl.SMALL_FP32
    x, dy, w = wl.fwd_bwd_inputs(c, DEV, seed=0)
    _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
    P.assert_ok(P.check_bwd(dy, x, w, rstd), c.name)


@pytest.mark.parametrize("compensated", [False, True])
def test_bwd_main_bf16_config(compensated):
    c = wl.MAIN_BF16
    x, dy, w = wl.fwd_bwd_inputs(c, DEV, seed=0)
    _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
    P.assert_ok(P.check_bwd(dy, x, w, rstd, compensated=compensated), c.name)


def test_bwd_special_rows():
    T, H = 130, 4096
    x, dy, w = wl.fwd_bwd_inputs(_wl(wl.MAIN_BF16, T, H), DEV, seed=9)
    x[0] = 0                       # zero row: dx = dy*w/sqrt(eps)
    x[1] = 2.0                     # constant row
    dy[2] = 0                      # zero gradient row
    x[3] = (x[3].float() * 1e3).to(torch.bfloat16)
    _, rstd = rmsn.rmsnorm_fwd(x, w, 1e-6)
    P.assert_ok(P.check_bwd(dy, x, w, rstd), "special rows")


@pytest.mark.parametrize("T,H,xd,wd", [(300, 4096, torch.bfloat16, torch.bfloat16),
                                       (700, 1536, torch.bfloat16, torch.float32),
                                       (65, 2048, torch.bfloat16, torch.float32),
                                       (257, 2048, torch.float32, torch.float32)])
def test_forward_then_backward_at_the_oracles_rstd(T, H, xd, wd):
    # end to end: the device's forward and then its backward (at the rstd the forward saved),
    # against the oracle's own chain (its FP64 rstd, then the backward at that rstd).  Beyond
    # the usual gates, dx may move by |d(dx)/d(rstd)| * |rstd_dev - rstd_ref| with
    # d(dx)/d(rstd) = g - 3 rstd^2 x mean(g x), bounded per element
    from oracle import gates
    import oracle
    x, dy, w = wl.fwd_bwd_inputs(_wl(wl.MAIN_BF16, T, H, xd, wd), DEV, seed=T + H)
    _, rstd = rmsn.rmsnorm_fwd(x, w, 1e-6)
    dx, dw = rmsn.rmsnorm_bwd(dy, x, w, rstd)
    torch.cuda.synchronize()
    X, DY, W = wl.to_oracle(x), wl.to_oracle(dy), wl.to_oracle(w)
    _, r_ref = oracle.rmsnorm_fwd(X, W, 1e-6)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(DY, X, W, r_ref)
    r_dev = rstd.cpu().numpy().astype(np.float64)
    assert gates.check_f32_rel(r_dev, r_ref)["n_fail"] == 0
    dec = oracle.bf16_bits_to_f64 if xd == torch.bfloat16 else (lambda a: np.asarray(a, np.float64))
    decw = oracle.bf16_bits_to_f64 if wd == torch.bfloat16 else (lambda a: np.asarray(a, np.float64))
    xf, dyf, wf = dec(X), dec(DY), decw(W)
    g = dyf * wf[None, :]
    S = np.mean(g * xf, axis=1, keepdims=True)
    dr = np.abs(r_dev - r_ref)[:, None]
    r = np.maximum(r_dev, r_ref)[:, None]
    moved = 1.01 * dr * (np.abs(g) + 3.0 * r * r * np.abs(xf) * np.abs(S))
    if xd == torch.bfloat16:
        depth = P.row_dot_depth(T, H, xd, wd, True)
        extra = gates.dx_fp32_bound(dyf, xf, wf, r_dev, dx_ref, depth) + moved
        res = gates.check_bf16(wl.to_oracle(dx), dx_ref, extra=extra)
    else:
        res = gates.check_f32_rel(wl.to_oracle(dx), dx_ref, row_rms_term=True)
    assert res["n_fail"] == 0, res
    assert gates.check_dw(dw.cpu().numpy(), dw_ref)["n_fail"] == 0


@pytest.mark.parametrize("T", [5, 300])  # the small-T route and the strip kernel
def test_row_beyond_fp32_range(T):
    # a row whose FP32 sum of squares overflows: rstd = 1/sqrt(inf) = 0 and y = 0 (the
    # pages' FP32 sum of squares; the FP64 oracle does not overflow there, so the forward of
    # the other rows is compared with it separately); the backward at the saved rstd gives
    # dx = 0 for that row and adds nothing to dW, which the oracle at the same rstd confirms
    H = 1024
    x, dy, w = wl.fwd_bwd_inputs(_wl(wl.MAIN_BF16, T, H), DEV, seed=12)
    x[2] = 1e20
    y, rstd = rmsn.rmsnorm_fwd(x, w, 1e-6)
    dx, dw = rmsn.rmsnorm_bwd(dy, x, w, rstd)
    torch.cuda.synchronize()
    assert rstd[2].item() == 0.0
    assert bool((y[2] == 0).all()) and bool((dx[2] == 0).all())
    keep = torch.tensor([i for i in range(T) if i != 2], device=DEV)
    P.assert_ok(P.check_fwd(x[keep].contiguous(), w, 1e-6), "forward of the other rows")
    P.assert_ok(P.gate_bwd(dy, x, w, rstd, dx, dw, deterministic=True, all_rows=True),
                "backward at the saved rstd")
    assert rmsn.rmsn_device_status() == 0


def test_bwd_t0_zeroes_dw():
    x = torch.empty(0, 256, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(256, device=DEV, dtype=torch.bfloat16)
    rstd = torch.empty(0, device=DEV)
    dw = torch.full((256,), float("nan"), device=DEV)
    rmsn.rmsnorm_bwd(x, x, w, rstd, dw=dw)
    torch.cuda.synchronize()
    assert bool((dw == 0).all())


# ---------------------------------------------------------- fused add + norm + quant
# (the last five: one CTA of 16 warps per SM, two stages up to H 12288, one above)
FUSED_SHAPES = [(1, 128), (2, 256), (7, 384), (63, 1024), (65, 2048), (129, 4096),
                (257, 5120), (31, 6144), (2047, 4096), (301, 8320), (333, 10240),
                (1000, 12288), (77, 14336), (5, 16384)]


@pytest.mark.parametrize("T,H", FUSED_SHAPES)
def test_fused_parity_shapes(T, H):
    x, res, w = wl.fused_inputs(_wl(wl.FUSED_QUANT, T, H), DEV, seed=T + H)
    P.assert_ok(P.check_fused(x, res, w, 1e-6, ld_pad=4), f"fused T={T} H={H}")


def test_fused_config():
    c = wl.FUSED_QUANT
    x, res, w = wl.fused_inputs(c, DEV, seed=0)
    P.assert_ok(P.check_fused(x, res, w, c.eps), c.name)


def test_fused_bench_shape():
    """The fused op at the shape the benchmark's step times (T = 8192, H = 4096)."""
    c = wl.FUSED_QUANT_MAIN
    x, res, w = wl.fused_inputs(c, DEV, seed=4)
    P.assert_ok(P.check_fused(x, res, w, c.eps), c.name)


def test_fused_zero_and_special_blocks():
    T, H = 12, 1024
    x, res, w = wl.fused_inputs(_wl(wl.FUSED_QUANT, T, H), DEV, seed=3)
    x[0] = 0
    res[0] = 0                     # whole zero row: rstd = 1/sqrt(eps), all blocks amax 0
    x[1, :128] = 0
    res[1, :128] = 0               # one zero block inside a normal row
    x[2] = 5.0
    res[2] = -1.0                  # constant row
    x[3] = (x[3].float() * 1e-3).to(torch.bfloat16)
    res[3] = 0                     # tiny row: E4M3 codes in the subnormal range
    P.assert_ok(P.check_fused(x, res, w, 1e-6), "special blocks")


def test_fused_t0_is_noop():
    x = torch.empty(0, 256, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(256, device=DEV, dtype=torch.bfloat16)
    q, s, n = rmsn.fused_add_rmsnorm_fp8_block_quant(x, x.clone(), w)
    assert q.shape == (0, 256)


# ------------------------------------------------------------------- error paths
def test_errors_on_device():
    x = torch.randn(16, 256, device=DEV).to(torch.bfloat16)
    w = torch.ones(256, device=DEV, dtype=torch.bfloat16)
    L = rmsn.load_library()
    y = torch.empty_like(x)
    r = torch.empty(16, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    # misaligned x (2 bytes off a 16-byte boundary)
    st = L.rmsnorm_fwd(x.data_ptr() + 2, 1, w.data_ptr(), 1, y.data_ptr(), r.data_ptr(), 15, 256,
                       1e-6, s)
    assert st == 3
    # workspace too small
    dw = torch.empty(256, device=DEV)
    ws = torch.empty(16, device=DEV, dtype=torch.uint8)
    st = L.rmsnorm_bwd(x.data_ptr(), x.data_ptr(), 1, w.data_ptr(), 1, r.data_ptr(), y.data_ptr(),
                       dw.data_ptr(), 16, 256, 1, 0, ws.data_ptr(), 16, s)
    assert st == 4
    with pytest.raises(rmsn.RmsnError):
        rmsn.fused_add_rmsnorm_fp8_block_quant(x[:, :200].contiguous(), x[:, :200].contiguous(),
                                               w[:200].contiguous())


def test_kernel_reuse_across_shared_memory_sizes():
    """The same kernel variant (bf16 x, fp32 w, 3 vectors per lane) runs at H = 5120 and
    H = 6144 with different shared-memory sizes; using the larger size again after the
    smaller one must still launch (the per-kernel limit is never lowered)."""
    for H in (5120, 6144, 5120):
        x, dy, w = wl.fwd_bwd_inputs(_wl(wl.MAIN_BF16, 40, H, torch.bfloat16, torch.float32), DEV,
                                     seed=H)
        r = P.check_fwd(x, w, 1e-6)
        P.assert_ok(r, f"fwd H={H}")
        P.assert_ok(P.check_bwd(dy, x, w, r["_rstd_dev"]), f"bwd H={H}")
