"""Pins of the FP64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute the same way:
closed forms, invariants of the definition, finite differences, exact rational or
correctly rounded sums, library routines (torch's bf16 and float8_e4m3fn casts), and
the values the pages print.  A dropped term, a wrong sign or index, or a transposed
operand in any oracle function fails at least one of them.
"""
import dataclasses
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rng(seed=0):
    return np.random.default_rng(seed)


def _fused(T, H, seed):
    wl = dataclasses.replace(workloads.FUSED_QUANT, T=T, H=H)
    return workloads.fused_inputs(wl, "cpu", seed=seed)


# ============================================================================ forward
def test_fwd_zero_row_closed_form():
    H, eps = 64, 1e-6
    x = np.zeros((2, H), np.float32)
    x[1] = _rng().standard_normal(H).astype(np.float32)
    w = (1 + 0.1 * _rng(1).standard_normal(H)).astype(np.float32)
    y, rstd = oracle.rmsnorm_fwd(x, w, eps)
    assert rstd[0] == 1.0 / math.sqrt(eps)
    assert np.all(y[0] == 0.0)


def test_fwd_constant_row_closed_form():
    H, eps, c = 96, 1e-6, 0.75
    x = np.full((1, H), c, np.float64)
    w = np.linspace(-2.0, 3.0, H)
    y, rstd = oracle.rmsnorm_fwd(x, w, eps)
    expect = c * w / math.sqrt(c * c + eps)
    np.testing.assert_allclose(y[0], expect, rtol=1e-14, atol=0)
    assert rstd[0] == pytest.approx(1.0 / math.sqrt(c * c + eps), rel=1e-15)


def test_fwd_one_hot_closed_form():
    H, eps, a, k = 256, 1e-6, -3.5, 17
    x = np.zeros((1, H), np.float32)
    x[0, k] = a
    w = np.ones(H, np.float32)
    y, rstd = oracle.rmsnorm_fwd(x, w, eps)
    r = 1.0 / math.sqrt(a * a / H + eps)
    assert rstd[0] == pytest.approx(r, rel=1e-15)
    assert y[0, k] == pytest.approx(a * r, rel=1e-15)
    assert np.count_nonzero(y[0]) == 1


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_fwd_unit_rms_invariant(eps):
    """mean((y/w)^2) = ms/(ms+eps): unit RMS of y/w at eps = 0."""
    T, H = 9, 200
    x = (_rng(2).standard_normal((T, H)) * 1.7).astype(np.float32)
    w = (1 + 0.1 * _rng(3).standard_normal(H)).astype(np.float32)
    y, _ = oracle.rmsnorm_fwd(x, w, eps)
    ms = np.mean(x.astype(np.float64) ** 2, axis=1)
    lhs = np.mean((y / w.astype(np.float64)) ** 2, axis=1)
    np.testing.assert_allclose(lhs, ms / (ms + eps), rtol=1e-13)


def test_fwd_scale_invariance_at_eps0():
    T, H, alpha = 5, 128, 37.25
    x = _rng(4).standard_normal((T, H))
    w = _rng(5).standard_normal(H)
    y1, r1 = oracle.rmsnorm_fwd(x, w, 0.0)
    y2, r2 = oracle.rmsnorm_fwd(alpha * x, w, 0.0)
    np.testing.assert_allclose(y2, y1, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r2 * alpha, r1, rtol=1e-14)


def test_fwd_mean_square_exact_rational():
    """1/rstd^2 - eps equals the exact rational mean of squares of the bf16 inputs."""
    T, H, eps = 4, 24, 1e-6
    xt = (torch.randn(T, H, generator=torch.Generator().manual_seed(7)) * 2).to(torch.bfloat16)
    xb = _bf16_bits(xt)
    w = _bf16_bits(torch.ones(H, dtype=torch.bfloat16))
    _, rstd = oracle.rmsnorm_fwd(xb, w, eps)
    xv = xt.double().numpy()
    for i in range(T):
        ms = sum(Fraction(float(v)) ** 2 for v in xv[i]) / H
        got = 1 / Fraction(float(rstd[i])) ** 2 - Fraction(eps)
        assert abs(float(got - ms)) <= 4e-15 * float(ms)


def test_fwd_row_and_column_indexing():
    """Each row uses its own rstd and column j uses w[j] (T != H, asymmetric values)."""
    T, H = 3, 8
    x = np.arange(1, T * H + 1, dtype=np.float64).reshape(T, H)
    w = np.arange(1, H + 1, dtype=np.float64) * 0.5
    y, rstd = oracle.rmsnorm_fwd(x, w, 0.0)
    for i in range(T):
        r = 1 / math.sqrt(sum(v * v for v in x[i]) / H)
        assert rstd[i] == pytest.approx(r, rel=1e-15)
        for j in range(H):
            assert y[i, j] == pytest.approx(x[i, j] * r * w[j], rel=1e-15)


# =========================================================================== backward
def _loss(x, w, dy, eps):
    y, _ = oracle.rmsnorm_fwd(x, w, eps)
    return float(np.sum(dy * y))


@pytest.mark.parametrize("eps", [1e-6, 0.3])
def test_bwd_dx_finite_differences(eps):
    """dx is the gradient of L = sum(dy * y(x)) (central differences, FP64)."""
    T, H, h = 3, 8, 1e-6
    x = _rng(10).standard_normal((T, H))
    dy = _rng(11).standard_normal((T, H))
    w = 1 + 0.1 * _rng(12).standard_normal(H)
    _, rstd = oracle.rmsnorm_fwd(x, w, eps)
    dx, _ = oracle.rmsnorm_bwd(dy, x, w, rstd)
    fd = np.zeros_like(x)
    for i in range(T):
        for j in range(H):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd[i, j] = (_loss(xp, w, dy, eps) - _loss(xm, w, dy, eps)) / (2 * h)
    np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-8)


def test_bwd_dw_finite_differences():
    T, H, h, eps = 4, 8, 1e-6, 1e-6
    x = _rng(13).standard_normal((T, H))
    dy = _rng(14).standard_normal((T, H))
    w = 1 + 0.1 * _rng(15).standard_normal(H)
    _, rstd = oracle.rmsnorm_fwd(x, w, eps)
    _, dw = oracle.rmsnorm_bwd(dy, x, w, rstd)
    for j in range(H):
        wp, wm = w.copy(), w.copy()
        wp[j] += h
        wm[j] -= h
        fd = (_loss(x, wp, dy, eps) - _loss(x, wm, dy, eps)) / (2 * h)
        assert dw[j] == pytest.approx(fd, rel=1e-7, abs=1e-9)


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_bwd_dx_orthogonality_invariant(eps):
    """sum_j x_ij dx_ij = H*c_i*eps/(ms_i+eps), c_i = mean_j(g*xhat): zero at eps = 0."""
    T, H = 6, 40
    x = _rng(16).standard_normal((T, H))
    dy = _rng(17).standard_normal((T, H))
    w = 1 + 0.1 * _rng(18).standard_normal(H)
    _, rstd = oracle.rmsnorm_fwd(x, w, eps)
    dx, _ = oracle.rmsnorm_bwd(dy, x, w, rstd)
    ms = np.mean(x * x, axis=1)
    c = np.mean(dy * w * x * rstd[:, None], axis=1)
    lhs = np.sum(x * dx, axis=1)
    rhs = H * c * eps / (ms + eps)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12 * H)


def test_bwd_zero_row_closed_form():
    H, eps = 32, 1e-6
    x = np.zeros((1, H))
    dy = _rng(19).standard_normal((1, H))
    w = _rng(20).standard_normal(H)
    _, rstd = oracle.rmsnorm_fwd(x, w, eps)
    dx, dw = oracle.rmsnorm_bwd(dy, x, w, rstd)
    np.testing.assert_allclose(dx[0], dy[0] * w / math.sqrt(eps), rtol=1e-14)
    assert np.all(dw == 0.0)


def test_bwd_scale_at_eps0():
    T, H, a = 3, 16, 8.5
    x = _rng(21).standard_normal((T, H))
    dy = _rng(22).standard_normal((T, H))
    w = _rng(23).standard_normal(H)
    _, r1 = oracle.rmsnorm_fwd(x, w, 0.0)
    _, r2 = oracle.rmsnorm_fwd(a * x, w, 0.0)
    dx1, dw1 = oracle.rmsnorm_bwd(dy, x, w, r1)
    dx2, dw2 = oracle.rmsnorm_bwd(dy, a * x, w, r2)
    np.testing.assert_allclose(dx2 * a, dx1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dw2, dw1, rtol=1e-13, atol=1e-14)


def test_bwd_dw_matches_fsum_bf16():
    """bf16 x, dy with an fp32 rstd: each dy*x*rstd is exact in binary64, so math.fsum
    of the column gives the correctly rounded exact sum."""
    T, H = 3000, 24
    g = torch.Generator().manual_seed(31)
    xt = torch.randn(T, H, generator=g).to(torch.bfloat16)
    dyt = torch.randn(T, H, generator=g).to(torch.bfloat16)
    rstd32 = (0.5 + torch.rand(T, generator=g)).to(torch.float32).numpy()
    w = np.ones(H, np.float32)
    _, dw = oracle.rmsnorm_bwd(_bf16_bits(dyt), _bf16_bits(xt), w, rstd32.astype(np.float64))
    xv, dyv = xt.double().numpy(), dyt.double().numpy()
    r = rstd32.astype(np.float64)
    for j in range(H):
        exact = math.fsum(float(dyv[i, j] * xv[i, j] * r[i]) for i in range(T))
        assert abs(dw[j] - exact) <= 2 * math.ulp(exact)


def test_bwd_bruteforce_rational_fp32():
    """dx and dw against exact rational arithmetic on a tiny fp32 case (given rstd)."""
    T, H = 3, 5
    x = _rng(24).standard_normal((T, H)).astype(np.float32)
    dy = _rng(25).standard_normal((T, H)).astype(np.float32)
    w = (1 + 0.1 * _rng(26).standard_normal(H)).astype(np.float32)
    rstd = np.array([0.75, 1.25, 2.0], np.float64)
    dx, dw = oracle.rmsnorm_bwd(dy, x, w, rstd)
    F = lambda v: Fraction(float(v))  # noqa: E731
    for i in range(T):
        r = F(rstd[i])
        xh = [F(x[i, j]) * r for j in range(H)]
        g = [F(dy[i, j]) * F(w[j]) for j in range(H)]
        c = sum(g[j] * xh[j] for j in range(H)) / H
        for j in range(H):
            ex = r * (g[j] - xh[j] * c)
            assert abs(float(F(dx[i, j]) - ex)) <= 1e-15 * max(1.0, abs(float(ex)))
    for j in range(H):
        ex = sum(F(dy[i, j]) * F(x[i, j]) * F(rstd[i]) for i in range(T))
        assert abs(float(F(dw[j]) - ex)) <= 1e-15 * max(1.0, abs(float(ex)))


def test_bwd_thread_count_independent():
    T, H = 257, 72
    x = _rng(27).standard_normal((T, H)).astype(np.float32)
    dy = _rng(28).standard_normal((T, H)).astype(np.float32)
    w = _rng(29).standard_normal(H).astype(np.float32)
    _, rstd = oracle.rmsnorm_fwd(x, w, 1e-6)
    a = oracle.rmsnorm_bwd(dy, x, w, rstd, nthreads=1)
    b = oracle.rmsnorm_bwd(dy, x, w, rstd, nthreads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ============================================================================ bf16 rounding
def test_bf16_round_matches_torch_cast():
    g = torch.Generator().manual_seed(3)
    v = torch.cat([
        torch.randn(4000, generator=g) * 10.0,
        torch.randn(500, generator=g) * 1e-39,           # bf16 / fp32 subnormals
        torch.randn(500, generator=g) * 3e38,            # near overflow
        torch.tensor([0.0, -0.0, 1.0, -1.0, 3.3895314e38, -3.3895314e38]),
    ]).to(torch.float32)
    ref = _bf16_bits(v.to(torch.bfloat16))
    got = oracle.bf16_round(v.double().numpy())
    assert np.array_equal(got, ref)


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert oracle.bf16_round([1.0 + 2.0 ** -8])[0] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert oracle.bf16_round([1.0 + 3 * 2.0 ** -8])[0] == 0x3F82
    # just above a tie rounds up
    assert oracle.bf16_round([1.0 + 2.0 ** -8 + 2.0 ** -40])[0] == 0x3F81


# ==================================================================================== E4M3
def _torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    ref = _torch_e4m3_decode_all()
    got = oracle.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_e4m3_encode_matches_torch_cast():
    g = torch.Generator().manual_seed(5)
    v = torch.cat([
        (torch.rand(20000, generator=g) * 2 - 1) * 448.0,
        (torch.rand(5000, generator=g) * 2 - 1) * 0.02,    # subnormal and small normals
        (torch.rand(2000, generator=g) * 2 - 1) * 2.0 ** -9,
    ]).to(torch.float32)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v.numpy())
    assert np.array_equal(got, ref)


def test_e4m3_midpoints_tie_to_even():
    vals = oracle.e4m3_decode(np.arange(0x00, 0x7E + 1))  # non-negative finite ladder
    for k in range(len(vals) - 1):
        mid = np.float32((np.float64(vals[k]) + np.float64(vals[k + 1])) / 2)
        code = int(oracle.e4m3_encode([mid])[0])
        even = k if k % 2 == 0 else k + 1
        assert code == even, (k, float(mid), code)


def test_e4m3_saturation_and_nan():
    facts = json.load(open(os.path.join(GOLDEN, "fused_quant_facts.json")))
    top = facts["e4m3_max_finite"]
    assert oracle.e4m3_decode([0x7E])[0] == top
    enc = oracle.e4m3_encode([448.0, 448.5, 470.0, 1e30, np.inf, -np.inf, -500.0, np.nan, -0.0])
    assert list(enc) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x80]


# ============================================================================ fused add+norm
def test_fused_residual_matches_torch_bf16_add():
    T, H = 7, 256
    x, r, w = _fused(T, H, 1)
    h, _, _ = oracle.fused_add_rmsnorm(_bf16_bits(x), _bf16_bits(r), _bf16_bits(w), 1e-6)
    assert np.array_equal(h, _bf16_bits(x + r))


def test_fused_zero_residual_reduces_to_forward():
    T, H = 5, 384
    x, _, w = _fused(T, H, 2)
    zero = torch.zeros(T, H, dtype=torch.bfloat16)
    h, n, rstd = oracle.fused_add_rmsnorm(_bf16_bits(x), _bf16_bits(zero), _bf16_bits(w), 1e-6)
    y, r2 = oracle.rmsnorm_fwd(_bf16_bits(x), _bf16_bits(w), 1e-6)
    assert np.array_equal(h, _bf16_bits(x))
    np.testing.assert_allclose(n, y, rtol=1e-15)
    np.testing.assert_allclose(rstd, r2, rtol=1e-15)


def test_fused_unit_rms_at_eps0():
    T, H = 4, 256
    x, r, w = _fused(T, H, 3)
    h, n, _ = oracle.fused_add_rmsnorm(_bf16_bits(x), _bf16_bits(r), _bf16_bits(w), 0.0)
    wv = w.double().numpy()
    np.testing.assert_allclose(np.mean((n / wv) ** 2, axis=1), 1.0, rtol=1e-13)


# ============================================================================ block quant
def test_quant_scale_layout_and_pads():
    """Scale of (row m, block b) sits at b*ld + m; entries m >= T stay untouched."""
    T, H, ld = 5, 384, workloads.round_up(5, 4) + 4
    n = np.zeros((T, H), np.float64)
    for m in range(T):
        for b in range(H // 128):
            n[m, b * 128 + (m * 7 + b * 13) % 128] = -(m + 1) * 10.0 - b  # block max magnitude
            n[m, b * 128 + (m * 3 + b) % 128 + 0] += 0.5
    bits = oracle.bf16_round(n.reshape(-1)).reshape(T, H)
    sentinel = np.full(((H // 128) * ld,), -7.0, np.float32)
    q, scale = oracle.block_quant_e4m3(bits, ld, scale_init=sentinel)
    dec = oracle.bf16_bits_to_f64(bits)
    for b in range(H // 128):
        for m in range(ld):
            s = scale[b * ld + m]
            if m >= T:
                assert s == -7.0
            else:
                amax = np.float32(np.max(np.abs(dec[m, b * 128:(b + 1) * 128])))
                assert s == np.float32(amax / np.float32(448.0))


def test_quant_block_max_encodes_to_448():
    T, H = 16, 512
    x, r, w = _fused(T, H, 4)
    _, n, _ = oracle.fused_add_rmsnorm(_bf16_bits(x), _bf16_bits(r), _bf16_bits(w), 1e-6)
    bits = oracle.bf16_round(n.reshape(-1)).reshape(T, H)
    q, _ = oracle.block_quant_e4m3(bits, workloads.round_up(T, 4))
    dec = oracle.bf16_bits_to_f64(bits)
    for m in range(T):
        for b in range(H // 128):
            blk = np.abs(dec[m, b * 128:(b + 1) * 128])
            k = int(np.argmax(blk))
            assert q[m, b * 128 + k] & 0x7F == 0x7E


def test_quant_dequant_error_bound():
    T, H = 32, 1024
    x, r, w = _fused(T, H, 5)
    _, n, _ = oracle.fused_add_rmsnorm(_bf16_bits(x), _bf16_bits(r), _bf16_bits(w), 1e-6)
    bits = oracle.bf16_round(n.reshape(-1)).reshape(T, H)
    ld = workloads.round_up(T, 4)
    q, scale = oracle.block_quant_e4m3(bits, ld)
    v = oracle.bf16_bits_to_f64(bits)
    dq = oracle.e4m3_decode(q.reshape(-1)).astype(np.float64).reshape(T, H)
    for b in range(H // 128):
        s = scale[b * ld: b * ld + T].astype(np.float64)[:, None]
        vb = v[:, b * 128:(b + 1) * 128] / s
        err = np.abs(dq[:, b * 128:(b + 1) * 128] - vb)
        normal = np.abs(vb) >= 2.0 ** -6
        assert np.all(err[normal] <= 2.0 ** -4 * np.abs(vb[normal]) * (1 + 1e-6))
        assert np.all(err[~normal] <= 2.0 ** -10 * (1 + 1e-6))


def test_quant_zero_block():
    T, H = 2, 256
    n = np.zeros((T, H))
    n[0, 5] = -0.0
    n[1, 130:140] = 1.5
    bits = oracle.bf16_round(n.reshape(-1)).reshape(T, H)
    bits[0, 5] = 0x8000  # negative zero
    q, scale = oracle.block_quant_e4m3(bits, 4)
    assert scale[0] == 0.0 and scale[1] == 0.0 and scale[4] == 0.0
    assert q[0, 5] == 0x80 and np.count_nonzero(q[0]) == 1
    assert np.all(q[1, :128] == 0)
    assert scale[4 + 1] == np.float32(1.5) / np.float32(448.0)


def test_quant_matches_torch_reference_path():
    """Same decisions as a plain torch fp32 path: amax, amax/448, cast of n/scale."""
    T, H = 64, 1024
    x, r, w = _fused(T, H, 6)
    _, n, _ = oracle.fused_add_rmsnorm(_bf16_bits(x), _bf16_bits(r), _bf16_bits(w), 1e-6)
    bits = oracle.bf16_round(n.reshape(-1)).reshape(T, H)
    ld = workloads.round_up(T, 4)
    q, scale = oracle.block_quant_e4m3(bits, ld)
    nt = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().view(T, H // 128, 128)
    amax = nt.abs().amax(dim=2)
    st = amax / 448.0
    qt = (nt / st[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).view(T, H).numpy()
    assert np.array_equal(q, qt)
    got_scale = scale.reshape(H // 128, ld)[:, :T].T
    assert np.array_equal(got_scale, st.numpy())


# ============================================================================ byte model
def test_fused_byte_model_against_page_example():
    """The page corrected its byte model (weight read once, not M x H) and printed the
    same run's bandwidth under both: 4397 -> 3599 GB/s at M=4096, H=8192."""
    f = json.load(open(os.path.join(GOLDEN, "fused_quant_facts.json")))["byte_model_fix_example"]
    M, H = f["M"], f["H"]
    new = workloads.fused_quant_bytes(M, H)
    old = new - 2 * H + 2 * M * H
    assert abs(f["gbps_weight_as_H"] * old / new - f["gbps_weight_as_MxH"]) < 0.001 * 4397


# ================================================================ residual variants
# FlashInfer PR #5741 "cake_rmsnorm_train", Design (forward with residual: h_new =
# bf16(x + residual) is normalized; backward: dx_total = dx + g_residual) and API.
def _res_loss(x, r, w, dy, g, eps):
    """L = sum(dy * y(x + r)) + sum(g * (x + r)): the loss whose gradient with respect to x
    (and to r) is dx_total (FP64, h unrounded)."""
    y, _, h = oracle.rmsnorm_fwd_residual(x, r, w, eps)
    return float(np.sum(dy * y) + np.sum(g * h))


@pytest.mark.parametrize("eps", [1e-6, 0.3])
def test_residual_dx_total_finite_differences(eps):
    T, H, step = 3, 8, 1e-6
    x = _rng(40).standard_normal((T, H))
    r = _rng(41).standard_normal((T, H))
    dy = _rng(42).standard_normal((T, H))
    g = _rng(43).standard_normal((T, H))
    w = 1 + 0.1 * _rng(44).standard_normal(H)
    _, rstd, h = oracle.rmsnorm_fwd_residual(x, r, w, eps)
    dxt, _ = oracle.rmsnorm_bwd_residual(dy, h, w, rstd, g)
    fdx, fdr = np.zeros_like(x), np.zeros_like(x)
    for i in range(T):
        for j in range(H):
            for arr, fd in ((x, fdx), (r, fdr)):
                ap, am = arr.copy(), arr.copy()
                ap[i, j] += step
                am[i, j] -= step
                args_p = (ap, r) if arr is x else (x, ap)
                args_m = (am, r) if arr is x else (x, am)
                fd[i, j] = (_res_loss(*args_p, w, dy, g, eps) -
                            _res_loss(*args_m, w, dy, g, eps)) / (2 * step)
    np.testing.assert_allclose(dxt, fdx, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dxt, fdr, rtol=1e-6, atol=1e-8)  # both inputs, one gradient


def test_residual_dw_finite_differences():
    T, H, step, eps = 4, 8, 1e-6, 1e-6
    x, r = _rng(45).standard_normal((T, H)), _rng(46).standard_normal((T, H))
    dy, g = _rng(47).standard_normal((T, H)), _rng(48).standard_normal((T, H))
    w = 1 + 0.1 * _rng(49).standard_normal(H)
    _, rstd, h = oracle.rmsnorm_fwd_residual(x, r, w, eps)
    _, dw = oracle.rmsnorm_bwd_residual(dy, h, w, rstd, g)
    for j in range(H):
        wp, wm = w.copy(), w.copy()
        wp[j] += step
        wm[j] -= step
        fd = (_res_loss(x, r, wp, dy, g, eps) - _res_loss(x, r, wm, dy, g, eps)) / (2 * step)
        assert dw[j] == pytest.approx(fd, rel=1e-7, abs=1e-9)


def test_residual_zero_reduces_to_plain_ops():
    x = _bf16_bits(torch.randn(5, 64, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16))
    w = _bf16_bits((1 + 0.1 * torch.randn(64, generator=torch.Generator().manual_seed(4))).to(torch.bfloat16))
    zero = np.zeros_like(x)
    y_r, rstd_r, h = oracle.rmsnorm_fwd_residual(x, zero, w, 1e-6)
    y, rstd = oracle.rmsnorm_fwd(x, w, 1e-6)
    assert np.array_equal(h, x)
    assert np.array_equal(y_r, y) and np.array_equal(rstd_r, rstd)
    dy = _bf16_bits(torch.randn(5, 64, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16))
    dxt, dw_r = oracle.rmsnorm_bwd_residual(dy, h, w, rstd, zero)
    dx, dw = oracle.rmsnorm_bwd(dy, x, w, rstd)
    assert np.array_equal(dxt, dx) and np.array_equal(dw_r, dw)


def test_residual_add_exact_and_rounded():
    # small integers: every sum is exact in bf16 and in binary32
    a = np.arange(-64, 64, dtype=np.float32).reshape(8, 16)
    b = a[::-1].copy()
    assert np.array_equal(oracle.residual_add(a, b), a + b)
    ab, bb = _bf16_bits(torch.from_numpy(a).to(torch.bfloat16)), _bf16_bits(torch.from_numpy(b).to(torch.bfloat16))
    assert np.array_equal(oracle.bf16_bits_to_f64(oracle.residual_add(ab, bb)), (a + b).astype(np.float64))
    # 1 + 2^-8 lies halfway between the bf16 neighbours 1 and 1 + 2^-7: ties to even gives 1;
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6 and ties to 1 + 2^-6
    one = _bf16_bits(torch.tensor([[1.0, 1.0]], dtype=torch.bfloat16))
    d = _bf16_bits(torch.tensor([[2.0 ** -8, 3 * 2.0 ** -8]], dtype=torch.bfloat16))
    got = oracle.bf16_bits_to_f64(oracle.residual_add(one, d))
    assert got.tolist() == [[1.0, 1.0 + 2.0 ** -6]]


def test_residual_g_only_shifts_dx():
    T, H = 3, 16
    x = _rng(50).standard_normal((T, H)).astype(np.float32)
    dy = _rng(51).standard_normal((T, H)).astype(np.float32)
    w = (1 + 0.1 * _rng(52).standard_normal(H)).astype(np.float32)
    _, rstd = oracle.rmsnorm_fwd(x, w, 1e-6)
    g = np.full((T, H), 0.25, np.float32)  # a constant gradient through the residual stream
    dxt, _ = oracle.rmsnorm_bwd_residual(dy, x, w, rstd, g)
    dx, _ = oracle.rmsnorm_bwd(dy, x, w, rstd)
    np.testing.assert_allclose(dxt - dx, 0.25, rtol=0, atol=1e-15)
