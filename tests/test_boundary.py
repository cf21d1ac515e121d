"""The C ABI without a GPU: the library loads and exports every function include/rmsn.h
declares; argument checks return their status before anything touches CUDA; the
launch planner (a pure host function) covers each row exactly and sizes the backward
workspace as documented."""
import ctypes
import os
import re

import pytest

import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
from rmsnorm_fwd_bwd_persistent_gb300 import build as rbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rmsn.h")

OK, INVALID, SHAPE, MISALIGNED, WS_SMALL, CUDA = 0, 1, 2, 3, 4, 5
A = 1 << 20  # a fake, 16-byte aligned "device" address: never dereferenced by these calls


@pytest.fixture(scope="module")
def lib():
    rbuild.build()
    return rmsn.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_function(lib):
    names = _declared_functions()
    assert {"rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes",
            "fused_add_rmsnorm_fp8_block_quant", "rmsn_status_string", "rmsn_plan",
            "rmsn_set_policy", "rmsn_device_status"} <= set(names)
    raw = ctypes.CDLL(rmsn.library_path())
    for n in names:
        assert hasattr(raw, n), f"{n} declared in rmsn.h but not exported"


def test_status_strings(lib):
    for s in range(0, 8):
        assert rmsn.rmsn_status_string(s) and rmsn.rmsn_status_string(s) != "unknown status"
    assert rmsn.rmsn_status_string(99) == "unknown status"


def test_fwd_argument_checks(lib):
    f = lib.rmsnorm_fwd
    assert f(A, 1, A, 1, A, A, 4, 7, 1e-6, None) == SHAPE          # H not a multiple of 8
    assert f(A, 0, A, 0, A, A, 4, 6, 1e-6, None) == SHAPE          # fp32: H % 4
    assert f(A, 1, A, 1, A, A, 4, 16392, 1e-6, None) == SHAPE      # above the maximum
    assert f(A, 1, A, 1, A, A, 4, 0, 1e-6, None) == SHAPE
    assert f(A, 2, A, 1, A, A, 4, 64, 1e-6, None) == INVALID       # dtype code
    assert f(A, 1, A, 1, A, A, -1, 64, 1e-6, None) == INVALID      # T < 0
    assert f(A, 1, A, 1, A, A, 4, 64, float("nan"), None) == INVALID
    assert f(A, 1, A, 1, A, A, 4, 64, -1.0, None) == INVALID
    assert f(A, 1, A, 1, A, A, 4, 64, float("inf"), None) == INVALID
    assert f(None, 1, A, 1, A, A, 4, 64, 1e-6, None) == INVALID
    assert f(A + 8, 1, A, 1, A, A, 4, 64, 1e-6, None) == MISALIGNED
    assert f(A, 1, A, 1, A + 4, A, 4, 64, 1e-6, None) == MISALIGNED
    assert f(A, 1, A, 1, A, A + 2, 4, 64, 1e-6, None) == MISALIGNED
    assert f(None, 1, None, 1, None, None, 0, 64, 1e-6, None) == OK   # T == 0: nothing to do


def test_bwd_argument_checks(lib):
    b = lib.rmsnorm_bwd
    assert b(A, A, 1, A, 0, A, A, A, 4, 12, 1, 0, A, 1 << 20, None) == SHAPE
    assert b(A, A, 1, A, 0, A, A, None, 4, 64, 1, 0, A, 1 << 20, None) == INVALID
    assert b(A, A, 1, A, 0, A, A, A + 4, 4, 64, 1, 0, A, 1 << 20, None) == MISALIGNED
    assert b(A, A, 3, A, 0, A, A, A, 4, 64, 1, 0, A, 1 << 20, None) == INVALID
    assert b(None, A, 1, A, 0, A, A, A, 4, 64, 1, 0, A, 1 << 20, None) == INVALID
    assert b(A, A + 2, 1, A, 0, A, A, A, 4, 64, 1, 0, A, 1 << 20, None) == MISALIGNED
    # both modes need the workspace (the atomic mode keeps its column sums there)
    assert b(A, A, 1, A, 0, A, A, A, 4, 64, 1, 0, None, 0, None) == WS_SMALL
    assert b(A, A, 1, A, 0, A, A, A, 4, 64, 0, 0, None, 0, None) == WS_SMALL
    assert b(A, A, 1, A, 0, A, A, A, 4, 64, 0, 0, A + 8, 1 << 20, None) == MISALIGNED


def test_fused_argument_checks(lib):
    f = lib.fused_add_rmsnorm_fp8_block_quant
    assert f(A, A, A, A, A, 8, A, 8, 200, 1e-6, None) == SHAPE     # H % 128
    assert f(A, A, A, A, A, 8, A, 8, 32768, 1e-6, None) == SHAPE   # above the maximum
    assert f(A, A, A, A, A, 4, A, 7, 256, 1e-6, None) == INVALID   # ld < round_up(T, 4) = 8
    assert f(A, A, A, A, A + 2, 8, A, 7, 256, 1e-6, None) == MISALIGNED
    assert f(A, A, A, A + 8, A, 8, A, 7, 256, 1e-6, None) == MISALIGNED
    assert f(A, None, A, A, A, 8, A, 7, 256, 1e-6, None) == INVALID
    assert f(None, None, None, None, None, 0, None, 0, 256, 1e-6, None) == OK


def test_residual_argument_checks(lib):
    f = lib.rmsnorm_fwd_residual
    assert f(A, A, 1, A, 1, A, A, A, 4, 7, 1e-6, None) == SHAPE        # H not a multiple of 8
    assert f(A, A, 3, A, 1, A, A, A, 4, 64, 1e-6, None) == INVALID     # dtype code
    assert f(A, None, 1, A, 1, A, A, A, 4, 64, 1e-6, None) == INVALID  # no residual
    assert f(A, A, 1, A, 1, A, None, A, 4, 64, 1e-6, None) == INVALID  # no h_new
    assert f(A, A + 8, 1, A, 1, A, A, A, 4, 64, 1e-6, None) == MISALIGNED
    assert f(A, A, 1, A, 1, A, A + 4, A, 4, 64, 1e-6, None) == MISALIGNED
    assert f(A, A, 1, A, 1, A, A, A, 4, 64, -1.0, None) == INVALID
    assert f(None, None, 1, None, 1, None, None, None, 0, 64, 1e-6, None) == OK
    b = lib.rmsnorm_bwd_residual
    assert b(A, A, 1, A, 0, A, A, A, A, 4, 12, 1, 0, A, 1 << 20, None) == SHAPE
    assert b(A, A, 1, A, 0, A, None, A, A, 4, 64, 1, 0, A, 1 << 20, None) == INVALID  # no g
    assert b(A, A, 1, A, 0, A, A, None, A, 4, 64, 1, 0, A, 1 << 20, None) == INVALID  # no dx
    assert b(A, A, 1, A, 0, A, A + 8, A, A, 4, 64, 1, 0, A, 1 << 20, None) == MISALIGNED
    assert b(A, A, 1, A, 0, A, A, A, A + 4, 4, 64, 1, 0, A, 1 << 20, None) == MISALIGNED
    assert b(A, A, 1, A, 0, A, A, A, A, 4, 64, 1, 0, None, 0, None) == WS_SMALL
    assert b(A, A, 1, A, 0, A, A, A, A, 4, 64, 0, 0, None, 0, None) == WS_SMALL  # atomic mode too


SM = 152


@pytest.mark.parametrize("op", [rmsn.OP_FWD, rmsn.OP_BWD, rmsn.OP_FUSED_QUANT,
                                rmsn.OP_FWD_RESIDUAL, rmsn.OP_BWD_RESIDUAL])
@pytest.mark.parametrize("H", [8, 128, 256, 1536, 2048, 4096, 4104, 5120, 6144, 8192, 16384])
@pytest.mark.parametrize("xd,wd", [(1, 1), (1, 0), (0, 0), (0, 1)])
def test_plan_covers_rows(lib, op, H, xd, wd):
    if op == rmsn.OP_FUSED_QUANT and (xd, wd) != (1, 1):
        with pytest.raises(rmsn.RmsnError):
            rmsn.rmsn_plan(op, 100, 4096, xd, wd)
        return
    vec = 8 if xd == 1 else 4
    if H % vec or (op == rmsn.OP_FUSED_QUANT and H % 128):
        with pytest.raises(rmsn.RmsnError):
            rmsn.rmsn_plan(op, 100, H, xd, wd)
        return
    is_bwd = op in (rmsn.OP_BWD, rmsn.OP_BWD_RESIDUAL)
    if is_bwd and xd == 0 and H > 8192:
        with pytest.raises(rmsn.RmsnError):
            rmsn.rmsn_plan(op, 100, H, xd, wd)
        return
    for T in (1, 65, 8192, 262144):
        p = rmsn.rmsn_plan(op, T, H, xd, wd, sm_count=SM)
        lanes = 32 * p["consumer_warps"]
        assert p["vec_elems"] == vec
        assert p["chunks_per_lane"] * lanes * vec >= H              # the row is covered
        producer = 0 if is_bwd else 32                              # bwd: thread 0 feeds the ring
        max_threads = 512 if is_bwd else (544 if op == rmsn.OP_FUSED_QUANT else 288)
        assert p["threads"] == lanes + producer and p["threads"] <= max_threads
        assert 1 <= p["grid"] <= min(T, SM * p["ctas_per_sm"])      # every CTA has a row
        row = H * (2 if xd == 1 else 4)
        rows = 1 if op == rmsn.OP_FWD else 2                        # rows per stage
        stage = -(-row // 128) * 128 * rows
        wpad = -(-(H * 4) // 128) * 128                           # w staged as FP32 in smem
        assert p["stages"] >= 1 and p["smem_bytes"] == 2048 + wpad + p["stages"] * stage
        assert p["ctas_per_sm"] * (p["smem_bytes"] + 1024) <= 233472  # fits the SM
        if is_bwd or (p["ctas_per_sm"] > 1 and op == rmsn.OP_FWD_RESIDUAL):
            assert p["stages"] >= 2                                 # bwd holds two rows
        if op == rmsn.OP_FWD:                                       # one stage above 4 KiB rows
            assert p["stages"] == (2 if row <= 4096 else 1)
        if op == rmsn.OP_FUSED_QUANT:
            assert p["stages"] == 1                                 # one stage, 3 CTAs per SM
        if op == rmsn.OP_FUSED_QUANT:
            assert lanes % 16 == 0                                  # 16 lanes hold one block


def test_plan_headline_geometry(lib):
    f = rmsn.rmsn_plan(rmsn.OP_FWD, 8192, 4096, 1, 1)
    assert (f["consumer_warps"], f["chunks_per_lane"], f["ctas_per_sm"], f["stages"]) == (4, 4, 6, 1)
    b = rmsn.rmsn_plan(rmsn.OP_BWD, 8192, 4096, 1, 1)
    assert (b["consumer_warps"], b["chunks_per_lane"], b["ctas_per_sm"]) == (8, 2, 2)
    assert b["grid"] == 2 * SM
    assert b["workspace_bytes"] == 2 * b["grid"] * 4096 * 4       # (high, low) rows per chunk
    q = rmsn.rmsn_plan(rmsn.OP_FUSED_QUANT, 8192, 4096, 1, 1)
    assert (q["consumer_warps"], q["chunks_per_lane"], q["ctas_per_sm"], q["stages"]) == (8, 2, 3, 1)


@pytest.mark.parametrize("H,xd,geom", [
    (1024, 1, (2, 2, 8)), (1536, 1, (3, 2, 5)), (2048, 1, (4, 2, 4)), (2560, 1, (5, 2, 3)),
    (3072, 1, (8, 2, 2)), (3584, 1, (7, 2, 2)), (4096, 1, (8, 2, 2)), (5120, 1, (8, 3, 2)),
    (6144, 1, (8, 3, 2)), (8192, 1, (16, 2, 1)), (16384, 1, (16, 4, 1)),
    (1280, 0, (5, 2, 3)), (2048, 0, (8, 2, 2)), (4096, 0, (16, 2, 1)), (8192, 0, (16, 4, 1))])
def test_plan_backward_geometry_by_row_length(lib, H, xd, geom):
    # 14-16 consumer warps per SM: 8 CTAs of 2 warps, 4 of 4, 2 of 8, one of 16 for rows of
    # at least 1024 16-byte vectors, or a count that is not a power of two (5 CTAs of 3,
    # 3 of 5, 2 of 7) for rows those fill at two vectors per lane; the residual backward
    # plans the same way
    for op in (rmsn.OP_BWD, rmsn.OP_BWD_RESIDUAL):
        p = rmsn.rmsn_plan(op, 65536, H, xd, 0)
        assert (p["consumer_warps"], p["chunks_per_lane"], p["ctas_per_sm"]) == geom
        assert 14 <= p["consumer_warps"] * p["ctas_per_sm"] <= 16
        assert p["grid"] == SM * p["ctas_per_sm"]
        assert p["workspace_bytes"] == 8 * H * p["grid"]


def test_plan_backward_warps_not_a_power_of_two(lib):
    # every width that takes a warp count other than a power of two: the row fills those
    # warps at two vectors per lane to at least 7/8, the power of two would have been
    # larger, and the SM holds at least 14 of the warps
    seen = set()
    for xd, vec in ((1, 8), (0, 4)):
        for H in range(vec, (16384 if xd else 8192) + 1, vec):  # fp32 rows up to 8192
            p = rmsn.rmsn_plan(rmsn.OP_BWD, 65536, H, xd, 0)
            nw, nvec = p["consumer_warps"], H // vec
            assert p["chunks_per_lane"] * 32 * nw >= nvec
            if nw & (nw - 1) == 0:
                continue
            seen.add(nw)
            assert p["chunks_per_lane"] == 2 and 8 * nvec >= 7 * 64 * nw and nvec <= 64 * nw
            assert nw * p["ctas_per_sm"] >= 14
            assert 1 << (nw - 1).bit_length() > nw  # the power of two it replaces
            assert rmsn.rmsn_plan(rmsn.OP_BWD_RESIDUAL, 65536, H, xd, 0)["consumer_warps"] == nw
    assert seen == {3, 5, 7}


def test_plan_backward_narrow_rows_over_short_strips(lib):
    # rows the plan gives 1 or 2 warps take twice the warps in half the CTAs while a chunk
    # would hold fewer than 8 rows (T < 8 * SMs * 16 / warps)
    for H, xd, long_geom, short_geom in [(512, 1, (1, 16), (2, 8)), (1024, 1, (2, 8), (4, 4)),
                                         (256, 0, (1, 16), (2, 8)), (4096, 1, (8, 2), (8, 2))]:
        nw = long_geom[0]
        limit = 8 * SM * (16 // nw)
        for op in (rmsn.OP_BWD, rmsn.OP_BWD_RESIDUAL):
            a = rmsn.rmsn_plan(op, limit, H, xd, 0)
            b = rmsn.rmsn_plan(op, limit - 1, H, xd, 0)
            assert (a["consumer_warps"], a["ctas_per_sm"]) == long_geom
            assert (b["consumer_warps"], b["ctas_per_sm"]) == short_geom


def test_plan_backward_warps_not_a_power_of_two_by_strip_length(lib):
    # rows the power of two fills to more than 5/8 (bf16 H 1536, 3584) change only over long
    # strips (T >= 16384); rows it fills to at most 5/8 (bf16 H 2304-2560, fp32 H 1280) at any T
    for H, xd, nw, nb in ((1536, 1, 4, 3), (3584, 1, 8, 7)):
        for op in (rmsn.OP_BWD, rmsn.OP_BWD_RESIDUAL):
            assert rmsn.rmsn_plan(op, 16383, H, xd, 0)["consumer_warps"] == nw
            assert rmsn.rmsn_plan(op, 16384, H, xd, 0)["consumer_warps"] == nb
    for H, xd in ((2304, 1), (2560, 1), (1280, 0)):
        assert rmsn.rmsn_plan(rmsn.OP_BWD, 300, H, xd, 0)["consumer_warps"] == 5


def test_plan_backward_short_strip_rule(lib):
    # bf16 rows of about three vectors per lane at 8 warps take one CTA of 16 warps per SM
    # over short strips (T <= 12288), the pair layout of 8 warps above; other widths keep theirs
    for H in (5632, 6144):
        for op in (rmsn.OP_BWD, rmsn.OP_BWD_RESIDUAL):
            short = rmsn.rmsn_plan(op, 12288, H, 1, 0)
            long_ = rmsn.rmsn_plan(op, 12289, H, 1, 0)
            assert (short["consumer_warps"], short["ctas_per_sm"]) == (16, 1)
            assert (long_["consumer_warps"], long_["ctas_per_sm"]) == (8, 2)
    for H in (4096, 5120):
        assert rmsn.rmsn_plan(rmsn.OP_BWD, 4096, H, 1, 0)["consumer_warps"] == 8
    assert rmsn.rmsn_plan(rmsn.OP_BWD, 4096, 6144, 0, 0)["consumer_warps"] == 16  # fp32 rows


def test_plan_forward_rows_in_flight(lib):
    # forward: 2 stages and 8 CTAs per SM for rows of at most 4 KiB, else one stage and
    # about 48 KiB of rows in flight per SM
    for H, xd, geom in [(1024, 1, (2, 8, 2)), (2048, 1, (2, 8, 2)), (4096, 1, (4, 6, 1)),
                        (6144, 1, (4, 4, 1)), (8192, 1, (8, 3, 1)), (2048, 0, (4, 6, 1)),
                        (4096, 0, (8, 3, 1)), (8192, 0, (8, 2, 1))]:
        p = rmsn.rmsn_plan(rmsn.OP_FWD, 65536, H, xd, xd)
        assert (p["consumer_warps"], p["ctas_per_sm"], p["stages"]) == geom, (H, xd, p)


def test_plan_residual_forward_rows_in_flight(lib):
    # the residual forward: 8 CTAs per SM for rows of at most 4 KiB, else 4 (fewer where
    # shared memory runs out), two stages
    for H, xd, cps in [(512, 1, 8), (1024, 1, 8), (2048, 1, 8), (1024, 0, 8), (3072, 1, 4),
                       (4096, 1, 4), (2048, 0, 4), (8192, 1, 2), (16384, 1, 1)]:
        p = rmsn.rmsn_plan(rmsn.OP_FWD_RESIDUAL, 65536, H, xd, xd)
        assert (p["ctas_per_sm"], p["stages"]) == (cps, 2), (H, xd, p)


def test_plan_fused_rows_in_flight(lib):
    # the fused quant: at most three vectors per lane; one stage per CTA; about 64 KiB of
    # stages in flight per SM, at least 2 CTAs, at most the CTAs whose warps (with the
    # producer) the register file holds at 72 registers per thread; fewer where shared
    # memory runs out
    # memory runs out; rows of more than 1024 vectors: one CTA of 16 warps, two stages up to
    # 48 KiB each
    for H, geom in [(512, (1, 14, 1)), (1024, (2, 9, 1)), (1536, (2, 9, 1)), (2048, (4, 5, 1)),
                    (3072, (4, 5, 1)), (4096, (8, 3, 1)), (6144, (8, 3, 1)), (8192, (8, 2, 1)),
                    (8320, (16, 1, 2)), (12288, (16, 1, 2)), (12416, (16, 1, 1)),
                    (16384, (16, 1, 1))]:
        p = rmsn.rmsn_plan(rmsn.OP_FUSED_QUANT, 65536, H, 1, 1)
        assert (p["consumer_warps"], p["ctas_per_sm"], p["stages"]) == geom, (H, p)
        assert p["chunks_per_lane"] <= 8 and p["chunks_per_lane"] * 32 * p["consumer_warps"] >= H // 8
        if p["consumer_warps"] <= 8:
            assert (p["consumer_warps"] + 1) * p["ctas_per_sm"] <= 65536 // (72 * 32)
        else:
            assert p["chunks_per_lane"] in (2, 3, 4) and p["threads"] == 544


def test_workspace_grows_with_t(lib):
    prev = 0
    for T in (1, 2, 3, 17, 100, 1000, 10 ** 4, 10 ** 5, 10 ** 6):
        p = rmsn.rmsn_plan(rmsn.OP_BWD, T, 2048, 1, 0, compensated=True)
        assert p["workspace_bytes"] >= prev
        assert p["grid"] <= min(T, SM * p["ctas_per_sm"])  # within the documented bound
        prev = p["workspace_bytes"]


def test_set_policy(lib):
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_policy(rmsn.OP_FWD, consumer_warps=3)
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_policy(rmsn.OP_FWD, consumer_warps=16)
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_policy(rmsn.OP_FWD, max_stages=33)
    try:
        rmsn.rmsn_set_policy(rmsn.OP_FWD, consumer_warps=8, ctas_per_sm=2, max_stages=3)
        p = rmsn.rmsn_plan(rmsn.OP_FWD, 8192, 4096, 1, 1)
        assert (p["threads"], p["ctas_per_sm"], p["stages"]) == (288, 2, 3)
    finally:
        rmsn.rmsn_set_policy(rmsn.OP_FWD)
    p = rmsn.rmsn_plan(rmsn.OP_FWD, 8192, 4096, 1, 1)
    assert (p["threads"], p["consumer_warps"]) == (160, 4)


def test_set_policy_backward_sixteen_warps(lib):
    # the backward ops and the fused quant take up to 16 consumer warps (one CTA per SM); the
    # forward ops do not
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_policy(rmsn.OP_FWD, consumer_warps=16)
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_policy(rmsn.OP_BWD, consumer_warps=32)
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_policy(rmsn.OP_BWD, consumer_warps=17)
    with pytest.raises(rmsn.RmsnError):
        rmsn.rmsn_set_policy(rmsn.OP_FWD_RESIDUAL, consumer_warps=6)
    try:  # any count up to 16 for the backward
        rmsn.rmsn_set_policy(rmsn.OP_BWD, consumer_warps=12)
        p = rmsn.rmsn_plan(rmsn.OP_BWD, 8192, 4096, 1, 1)
        assert (p["consumer_warps"], p["threads"], p["chunks_per_lane"]) == (12, 384, 2)
    finally:
        rmsn.rmsn_set_policy(rmsn.OP_BWD)
    for op in (rmsn.OP_BWD, rmsn.OP_BWD_RESIDUAL):
        try:
            rmsn.rmsn_set_policy(op, consumer_warps=16)
            p = rmsn.rmsn_plan(op, 8192, 4096, 1, 1)
            assert (p["consumer_warps"], p["ctas_per_sm"], p["threads"]) == (16, 1, 512)
            assert p["chunks_per_lane"] == 1 and p["grid"] == SM
        finally:
            rmsn.rmsn_set_policy(op)
        p = rmsn.rmsn_plan(op, 8192, 4096, 1, 1)
        assert (p["consumer_warps"], p["ctas_per_sm"]) == (8, 2)


def test_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.randn(4, 64)
    with pytest.raises(ValueError):
        rmsn.rmsnorm_fwd(x, torch.ones(64))


def test_product_never_imports_oracle():
    """The product package does not import, load or name the oracle."""
    pkg = os.path.join(ROOT, "rmsnorm_fwd_bwd_persistent_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "liboracle" not in src and "rmsnorm_oracle" not in src, fn
