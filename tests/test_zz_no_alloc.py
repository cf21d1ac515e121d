"""The allocation-free backward (rmsnorm_bwd_noalloc), called through the C ABI.

Some callers cannot allocate device memory where they call the backward (a framework
that hands out all device memory up front from its own pool, a latency-critical loop in
which cudaMalloc's implicit synchronization would stall, a plain C caller with no
allocator for a workspace).  rmsnorm_bwd_noalloc keeps its scratch in a fixed array the
library owns.  It runs the same kernels as rmsnorm_bwd (deterministic, caller
workspace), so on two calls in a row its dx and dW must be bit-identical to that call's.
The cases cover the strip route, the one-launch small-T route (which needs no scratch,
so it accepts widths whose strip plan would not fit), a strip plan whose scratch is the
largest that still fits the fixed array, and the rejection one width above it.  This
file is collected last; it passes alone in a fresh process and after the other tests.
"""
import pytest
import torch

import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
SCRATCH_LIMIT = 7  # RMSN_ERR_SCRATCH_LIMIT
SCRATCH_BYTES = 16 << 20  # RMSN_NOALLOC_SCRATCH_BYTES


def _noalloc(dy, x, w, rstd, dx, dw, compensated):
    L = rmsn.load_library()
    T, H = x.shape
    return L.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), rmsn.RMSN_BF16 if x.dtype == torch.bfloat16 else rmsn.RMSN_F32,
                                 w.data_ptr(), rmsn.RMSN_BF16 if w.dtype == torch.bfloat16 else rmsn.RMSN_F32,
                                 rstd.data_ptr(), dx.data_ptr(), dw.data_ptr(), T, H, int(compensated),
                                 torch.cuda.current_stream().cuda_stream)


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _strip_scratch(T, H):
    return rmsn.rmsn_plan(rmsn.OP_BWD, T, H, rmsn.RMSN_BF16, rmsn.RMSN_BF16,
                          sm_count=_sm_count())["workspace_bytes"]


def _widest_fitting_h(T):
    """The largest bf16 width whose strip plan at T rows fits the fixed scratch, and the
    next width (a multiple of 8) above it, which does not."""
    best = None
    for H in range(8, rmsn.RMSN_MAX_H + 1, 8):
        if _strip_scratch(T, H) <= SCRATCH_BYTES:
            best = H
    return best, best + 8


def _check_bitwise(T, H, wd, compensated):
    c = wl.Workload("noalloc", T, H, torch.bfloat16, wd)
    x, dy, w = wl.fwd_bwd_inputs(c, "cuda", seed=T + H)
    _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
    dx_ref, dw_ref = rmsn.rmsnorm_bwd(dy, x, w, rstd, deterministic=True, compensated=compensated)
    for call in range(2):
        dx = torch.full_like(x, float("nan"))
        dw = torch.full((H,), float("nan"), device="cuda")
        st = _noalloc(dy, x, w, rstd, dx, dw, compensated)
        assert st == 0, rmsn.rmsn_status_string(st)
        torch.cuda.synchronize()
        assert rmsn.rmsn_device_status() == 0
        assert torch.equal(dx.view(torch.int16), dx_ref.view(torch.int16)), (call, "dx bits")
        assert torch.equal(dw.view(torch.int32), dw_ref.view(torch.int32)), (call, "dw bits")


@pytest.mark.parametrize("T,H,wd,compensated", [(8192, 4096, torch.bfloat16, False),
                                                 (4097, 6144, torch.float32, True),
                                                 (63, 1536, torch.float32, False)])
def test_noalloc_bitwise_equals_workspace_backward_twice(T, H, wd, compensated):
    _check_bitwise(T, H, wd, compensated)


def test_noalloc_small_t_route_needs_no_scratch():
    # a width whose strip plan would not fit, at a T the one-launch route takes
    T, H = 200, 16384
    assert T <= rmsn.rmsn_small_t_max()
    assert _strip_scratch(T, H) > SCRATCH_BYTES
    _check_bitwise(T, H, torch.bfloat16, False)


def test_noalloc_at_the_scratch_boundary():
    T = 4 * _sm_count() * 4  # more rows than chunks: the strip route with its largest grid
    h_fit, h_over = _widest_fitting_h(T)
    assert _strip_scratch(T, h_fit) > SCRATCH_BYTES * 0.9  # close to the limit
    _check_bitwise(T, h_fit, torch.bfloat16, False)
    x = torch.zeros(T, h_over, device="cuda", dtype=torch.bfloat16)
    w = torch.ones(h_over, device="cuda", dtype=torch.bfloat16)
    rstd = torch.ones(T, device="cuda")
    dx = torch.empty_like(x)
    dw = torch.empty(h_over, device="cuda")
    assert _noalloc(x, x, w, rstd, dx, dw, False) == SCRATCH_LIMIT


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T, H = 4096, 16384  # needs 8 * H * min(T, SMs * CTAs per SM) bytes, well above 16 MiB
    x = torch.zeros(T, H, device="cuda", dtype=torch.bfloat16)
    w = torch.ones(H, device="cuda", dtype=torch.bfloat16)
    rstd = torch.ones(T, device="cuda")
    dx = torch.empty_like(x)
    dw = torch.empty(H, device="cuda")
    assert _noalloc(x, x, w, rstd, dx, dw, False) == SCRATCH_LIMIT
    assert "16 MiB" in rmsn.rmsn_status_string(SCRATCH_LIMIT)
