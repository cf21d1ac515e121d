"""The allocation-free backward (rmsnorm_bwd_noalloc), called through the C ABI.

Some callers cannot allocate device memory where they call the backward (a framework
that hands out all device memory up front from its own pool, a latency-critical loop in
which cudaMalloc's implicit synchronization would stall, a plain C caller with no
allocator for a workspace).  rmsnorm_bwd_noalloc keeps its scratch in a fixed array the
library owns.  These tests check, on two calls in a row, that it returns what
rmsnorm_bwd (deterministic, caller workspace) returns, within the parity tolerances
(dx within one bf16 ulp, dW within atol 1e-4 + rtol 1e-4), and that a call needing more
than the fixed scratch is rejected.  This file is collected last; it passes alone in a
fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

from oracle import gates
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
SCRATCH_LIMIT = 7  # RMSN_ERR_SCRATCH_LIMIT


def _noalloc(dy, x, w, rstd, dx, dw, compensated):
    L = rmsn.load_library()
    T, H = x.shape
    return L.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), rmsn.RMSN_BF16 if x.dtype == torch.bfloat16 else rmsn.RMSN_F32,
                                 w.data_ptr(), rmsn.RMSN_BF16 if w.dtype == torch.bfloat16 else rmsn.RMSN_F32,
                                 rstd.data_ptr(), dx.data_ptr(), dw.data_ptr(), T, H, int(compensated),
                                 torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("T,H,wd,compensated", [(8192, 4096, torch.bfloat16, False),
                                                 (4097, 6144, torch.float32, True),
                                                 (63, 1536, torch.float32, False)])
def test_noalloc_matches_workspace_backward_twice(T, H, wd, compensated):
    c = wl.Workload("noalloc", T, H, torch.bfloat16, wd)
    x, dy, w = wl.fwd_bwd_inputs(c, "cuda", seed=T + H)
    _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
    dx_ref, dw_ref = rmsn.rmsnorm_bwd(dy, x, w, rstd, deterministic=True, compensated=compensated)
    dx_ref_b = wl.to_oracle(dx_ref)
    dw_ref_h = dw_ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        dx = torch.full_like(x, float("nan"))
        dw = torch.full((H,), float("nan"), device="cuda")
        st = _noalloc(dy, x, w, rstd, dx, dw, compensated)
        assert st == 0, rmsn.rmsn_status_string(st)
        torch.cuda.synchronize()
        assert rmsn.rmsn_device_status() == 0
        rdx = gates.check_bf16(wl.to_oracle(dx), gates.bf16_to_f64(dx_ref_b))
        rdw = gates.check_dw(dw.cpu().numpy(), dw_ref_h)
        assert rdx["n_fail"] == 0, (call, rdx)
        assert rdw["n_fail"] == 0, (call, rdw)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T, H = 4096, 16384  # needs 8 * H * min(T, SMs * CTAs per SM) bytes, well above 16 MiB
    x = torch.zeros(T, H, device="cuda", dtype=torch.bfloat16)
    w = torch.ones(H, device="cuda", dtype=torch.bfloat16)
    rstd = torch.ones(T, device="cuda")
    dx = torch.empty_like(x)
    dw = torch.empty(H, device="cuda")
    assert _noalloc(x, x, w, rstd, dx, dw, False) == SCRATCH_LIMIT
    assert "16 MiB" in rmsn.rmsn_status_string(SCRATCH_LIMIT)
