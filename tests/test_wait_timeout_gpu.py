"""The bounded waits end and report instead of hanging.  A self-test CTA waits on an
mbarrier that nothing completes (no copy in flight); after its limit the wait gives up,
the device error word reports it, the status call clears it, and the context stays usable
(a normal call afterwards is correct and reports no timeout)."""
import time

import pytest
import torch

import _parity as P
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_that_never_completes_reports_and_clears():
    assert rmsn.rmsn_device_status() == 0
    t0 = time.perf_counter()
    rmsn.rmsn_selftest_wait_timeout(2_000_000)  # 2 ms
    flags = rmsn.rmsn_device_status()           # synchronizes
    elapsed = time.perf_counter() - t0
    assert flags & 1, "the wait should have run out and set bit 0"
    assert elapsed < 5.0                          # it ended by itself
    assert rmsn.rmsn_device_status() == 0         # read-and-clear


def test_context_usable_after_timeout():
    rmsn.rmsn_selftest_wait_timeout(1_000_000)
    assert rmsn.rmsn_device_status() & 1
    x, _, w = wl.fwd_bwd_inputs(wl.SMALL_FP32, DEV, seed=0)
    P.assert_ok(P.check_fwd(x, w, 1e-6), "forward after a timed-out self-test")


def test_selftest_rejects_bad_limits():
    for bad in (0, 10 ** 10):
        with pytest.raises(rmsn.RmsnError):
            rmsn.rmsn_selftest_wait_timeout(bad)
