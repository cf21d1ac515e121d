import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Widening statistics of the bf16 dx gates (elements that needed the a-priori FP32
    bound on top of one ulp, and their error in bf16 ulps of their row's RMS), and the
    weight-gradient budget figures of every dW comparison."""
    mod = sys.modules.get("_parity")
    dwr = getattr(mod, "DW_BUDGET", None) if mod else None
    if dwr:
        tr = terminalreporter
        w = max(dwr, key=lambda r: r["worst"])
        tr.section("dW budget")
        tr.write_line(f"{len(dwr)} dW comparisons, {sum(r['n'] for r in dwr)} elements: worst "
                      f"|dw - ref| / (1e-4 + 1e-4 |ref|) = {w['worst']:.4f} (limit 1) at "
                      f"{w['what']}; max rel-L2 {max(r['rel_l2'] for r in dwr):.2e}")
    rec = getattr(mod, "WIDENING", None) if mod else None
    if not rec:
        return
    n = sum(r["n"] for r in rec)
    nw = sum(r["n_widened"] for r in rec)
    worst = max(rec, key=lambda r: r["n_widened"] / max(r["n"], 1))
    tr = terminalreporter
    tr.section("bf16 dx gate widening")
    tr.write_line(f"{len(rec)} bf16 dx comparisons, {n} elements: {nw} widened "
                  f"({nw / max(n, 1):.2e}); max error of unwidened elements "
                  f"{max(r['max_err_in_ulp'] for r in rec):.3f} ulp; max widened error "
                  f"{max(r['max_widened_err_row_ulp'] for r in rec):.3e} row-RMS ulp")
    tr.write_line(f"largest widened fraction: {worst['what']}: {worst['n_widened']} of "
                  f"{worst['n']}")
