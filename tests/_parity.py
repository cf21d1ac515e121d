"""Parity checks of the CUDA path against the FP64 oracle (helpers for the GPU tests).

Outputs are NaN-poisoned before each call (an element the kernel leaves unwritten
fails the gate) and sit inside guard bands filled with a sentinel (a write outside the
output fails the guard check).  Large cases compare a sample of rows elementwise and
the whole weight gradient.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import gates
import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
import workloads as wl

GUARD = 64  # elements of guard band on each side (a multiple of 16 bytes for any dtype)
FULL_LIMIT = 1 << 25  # compare every element up to this many; sample rows above
CHUNK_ELEMS = 1 << 25  # rows compared per oracle call when every row is compared
MAX_FRAC_WIDENED = 0.005  # bf16 dx elements that may need the FP32 bound on top of 1 ulp
MAX_WIDENED_ROW_ULP = 1.0  # and their error, in bf16 ulps of the row's RMS

# Widening statistics of every bf16 dx gate evaluated in this process (printed by the
# terminal summary in conftest.py).
WIDENING: list = []
DW_BUDGET: list = []  # every dW comparison: worst |dw - ref| / (1e-4 + 1e-4 |ref|), rel-L2


def guarded(shape, dtype, device, fill=float("nan")):
    """A contiguous tensor of `shape` inside a buffer with GUARD sentinel elements around it."""
    n = int(np.prod(shape)) if len(shape) else 1
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
    if dtype == torch.uint8:
        buf.fill_(0xA5)
    else:
        buf.fill_(-12288.0)
    body = buf[GUARD:GUARD + n].view(*shape)
    if dtype == torch.uint8:
        body.fill_(0xFF)  # E4M3 NaN code: any unwritten byte fails
    else:
        body.fill_(fill)
    return buf, body


def guards_ok(buf: torch.Tensor) -> bool:
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    if buf.dtype == torch.uint8:
        return bool((g == 0xA5).all())
    return bool((g == -12288.0).all())


def _rows(T: int, H: int, nsample: int = 192, seed: int = 0) -> np.ndarray:
    if T * H <= FULL_LIMIT:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    pick = rng.choice(T, size=min(nsample, T), replace=False)
    return np.unique(np.concatenate([pick, [0, 1, T - 2, T - 1]]))


def _row_chunks(T: int, H: int, all_rows: bool):
    """Row index arrays to compare: every row (in chunks of about CHUNK_ELEMS elements) when
    all_rows or when the tensor is small, else one sample of rows."""
    if not all_rows:
        return [_rows(T, H)]
    step = max(1, CHUNK_ELEMS // H)
    return [np.arange(a, min(a + step, T)) for a in range(0, T, step)]


def _merge(parts: list) -> dict:
    """Combines gate results over row chunks (counts add, worst values take the max)."""
    out = {}
    for r in parts:
        for k, v in r.items():
            if k == "first_fail":
                out.setdefault(k, None)
                if out[k] is None and v is not None:
                    out[k] = v
            elif k in ("n", "n_fail", "n_widened"):
                out[k] = out.get(k, 0) + v
            elif isinstance(v, (int, float)):
                out[k] = max(out.get(k, v), v)
    if "n_widened" in out:
        out["frac_widened"] = out["n_widened"] / out["n"] if out["n"] else 0.0
    return out


def row_dot_depth(T: int, H: int, x_dtype, w_dtype, deterministic: bool,
                  residual: bool = False) -> int:
    """Roundings on the longest path of the device's row-dot tree for this call (the
    launch plan's warps and vectors per lane; the one-launch small-T route's 256-thread
    row task when it takes the call)."""
    xd = rmsn.RMSN_BF16 if x_dtype == torch.bfloat16 else rmsn.RMSN_F32
    wd = rmsn.RMSN_BF16 if w_dtype == torch.bfloat16 else rmsn.RMSN_F32
    vec = 8 if xd == rmsn.RMSN_BF16 else 4
    if deterministic and T <= rmsn.rmsn_small_t_max():
        return gates.row_dot_depth(-(-(H // vec) // 256) * (vec // 2), 8)
    op = rmsn.OP_BWD_RESIDUAL if residual else rmsn.OP_BWD
    p = rmsn.rmsn_plan(op, T, H, xd, wd)
    return gates.row_dot_depth(p["chunks_per_lane"] * (vec // 2), p["consumer_warps"])


def _widening(r: dict, what: str) -> dict:
    """Records a bf16 dx gate's widening statistics and turns the limits into a check."""
    WIDENING.append({"what": what, "n": r["n"], "n_widened": r["n_widened"],
                     "max_err_in_ulp": r["max_err_in_ulp"],
                     "max_widened_err_row_ulp": r["max_widened_err_row_ulp"]})
    bad = (r["frac_widened"] > MAX_FRAC_WIDENED or
           r["max_widened_err_row_ulp"] > MAX_WIDENED_ROW_ULP)
    return {"n_fail": int(bad), "frac_widened": r["frac_widened"],
            "max_widened_err_row_ulp": r["max_widened_err_row_ulp"]}


def _dw_record(r: dict, what: str) -> dict:
    """Records a dW comparison's budget figures for the end-of-run summary."""
    DW_BUDGET.append({"what": what, "n": r["n"], "worst": r["worst"], "rel_l2": r["rel_l2"]})
    return r


def _f64(a: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def gate_fwd(x, w, eps, y, rstd, all_rows: bool = False) -> dict:
    """Forward outputs already on the device (y, rstd) against the oracle."""
    T, H = x.shape
    W = wl.to_oracle(w)
    r_all = rstd.cpu().numpy()
    pr, py = [], []
    for rows in _row_chunks(T, H, all_rows):
        ridx = torch.from_numpy(rows).to(x.device)
        y_ref, r_ref = oracle.rmsnorm_fwd(wl.to_oracle(x[ridx]), W, eps)
        y_dev = wl.to_oracle(y[ridx])
        pr.append(gates.check_f32_rel(r_all[rows], r_ref))
        py.append(gates.check_bf16(y_dev, y_ref) if x.dtype == torch.bfloat16
                  else gates.check_f32_rel(y_dev, y_ref))
    return {"rstd": _merge(pr), "y": _merge(py)}


def check_fwd(x: torch.Tensor, w: torch.Tensor, eps: float, all_rows: bool = False) -> dict:
    T, H = x.shape
    ybuf, y = guarded((T, H), x.dtype, x.device)
    rbuf, rstd = guarded((T,), torch.float32, x.device)
    rmsn.rmsnorm_fwd(x, w, eps, y=y, rstd=rstd)
    torch.cuda.synchronize()
    out = gate_fwd(x, w, eps, y, rstd, all_rows)
    out["guards"] = {"n_fail": int(not (guards_ok(ybuf) and guards_ok(rbuf)))}
    out["device_status"] = {"n_fail": rmsn.rmsn_device_status()}
    out["_rstd_dev"] = rstd
    return out


def gate_bwd(dy, x, w, rstd, dx, dw, deterministic: bool, all_rows: bool = False,
             full_dw: bool = True) -> dict:
    """Backward outputs already on the device (dx, dw) against the oracle at the saved
    rstd."""
    T, H = x.shape
    W = wl.to_oracle(w)
    r_all = rstd.cpu().numpy().astype(np.float64)
    depth = row_dot_depth(T, H, x.dtype, w.dtype, deterministic)
    parts = []
    for rows in _row_chunks(T, H, all_rows):
        ridx = torch.from_numpy(rows).to(x.device)
        DYs, Xs = wl.to_oracle(dy[ridx]), wl.to_oracle(x[ridx])
        dx_ref, _ = oracle.rmsnorm_bwd(DYs, Xs, W, r_all[rows], want_dw=False)
        dx_dev = wl.to_oracle(dx[ridx])
        if x.dtype == torch.bfloat16:
            extra = gates.dx_fp32_bound(_f64(DYs), _f64(Xs), _f64(W), r_all[rows], dx_ref, depth)
            parts.append(gates.check_bf16(dx_dev, dx_ref, extra=extra))
        else:
            parts.append(gates.check_f32_rel(dx_dev, dx_ref, row_rms_term=True))
    out = {"dx": _merge(parts)}
    if x.dtype == torch.bfloat16:
        out["dx_widening"] = _widening(out["dx"], f"bwd T={T} H={H} det={int(deterministic)}")
    if full_dw:
        _, dw_ref = oracle.rmsnorm_bwd(wl.to_oracle(dy), wl.to_oracle(x), W, r_all, want_dx=False)
        out["dw"] = _dw_record(gates.check_dw(dw.cpu().numpy(), dw_ref),
                               f"bwd T={T} H={H} det={int(deterministic)}")
    return out


def check_bwd(dy, x, w, rstd, deterministic=True, compensated=False, full_dw=True,
              workspace=None, all_rows=False) -> dict:
    T, H = x.shape
    dxbuf, dx = guarded((T, H), x.dtype, x.device)
    dwbuf, dw = guarded((H,), torch.float32, x.device)
    if workspace is None:  # NaN-poisoned: no call may depend on what it held before
        n = rmsn.rmsnorm_bwd_workspace_bytes(T, H, compensated, x.device)
        workspace = torch.full((max(n, 16) // 4,), float("nan"), device=x.device,
                               dtype=torch.float32)
    rmsn.rmsnorm_bwd(dy, x, w, rstd, deterministic=deterministic, compensated=compensated,
                     workspace=workspace, dx=dx, dw=dw)
    torch.cuda.synchronize()
    out = gate_bwd(dy, x, w, rstd, dx, dw, deterministic, all_rows, full_dw)
    out["guards"] = {"n_fail": int(not (guards_ok(dxbuf) and guards_ok(dwbuf)))}
    out["device_status"] = {"n_fail": rmsn.rmsn_device_status()}
    out["_dw_dev"] = dw
    return out


def check_fwd_residual(x, res, w, eps, inplace: bool = False) -> dict:
    """rmsnorm_fwd_residual against the oracle: h_new bit-exact (one rounding of an exact
    sum), y and rstd as the forward.  inplace: h_new is written over `res`."""
    T, H = x.shape
    res_in = res.clone()
    ybuf, y = guarded((T, H), x.dtype, x.device)
    rbuf, rstd = guarded((T,), torch.float32, x.device)
    if inplace:
        hbuf, h = None, res
    else:
        hbuf, h = guarded((T, H), x.dtype, x.device)
    rmsn.rmsnorm_fwd_residual(x, res, w, eps, y=y, h_new=h, rstd=rstd)
    torch.cuda.synchronize()
    rows = _rows(T, H)
    ridx = torch.from_numpy(rows).to(x.device)
    y_ref, r_ref, h_ref = oracle.rmsnorm_fwd_residual(wl.to_oracle(x[ridx]), wl.to_oracle(res_in[ridx]),
                                                      wl.to_oracle(w), eps)
    h_dev = wl.to_oracle(h[ridx])
    out = {"h_new": {"n_fail": int(np.count_nonzero(h_dev.view(np.uint16 if h_dev.dtype == np.uint16 else np.uint32)
                                                    != h_ref.view(np.uint16 if h_ref.dtype == np.uint16 else np.uint32)))},
           "rstd": gates.check_f32_rel(rstd.cpu().numpy()[rows], r_ref)}
    y_dev = wl.to_oracle(y[ridx])
    out["y"] = gates.check_bf16(y_dev, y_ref) if x.dtype == torch.bfloat16 else gates.check_f32_rel(y_dev, y_ref)
    bufs = [ybuf, rbuf] + ([hbuf] if hbuf is not None else [])
    out["guards"] = {"n_fail": int(not all(guards_ok(b) for b in bufs))}
    out["device_status"] = {"n_fail": rmsn.rmsn_device_status()}
    out["_h"], out["_rstd_dev"] = h, rstd
    return out


def check_bwd_residual(dy, h, w, rstd, g_res, deterministic=True, compensated=False,
                       alias: str | None = None) -> dict:
    """rmsnorm_bwd_residual against the oracle: dx_total = dx + g_residual (bf16 within one
    ulp, widened by the a-priori FP32 bound of dx plus the rounding of the FP32 sum), dw as
    rmsnorm_bwd.  alias: 'g' writes dx_total over g_residual, 'dy' over dy."""
    T, H = h.shape
    dy_in, g_in = dy.clone(), g_res.clone()
    dwbuf, dw = guarded((H,), torch.float32, h.device)
    if alias == "g":
        dxbuf, dxt = None, g_res
    elif alias == "dy":
        dxbuf, dxt = None, dy
    else:
        dxbuf, dxt = guarded((T, H), h.dtype, h.device)
    n = rmsn.rmsnorm_bwd_workspace_bytes(T, H, compensated, h.device)
    ws = torch.full((max(n, 16) // 4,), float("nan"), device=h.device, dtype=torch.float32)
    rmsn.rmsnorm_bwd_residual(dy, h, w, rstd, g_res, deterministic=deterministic,
                              compensated=compensated, workspace=ws, dx_total=dxt, dw=dw)
    torch.cuda.synchronize()
    rows = _rows(T, H)
    ridx = torch.from_numpy(rows).to(h.device)
    W = wl.to_oracle(w)
    r_all = rstd.cpu().numpy().astype(np.float64)
    DYs, Hs, Gs = wl.to_oracle(dy_in[ridx]), wl.to_oracle(h[ridx]), wl.to_oracle(g_in[ridx])
    dxt_ref, _ = oracle.rmsnorm_bwd_residual(DYs, Hs, W, r_all[rows], Gs, want_dw=False)
    dx_dev = wl.to_oracle(dxt[ridx])
    out = {}
    if h.dtype == torch.bfloat16:
        # dx_total = RN(o + g) with o the FP32 dx (error <= B): |error| <= (1+u) B + u |dx_total|
        dx_plain, _ = oracle.rmsnorm_bwd(DYs, Hs, W, r_all[rows], want_dw=False)
        depth = row_dot_depth(T, H, h.dtype, w.dtype, deterministic, residual=True)
        extra = gates.dx_fp32_bound(_f64(DYs), _f64(Hs), _f64(W), r_all[rows], dx_plain, depth) \
            * (1.0 + gates.U32) + gates.U32 * np.abs(dxt_ref)
        out["dx_total"] = gates.check_bf16(dx_dev, dxt_ref, extra=extra)
        out["dx_widening"] = _widening(out["dx_total"], f"bwd_residual T={T} H={H}")
    else:
        out["dx_total"] = gates.check_f32_rel(dx_dev, dxt_ref, row_rms_term=True)
    _, dw_ref = oracle.rmsnorm_bwd_residual(wl.to_oracle(dy_in), wl.to_oracle(h), W, r_all,
                                            wl.to_oracle(g_in), want_dx=False)
    out["dw"] = _dw_record(gates.check_dw(dw.cpu().numpy(), dw_ref), f"bwd_residual T={T} H={H}")
    bufs = [dwbuf] + ([dxbuf] if dxbuf is not None else [])
    out["guards"] = {"n_fail": int(not all(guards_ok(b) for b in bufs))}
    out["device_status"] = {"n_fail": rmsn.rmsn_device_status()}
    out["_dw_dev"] = dw
    return out


def gate_fused(x, res_in, w, eps, q, scale, normed, res_out) -> dict:
    """Fused outputs already on the device against the oracle: residual bit-exact, normed
    within one bf16 ulp, codes and scales bit-exact when the oracle quantizes the device's
    own normed output.  res_in: the residual before the call (oracle format)."""
    T, H = x.shape
    ld = scale.shape[1]
    h_ref, n_ref, _ = oracle.fused_add_rmsnorm(wl.to_oracle(x), res_in, wl.to_oracle(w), eps)
    nb = wl.to_oracle(normed)
    s_dev = scale.cpu().numpy().reshape(-1)
    q_ref, s_ref = oracle.block_quant_e4m3(nb, ld)
    valid = np.zeros((H // 128, ld), bool)
    valid[:, :T] = True
    valid = valid.reshape(-1)
    return {
        "residual": {"n_fail": int(np.count_nonzero(wl.to_oracle(res_out) != h_ref))},
        "normed": gates.check_bf16(nb, n_ref),
        "q": {"n_fail": int(np.count_nonzero(q.cpu().numpy() != q_ref))},
        "scale": {"n_fail": int(np.count_nonzero(s_dev[valid].view(np.uint32) !=
                                                 s_ref[valid].view(np.uint32)))},
        "_scale_flat": s_dev, "_valid": valid,
    }


def check_fused(x, res, w, eps, ld_pad: int = 0) -> dict:
    T, H = x.shape
    ld = wl.round_up(T, 4) + ld_pad
    res_in = wl.to_oracle(res).copy()
    qbuf, q = guarded((T, H), torch.uint8, x.device)
    sbuf, scale = guarded((H // 128, ld), torch.float32, x.device)
    nbuf, normed = guarded((T, H), torch.bfloat16, x.device)
    rmsn.fused_add_rmsnorm_fp8_block_quant(x, res, w, eps, q=q, block_scale=scale, normed=normed)
    torch.cuda.synchronize()
    out = gate_fused(x, res_in, w, eps, q, scale, normed, res)
    s_dev, valid = out["_scale_flat"], out["_valid"]
    # pad entries m in [T, ld) keep the poison (NaN) the test wrote
    out["scale_pads"] = {"n_fail": int(np.count_nonzero(~np.isnan(s_dev[~valid])))}
    out["guards"] = {"n_fail": int(not (guards_ok(qbuf) and guards_ok(sbuf) and guards_ok(nbuf)))}
    out["device_status"] = {"n_fail": rmsn.rmsn_device_status()}
    return out


def assert_ok(res: dict, what: str = ""):
    bad = {k: v for k, v in res.items() if not k.startswith("_") and v.get("n_fail")}
    assert not bad, f"{what}: parity failed: {bad}"
