"""Benchmark: achieved HBM GB/s (and % of the GB300 bandwidth roofline) and us/call of
the RMSNorm hot path at T=8192, H=4096, bf16.

One step = forward + deterministic fused backward (main strip kernel + dW column
reduce) + fused residual-add/RMSNorm/E4M3 1x128 block quant, each on its own seeded
synthetic inputs of the headline shape, with L2 flushed (512 MiB written, 256 MiB read) before every
op and each op timed with CUDA events on its stream (the pages' protocol: kernel time,
cold L2, FlashInfer PR #5741 Performance; miles-ext-kernels PR #15 Performance).
The bandwidth is the logical-byte model of the same pages divided by the step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an independent replica on
its own GPU (the path needs no exchange between GPUs); the value is the bytes of all
ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "achieved HBM GB/s (% of GB300 peak) and us/call, RMSNorm fwd+fused bwd"
UNIT = "GB/s"
T_MAIN, H_MAIN = 8192, 4096
WORKLOAD = ("RMSNorm forward + fused dX/dW backward (deterministic) + fused residual-add/"
            "RMSNorm/E4M3 1x128 block quant, T=8192 H=4096 bf16 (fp32 rstd, dW, scales)")
FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------- helpers
def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(local_ms: float, local_bytes: int, world: int):
    """Max step time over ranks and total bytes of all ranks (the replicas' whole job)."""
    if world == 1:
        return local_ms, local_bytes
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    b = torch.tensor([float(local_bytes)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: copy, burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 copy measurement)"


def _source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "rmsnorm_fwd_bwd_persistent_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(op: str):
    """DRAM bytes (read + write) per launch of `op` from the committed ncu summary, if it
    was taken on the current sources of that op's kernels; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)[op]
        if d.get("source_digest") == _source_digest(d["sources"]):
            return int(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------- our arm
class Step:
    """Device buffers of one step at the headline shape (inputs resident in HBM)."""

    def __init__(self, dev, seed=0):
        import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
        self.rmsn = rmsn
        c = wl.MAIN_BF16
        self.x, self.dy, self.w = wl.fwd_bwd_inputs(c, dev, seed)
        self.y = torch.empty_like(self.x)
        self.rstd = torch.empty(c.T, device=dev)
        self.dx = torch.empty_like(self.x)
        self.dw = torch.empty(c.H, device=dev)
        nws = rmsn.rmsnorm_bwd_workspace_bytes(c.T, c.H, False, dev)
        self.ws = torch.empty(max(nws, 16), device=dev, dtype=torch.uint8)
        f = wl.FUSED_QUANT_MAIN
        self.fx, self.fres, self.fw = wl.fused_inputs(f, dev, seed + 1)
        self.q = torch.empty(f.T, f.H, device=dev, dtype=torch.uint8)
        self.scale = torch.empty(f.H // 128, wl.round_up(f.T, 4), device=dev)
        self.normed = torch.empty_like(self.fx)
        self.eps = c.eps
        self.flush_buf = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
        self.flush_rd = self.flush_buf.view(torch.float32)[: (FLUSH_BYTES // 2) // 4]
        self.bytes = {
            "fwd": wl.fwd_bytes(c.T, c.H, c.x_dtype, c.w_dtype),
            "bwd": wl.bwd_bytes(c.T, c.H, c.x_dtype, c.w_dtype),
            "fused_quant": wl.fused_quant_bytes(f.T, f.H),
        }
        # the residual training variant at the same shape (timed apart from the step)
        r = wl.RESIDUAL_MAIN
        self.rx, self.rres, self.rdy, self.rg, self.rw = wl.residual_inputs(r, dev, seed + 2)
        self.ry, self.rh, self.rdx = (torch.empty_like(self.rx) for _ in range(3))
        self.rrstd = torch.empty(r.T, device=dev)
        self.rdw = torch.empty(r.H, device=dev)
        self.bytes_extra = {
            "fwd_residual": wl.fwd_residual_bytes(r.T, r.H, r.x_dtype, r.w_dtype),
            "bwd_residual": wl.bwd_residual_bytes(r.T, r.H, r.x_dtype, r.w_dtype),
        }
        rmsn.rmsnorm_fwd_residual(self.rx, self.rres, self.rw, r.eps, y=self.ry, h_new=self.rh,
                                  rstd=self.rrstd)
        # fwd writes rstd for the bwd once, so the bwd sees the forward's saved value
        rmsn.rmsnorm_fwd(self.x, self.w, self.eps, y=self.y, rstd=self.rstd)

    def flush(self):
        """Evicts L2: writes 512 MiB, then reads 256 MiB of it so that L2 holds clean lines
        (no write-back of flush data lands inside the next timed op)."""
        self.flush_buf.zero_()
        self.flush_rd.sum()

    def fwd(self):
        self.rmsn.rmsnorm_fwd(self.x, self.w, self.eps, y=self.y, rstd=self.rstd)

    def bwd(self):
        self.rmsn.rmsnorm_bwd(self.dy, self.x, self.w, self.rstd, deterministic=True,
                              compensated=False, workspace=self.ws, dx=self.dx, dw=self.dw)

    def fused(self):
        self.rmsn.fused_add_rmsnorm_fp8_block_quant(self.fx, self.fres, self.fw, self.eps,
                                                    q=self.q, block_scale=self.scale,
                                                    normed=self.normed)

    def fwd_residual(self):
        self.rmsn.rmsnorm_fwd_residual(self.rx, self.rres, self.rw, self.eps, y=self.ry,
                                       h_new=self.rh, rstd=self.rrstd)

    def bwd_residual(self):
        self.rmsn.rmsnorm_bwd_residual(self.rdy, self.rh, self.rw, self.rrstd, self.rg,
                                       deterministic=True, compensated=False, workspace=self.ws,
                                       dx_total=self.rdx, dw=self.rdw)

    OPS = ("fwd", "bwd", "fused_quant")
    EXTRA_OPS = ("fwd_residual", "bwd_residual")
    LAUNCHES = {"fwd": 1, "bwd": 2, "fused_quant": 1, "fwd_residual": 1, "bwd_residual": 2}

    def run_op(self, name):
        {"fwd": self.fwd, "bwd": self.bwd, "fused_quant": self.fused,
         "fwd_residual": self.fwd_residual, "bwd_residual": self.bwd_residual}[name]()


def time_steps(step: Step, steps: int, warmup: int, world: int):
    ev = {op: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)] for op in Step.OPS}
    for _ in range(warmup):
        for op in Step.OPS:
            step.flush()
            step.run_op(op)
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        for op in Step.OPS:
            step.flush()  # L2 flush between timed ops (outside the events)
            s, e = ev[op][i]
            s.record()
            step.run_op(op)
            e.record()
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    per_op = {op: [s.elapsed_time(e) for s, e in ev[op]] for op in Step.OPS}
    return per_op, wall


def time_extra(step: Step, steps: int, warmup: int):
    """The residual training variant (not part of the step), same protocol: L2 flushed
    before each op, CUDA events around each call; mean us per op."""
    for _ in range(warmup):
        for op in Step.EXTRA_OPS:
            step.flush()
            step.run_op(op)
    ev = {op: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)] for op in Step.EXTRA_OPS}
    torch.cuda.synchronize()
    for i in range(steps):
        for op in Step.EXTRA_OPS:
            step.flush()
            s, e = ev[op][i]
            s.record()
            step.run_op(op)
            e.record()
    torch.cuda.synchronize()
    out = {}
    for op in Step.EXTRA_OPS:
        ms = statistics.mean(s.elapsed_time(e) for s, e in ev[op])
        gbs = step.bytes_extra[op] / (ms * 1e-3) / 1e9
        out[op] = {"us_mean": ms * 1e3, "gbs": gbs, "bytes": step.bytes_extra[op],
                   "launches": Step.LAUNCHES[op]}
    return out


def time_long_strip(dev, steps: int, warmup: int, peak: float):
    """The deterministic backward over a long strip (T=65536, H=4096 bf16: 216 rows per CTA
    instead of 27), where the per-call fixed costs amortise; same protocol (L2 flushed before
    each call, CUDA events around it)."""
    import dataclasses
    import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
    c = dataclasses.replace(wl.MAIN_BF16, T=65536)
    x, dy, w = wl.fwd_bwd_inputs(c, dev, 3)
    _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
    dx, dw = torch.empty_like(x), torch.empty(c.H, device=dev)
    ws = torch.empty(rmsn.rmsnorm_bwd_workspace_bytes(c.T, c.H, False, dev), device=dev,
                     dtype=torch.uint8)
    flush = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
    rd = flush.view(torch.float32)[: (FLUSH_BYTES // 2) // 4]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(warmup + steps):
        flush.zero_()
        rd.sum()
        if i >= warmup:
            ev[i - warmup][0].record()
        rmsn.rmsnorm_bwd(dy, x, w, rstd, True, False, ws, dx, dw)
        if i >= warmup:
            ev[i - warmup][1].record()
    torch.cuda.synchronize()
    us = statistics.mean(s.elapsed_time(e) for s, e in ev) * 1e3
    by = wl.bwd_bytes(c.T, c.H, c.x_dtype, c.w_dtype)
    return {"workload": "deterministic bwd, T=65536 H=4096 bf16", "us_mean": us,
            "gbs": by / (us * 1e-6) / 1e9, "frac": by / (us * 1e-6) / 1e9 / peak, "bytes": by}


def _mean_us(fn, steps: int, warmup: int, flush, rd) -> float:
    """Mean CUDA-event time of fn in us, L2 flushed (outside the events) before each call."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(warmup + steps):
        flush.zero_()
        rd.sum()
        if i >= warmup:
            ev[i - warmup][0].record()
        fn()
        if i >= warmup:
            ev[i - warmup][1].record()
    torch.cuda.synchronize()
    return statistics.mean(s.elapsed_time(e) for s, e in ev) * 1e3


def time_configs(dev, steps: int, warmup: int, peak: float):
    """Every other workload of the method, each alone, same protocol as the step's ops:
    T=64 H=256 fp32 forward and backward; the fused add+norm+E4M3 quant at T=2048 H=4096;
    the deterministic backward sweep (bf16 x/dy, fp32 w; T=65 is the small-T leg) and the
    compensated backward at T=262144 H=5120."""
    import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
    flush = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
    rd = flush.view(torch.float32)[: (FLUSH_BYTES // 2) // 4]
    out = {}

    def rec(name, us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"us_mean": us, "gbs": gbs, "frac": gbs / peak, "bytes": nbytes}

    def bwd_case(c, compensated, n):
        x, dy, w = wl.fwd_bwd_inputs(c, dev, 0)
        _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
        dx, dw = torch.empty_like(x), torch.empty(c.H, device=dev)
        ws = torch.empty(max(rmsn.rmsnorm_bwd_workspace_bytes(c.T, c.H, compensated, dev), 16),
                         device=dev, dtype=torch.uint8)
        us = _mean_us(lambda: rmsn.rmsnorm_bwd(dy, x, w, rstd, True, compensated, ws, dx, dw),
                      n, warmup, flush, rd)
        rec(c.name + ("_compensated" if compensated else ""), us,
            wl.bwd_bytes(c.T, c.H, c.x_dtype, c.w_dtype))

    c = wl.SMALL_FP32
    x, dy, w = wl.fwd_bwd_inputs(c, dev, 0)
    y, rstd = torch.empty_like(x), torch.empty(c.T, device=dev)
    rec(c.name + "_fwd", _mean_us(lambda: rmsn.rmsnorm_fwd(x, w, c.eps, y=y, rstd=rstd), steps,
                                  warmup, flush, rd), wl.fwd_bytes(c.T, c.H, c.x_dtype, c.w_dtype))
    bwd_case(c, False, steps)
    f = wl.FUSED_QUANT
    fx, fres, fw = wl.fused_inputs(f, dev, 0)
    q = torch.empty(f.T, f.H, device=dev, dtype=torch.uint8)
    sc = torch.empty(f.H // 128, wl.round_up(f.T, 4), device=dev)
    nm = torch.empty_like(fx)
    rec(f.name, _mean_us(lambda: rmsn.fused_add_rmsnorm_fp8_block_quant(fx, fres, fw, f.eps, q, sc,
                                                                        nm),
                         steps, warmup, flush, rd), wl.fused_quant_bytes(f.T, f.H))
    for c in wl.DET_SWEEP:
        if c.T > 65:
            bwd_case(c, False, max(5, min(steps, 20)))
            torch.cuda.empty_cache()
    bwd_case(wl.TWOSUM_LARGE, True, max(5, min(steps, 10)))
    torch.cuda.empty_cache()
    return out


def time_graph(step: Step, steps: int):
    """The step (three ops, each after an L2 flush) captured once in a CUDA graph and
    replayed: per-step time of the ops = (replays of [flush, op] x 3 - replays of the three
    flushes alone) / replays, with CUDA events around each batch of replays."""
    def ops():
        for op in Step.OPS:
            step.flush()
            step.run_op(op)

    def flushes():
        for _ in Step.OPS:
            step.flush()

    graphs = []
    for fn in (ops, flushes):
        fn()  # every one-time set-up happens before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    times = []
    for g in graphs:
        for _ in range(3):
            g.replay()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s.record()
        for _ in range(steps):
            g.replay()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e) / steps)
    return {"ms_per_step": times[0] - times[1], "replays": steps,
            "note": "ops of one step from CUDA-graph replay, flush time subtracted"}


def time_small_t(dev, steps: int, warmup: int):
    """The determinism sweep's T=65 rows (bf16 x/dy, fp32 w) through the deterministic
    backward, on the one-launch small-T route and on the strip route; mean us per call,
    L2 flushed before each call."""
    import dataclasses
    import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
    flush = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
    rd = flush.view(torch.float32)[: (FLUSH_BYTES // 2) // 4]
    old = rmsn.rmsn_small_t_max()
    out = {}
    try:
        for H in wl.DET_SWEEP_H:
            c = dataclasses.replace(wl.DET_SWEEP[0], T=65, H=H)
            x, dy, w = wl.fwd_bwd_inputs(c, dev, 0)
            _, rstd = rmsn.rmsnorm_fwd(x, w, c.eps)
            dx, dw = torch.empty_like(x), torch.empty(H, device=dev)
            ws = torch.empty(max(rmsn.rmsnorm_bwd_workspace_bytes(65, H, False, dev), 16),
                             device=dev, dtype=torch.uint8)
            row = {}
            for route, t_max in (("small_t", old if old > 0 else 256), ("strip", 0)):
                rmsn.rmsn_set_small_t_max(t_max)
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(steps)]
                for i in range(warmup + steps):
                    flush.zero_()
                    rd.sum()
                    if i >= warmup:
                        ev[i - warmup][0].record()
                    rmsn.rmsnorm_bwd(dy, x, w, rstd, True, False, ws, dx, dw)
                    if i >= warmup:
                        ev[i - warmup][1].record()
                torch.cuda.synchronize()
                row[route] = statistics.mean(s.elapsed_time(e) for s, e in ev) * 1e3
            out[f"T65_H{H}"] = {"us_small_t": row["small_t"], "us_strip": row["strip"],
                                "bytes": wl.bwd_bytes(65, H, c.x_dtype, c.w_dtype)}
    finally:
        rmsn.rmsn_set_small_t_max(old)
    return out


def time_e2e(step: Step, steps: int, warmup: int):
    """The same step through the public API from pinned host buffers: every step copies
    all its inputs host->device, runs the three ops and copies every output device->host.
    Steps are pipelined over two sets of device buffers and three streams (inputs of step
    i+1 and outputs of step i-1 move while step i computes); events order each set's
    reuse.  Returns (ms per step, H2D bytes per step, D2H bytes per step)."""
    dev = step.x.device
    in_names = ("x", "dy", "w", "fx", "fres", "fw")
    out_names = ("y", "rstd", "dx", "dw", "q", "scale", "normed", "fres")
    h_in = {k: getattr(step, k).cpu().pin_memory() for k in in_names}
    sets = []
    for _ in range(2):
        d = {k: torch.empty_like(getattr(step, k)) for k in set(in_names) | set(out_names)}
        d["ws"] = torch.empty_like(step.ws)
        d["h_out"] = {k: torch.empty(getattr(step, k).shape, dtype=getattr(step, k).dtype,
                                     pin_memory=True) for k in out_names}
        sets.append(d)
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in sets[0]["h_out"].values())
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    rmsn = step.rmsn

    def one(i, ev):
        d = sets[i % 2]
        e_free = ev.get(("out", i - 2))      # set reusable once step i-2's outputs left
        with torch.cuda.stream(s_in):
            if e_free is not None:
                s_in.wait_event(e_free)
            for k in in_names:
                d[k].copy_(h_in[k], non_blocking=True)
            ev[("in", i)] = torch.cuda.Event()
            ev[("in", i)].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev[("in", i)])
            rmsn.rmsnorm_fwd(d["x"], d["w"], step.eps, y=d["y"], rstd=d["rstd"])
            rmsn.rmsnorm_bwd(d["dy"], d["x"], d["w"], d["rstd"], True, False, d["ws"], d["dx"], d["dw"])
            rmsn.fused_add_rmsnorm_fp8_block_quant(d["fx"], d["fres"], d["fw"], step.eps, d["q"],
                                                   d["scale"], d["normed"])
            ev[("comp", i)] = torch.cuda.Event()
            ev[("comp", i)].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev[("comp", i)])
            for k in out_names:
                d["h_out"][k].copy_(d[k], non_blocking=True)
            ev[("out", i)] = torch.cuda.Event()
            ev[("out", i)].record(s_out)

    ev = {}
    for i in range(warmup):
        one(i, ev)
    torch.cuda.synchronize()
    ev = {}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        one(i, ev)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    t1.synchronize()
    del dev
    return t0.elapsed_time(t1) / steps, h2d, d2h


# --------------------------------------------------------------------- oracle legs
def oracle_sample_step(rows: int, seed: int = 0):
    """One pass of the FP64 oracle over `rows` rows of each op of the step (CPU)."""
    import dataclasses
    import oracle
    c = dataclasses.replace(wl.MAIN_BF16, T=rows)
    x, dy, w = wl.fwd_bwd_inputs(c, "cpu", seed)
    f = dataclasses.replace(wl.FUSED_QUANT_MAIN, T=rows)
    fx, fres, fw = wl.fused_inputs(f, "cpu", seed + 1)
    X, DY, W = wl.to_oracle(x), wl.to_oracle(dy), wl.to_oracle(w)
    FX, FR, FW = wl.to_oracle(fx), wl.to_oracle(fres), wl.to_oracle(fw)
    nbytes = (wl.fwd_bytes(rows, c.H, c.x_dtype, c.w_dtype) +
              wl.bwd_bytes(rows, c.H, c.x_dtype, c.w_dtype) + wl.fused_quant_bytes(rows, f.H))

    def run():
        _, r = oracle.rmsnorm_fwd(X, W, c.eps)
        oracle.rmsnorm_bwd(DY, X, W, r)
        _, n, _ = oracle.fused_add_rmsnorm(FX, FR, FW, f.eps)
        nb = oracle.bf16_round(n).reshape(n.shape)
        oracle.block_quant_e4m3(nb, wl.round_up(rows, 4))
    return run, nbytes


def cpu_baseline(budget_s: float = 12.0):
    import oracle
    rows = 256
    run, nbytes = oracle_sample_step(rows)
    run()  # builds/loads the oracle
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        run()
        n += 1
    dt = time.perf_counter() - t0
    return {"value": nbytes * n / dt / 1e9, "unit": UNIT, "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": f"{n} passes of the FP64 oracle over {rows} rows (H=4096) of each op of the "
                      f"step: fwd, bwd (dx and dW), fused add+norm+E4M3 quant; {dt:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    run, nbytes = oracle_sample_step(8)
    run()
    t = time.perf_counter()
    run()
    one = max(time.perf_counter() - t, 1e-4)
    budget = 90.0 / max(args.steps + args.warmup, 1)
    rows = int(max(8, min(2048, 8 * budget / one)))
    run, nbytes = oracle_sample_step(rows)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    sample = (f"each step: the FP64 oracle over {rows} of the T=8192 rows (H=4096) of each op: "
              f"fwd, bwd (dx and dW), fused add+norm+E4M3 quant")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; x, dy ~ N(0,1), residual ~ N(0,2), w = 1 + 0.1 N(0,1))",
        "config": {"workload": WORKLOAD, "T": T_MAIN, "H": H_MAIN, "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.default_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------- one op alone
ONLY_OPS = ("fwd", "bwd", "bwd_fast", "fused_quant", "fwd_residual", "bwd_residual")


def run_only(args):
    """One op at T x H bf16 (inputs seeded as in the step), --warmup + --launches calls,
    nothing else allocated: what a profiler captures when it needs one kernel at a time."""
    import dataclasses
    import rmsnorm_fwd_bwd_persistent_gb300 as rmsn
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T, H, op = args.T, args.H, args.only
    if op == "fused_quant":
        c = dataclasses.replace(wl.FUSED_QUANT_MAIN, T=T, H=H)
        x, res, w = wl.fused_inputs(c, dev, 1)
        q = torch.empty(T, H, device=dev, dtype=torch.uint8)
        sc = torch.empty(H // 128, wl.round_up(T, 4), device=dev)
        nm = torch.empty_like(x)
        fn = lambda: rmsn.fused_add_rmsnorm_fp8_block_quant(x, res, w, c.eps, q, sc, nm)  # noqa
    elif op in ("fwd_residual", "bwd_residual"):
        c = dataclasses.replace(wl.RESIDUAL_MAIN, T=T, H=H)
        x, res, dy, g, w = wl.residual_inputs(c, dev, 2)
        y, h = torch.empty_like(x), torch.empty_like(x)
        rstd = torch.empty(T, device=dev)
        rmsn.rmsnorm_fwd_residual(x, res, w, c.eps, y=y, h_new=h, rstd=rstd)
        if op == "fwd_residual":
            fn = lambda: rmsn.rmsnorm_fwd_residual(x, res, w, c.eps, y=y, h_new=h, rstd=rstd)  # noqa
        else:
            dxt, dw = torch.empty_like(x), torch.empty(H, device=dev)
            ws = torch.empty(rmsn.rmsnorm_bwd_workspace_bytes(T, H, False, dev), device=dev,
                             dtype=torch.uint8)
            fn = lambda: rmsn.rmsnorm_bwd_residual(dy, h, w, rstd, g, True, False, ws, dxt, dw)  # noqa
    else:
        c = dataclasses.replace(wl.MAIN_BF16, T=T, H=H)
        x, dy, w = wl.fwd_bwd_inputs(c, dev, 0)
        y, rstd = torch.empty_like(x), torch.empty(T, device=dev)
        rmsn.rmsnorm_fwd(x, w, c.eps, y=y, rstd=rstd)
        if op == "fwd":
            fn = lambda: rmsn.rmsnorm_fwd(x, w, c.eps, y=y, rstd=rstd)  # noqa
        else:
            det = op == "bwd"
            dx, dw = torch.empty_like(x), torch.empty(H, device=dev)
            ws = torch.empty(max(rmsn.rmsnorm_bwd_workspace_bytes(T, H, False, dev), 16),
                             device=dev, dtype=torch.uint8)
            fn = lambda: rmsn.rmsnorm_bwd(dy, x, w, rstd, det, False, ws, dx, dw)  # noqa
    for _ in range(args.warmup + args.launches):
        fn()
    torch.cuda.synchronize()
    st = rmsn.rmsn_device_status()
    print(json.dumps({"only": op, "T": T, "H": H, "calls": args.warmup + args.launches,
                      "device_status": st}), flush=True)
    return 0 if st == 0 else 1


# ------------------------------------------------------------------------------ main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=sorted(ONLY_OPS),
                    help="run one op alone at --T x --H (bf16) for --launches calls after "
                         "--warmup calls, allocating only its own buffers (a small process "
                         "for a profiler to capture); prints one line, times nothing")
    ap.add_argument("--T", type=int, default=T_MAIN)
    ap.add_argument("--H", type=int, default=H_MAIN)
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args(argv)
    if args.only:
        return run_only(args)
    args.warmup = max(args.warmup, 3)

    world, rank, local = _dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


def run_ours(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    step = Step(dev)
    peak, peak_src = measured_peak()

    clocks = ClockSampler(local)
    clocks.start()
    per_op, wall = time_steps(step, args.steps, args.warmup, world)
    clk = clocks.stop()

    op_ms = {op: statistics.mean(v) for op, v in per_op.items()}
    step_ms = sum(op_ms.values())
    step_bytes = sum(step.bytes.values())
    max_ms, total_bytes = aggregate(step_ms, step_bytes, world)
    value = total_bytes / (max_ms * 1e-3) / 1e9

    extra = time_extra(step, min(args.steps, 200), 3)
    small = time_small_t(dev, min(args.steps, 200), 3)
    graph = time_graph(step, min(args.steps, 200))
    long_strip = time_long_strip(dev, min(args.steps, 100), 3, peak)
    configs = time_configs(dev, min(args.steps, 100), 3, peak)
    e2e_ms, h2d, d2h = time_e2e(step, args.e2e_steps, 3)
    e2e_ms_max, _ = aggregate(e2e_ms, step_bytes, world)
    e2e_value = total_bytes / (e2e_ms_max * 1e-3) / 1e9

    ops = {}
    for op in Step.OPS:
        us = statistics.median(per_op[op]) * 1e3
        gbs = step.bytes[op] / (op_ms[op] * 1e-3) / 1e9
        ops[op] = {"us_median": us, "us_mean": op_ms[op] * 1e3, "gbs": gbs, "frac": gbs / peak,
                   "bytes": step.bytes[op], "launches": Step.LAUNCHES[op]}
    per_op = {op: {"us_mean": ops[op]["us_mean"], "gbs": ops[op]["gbs"], "frac": ops[op]["frac"],
                   "bytes": ops[op]["bytes"]} for op in Step.OPS}
    dom = max(Step.OPS, key=lambda o: op_ms[o])
    achieved = step.bytes[dom] / (op_ms[dom] * 1e-3) / 1e9
    traffic = recorded_traffic(dom)

    if rank != 0:
        return 0
    cpu = None if args.no_cpu_baseline or world > 1 else cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; x, dy ~ N(0,1), residual ~ N(0,2), w = 1 + 0.1 N(0,1))",
        "config": {"workload": WORKLOAD, "T": T_MAIN, "H": H_MAIN, "x_dtype": "bf16",
                   "w_dtype": "bf16", "accumulate": "fp32", "bwd_mode": "deterministic",
                   "l2": "flush (512 MiB write + 256 MiB read) ahead of each timed op, outside "
                         "the events",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "ops": ops,
        "roofline": {"bound": "hbm", "kernel": {"bwd": "rmsnorm_bwd (main strip kernel + dW "
                                                       "column reduce)",
                                                "fwd": "rmsnorm_fwd_kernel",
                                                "fused_quant": "fused_add_rmsnorm_fp8_kernel"}[dom],
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes": step.bytes[dom],
                     "peak_source": peak_src, "per_op": per_op},
        "ops_residual_variant": {k: dict(v, frac=v["gbs"] / peak) for k, v in extra.items()},
        "bwd_small_t_route": small,
        "bwd_long_strip": long_strip,
        "other_configs": configs,
        "graph_replay": dict(graph, eager_ms_per_step=max_ms,
                             gbs=step_bytes / (graph["ms_per_step"] * 1e-3) / 1e9),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_max},
        "gpu_launches": sum(Step.LAUNCHES[o] for o in Step.OPS) * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
