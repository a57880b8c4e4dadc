#!/usr/bin/env python
"""Benchmark of the fused chunked linear cross-entropy forward+backward.

One step = one lce_fused_fwd_bwd call (loss, lse, grad_X, grad_W) on the
Qwen3-8B head shape: N = 131072 rows (one sequence), H = 4096, V = 151936,
no bias, labels Zipf(1.1) with 5% ignored, chunk size chosen by the library.
Inputs are seeded synthetic draws of that shape (lce_inputs).

Prints one JSON line:
  value     tokens/s with the inputs already resident in HBM (device-timed,
            CUDA events on the call's stream, W warm-up steps, then K steps)
  e2e       the same metric with the inputs in pinned host memory: each step
            copies X, W, y to the device, runs the call, and copies loss, lse,
            grad_X and grad_W back, all inside the timed region
  roofline  the dominant kernel (by device time) against the measured tensor
            peak: algorithmic FLOPs per launch / mean launch duration, timed
            live with the library's per-kernel CUDA events in a second pass
            of the same K steps right after the timed region (the events add
            a bubble per launch, so the timed region itself runs without them)
  cpu_baseline  the FP64 CPU oracle on a bounded sample of the same rows
  clocks    nvidia-smi SM clock samples taken during the timed region

`--impl reference` times the FP64 CPU oracle instead, on the host cores,
each step a bounded sample of the same workload (the oracle is the only
reference this method has).  With several GPUs (torchrun), every rank runs
its own replica of the whole workload; value is the sum over ranks of rows
processed divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

# The oracle's BLAS uses every host core; must be set before numpy loads.
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s fused LCE fwd+bwd (Qwen3-8B head) and % of BF16 tensor peak"
WORKLOAD = "qwen3-8b-head-N131072-H4096-V151936"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# DRAM bytes (read + write) of one full-size launch of the dominant GEMM role
# on this workload.  ncu multi-metric captures stay on small cases, so the
# figure is scaled: the forward logits launch of an 8192-row chunk (keeping E
# and rescaling the previous chunk's) was captured at V = 16384, 32768 and
# 65536, its traffic grew linearly in V (least squares: 84,573 bytes per
# vocabulary row, minus 0.165 GB), and the line gives 12.69 GB at V = 151936
# (11.40-11.54 GB in three earlier captures of the same kernels: DRAM reads
# vary from run to run with what L2 holds).
# The figure holds only for the sources it was captured with:
# DRAM_BYTES_SOURCES lists the files that decide a GEMM launch's traffic and
# DRAM_BYTES_DIGEST their SHA-256 at capture time.  When the digest no longer
# matches, roofline.traffic is reported as null.
DRAM_BYTES_PER_LAUNCH = {"logits_lse": 12.69e9, "grad_w": None, "grad_x": None, "recomputed_logits_softmax": None}
DRAM_BYTES_CHUNK_ROWS = 8192  # the chunk size those launches ran with
DRAM_BYTES_FORM = "pair"  # and their GEMM form
DRAM_BYTES_SOURCES = ["csrc/lce_gemm.cuh", "csrc/lce_gemm_pair.cuh", "csrc/lce_internal.cuh", "csrc/lce_ptx.cuh",
                      "csrc/lce_api.cu", "csrc/lce_gemm_logits.cu", "csrc/lce_gemm_grads.cu",
                      "csrc/lce_gemm_gradx_wide.cu"]
DRAM_BYTES_DIGEST = "a6e09c7325ab60d9"


def gemm_source_digest() -> str:
    h = hashlib.sha256()
    for rel in DRAM_BYTES_SOURCES:
        with open(os.path.join(ROOT, "lm_head_linear_chunked_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def role_bytes(H: int, V: int, rows, valid, overlapped: bool) -> dict:
    """Algorithmic DRAM bytes per step of each GEMM role of the fused call:
    each operand read once, each result written once, per chunk.  rows[c] and
    valid[c]: chunk c's rows and valid rows (the backward runs on valid rows
    only).
      logits_lse: X_c, W, E of the valid rows written; with the overlapped
        schedule also the previous chunk's E read and P written (its side job;
        the last chunk's rescale is a separate kernel).
      grad_x: P and W16 read, grad_X rows written (nothing for a chunk without
        valid rows).
      grad_w: P and X16 read; the FP32 accumulator written (first chunk), read
        and written (later chunks), plus its bf16 cast written (last chunk); a
        chunk between the first and the last without valid rows adds nothing."""
    n = len(rows)
    fwd = sum(2 * r * H + 2 * V * H + 2 * v * V for r, v in zip(rows, valid))
    if overlapped:
        fwd += sum(4 * v * V for v in valid[:-1])
    gx = sum(2 * v * V + 2 * V * H + 2 * v * H for v in valid if v > 0)
    gw = 0
    for c, v in enumerate(valid):
        first, last = c == 0, c == n - 1
        if v == 0 and not first and not last:
            continue
        acc = (4 if first else 8) * V * H + (2 * V * H if last else 0)
        gw += 2 * v * V + 2 * v * H + acc
    return {"logits_lse": float(fwd), "grad_x": float(gx), "grad_w": float(gw)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(seconds: float) -> float:
    """The slowest rank's time (every rank gets it); the local time alone
    without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return seconds
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(rows_per_rank: int, world: int, slowest_seconds: float) -> float:
    """Whole-job rate of independent replicas: every rank's rows over the slowest rank's time."""
    return world * rows_per_rank / slowest_seconds


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(w, rows: int, X=None, W_bits=None, y=None):
    """Runs the FP64 oracle, as it stands, on the first `rows` rows of the
    workload (all of W): returns (seconds, rows)."""
    import numpy as np

    import lce_inputs as L
    import oracle

    if W_bits is None:
        W_bits = np.empty((w.V, w.H), dtype=np.uint16)
        L.w_into(w, W_bits.ctypes.data)
    if y is None:
        y = L.labels(w)
    b_bits = None
    if w.has_bias:
        b_bits = np.empty(w.V, dtype=np.uint16)
        L.b_into(w, b_bits.ctypes.data)
    Xr = L.x_rows(w, np.arange(rows))
    t0 = time.perf_counter()
    oracle.fused(Xr, W_bits, b_bits, y[:rows])
    return time.perf_counter() - t0, rows


def cpu_baseline(w, rows=256):
    import numpy as np

    import lce_inputs as L
    W_bits = np.empty((w.V, w.H), dtype=np.uint16)
    L.w_into(w, W_bits.ctypes.data)
    y = L.labels(w)
    t, n = oracle_sample(w, rows, W_bits=W_bits, y=y)
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    out = {"value": n / t, "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "sample": f"FP64 oracle forward+backward (numpy, float64 BLAS) on the first {n} of {w.N} rows "
                     f"with all of W [{w.V}x{w.H}], {t:.1f} s; tokens/s extrapolated from that sample",
           "host_cores": os.cpu_count()}
    one = cpu_baseline_one_thread(w, max(1, rows // 16))
    if one is not None:
        out["one_thread"] = one
    return out


def cpu_baseline_one_thread(w, rows):
    """The same oracle on one host thread (BLAS limited to one thread), in a
    fresh interpreter so the limit takes effect: {"value", "rows", "seconds"}."""
    import subprocess
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, json; sys.path.insert(0, %r); import bench, lce_inputs as L; "
            "w = [x for x in L.WORKLOADS if x.name == %r][0]; t, n = bench.oracle_sample(w, %d); "
            "print(json.dumps({'seconds': t, 'rows': n}))") % (ROOT, w.name, rows)
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        d = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return {"value": d["rows"] / d["seconds"], "unit": "tokens/s", "rows": d["rows"], "seconds": d["seconds"]}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import lce_inputs as L
    W_bits = np.empty((w.V, w.H), dtype=np.uint16)
    L.w_into(w, W_bits.ctypes.data)
    y = L.labels(w)
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(w, rows, W_bits=W_bits, y=y)
    times = []
    for _ in range(args.steps):
        t, _n = oracle_sample(w, rows, W_bits=W_bits, y=y)
        times.append(t)
    t_step = sum(times) / len(times)
    value = rows / t_step
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "N": w.N, "H": w.H, "V": w.V, "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: FP64 oracle forward+backward on the first {rows} of {w.N} rows "
                                   f"with all of W"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        for r in rows:
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"],
                                 r[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "power_w_mean": statistics.mean(pw) if pw else None,
                "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our library

def run_ours(args, w):
    import numpy as np
    import torch

    import __graft_entry__
    import lce_inputs as L
    import lm_head_linear_chunked_gb300 as lce

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    prev_form = lce.lce_set_gemm_form(args.gemm_form or "single")
    if not args.gemm_form:
        lce.lce_set_gemm_form(prev_form)  # keep the library's default
    gemm_form = args.gemm_form or {lce.GEMM_SINGLE: "single", lce.GEMM_PAIR: "pair"}[prev_form]
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    __graft_entry__.build()

    N, H, V = w.N, w.H, w.V
    chunk = args.chunk_rows if args.chunk_rows is not None else w.chunk_rows
    # seeded inputs, generated on the host into pinned memory
    Xh = torch.empty((N, H), dtype=torch.bfloat16, pin_memory=True)
    Wh = torch.empty((V, H), dtype=torch.bfloat16, pin_memory=True)
    L.x_into(w, Xh.data_ptr())
    L.w_into(w, Wh.data_ptr())
    yh = torch.from_numpy(L.labels(w)).pin_memory()
    bh = None
    if w.has_bias:
        bh = torch.empty(V, dtype=torch.bfloat16, pin_memory=True)
        L.b_into(w, bh.data_ptr())
    has_b = bh is not None

    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        X = Xh.to(dev, non_blocking=True)
        W = Wh.to(dev, non_blocking=True)
        y = yh.to(dev, non_blocking=True)
        b = bh.to(dev, non_blocking=True) if has_b else None
        nws = lce.lce_workspace_size(N, H, V, chunk, has_b, lce.WS_FUSED)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
        gX = torch.empty_like(X)
        gW = torch.empty_like(W)
        gW_acc = torch.empty((V, H), dtype=torch.float32, device=dev)
        gb = torch.empty(V, dtype=torch.bfloat16, device=dev) if has_b else None
        gb_acc = torch.empty(V, dtype=torch.float32, device=dev) if has_b else None
    s.synchronize()

    def step():
        lce.lce_fused_fwd_bwd(N, H, V, X, W, b, y, -100, chunk, 1.0, None, loss, lse, n_valid, gX, gW, gb,
                              gW_acc, gb_acc, ws, nws, s)

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    st = lce.lce_check_status(ws, s)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {lce.STATUS[st]}")

    # ---- device-resident timing: the timed region, K steps with nothing but
    # the two bracketing events on the call's stream
    barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(s)
        for _ in range(args.steps):
            step()
        ev1.record(s)
        torch.cuda.synchronize(dev)
    barrier()
    clocks = clk.summary()
    t_step = ev0.elapsed_time(ev1) / 1e3 / args.steps
    st = lce.lce_check_status(ws, s)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {lce.STATUS[st]}")
    t_step = max_over_ranks(t_step)

    # ---- the same K steps again with every kernel bracketed by CUDA events
    # (the library's profiler), for the per-kernel times and the roofline.
    # The events add a pipeline bubble per launch, which shows on small
    # problems as a longer step; the kernels' own durations are unchanged.
    barrier()
    torch.cuda.synchronize(dev)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    lce.lce_profile_begin()
    p0.record(s)
    for _ in range(args.steps):
        step()
    p1.record(s)
    torch.cuda.synchronize(dev)
    prof = lce.lce_profile_end()
    barrier()
    t_prof = max_over_ranks(p0.elapsed_time(p1) / 1e3 / args.steps)

    # ---- the forward and the backward entry points on their own (2NHV and 6NHV)
    split = None
    if not args.no_split:
        nws_f = lce.lce_workspace_size(N, H, V, chunk, has_b, lce.WS_FORWARD)
        nws_b = lce.lce_workspace_size(N, H, V, chunk, has_b, lce.WS_BACKWARD)
        ws_f = torch.empty(nws_f, dtype=torch.uint8, device=dev)
        ws_b = torch.empty(nws_b, dtype=torch.uint8, device=dev)

        def fwd():
            lce.lce_forward(N, H, V, X, W, b, y, -100, chunk, loss, lse, n_valid, ws_f, nws_f, s)

        def bwd():
            lce.lce_backward(N, H, V, X, W, b, y, -100, chunk, lse, 1.0, None, gX, gW, gb, gW_acc, gb_acc,
                             ws_b, nws_b, s)

        split = {}
        nv_rows = int((yh != -100).sum().item())  # the gradient products run over the valid rows only
        for name, fn, fl in (("forward", fwd, 2.0 * N * H * V), ("backward", bwd, 2.0 * (N + 2 * nv_rows) * H * V)):
            for _ in range(2):
                fn()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(s)
            for _ in range(args.steps):
                fn()
            a1.record(s)
            torch.cuda.synchronize(dev)
            t = a0.elapsed_time(a1) / 1e3 / args.steps
            split[name] = {"ms": 1e3 * t, "tokens_per_s": N / t, "tflops": fl / t / 1e12}
        st = lce.lce_check_status(ws_b, s)
        if st != 0:
            raise RuntimeError(f"device status after lce_backward: {lce.STATUS[st]}")
        del ws_f, ws_b

    # ---- end to end: host buffers, copies inside the timed region.  Two sets
    # of device buffers: step k+1's inputs are copied in while step k
    # computes, and step k's results are copied out while step k+1 computes.
    e2e = None
    if not args.no_e2e:
        def device_set():
            return {"X": torch.empty_like(X), "W": torch.empty_like(W), "y": torch.empty_like(y),
                    "loss": torch.empty_like(loss), "lse": torch.empty_like(lse), "n_valid": torch.empty_like(n_valid),
                    "gX": torch.empty_like(gX), "gW": torch.empty_like(gW), "gW_acc": torch.empty_like(gW_acc),
                    "b": torch.empty_like(b) if has_b else None, "gb": torch.empty_like(gb) if has_b else None,
                    "gb_acc": torch.empty_like(gb_acc) if has_b else None, "ws": torch.empty_like(ws)}

        def host_set():
            return {"loss": torch.empty(1, dtype=torch.float32, pin_memory=True),
                    "lse": torch.empty(N, dtype=torch.float32, pin_memory=True),
                    "gX": torch.empty((N, H), dtype=torch.bfloat16, pin_memory=True),
                    "gW": torch.empty((V, H), dtype=torch.bfloat16, pin_memory=True),
                    "gb": torch.empty(V, dtype=torch.bfloat16, pin_memory=True) if has_b else None}

        dsets = [device_set(), device_set()]
        hsets = [host_set(), host_set()]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def run_steps(k_steps, t0=None, t1=None):
            comp_done, out_done = [], []
            if t0 is not None:
                t0.record(s_in)
            for k in range(k_steps):
                d, h = dsets[k % 2], hsets[k % 2]
                if k >= 2:
                    s_in.wait_event(comp_done[k - 2])       # set's inputs no longer read
                with torch.cuda.stream(s_in):
                    d["X"].copy_(Xh, non_blocking=True)
                    d["W"].copy_(Wh, non_blocking=True)
                    d["y"].copy_(yh, non_blocking=True)
                    if has_b:
                        d["b"].copy_(bh, non_blocking=True)
                    in_done = torch.cuda.Event()
                    in_done.record(s_in)
                s.wait_event(in_done)
                if k >= 2:
                    s.wait_event(out_done[k - 2])           # set's results already copied out
                lce.lce_fused_fwd_bwd(N, H, V, d["X"], d["W"], d["b"], d["y"], -100, chunk, 1.0, None, d["loss"],
                                      d["lse"], d["n_valid"], d["gX"], d["gW"], d["gb"], d["gW_acc"], d["gb_acc"],
                                      d["ws"], nws, s)
                ev = torch.cuda.Event()
                ev.record(s)
                comp_done.append(ev)
                s_out.wait_event(ev)
                with torch.cuda.stream(s_out):
                    h["loss"].copy_(d["loss"], non_blocking=True)
                    h["lse"].copy_(d["lse"], non_blocking=True)
                    h["gX"].copy_(d["gX"], non_blocking=True)
                    h["gW"].copy_(d["gW"], non_blocking=True)
                    if has_b:
                        h["gb"].copy_(d["gb"], non_blocking=True)
                    ev2 = torch.cuda.Event()
                    ev2.record(s_out)
                out_done.append(ev2)
            if t1 is not None:
                t1.record(s_out)

        run_steps(2)
        torch.cuda.synchronize(dev)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        run_steps(args.steps, e0, e1)
        torch.cuda.synchronize(dev)
        barrier()
        for d in dsets:
            st = lce.lce_check_status(d["ws"], s)
            if st != 0:
                raise RuntimeError(f"device status after end-to-end steps: {lce.STATUS[st]}")
        t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps)
        h2d = Xh.numel() * 2 + Wh.numel() * 2 + yh.numel() * 8 + (V * 2 if has_b else 0)
        d2h = 4 + N * 4 + N * H * 2 + V * H * 2 + (V * 2 if has_b else 0)
        e2e = {"value": replica_rate(N, ws_n, t_e2e), "unit": "tokens/s", "ms_per_step": 1e3 * t_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "lce_fused_fwd_bwd via the Python binding; inputs copied from pinned host memory and "
                       "loss, lse, grad_X, grad_W copied back every step, double-buffered so a step's copies "
                       "overlap its neighbours' compute"}
        loss_v = float(hsets[(args.steps - 1) % 2]["loss"].item())
    else:
        loss_v = float(loss.item())

    if rank != 0:
        if ws_n > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    flops = w.flops_fused()
    tflops = flops / t_step / 1e12
    C = lce.lce_chunk_rows(N, H, V, chunk)
    n_chunks = -(-N // C)
    # dominant kernel: the GEMM role with the most device time
    gemm_kinds = ["logits_lse", "recomputed_logits_softmax", "grad_x", "grad_w"]
    dom = max(gemm_kinds, key=lambda k: prof[k][0])
    # the fused call's schedule: the forward rescales the previous chunk (no p_rescale launches but the last)
    overlapped = nws > lce.lce_workspace_size(N, H, V, chunk, has_b, lce.WS_FUSED_MIN)
    # FLOPs each role executes per step: the logits passes run over all N rows
    # (lse is written for every row), the gradient products over the valid rows
    # only (ignored rows are compacted away)
    n_valid_rows = int((yh != -100).sum().item())
    role_flops = {k: 2.0 * (n_valid_rows if k in ("grad_x", "grad_w") else N) * H * V for k in gemm_kinds}
    executed = sum(role_flops[k] for k in gemm_kinds if prof[k][1] > 0)
    dom_ms, dom_n = prof[dom]
    # each GEMM role runs once per chunk; a split grad_X product adds its
    # reduction kernel to the role, so time is counted per chunk, not per launch
    role_chunks = args.steps * n_chunks
    dom_flops_per_launch = role_flops[dom] / n_chunks
    dom_tflops = dom_flops_per_launch / (dom_ms / role_chunks / 1e3) / 1e12
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    total_launches = sum(v[1] for v in prof.values())
    # Which peak bounds each role: the time its FLOPs take at the sustained
    # tensor peak against the time its algorithmic bytes take at the measured
    # copy bandwidth (small chunks make grad_W, for one, bandwidth-bound).
    chunk_rows = [min(C, N - r0) for r0 in range(0, N, C)]
    yv = (yh != -100)
    chunk_valid = [int(yv[r0:r0 + C].sum().item()) for r0 in range(0, N, C)]
    rbytes = role_bytes(H, V, chunk_rows, chunk_valid, overlapped)
    role_bound = {k: ("hbm" if rbytes[k] / (hbm * 1e9) > role_flops[k] / (sustained * 1e12) else "tensor")
                  for k in rbytes}
    dom_bound = role_bound.get(dom, "tensor")
    dom_gbs = rbytes.get(dom, 0.0) / (dom_ms / args.steps / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": replica_rate(N, ws_n, t_step), "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "N": N, "H": H, "V": V, "chunk_rows": C, "chunks": n_chunks,
                   "gemm_form": gemm_form,
                   "bias": has_b, "ignored_rows": int((yh == -100).sum().item()),
                   "l2": f"inputs larger than L2 (X {N * H * 2 / 1e9:.2f} GB, W {V * H * 2 / 1e9:.2f} GB; L2 129 MB)",
                   "parallelism": "replicas" if ws_n > 1 else "single GPU"},
        "tflops": tflops,
        "flops_per_step": flops,
        "flops_note": "8*N*H*V counted (forward, recomputed logits, grad_X, grad_W); the fused call skips the "
                      "recompute, see tflops_executed",
        "tflops_executed": executed / t_step / 1e12,
        "frac_of_peak": {"measured_burst_bf16": tflops / burst, "measured_sustained_bf16": tflops / sustained,
                         "nominal_dense_bf16_2250": tflops / 2250.0, "peak_source": peak_src,
                         "flops": "8*N*H*V counted; above 1 because the recompute is not executed"},
        "frac_of_peak_executed": {"measured_burst_bf16": executed / t_step / 1e12 / burst,
                                  "measured_sustained_bf16": executed / t_step / 1e12 / sustained,
                                  "nominal_dense_bf16_2250": executed / t_step / 1e12 / 2250.0,
                                  "peak_source": peak_src,
                                  "flops": "tensor-core FLOPs the step executes: 2*N*H*V for the logits pass and "
                                           "2*n_valid*H*V for each gradient product, which run over the valid rows "
                                           "only (2*N*H*V + 4*n_valid*H*V in the fused call)"},
        "workspace_note": "the fused call keeps each chunk's fp16 exponentials in the workspace instead of "
                          "recomputing the logits tile in the backward",
        "roofline": {"bound": "tensor", "achieved": dom_tflops, "peak": sustained, "unit": "TFLOP/s",
                     "frac": dom_tflops / sustained, "peak_kind": f"{peak_src} sustained bf16",
                     "traffic": DRAM_BYTES_PER_LAUNCH.get(dom) if args.workload == WORKLOAD and not args.shape
                     and C == DRAM_BYTES_CHUNK_ROWS and gemm_form == DRAM_BYTES_FORM
                     and gemm_source_digest() == DRAM_BYTES_DIGEST else None,
                     "traffic_source": f"ncu dram__bytes_read.sum + dram__bytes_write.sum of this launch at V = 16384, "
                                       f"32768 and 65536 (8192-row chunks, H = 4096), scaled linearly in V to the full "
                                       f"vocabulary; sources {DRAM_BYTES_DIGEST} at capture, these sources "
                                       f"{gemm_source_digest()}",
                     "algorithmic_bytes": (2.0 * C * H + 2.0 * V * H + 2.0 * C * V + 4.0 * C * V
                                           if dom == "logits_lse" and overlapped else None),
                     "kernel": f"{'gemm_pair_kernel' if gemm_form == 'pair' else 'gemm_kernel'} ({dom})" + (
                         ", which also turns the previous chunk's kept exponentials into the softmax (4*C*V bytes) "
                         "with its epilogue warps" if dom == "logits_lse" and overlapped else ""),
                     "roles": {k: {"tflops": role_flops[k] / n_chunks / (prof[k][0] / role_chunks / 1e3) / 1e12,
                                   "frac": role_flops[k] / n_chunks / (prof[k][0] / role_chunks / 1e3) / 1e12 /
                                   sustained, "ms_per_chunk": prof[k][0] / role_chunks,
                                   "launches_per_chunk": prof[k][1] / role_chunks}
                               for k in gemm_kinds if prof[k][1] > 0},
                     "roles_note": "per chunk: the role's GEMM launch and, for grad_x, the kernel that adds the "
                                   "partial sums of a product split over the vocabulary",
                     "flops_per_launch": dom_flops_per_launch, "launches": dom_n,
                     "mean_launch_ms": dom_ms / role_chunks,
                     "peak_source": f"{peak_src} sustained bf16 (fp16 operands run at the bf16 rate)"},
        "kernels_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
        "profiled_pass": {"value": replica_rate(N, ws_n, t_prof), "ms_per_step": 1e3 * t_prof,
                          "note": "the same K steps again with every kernel bracketed by CUDA events; "
                                  "kernels_ms_per_step, roofline and gpu_launches come from this pass"},
        "gpu_launches": total_launches,
        "loss": loss_v,
        "workspace_bytes": nws,
        "logits_bytes_avoided": N * V * 2,
        "clocks": clocks,
        # energy of one step from the power samples of the timed region (board power as nvidia-smi reports it);
        # under the power cap, time per step follows energy per step
        "joules_per_step": clocks["power_w_mean"] * t_step if clocks.get("power_w_mean") else None,
        "e2e": e2e,
        "separate_entry_points": split,
    }
    for k, r in line["roofline"]["roles"].items():  # each role's bound and its bandwidth figure
        if k in rbytes:
            r["bound"] = role_bound[k]
            r["gbs"] = rbytes[k] / (prof[k][0] / args.steps / 1e3) / 1e9
            r["frac_hbm"] = r["gbs"] / hbm
    if dom_bound == "hbm":
        # the dominant role is bandwidth-bound (e.g. grad_W at small chunks): the
        # roofline is its algorithmic bytes against the measured copy rate, and the
        # tensor figures stay beside it
        tensor_view = line["roofline"]
        line["roofline"] = {
            "bound": "hbm", "achieved": dom_gbs, "peak": hbm, "unit": "GB/s", "frac": dom_gbs / hbm,
            "peak_kind": f"{peak_src} HBM copy rate",
            "algorithmic_bytes": rbytes[dom] / n_chunks,
            "algorithmic_bytes_note": "per launch: the mean over the step's chunks of the operands read once, the "
                                      "results written once, and the FP32 grad_W accumulator read and written per "
                                      "chunk",
            "traffic": None, "traffic_source": "no ncu capture for this workload's launches",
            "kernel": tensor_view["kernel"], "roles": tensor_view.pop("roles"),
            "tensor_view": tensor_view,
        }
    if not args.no_cpu_baseline and ws_n == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_rows)
    print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_gemm(args):
    """Times the library's bare tensor-core GEMM (lce_debug_gemm) on one shape."""
    import torch

    import __graft_entry__
    import lm_head_linear_chunked_gb300 as lce
    __graft_entry__.build()
    if args.gemm_form:
        lce.lce_set_gemm_form(args.gemm_form)
    M, N, K, layout = (int(x) for x in args.gemm.split(","))
    torch.manual_seed(0)
    a_shape = (M, K) if layout in (0, 1) else (K, M)
    b_shape = (N, K) if layout == 0 else (K, N)
    A = torch.randn(a_shape, device="cuda").to(torch.bfloat16)
    B = torch.randn(b_shape, device="cuda").to(torch.bfloat16)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(args.warmup):
        lce.lce_debug_gemm(layout, M, N, K, A, B, D, ws, ws.numel(), s)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.steps):
        lce.lce_debug_gemm(layout, M, N, K, A, B, D, ws, ws.numel(), s)
    e1.record(s)
    torch.cuda.synchronize()
    assert lce.lce_check_status(ws, s) == 0
    t = e0.elapsed_time(e1) / 1e3 / args.steps
    print(json.dumps({"gemm": [M, N, K, layout], "ms": 1e3 * t, "tflops": 2.0 * M * N * K / t / 1e12}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--shape", default=None,
                    help="N,H,V: a custom shape with the same input recipe (for profiling small cases)")
    ap.add_argument("--chunk-rows", type=int, default=None)
    ap.add_argument("--cpu-rows", type=int, default=256, help="rows of the CPU-oracle baseline sample")
    ap.add_argument("--ref-rows", type=int, default=32, help="rows per step of --impl reference")
    ap.add_argument("--gemm", default=None, help="M,N,K,layout: time the bare GEMM core instead")
    ap.add_argument("--gemm-form", choices=["single", "pair"], default=None,
                    help="tensor-core GEMM form (default: the library's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-split", action="store_true", help="skip timing lce_forward and lce_backward alone")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    import lce_inputs as L
    w = L.BY_NAME[args.workload]
    if args.shape:
        n, h, v = (int(x) for x in args.shape.split(","))
        w = L.Workload(f"custom-N{n}-H{h}-V{v}", n, 1, h, v, None, "random", 0.05, 0, 7)
    if args.gemm:
        run_gemm(args)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
