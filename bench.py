#!/usr/bin/env python3
"""Benchmark of the causal GQA prefill attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 5] [--impl ours|reference]

One step = one forward pass (the whole hot path: one kernel launch) over the
workload's synthetic bf16 inputs, already resident in device memory. L2 is
flushed (a 256 MiB device write) before every step, outside the timed
interval; each step is timed with CUDA events on the launching stream. The
default workload is the largest single-GPU layer, the long-context 36-head
shape (B=1, L=131072, n_q=36, n_kv=6, d_h=128; about 0.1 s per step, so the
default 20 steps make a timed window of about 2 s that the clock sampler
sees); the other workloads are chosen with --workload N (give short ones
more steps).

Under torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (units are independent; no collective on the data path): "scaling"
is weak and ``value`` is the total over ranks divided by the slowest rank's
time. Rank 0 prints one JSON line.

``--impl reference`` times the fp64 CPU oracle instead (rank 0 only), each
step a bounded sample of query rows of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal prefill attention TFLOP/s (2·n_q·d_h·L²) on 1 GB300; % of bf16 peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 * 10**6   # GB300 L2 capacity (nominal)
FALLBACK_BF16_TFLOPS = 1900.0


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


class Dist:
    def __init__(self):
        self.world = _env_int("WORLD_SIZE", 1)
        self.rank = _env_int("RANK", 0)
        self.local_rank = _env_int("LOCAL_RANK", 0)
        self.pg = None
        if self.world > 1:
            import datetime
            import torch.distributed as dist
            # host-side barrier / max only; BENCH_PG_TIMEOUT_S bounds how long a
            # rank waits for a peer that never arrives
            timeout = datetime.timedelta(seconds=_env_int("BENCH_PG_TIMEOUT_S", 1800))
            dist.init_process_group("gloo", timeout=timeout)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background.

    Only samples whose timestamp falls inside the timed window are summarised;
    if the window is too short to catch one, the samples of the warm-up plus
    the timed window are used and the summary says so.
    """

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t_start = None
        self.window = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        self.t_start = time.time()

    def mark_window(self, t0: float, t1: float):
        self.window = (t0, t1)

    def stop(self) -> dict:
        import datetime

        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
                except ValueError:
                    continue
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        span = "timed"
        sel = [r for r in rows if self.window and self.window[0] <= r[0] <= self.window[1]]
        if not sel:
            span = "warm-up + timed (timed window shorter than the 100 ms sampling period)"
            lo = self.t_start if self.t_start else rows[0][0]
            hi = self.window[1] if self.window else rows[-1][0]
            sel = [r for r in rows if lo <= r[0] <= hi] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(sel), "window": span,
                "power_w_median": statistics.median(r[3] for r in sel)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def kernel_source(w) -> str:
    """The CUDA source file that holds the kernels this workload times."""
    name = ("attn_decode.cu" if w.decode else "attn_backward.cu" if w.backward
            else "attn_prefill.cu")
    return os.path.join(ROOT, "causal_gqa_prefill_gb300", "csrc", name)


def kernel_source_hash(w) -> str:
    with open(kernel_source(w), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(w):
    """DRAM bytes per launch (per step for multi-launch steps) from the
    committed ncu summaries, if they were taken on the current source of this
    workload's kernels (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash(w)
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split("\t")
            if len(parts) >= 3 and parts[0] == str(w.number) and parts[1] == src:
                return float(parts[2])
    return None


def oracle_sample(w, q_host, k_host, v_host, rng, rows_per_chunk, seconds=None, chunks=None):
    """Times the fp64 oracle on random query rows; returns (flops, seconds, rows)."""
    import numpy as np
    import oracle

    flops = 0.0
    spent = 0.0
    nrows = 0
    done = 0
    while True:
        b = rng.integers(0, w.B, rows_per_chunk)
        h = rng.integers(0, w.n_q, rows_per_chunk)
        i = rng.integers(0, w.L, rows_per_chunk)
        rows = np.stack([b, h, i], axis=1)
        qv = q_host[b, i, h]
        t0 = time.perf_counter()
        oracle.attention_rows(qv, k_host, v_host, rows, causal=w.causal, scale=w.scale, n_q=w.n_q,
                              lq=w.L)
        spent += time.perf_counter() - t0
        keys = (i + w.offset + 1) if w.causal else np.full_like(i, w.keys)
        flops += float((4.0 * w.d_h * keys).sum())
        nrows += rows_per_chunk
        done += 1
        if seconds is not None and spent >= seconds:
            break
        if chunks is not None and done >= chunks:
            break
    return flops, spent, nrows


def oracle_backward_sample(w, q_host, k_host, v_host, do_host, rng, rows, seconds=None,
                           calls=None):
    """Times the fp64 backward oracle on causal prefixes of ``rows`` positions of
    random (batch, K/V head) groups; returns (flops, seconds, calls). A prefix
    of a causal problem is a complete smaller problem; its metric count is
    2.5 x the forward's 2*g*d_h*rows^2."""
    import oracle

    flops, spent, done = 0.0, 0.0, 0
    g = w.g
    while True:
        b = int(rng.integers(0, w.B))
        kvh = int(rng.integers(0, w.n_kv))
        hs = slice(kvh * g, (kvh + 1) * g)
        args = (q_host[b:b + 1, :rows, hs], k_host[b:b + 1, :rows, kvh:kvh + 1],
                v_host[b:b + 1, :rows, kvh:kvh + 1], do_host[b:b + 1, :rows, hs])
        t0 = time.perf_counter()
        oracle.attention_backward(*args, causal=w.causal, scale=w.scale)
        spent += time.perf_counter() - t0
        per = 2 * g * w.d_h * rows * rows * (1 if w.causal else 2)
        flops += per * 5 / 2
        done += 1
        if seconds is not None and spent >= seconds:
            break
        if calls is not None and done >= calls:
            break
    return flops, spent, done


def cpu_model() -> str:
    """The host CPU's model name (x86) or implementer and part codes (Arm)."""
    import platform

    try:
        with open("/proc/cpuinfo") as f:
            fields = [ln.split(":", 1) for ln in f.read().splitlines() if ":" in ln]
    except OSError:
        return platform.machine()
    kv = {}
    for k, v in fields:
        kv.setdefault(k.strip(), v.strip())
    if "model name" in kv:
        return kv["model name"]
    if "CPU part" in kv:
        return "%s, CPU implementer %s, part %s" % (
            platform.machine(), kv.get("CPU implementer", "?"), kv["CPU part"])
    return platform.machine()


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads") for p in threadpool_info() if p.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def host_inputs(w):
    """The workload's seeded inputs as host arrays (drawn on the GPU if one is
    present, exactly as the CUDA path sees them): float64, except the forward's
    Q in float32 (exact for bf16; the oracle upcasts the rows it reads)."""
    import numpy as np
    import torch
    from causal_gqa_prefill_gb300 import workloads as W

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    q, k, v = W.make_inputs(w, dev)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    if w.backward:
        return f(q), f(k), f(v), f(W.make_grad(w, dev))
    # the forward oracle reads Q only at the sampled rows (converted to float64
    # there); float32 holds the bf16 values exactly at half the host memory
    return q.float().cpu().numpy(), f(k), f(v)


def run_reference(args, w, dist):
    import numpy as np

    if dist.rank != 0:
        return 0
    if w.backward:
        return run_reference_backward(args, w)
    q, k, v = host_inputs(w)
    rng = np.random.default_rng(w.seed)
    # Size each step so that warm-up plus timed steps take about
    # --ref-seconds of oracle time in total (calibrated on one chunk).
    f, s, n = oracle_sample(w, q, k, v, rng, 64, chunks=1)
    per_row = s / n
    budget = args.ref_seconds / (args.steps + args.warmup)
    rows_per_step = int(min(args.ref_rows, max(8, budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, rng, rows_per_step, chunks=1)
    total_flops, total_s = 0.0, 0.0
    step_ms = []
    for _ in range(args.steps):
        f, s, _ = oracle_sample(w, q, k, v, rng, rows_per_step, chunks=1)
        total_flops += f
        total_s += s
        step_ms.append(s * 1e3)
    value = total_flops / total_s / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(step_ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(w.describe()),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{rows_per_step} random query rows per step of {w.name}; "
                                   "fp64 NumPy oracle on the host cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def backward_prefix_rows(w, q, k, v, do, rng, target_s):
    """Prefix length whose backward oracle call takes about ``target_s`` seconds."""
    rows = min(w.L, 512)
    while True:
        _, s, _ = oracle_backward_sample(w, q, k, v, do, rng, rows, calls=1)
        if s >= target_s or rows >= w.L:
            return rows
        rows = min(w.L, int(rows * max(1.25, min(4.0, (target_s / max(s, 1e-6)) ** 0.5))))
        rows = max(128, rows // 128 * 128)


def run_reference_backward(args, w):
    import numpy as np

    q, k, v, do = host_inputs(w)
    rng = np.random.default_rng(w.seed)
    budget = args.ref_seconds / (args.steps + args.warmup)
    rows = backward_prefix_rows(w, q, k, v, do, rng, budget)
    for _ in range(args.warmup):
        oracle_backward_sample(w, q, k, v, do, rng, rows, calls=1)
    total_flops, total_s, step_ms = 0.0, 0.0, []
    for _ in range(args.steps):
        f, s, _ = oracle_backward_sample(w, q, k, v, do, rng, rows, calls=1)
        total_flops += f
        total_s += s
        step_ms.append(s * 1e3)
    value = total_flops / total_s / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(step_ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(w.describe()),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"backward of the first {rows} positions of one random "
                                   f"(batch, K/V head) group per step of {w.name}; fp64 NumPy "
                                   "oracle on the host cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w, dist):
    import numpy as np
    import torch
    import causal_gqa_prefill_gb300 as cg
    from causal_gqa_prefill_gb300 import workloads as W

    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    q, k, v = W.make_inputs(w, dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.n_q, w.L), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    # A decode step reads a K/V cache several times the L2 size once, front to
    # back, so nothing of one step survives in L2 for the next: those steps
    # run without the flush, whose dirty lines would otherwise be written back
    # to HBM while the (bandwidth-bound) step reads.
    kv_bytes = 2 * w.B * w.keys * w.n_kv * w.d_h * 2
    flush_steps = not (w.decode and kv_bytes > 3 * L2_BYTES)
    stream = torch.cuda.current_stream(dev)
    sh = int(stream.cuda_stream)

    ws = None
    if w.decode:
        ws = torch.empty(cg.attn_decode_workspace_bytes(w.B, w.keys, w.n_q, w.n_kv, w.d_h),
                         dtype=torch.uint8, device=dev)

    def fwd(q_, k_, v_, o_, l_):
        # one call of the C entry point for this workload (chunked when Lk > L)
        if w.decode:
            st = cg.attn_decode_fwd(q_, k_, v_, o_, l_, ws, ws.numel(), w.B, w.keys, w.n_q,
                                    w.n_kv, w.d_h, w.scale, sh)
        elif w.dtype == "e4m3":
            st = cg.attn_prefill_fwd_fp8(q_, k_, v_, o_, l_, w.B, w.L, w.keys, w.n_q, w.n_kv,
                                         w.d_h, int(w.causal), w.scale, 1.0, 1.0, 1.0, sh)
        elif w.keys == w.L:
            st = cg.attn_prefill_fwd(q_, k_, v_, o_, l_, w.B, w.L, w.n_q, w.n_kv, w.d_h,
                                     int(w.causal), w.scale, sh)
        else:
            st = cg.attn_prefill_fwd_chunk(q_, k_, v_, o_, l_, w.B, w.L, w.keys, w.n_q, w.n_kv,
                                           w.d_h, int(w.causal), w.scale, sh)
        if st != cg.ATTN_OK:
            raise cg.AttnError(st, "attention forward")

    bwd_ws = dout = grads = None
    if w.backward:
        # the forward's outputs are inputs of the backward step: computed once here
        fwd(q, k, v, o, lse)
        dout = W.make_grad(w, dev)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        bwd_ws = torch.empty(cg.attn_prefill_bwd_workspace_bytes(w.B, w.L, w.n_q, w.n_kv, w.d_h),
                             dtype=torch.uint8, device=dev)

    def bwd(q_, k_, v_, o_, l_, do_, dq_, dk_, dv_):
        st = cg.attn_prefill_bwd(q_, k_, v_, o_, l_, do_, dq_, dk_, dv_, bwd_ws, bwd_ws.numel(),
                                 w.B, w.L, w.n_q, w.n_kv, w.d_h, int(w.causal), w.scale, sh)
        if st != cg.ATTN_OK:
            raise cg.AttnError(st, "attention backward")

    def step():
        if w.backward:
            bwd(q, k, v, o, lse, dout, *grads)
        else:
            fwd(q, k, v, o, lse)

    sampler = ClockSampler(dist.local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    for _ in range(args.warmup):
        if flush_steps:
            flush.zero_()
        step()
    st = cg.attn_device_check(sh)
    if st != cg.ATTN_OK:
        raise cg.AttnError(st, "warm-up")

    # Steps with an L2 flush are timed one by one (an event pair around each
    # step, the flush outside it). Steps without one run back to back and are
    # timed as one window of K steps: an event recorded between two steps would
    # stop the next step's launch from overlapping the previous one's end.
    window = not flush_steps
    n_ev = 1 if window else args.steps
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_ev)]
    dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    t_epoch0 = time.time()
    if window:
        events[0][0].record(stream)
        for _ in range(args.steps):
            step()
        events[0][1].record(stream)
    else:
        for s, e in events:
            flush.zero_()
            s.record(stream)
            step()
            e.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    t_wall = time.perf_counter() - t_wall
    sampler.mark_window(t_epoch0, time.time())
    clocks = sampler.stop()
    st = cg.attn_device_check(sh)
    if st != cg.ATTN_OK:
        raise cg.AttnError(st, "timed steps")
    step_ms = ([events[0][0].elapsed_time(events[0][1]) / args.steps] if window else
               [s.elapsed_time(e) for s, e in events])
    mean_ms = dist.max(statistics.mean(step_ms))
    flops = w.metric_flops()
    value = dist.world * flops / (mean_ms * 1e-3) / 1e12

    # End to end through the public API: every step copies its inputs from
    # pinned host memory and its outputs back to pinned host memory (forward:
    # Q, K, V in, O and LSE out; backward: Q, K, V, O, LSE, dO in, dQ, dK, dV
    # out). Copies run on their own streams with two device buffer sets, so
    # step i+1's upload and step i-1's download overlap step i's compute (a
    # pipelined loop); the timed region spans all K steps' copies.
    dev_in = [q, k, v] + ([o, lse, dout] if w.backward else [])
    dev_out = list(grads) if w.backward else [o, lse]
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out]
                for _ in range(3)]
    bufs_in = [dev_in, [t.clone() for t in dev_in]]
    bufs_out = [dev_out, [torch.empty_like(t) for t in dev_out]]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def call(b):
        if w.backward:
            bwd(*bufs_in[b], *bufs_out[b])
        else:
            fwd(*bufs_in[b], *bufs_out[b])

    # bf16 prefill (square or chunked) goes end to end through the host-buffer
    # C entry point: each call enqueues its own input copies, the forward and
    # the result copies; steps rotate over three streams and three staging
    # buffers so that one step's copies overlap its neighbours' work
    host_entry = not w.backward and not w.decode and w.dtype == "bf16"
    if host_entry:
        stage_bytes = cg.attn_prefill_host_staging_bytes(w.B, w.L, w.keys, w.n_q, w.n_kv, w.d_h)
        staging = [torch.empty(stage_bytes, dtype=torch.uint8, device=dev) for _ in range(3)]
        host_streams = [torch.cuda.Stream(dev) for _ in range(3)]

    def e2e_run_host(nsteps):
        ev0 = torch.cuda.Event()
        ev0.record(stream)
        for s_ in host_streams:
            s_.wait_event(ev0)
        for i in range(nsteps):
            b = i % 3
            st = cg.attn_prefill_fwd_host(*host_in, *host_out[b], staging[b], stage_bytes, w.B,
                                          w.L, w.keys, w.n_q, w.n_kv, w.d_h, int(w.causal),
                                          w.scale, host_streams[b])
            if st != cg.ATTN_OK:
                raise cg.AttnError(st, "attn_prefill_fwd_host")
        for s_ in host_streams:
            stream.wait_stream(s_)

    def e2e_run(nsteps):
        ev_up = [torch.cuda.Event() for _ in range(nsteps)]
        ev_fw = [torch.cuda.Event() for _ in range(nsteps)]
        ev_dn = [torch.cuda.Event() for _ in range(nsteps)]
        for i in range(nsteps):
            b = i % 2
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(ev_fw[i - 2])
                for d_, h_ in zip(bufs_in[b], host_in):
                    d_.copy_(h_, non_blocking=True)
                ev_up[i].record(s_up)
            stream.wait_event(ev_up[i])
            if i >= 2:
                stream.wait_event(ev_dn[i - 2])
            call(b)
            ev_fw[i].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_fw[i])
                for h_, d_ in zip(host_out[b], bufs_out[b]):
                    h_.copy_(d_, non_blocking=True)
                ev_dn[i].record(s_down)
        stream.wait_event(ev_dn[nsteps - 1])

    run_e2e = e2e_run_host if host_entry else e2e_run
    run_e2e(args.warmup)
    torch.cuda.synchronize()
    dist.barrier()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    run_e2e(args.steps)
    e_end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    e2e_ms = dist.max(e_start.elapsed_time(e_end) / args.steps)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    e2e_value = dist.world * flops / (e2e_ms * 1e-3) / 1e12

    # The host link alone, one cudaMemcpyAsync per tensor (the same pinned
    # buffers and sizes as a step): uploads alone, downloads alone, and both at
    # once on two streams. A pipelined step cannot beat max(kernel time, time
    # of both directions together).
    def timed_copies(up, down, reps=3):
        best = float("inf")
        for _ in range(reps):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            s_up.wait_event(t0)
            s_down.wait_event(t0)
            if up:
                with torch.cuda.stream(s_up):
                    for d_, h_ in zip(bufs_in[0], host_in):
                        d_.copy_(h_, non_blocking=True)
            if down:
                with torch.cuda.stream(s_down):
                    for h_, d_ in zip(host_out[0], bufs_out[0]):
                        h_.copy_(d_, non_blocking=True)
            stream.wait_stream(s_up)
            stream.wait_stream(s_down)
            t1.record(stream)
            torch.cuda.synchronize()
            best = min(best, t0.elapsed_time(t1))
        return best

    h2d_ms = timed_copies(True, False)
    d2h_ms = timed_copies(False, True)
    both_ms = timed_copies(True, True)
    kernel_ms = statistics.mean(step_ms)
    link = {"h2d_ms": h2d_ms, "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9,
            "d2h_ms": d2h_ms, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
            "both_ms": both_ms, "both_gbs": (h2d + d2h) / (both_ms * 1e-3) / 1e9,
            "bound_ms": max(kernel_ms, both_ms),
            "e2e_over_bound": e2e_ms / max(kernel_ms, both_ms),
            "how": "best of 3, pinned host buffers, one cudaMemcpyAsync per tensor; bound = "
                   "max(device step, uploads and downloads together)"}

    peaks, peak_src = measured_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    ratio = 1.0
    if w.dtype == "e4m3":
        # an e4m3 contraction: the measured bf16 rate times the nominal fp8/bf16 ratio (2)
        ratio = 2.0
        burst, sustained = 2.0 * burst, 2.0 * sustained
    # A timed window long enough to hit the power cap is a sustained run: it
    # is compared with the dense bf16 rate measured under the same cap.
    capped = "sw_power_cap" in clocks.get("reasons", []) and clocks.get("window") == "timed"
    peak = sustained if capped else burst
    peak_note = (f"bf16_tflops_sustained ({peak_src}; power cap active in the timed window)"
                 if capped else f"bf16_tflops ({peak_src}, burst)")
    if ratio != 1.0:
        peak_note += " x 2 (nominal e4m3/bf16 tensor-rate ratio)"
    achieved = flops / (statistics.mean(step_ms) * 1e-3) / 1e12
    traffic = recorded_traffic(w)
    if w.decode:
        # a decode step is bound by reading the K/V cache once: HBM roofline
        hbm = float(peaks.get("hbm_gbs", 6800.0))
        gbs = w.io_bytes() / (statistics.mean(step_ms) * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "peak_source": f"hbm_gbs ({peak_src})", "traffic": traffic,
                "algorithmic_bytes_per_launch": w.io_bytes()}
    elif w.backward:
        # the step is three launches (row statistics, dK/dV, dQ): timed as one
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "peak_source": peak_note, "traffic": traffic,
                "kernel": "backward step (rowdot + dkdv + dq launches), 2.5x forward FLOPs"}
    else:
        roof = None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if w.dtype == "e4m3" else "bf16",
        "data": "synthetic",
        "config": dict(w.describe(), parallelism=f"replicas x{dist.world}",
                       **({"flop_count": "2.5 x 2*n_q*d_h*L^2*B (five products of the forward's "
                                         "size against two)"} if w.backward else {}),
                       l2=("flushed before every step (256 MiB device write, outside the timed "
                           "interval)" if flush_steps else
                           "no flush: each step streams a K/V cache of %.0f MB, more than 3x "
                           "the 129 MB L2" % (kv_bytes / 1e6)),
                       timing=("one CUDA event pair around the K back-to-back steps" if window
                               else "a CUDA event pair around each step")),
        "pct_of_peak": 100.0 * achieved / peak,
        "pct_of_burst": 100.0 * achieved / burst,
        "pct_of_sustained": 100.0 * achieved / sustained,
        "gbs_io": w.io_bytes() / (statistics.mean(step_ms) * 1e-3) / 1e9,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "host_link": link,
                "note": ("through attn_prefill_fwd_host (copies in, forward, copies out in one "
                         "C call); pinned host buffers; steps rotate over three streams and "
                         "three staging buffers; no L2 flush") if host_entry else
                        ("pinned host buffers; uploads, compute and downloads on three streams, "
                         "two device buffer sets, no L2 flush")},
        "gpu_launches": args.steps * (2 if w.decode else 3 if w.backward else 1),
        "roofline": roof or {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                             "frac": achieved / peak, "peak_source": peak_note,
                             "traffic": traffic},
        "step_ms_min": None if window else min(step_ms),
        "step_ms_median": None if window else statistics.median(step_ms), "wall_s_timed": t_wall,
        "grid": cg.attn_prefill_grid_size(w.B, w.L, w.n_q, w.n_kv, w.d_h, w.causal),
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and w.backward:
        fq, fk, fv, fd = (t.float().cpu().numpy().astype(np.float64) for t in (q, k, v, dout))
        rng = np.random.default_rng(w.seed)
        rows = backward_prefix_rows(w, fq, fk, fv, fd, rng, args.cpu_seconds / 4)
        f, s, n = oracle_backward_sample(w, fq, fk, fv, fd, rng, rows, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": f / s / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"backward of the first {rows} positions of {n} random (batch, K/V head) "
                      f"groups of {w.name} (fp64 NumPy oracle), {s:.1f} s"}
    elif dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        fq = q.float().cpu().numpy()     # exact; the oracle upcasts the rows it reads
        fk, fv = (t.float().cpu().numpy().astype(np.float64) for t in (k, v))
        rng = np.random.default_rng(w.seed)
        f, s, n = oracle_sample(w, fq, fk, fv, rng, 256, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": f / s / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{n} random query rows of {w.name} (fp64 NumPy oracle), {s:.1f} s"}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=4096, help="upper bound on rows per step")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="oracle time budget of the whole reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from causal_gqa_prefill_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    dist = Dist()
    try:
        if args.impl == "reference":
            return run_reference(args, w, dist)
        return run_ours(args, w, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
