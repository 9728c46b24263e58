"""Benchmark of the attention hot path: one step = fa_fwd + fa_bwd over one
batch of synthetic input, at the slides' largest forward-sweep size with
d = 128 (B=8, H=16, N=8192, non-causal, scale 1/sqrt(d)).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  FLOPs follow the pages' count: forward
4*B*H*N^2*d (two S x S x d matmuls per head, cs2680 Lecture 9 sec. 9.2),
halved when causal; backward 2.5x the forward.  ``value`` is whole-job
TFLOPS with the inputs resident in HBM; ``e2e`` is the same metric with each
step's inputs copied from pinned host memory and all its outputs copied back
inside the timed region, pipelined as a user streaming batches would run it
(step k+1's upload and step k-1's download overlap step k's kernels).
Every rank (one per GPU, launched by torchrun) runs its own independent
batch (weak scaling, no data-path collective); timing is the max over
ranks, exchanged over gloo.  Each of the headline's inputs is larger than
L2; for workloads whose inputs fit in L2 (``--workload``), L2 is flushed
before every timed step outside that step's CUDA events.

``--impl reference`` times the fp64 CPU oracle (the reference arm of this
build) on a bounded sample of the same workload on the host cores.

The default (N = 1) line also reports ``n_sweep_d128``: forward and backward
TFLOPS at N = 1K, 2K, 4K and 16K (B=8, H=16, d=128), measured after the timed
region (``--no-sweep`` skips it).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS (bf16, d=128, N=1K-16K) and % of GB300 bf16 tensor peak"
UNIT = "TFLOPS"
WORKLOAD = dict(name="sweep_N8192_d128", B=8, H=16, N=8192, d=128, causal=False)
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
FLUSH_NOTE = ("inputs smaller than L2 (each of Q, K, V, dO is %d MiB): L2 flushed before every "
              "timed step by writing a " + str(2 * L2_BYTES >> 20) + " MiB buffer outside the "
              "step's events")


# Nominal dense tensor-core rate per SM and clock, and NVIDIA's published
# dense per-GPU figures.  8192 bf16 FLOP/clk/SM is the rate at which ncu's
# sm__pipe_tensor_cycles_active counts a tcgen05 kind::f16 product as busy
# (the tensor-pipe percentage of every capture under profiles/ equals the
# achieved FLOP/s over 8192 x 152 SMs x the capture's SM clock); with 152
# SMs it gives NVIDIA's 2.25 PFLOP/s dense bf16 at 1.807 GHz.  E4M3
# (kind::f8f6f4) runs at twice that rate (4.5 PFLOP/s published).
NOMINAL_FLOP_PER_CLK_SM = {"bf16": 8192.0, "e4m3": 16384.0}
DATASHEET_TFLOPS = {"bf16": 2250.0, "e4m3": 4500.0}


def tensor_peaks(dev, sm_mhz, dtype="bf16"):
    """The nominal tensor peak at the sampled SM clock and the datasheet
    peak, in TFLOP/s, with how they were obtained."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"datasheet": DATASHEET_TFLOPS[dtype], "sm_count": sms}
    if sm_mhz:
        out["nominal_at_clock"] = NOMINAL_FLOP_PER_CLK_SM[dtype] * sms * sm_mhz * 1e6 / 1e12
        out["clock_mhz"] = sm_mhz
    return out


def add_peak_fracs(roof, achieved, tp, dtype="bf16"):
    """Beside a roofline's measured-peak fraction, the fractions of the
    nominal peak at the sampled clock and of the datasheet peak."""
    roof["peak_datasheet"] = tp["datasheet"]
    roof["frac_datasheet"] = achieved / tp["datasheet"]
    if "nominal_at_clock" in tp:
        roof["peak_nominal_at_clock"] = tp["nominal_at_clock"]
        roof["frac_nominal"] = achieved / tp["nominal_at_clock"]
        roof["nominal_note"] = ("%d %s FLOP/clk/SM x %d SMs x %.0f MHz (median SM clock sampled "
                                "in the timed region)" % (NOMINAL_FLOP_PER_CLK_SM[dtype], dtype,
                                                          tp["sm_count"], tp["clock_mhz"]))
    return roof


def copy_rates(dev, nbytes=1 << 30, reps=3):
    """Pinned host <-> device copy rates in GB/s (cudaMemcpyAsync through
    torch): each direction alone, then both at once on two streams (as the
    pipelined end-to-end run overlaps them).  Best of `reps`."""
    import torch
    h_src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn_list):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            evs = []
            for st, fn in fn_list:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(st)
                with torch.cuda.stream(st):
                    fn()
                e1.record(st)
                evs.append((e0, e1))
            torch.cuda.synchronize(dev)
            t = [a.elapsed_time(b) / 1e3 for a, b in evs]
            best = t if best is None else [min(x, y) for x, y in zip(best, t)]
        return best

    h2d = timed([(up, lambda: d_a.copy_(h_src, non_blocking=True))])[0]
    d2h = timed([(down, lambda: h_dst.copy_(d_b, non_blocking=True))])[0]
    both = timed([(up, lambda: d_a.copy_(h_src, non_blocking=True)),
                  (down, lambda: h_dst.copy_(d_b, non_blocking=True))])
    del h_src, h_dst, d_a, d_b
    return {"h2d": nbytes / h2d / 1e9, "d2h": nbytes / d2h / 1e9,
            "h2d_concurrent": nbytes / both[0] / 1e9, "d2h_concurrent": nbytes / both[1] / 1e9,
            "bytes_per_copy": nbytes}


def fp8_matmul_peak(dev, n=8192, reps=10):
    """Burst E4M3 matmul rate (torch._scaled_mm, cuBLASLt) in TFLOP/s, best
    of `reps`, or None where that call is unavailable."""
    import torch
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.tensor(1.0, device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = None
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize(dev)
            t = e0.elapsed_time(e1) / 1e3
            best = t if best is None else min(best, t)
        return 2.0 * n ** 3 / best / 1e12
    except Exception:  # an older torch or cuBLASLt without E4M3 matmuls
        return None


def l2_flush_buffer(dev):
    import torch
    return torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)


# ----------------------------------------------------------------- host logic

def fwd_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f * 0.5 if causal else f


def step_flops(w):
    f = fwd_flops(w["B"], w["H"], w["N"], w["d"], w["causal"])
    return f, 2.5 * f


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch: a disjoint stream of the same recipe."""
    return base + 1000003 * rank


def aggregate(per_rank_flops: float, world: int, max_seconds: float) -> float:
    """Whole-job TFLOPS: all ranks' FLOPs over the slowest rank's time."""
    return per_rank_flops * world / max_seconds / 1e12


def reduce_max(value: float, group=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def barrier(group=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier(group=group)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def source_hash(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, if it
    was captured on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        ent = t[kernel_key]
        src = os.path.join(ROOT, ent["source"])
        if source_hash(src) != ent["source_sha256_16"]:
            return None
        return float(ent["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None


def gpu_selector(local_rank: int) -> str:
    """nvidia-smi -i argument for this rank's GPU (its UUID when torch knows it)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        if u and u != "None":
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    return str(local_rank)


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampler running during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[2:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_dict(name: str):
    from io_aware_exact_02_gb300 import synth
    if name == WORKLOAD["name"]:
        return dict(WORKLOAD)
    wl = synth.by_name(name)
    return dict(name=wl.name, B=wl.B, H=wl.H, N=wl.N, d=wl.d, causal=wl.causal)


# ------------------------------------------------------------ reference arm

def cpu_sample(w, heads: int, seed: int = 0):
    """Time the fp64 oracle on `heads` whole heads of the workload (fwd + bwd).

    Returns (TFLOPS by the workload's FLOP count for that sample, seconds,
    threads)."""
    import oracle
    from io_aware_exact_02_gb300 import synth
    q, k, v, do = synth.draw(1, heads, w["N"], w["d"], seed=seed)
    scale = 1.0 / math.sqrt(w["d"])
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, w["causal"], scale)
    oracle.attn_bwd(q, k, v, do, w["causal"], scale)
    dt = time.perf_counter() - t0
    ff, bf = step_flops(dict(w, B=1, H=heads))
    return (ff + bf) / dt / 1e12, dt, oracle.num_threads()


def cpu_single_thread_rows(w, rows: int = 256, seed: int = 0):
    """The oracle's forward on `rows` query rows of one head with one thread:
    (TFLOPS, seconds).  A single-thread reference point beside the all-core
    figure."""
    import oracle
    from io_aware_exact_02_gb300 import synth
    import numpy as np
    q, k, v, _ = synth.draw(1, 1, w["N"], w["d"], seed=seed, with_dout=False)
    sel = np.linspace(0, w["N"] - 1, rows).astype(np.int64)
    heads = np.zeros(rows, dtype=np.int64)
    before = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(q, k, v, w["causal"], 1.0 / math.sqrt(w["d"]), heads, sel)
        dt = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(before)
    keys = sum(min(int(i) + 1, w["N"]) if w["causal"] else w["N"] for i in sel)
    return 4.0 * keys * w["d"] / dt / 1e12, dt


def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    heads = args.ref_heads
    for _ in range(args.warmup):
        cpu_sample(w, heads)
    times = []
    threads = 1
    for _ in range(args.steps):
        _, dt, threads = cpu_sample(w, heads)
        times.append(dt)
    ff, bf = step_flops(dict(w, B=1, H=heads))
    sec = statistics.mean(times)
    value = (ff + bf) / sec / 1e12
    sample = ("fwd+bwd of %d of %d heads (N=%d, d=%d, %s) per step, fp64 oracle on host cores"
              % (heads, w["B"] * w["H"], w["N"], w["d"], "causal" if w["causal"] else "non-causal"))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w["name"], "B": w["B"], "H": w["H"], "N": w["N"], "d": w["d"],
                   "causal": w["causal"], "sample_heads": heads},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

SWEEP_N = (1024, 2048, 4096, 16384)


def n_sweep(dev, seed, steps=5, warmup=3):
    """The metric's range at d = 128 (B=8, H=16, non-causal): forward and
    backward TFLOPS per N, each kernel call timed with CUDA events on the
    launching stream, L2 flushed before every call whose inputs fit in it."""
    import torch
    from io_aware_exact_02_gb300 import fa, synth
    out = {}
    flush = None
    for N in SWEEP_N:
        B, H, d = 8, 16, 128
        q, k, v, do = synth.draw(B, H, N, d, seed=seed, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        ws = torch.empty(fa.bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        small = q.numel() * q.element_size() <= L2_BYTES
        if small and flush is None:
            flush = l2_flush_buffer(dev)
        stream = torch.cuda.current_stream(dev)

        def call(which):
            if which == 0:
                fa.fwd(q, k, v, out=o, lse=lse)
            else:
                fa.bwd(q, k, v, o, do, lse, dq=dq, dk=dk, dv=dv, workspace=ws)

        times = [0.0, 0.0]
        for it in range(warmup + steps):
            for which in (0, 1):
                if small:
                    flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call(which)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                if it >= warmup:
                    times[which] += e0.elapsed_time(e1) / 1e3
        fa.check_device_status()
        ff = fwd_flops(B, H, N, d, False)
        out["N%d" % N] = {"fwd_tflops": ff * steps / times[0] / 1e12,
                          "bwd_tflops": 2.5 * ff * steps / times[1] / 1e12}
        del q, k, v, do, o, lse, dq, dk, dv, ws
    return out


def run_gpu(args, w, rank, world, local_rank):
    import torch
    from io_aware_exact_02_gb300 import fa, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa.load()
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    scale = 1.0 / math.sqrt(d)
    seed = rank_seed(args.seed, rank)
    q, k, v, do = synth.draw(B, H, N, d, seed=seed, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(fa.bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    in_bytes = q.numel() * q.element_size()
    # Inputs that fit in L2 would stay there from one timed step to the next:
    # then a buffer of twice the L2 size is written before every timed step,
    # outside the step's events, and the step time is the sum of those events.
    flush = l2_flush_buffer(dev) if in_bytes <= L2_BYTES else None
    l2_note = ("inputs larger than L2 (each of Q, K, V, dO is %d MiB > 129 MB)" % (in_bytes >> 20)
               if flush is None else FLUSH_NOTE % (in_bytes >> 20))

    def step(events=None):
        if events is not None:
            events[0].record(stream)
        fa.fwd(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
        if events is not None:
            events[1].record(stream)
        fa.bwd(q, k, v, o, do, lse, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv,
               workspace=ws, phases=1)
        if events is not None:
            events[2].record(stream)
        fa.bwd(q, k, v, o, do, lse, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv,
               workspace=ws, phases=2)
        if events is not None:
            events[3].record(stream)
        fa.bwd(q, k, v, o, do, lse, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv,
               workspace=ws, phases=4)
        if events is not None:
            events[4].record(stream)

    launches_per_step = 4  # fwd, bwd prep, bwd main, dQ convert
    for _ in range(args.warmup):
        step()
    fa.check_device_status()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    sampler = ClockSampler(gpu_selector(local_rank))
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        if flush is not None:
            flush.zero_()
        step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    fa.check_device_status()
    if flush is None:
        elapsed = t_start.elapsed_time(t_end) / 1e3
    else:
        elapsed = sum(evs[s][0].elapsed_time(evs[s][4]) for s in range(args.steps)) / 1e3
    per_kernel = {"fwd": 0.0, "bwd_prep": 0.0, "bwd_main": 0.0, "bwd_convert": 0.0}
    names = list(per_kernel)
    for s in range(args.steps):
        for i, nm in enumerate(names):
            per_kernel[nm] += evs[s][i].elapsed_time(evs[s][i + 1]) / 1e3
    max_elapsed = reduce_max(elapsed)
    ff, bf = step_flops(w)
    value = aggregate((ff + bf) * args.steps, world, max_elapsed)

    # ---------------------------------------------------------- end to end
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        hq, hk, hv, hdo = (t.to("cpu").pin_memory() for t in (q, k, v, do))
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        hdq, hdk, hdv = (torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3))

        # Pipelined like a user streaming batches: `--e2e-sets` sets of
        # device buffers (three by default); step k's inputs go up while the
        # compute stream runs step k-1 and its results come back while it
        # runs step k+1.  A set is reused every sets-th step, once its
        # results have come back: with two sets the upload of step k waits
        # for the download of step k-2, so the two directions take turns on
        # the link; with three they overlap.  With
        # --e2e-copy-streams > 1 each copy direction is spread over that many
        # streams (tensors round-robin), so that several copy engines can move
        # the step's gigabyte.  Every step still copies its own inputs in and
        # all of its outputs out inside the timed region.
        sets = [(q, k, v, do, o, lse, dq, dk, dv, ws)]
        nsets = max(2, args.e2e_sets)
        for _ in range(nsets - 1):
            sets.append(tuple(torch.empty_like(t) for t in sets[0]))
        nc = max(1, args.e2e_copy_streams)
        ups = [torch.cuda.Stream(dev) for _ in range(nc)]
        downs = [torch.cuda.Stream(dev) for _ in range(nc)]
        comp = torch.cuda.Stream(dev)

        def timing_event(stream):
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            return ev

        stage_events = []  # per step: (h2d start, h2d end, compute start, end, d2h start, end)

        def e2e_run(n):
            stage_events.clear()
            done_down = [[] for _ in range(nsets)]  # set b's last D2H events (then it is free)
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(ups[0])
            for u in ups[1:]:
                u.wait_event(start)
            for step in range(n):
                b = step % nsets
                bq, bk, bv, bdo, bo, blse, bdq, bdk, bdv, bws = sets[b]
                loaded = []
                stamps = []
                for i, (dst, src) in enumerate(((bq, hq), (bk, hk), (bv, hv), (bdo, hdo))):
                    u = ups[i % nc]
                    for ev in done_down[b]:
                        u.wait_event(ev)
                    if i == 0:
                        stamps.append(timing_event(u))
                    with torch.cuda.stream(u):
                        dst.copy_(src, non_blocking=True)
                        ev = torch.cuda.Event(enable_timing=(i == 3))
                        ev.record(u)
                    loaded.append(ev)
                stamps.append(loaded[-1])
                for ev in loaded:
                    comp.wait_event(ev)
                stamps.append(timing_event(comp))
                with torch.cuda.stream(comp):
                    fa.fwd(bq, bk, bv, causal=causal, scale=scale, out=bo, lse=blse)
                    fa.bwd(bq, bk, bv, bo, bdo, blse, causal=causal, scale=scale, dq=bdq, dk=bdk,
                           dv=bdv, workspace=bws)
                    computed = torch.cuda.Event(enable_timing=True)
                    computed.record(comp)
                stamps.append(computed)
                done_down[b] = []
                for j, (dst, src) in enumerate(((hdq, bdq), (hdk, bdk), (hdv, bdv), (ho, bo),
                                                (hlse, blse))):
                    dn = downs[j % nc]
                    dn.wait_event(computed)
                    if j == 0:
                        stamps.append(timing_event(dn))
                    with torch.cuda.stream(dn):
                        dst.copy_(src, non_blocking=True)
                        ev = torch.cuda.Event(enable_timing=(j == 4))
                        ev.record(dn)
                    done_down[b].append(ev)
                stamps.append(done_down[b][-1])
                stage_events.append(stamps)
            for ev in sum(done_down, []):
                downs[0].wait_event(ev)
            end.record(downs[0])
            return start, end

        e2e_run(2)
        torch.cuda.synchronize(dev)
        barrier()
        e0, e1 = e2e_run(e2e_steps)
        torch.cuda.synchronize(dev)
        barrier()
        fa.check_device_status(stream=comp.cuda_stream)
        e2e_sec = reduce_max(e0.elapsed_time(e1) / 1e3)
        # Mean duration of each stage of a step (with one copy stream per
        # direction the stage is contiguous on its stream): what the copies
        # and the kernels took while running together.
        stage_ms = None
        if nc == 1:
            stage_ms = {name: statistics.mean(st[2 * i].elapsed_time(st[2 * i + 1])
                                              for st in stage_events)
                        for i, name in enumerate(("h2d", "kernels", "d2h"))}
        h2d = 4 * in_bytes
        d2h = 4 * in_bytes + lse.numel() * 4
        e2e = {"value": aggregate((ff + bf) * e2e_steps, world, e2e_sec), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "pipelined": "H2D of step k+1 and D2H of step k-1 overlap step k's kernels "
                            "(%d device buffer sets, %d copy streams per direction)"
                            % (nsets, nc)}
        # The host link, measured on this machine in this run: a pipelined step
        # can be no shorter than its kernels or than either direction's
        # copies at the rate both directions reach together.
        del sets
        rates = copy_rates(dev)
        kern_ms = elapsed / args.steps * 1e3
        h2d_ms = h2d / (rates["h2d_concurrent"] * 1e9) * 1e3
        d2h_ms = d2h / (rates["d2h_concurrent"] * 1e9) * 1e3
        bound = max(kern_ms, h2d_ms, d2h_ms)
        e2e_ms = e2e_sec / e2e_steps * 1e3
        e2e.update({"ms_per_step": e2e_ms, "stage_ms_in_pipeline": stage_ms, "copy_gbs": rates,
                    "bound_ms": bound,
                    "bound_parts_ms": {"kernels": kern_ms, "h2d": h2d_ms, "d2h": d2h_ms},
                    "frac_of_bound": bound / e2e_ms})

    # ------------------------------------------------------------ roofline
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    main_avg = per_kernel["bwd_main"] / args.steps
    fwd_avg = per_kernel["fwd"] / args.steps
    achieved = bf / main_avg / 1e12
    roofline = {"bound": "tensor", "kernel": "fa_bwd_main_kernel<%d>" % d, "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": "%s burst bf16 (MEASURED_PEAKS.json bf16_tflops)" % peak_kind
                if peak_kind == "measured" else "fallback burst bf16",
                "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
                "traffic": profiled_traffic("fa_bwd_main_kernel_d%d_%s" % (d, w["name"]))}
    tp = tensor_peaks(dev, clocks.get("sm_mhz") or clocks.get("sm_max_mhz"))
    add_peak_fracs(roofline, achieved, tp)
    kernels = {nm: {"ms_per_launch": per_kernel[nm] / args.steps * 1e3} for nm in names}
    kernels["fwd"]["tflops"] = ff / fwd_avg / 1e12
    kernels["fwd"]["frac_of_peak"] = ff / fwd_avg / 1e12 / peak
    if "nominal_at_clock" in tp:
        kernels["fwd"]["frac_nominal"] = ff / fwd_avg / 1e12 / tp["nominal_at_clock"]
    kernels["fwd"]["frac_datasheet"] = ff / fwd_avg / 1e12 / tp["datasheet"]
    kernels["bwd_main"]["tflops"] = achieved
    bwd_total = (per_kernel["bwd_prep"] + per_kernel["bwd_main"] + per_kernel["bwd_convert"]) / args.steps
    # The trade the backward pass makes (cs2680 Lecture 9 sec. 9.6): recompute
    # S and P instead of writing the N x N probabilities in the forward pass
    # and reading them back, 2 * B*H*N^2 bf16 bytes at the HBM copy rate.
    p_bytes = 2.0 * 2.0 * B * H * N * N
    kernels["stored_p_equivalent"] = {
        "bytes": p_bytes,
        "ms_at_hbm_peak": p_bytes / (float(load_peaks()[0]["hbm_gbs"]) * 1e9) * 1e3}
    kernels["bwd_total"] = {"ms_per_call": bwd_total * 1e3, "tflops": bf / bwd_total / 1e12,
                            "frac_of_peak": bf / bwd_total / 1e12 / peak}
    if "nominal_at_clock" in tp:
        kernels["bwd_total"]["frac_nominal"] = bf / bwd_total / 1e12 / tp["nominal_at_clock"]
    # The backward pass as one fa_bwd call, after the timed region (as the N
    # sweep measures it): its three kernels back to back, each launched with
    # programmatic dependent launch.  The per-kernel events of the timed step
    # keep each launch from overlapping the end of the kernel before it,
    # which at short lengths costs a few microseconds per call.
    call_s = []
    for it in range(7):
        if flush is not None:
            flush.zero_()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        fa.bwd(q, k, v, o, do, lse, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)
        c1.record(stream)
        torch.cuda.synchronize(dev)
        if it >= 2:
            call_s.append(c0.elapsed_time(c1) / 1e3)
    fa.check_device_status()
    bwd_call = sum(call_s) / len(call_s)
    kernels["bwd_call"] = {"ms_per_call": bwd_call * 1e3, "tflops": bf / bwd_call / 1e12,
                           "frac_of_peak": bf / bwd_call / 1e12 / peak,
                           "note": "one fa_bwd call, L2 flushed before it when the inputs fit "
                                   "in L2, after the timed region"}
    hbm_bytes = 8.0 * B * H * N * d + 4.0 * B * H * N  # fwd: Q, K, V read, O written, lse
    kernels["fwd"]["algorithmic_hbm_gbs"] = hbm_bytes / fwd_avg / 1e9

    # ------------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, dt, threads = cpu_sample(w, args.cpu_heads)
        st_val, st_dt = cpu_single_thread_rows(w)
        cpu = {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "fwd+bwd of %d of %d heads (N=%d, d=%d), fp64 oracle, %.1f s"
                         % (args.cpu_heads, B * H, N, d, dt),
               "single_thread": {"value": st_val, "unit": UNIT,
                                 "sample": "forward of 256 query rows of one head, 1 thread, "
                                           "%.2f s" % st_dt}}

    sweep = None
    if world == 1 and not args.no_sweep and w["name"] == WORKLOAD["name"]:
        sweep = n_sweep(dev, seed)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": max_elapsed / args.steps * 1e3,
            "ms_per_step_median": statistics.median(
                evs[s][0].elapsed_time(evs[s][4]) for s in range(args.steps)),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w["name"], "B": B, "H": H, "N": N, "d": d,
                       "causal": causal, "scale": scale, "step": "fa_fwd + fa_bwd",
                       "parallelism": "replicas x%d (independent batches per GPU)" % world,
                       "l2": l2_note, "seed": args.seed},
            "clocks": clocks, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "roofline": roofline, "cpu_baseline": cpu, "kernels": kernels,
        }
        if sweep is not None:
            line["n_sweep_d128"] = dict(sweep, note="B=8 H=16 d=128 non-causal, per kernel "
                                        "call, L2 flushed when the inputs fit in it; outside "
                                        "the timed region")
        print(json.dumps(line), flush=True)
    return 0


def run_gqa(args, wl, rank, world, local_rank):
    """A general-form workload: decode (HBM-bound, GB/s) or GQA prefill
    (TFLOPS), timed through fa_fwd_gqa with the library's split choice."""
    import torch
    from io_aware_exact_02_gb300 import fa, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa.load()
    q, k, v = synth.draw_gqa(wl, seed=rank_seed(args.seed, rank), device=dev)
    splits = fa.fwd_gqa_splits(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nkv, wl.d, wl.causal)
    o = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, wl.Nq), dtype=torch.float32, device=dev)
    ws_bytes = fa.fwd_gqa_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nkv, wl.d, splits)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fwd_gqa(q, k, v, causal=wl.causal, scale=wl.softmax_scale, num_splits=splits,
                   out=o, lse=lse, workspace=ws if ws_bytes else None)

    kv_bytes = 2.0 * wl.B * wl.Hkv * wl.Nkv * wl.d * 2
    # K and V are the re-read streams: when one fits in L2, L2 is flushed
    # before every timed call, outside that call's events.
    flush = l2_flush_buffer(dev) if kv_bytes / 2 <= L2_BYTES else None
    for _ in range(args.warmup):
        step()
    fa.check_device_status()
    sampler = ClockSampler(gpu_selector(local_rank))
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for e0, e1 in evs:
        if flush is not None:
            flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    fa.check_device_status()
    sec = reduce_max(sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3)
    per_call = sec / args.steps
    qo_bytes = 2.0 * wl.B * wl.Hq * wl.Nq * wl.d * 2 + 4.0 * wl.B * wl.Hq * wl.Nq
    alg_bytes = kv_bytes + qo_bytes
    flops = 4.0 * wl.B * wl.Hq * wl.Nq * wl.Nkv * wl.d
    if wl.causal and wl.Nq == wl.Nkv:
        flops *= 0.5
    peaks, peak_kind = load_peaks()
    decode = wl.Nq <= 16
    if decode:
        value = world * alg_bytes / per_call / 1e9
        unit, metric = "GB/s", "decode attention HBM GB/s (algorithmic bytes: Q, K, V read, O, lse written)"
        peak = float(peaks["hbm_gbs"])
        roofline = {"bound": "hbm", "kernel": "fa_fwd_kernel (general) + fa_combine_kernel",
                    "achieved": value / world, "peak": peak, "unit": "GB/s",
                    "frac": value / world / peak, "peak_kind": "%s HBM copy" % peak_kind,
                    "traffic": profiled_traffic("fa_fwd_general_and_combine_" + wl.name)}
    else:
        value = world * flops / per_call / 1e12
        unit, metric = "TFLOPS", "GQA prefill attention TFLOPS (bf16)"
        peak = float(peaks["bf16_tflops"])
        roofline = {"bound": "tensor", "kernel": "fa_fwd_kernel (general)",
                    "achieved": value / world, "peak": peak, "unit": "TFLOP/s",
                    "frac": value / world / peak, "peak_kind": "%s burst bf16" % peak_kind,
                    "traffic": profiled_traffic("fa_fwd_general_" + wl.name)}
        add_peak_fracs(roofline, value / world,
                       tensor_peaks(dev, clocks.get("sm_mhz") or clocks.get("sm_max_mhz")))
    if rank == 0:
        print(json.dumps({
            "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_call * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "Nq": wl.Nq,
                       "Nkv": wl.Nkv, "d": wl.d, "causal": wl.causal, "splits": splits,
                       "step": "fa_fwd_gqa",
                       "l2": ("K and V are %d MiB together; " % (kv_bytes / 2**20))
                       + ("inputs larger than L2" if flush is None
                          else "L2 flushed before every timed call (a %d MiB buffer written "
                               "outside the call's events)" % (2 * L2_BYTES >> 20)),
                       "workspace_bytes": ws_bytes},
            "clocks": clocks, "gpu_launches": args.steps * (2 if splits > 1 else 1),
            "roofline": roofline, "tflops": flops / per_call / 1e12,
            "hbm_gbs_algorithmic": alg_bytes / per_call / 1e9}), flush=True)
    return 0


def visible_pairs(mask, N, causal):
    """(query, key) pairs a block mask leaves visible in one head: the
    algorithmic work of the block-sparse passes is proportional to it."""
    nb = len(mask)
    total = 0
    for r in range(nb):
        r0, r1 = r * 128, min(N, (r + 1) * 128)
        for c in range(nb):
            if not mask[r][c]:
                continue
            c0, c1 = c * 128, min(N, (c + 1) * 128)
            if not causal:
                total += (r1 - r0) * (c1 - c0)
            else:  # keys j <= i, row by row
                for i in range(r0, r1):
                    total += max(0, min(c1, i + 1) - c0)
    return total


def run_blocksparse(args, wl, rank, world, local_rank):
    """Block-sparse fwd + bwd step (TFLOPS counted over the visible pairs)."""
    import torch
    from io_aware_exact_02_gb300 import fa, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa.load()
    dense = synth.Workload(wl.name, wl.B, wl.H, wl.N, wl.d, wl.causal)
    q, k, v, do = synth.draw_workload(dense, seed=rank_seed(args.seed, rank), device=dev)
    mask_cpu = synth.draw_block_mask(wl.n_blocks, wl.density, seed=args.seed)
    mask = mask_cpu.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.bwd_workspace_size(wl.B, wl.H, wl.N, wl.d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    fwd_ms, bwd_ms = [], []

    def step(record=False):
        if record:
            ev[0].record(stream)
        fa.fwd_blocksparse(q, k, v, mask, causal=wl.causal, scale=wl.softmax_scale, out=o,
                           lse=lse)
        if record:
            ev[1].record(stream)
        fa.bwd_blocksparse(q, k, v, o, do, lse, mask, causal=wl.causal, scale=wl.softmax_scale,
                           dq=dq, dk=dk, dv=dv, workspace=ws)
        if record:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    fa.check_device_status()
    sampler = ClockSampler(gpu_selector(local_rank))
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    # Per-pass split, measured in separate steps after the timed region.
    for _ in range(3):
        step(record=True)
        torch.cuda.synchronize(dev)
        fwd_ms.append(ev[0].elapsed_time(ev[1]))
        bwd_ms.append(ev[1].elapsed_time(ev[2]))
    fa.check_device_status()
    sec = reduce_max(e0.elapsed_time(e1) / 1e3)
    per_step = sec / args.steps
    pairs = visible_pairs(mask_cpu.tolist(), wl.N, wl.causal)
    f_fwd = 4.0 * wl.B * wl.H * pairs * wl.d
    f_bwd = 2.5 * f_fwd
    value = world * (f_fwd + f_bwd) / per_step / 1e12
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    t_fwd, t_bwd = statistics.median(fwd_ms) / 1e3, statistics.median(bwd_ms) / 1e3
    if rank == 0:
        print(json.dumps({
            "metric": "block-sparse attention fwd+bwd TFLOPS (bf16, FLOPs over visible pairs)",
            "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d,
                       "causal": wl.causal, "density": wl.density,
                       "active_blocks": int(mask_cpu.sum()), "blocks": wl.n_blocks ** 2,
                       "step": "fa_fwd_blocksparse + fa_bwd_blocksparse",
                       "l2": "inputs larger than L2"},
            "clocks": clocks, "gpu_launches": args.steps * 4,
            "roofline": add_peak_fracs(
                {"bound": "tensor", "kernel": "fa_bwd_main_kernel (sparse)",
                 "achieved": f_bwd / t_bwd / 1e12, "peak": peak, "unit": "TFLOP/s",
                 "frac": f_bwd / t_bwd / 1e12 / peak, "peak_kind": "%s burst bf16" % peak_kind,
                 "traffic": profiled_traffic("fa_bwd_main_kernel_sparse_" + wl.name)},
                f_bwd / t_bwd / 1e12,
                tensor_peaks(dev, clocks.get("sm_mhz") or clocks.get("sm_max_mhz"))),
            "fwd_tflops": f_fwd / t_fwd / 1e12, "bwd_tflops": f_bwd / t_bwd / 1e12,
            "fwd_ms": t_fwd * 1e3, "bwd_ms": t_bwd * 1e3}), flush=True)
    return 0


FP8_WORKLOAD = dict(name="fp8_hadamard_B8_H16_N8192_d128", B=8, H=16, N=8192, d=128,
                    causal=False)


def run_fp8(args, w, rank, world, local_rank):
    """FP8 forward step: quantisation (with the Hadamard rotation) + FP8
    attention, TFLOPS by the forward FLOP count."""
    import torch
    from io_aware_exact_02_gb300 import fa, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa.load()
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    wl = synth.Workload(w["name"], B, H, N, d, causal)
    q, k, v, _ = synth.draw_workload(wl, seed=rank_seed(args.seed, rank), device=dev,
                                     with_dout=False)
    ws = torch.empty(fa.fwd_fp8_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    q_ms, a_ms = [], []

    def step(record=False):
        if record:
            ev[0].record(stream)
        fa.fp8_quantize(q, k, v, hadamard=True, workspace=ws)
        if record:
            ev[1].record(stream)
        fa.fwd_fp8_quantized(ws, B, H, N, d, causal=causal, scale=wl.softmax_scale,
                             hadamard=True, out=o, lse=lse)
        if record:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    fa.check_device_status()
    sampler = ClockSampler(gpu_selector(local_rank))
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    for _ in range(3):
        step(record=True)
        torch.cuda.synchronize(dev)
        q_ms.append(ev[0].elapsed_time(ev[1]))
        a_ms.append(ev[1].elapsed_time(ev[2]))
    fa.check_device_status()
    sec = reduce_max(e0.elapsed_time(e1) / 1e3)
    per_step = sec / args.steps
    flops = fwd_flops(B, H, N, d, causal)
    value = world * flops / per_step / 1e12
    # Denominators: a burst E4M3 matmul measured here (cuBLASLt through
    # torch._scaled_mm), the nominal E4M3 rate at the sampled clock and the
    # datasheet figure.
    fp8_peak = fp8_matmul_peak(dev)
    tp = tensor_peaks(dev, clocks.get("sm_mhz") or clocks.get("sm_max_mhz"), "e4m3")
    if fp8_peak is not None:
        peak, peak_kind = fp8_peak, "measured burst E4M3 matmul (torch._scaled_mm 8192^3, this run)"
    else:
        peak = tp.get("nominal_at_clock", tp["datasheet"])
        peak_kind = ("nominal E4M3 at the sampled clock (no E4M3 matmul available to measure)"
                     if "nominal_at_clock" in tp else "datasheet E4M3")
    t_q, t_a = statistics.median(q_ms) / 1e3, statistics.median(a_ms) / 1e3
    in_bytes = 3.0 * B * H * N * d * 2
    if rank == 0:
        print(json.dumps({
            "metric": "FP8 attention forward TFLOPS (E4M3, Hadamard rotation, quantisation "
                      "included)",
            "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": w["name"], "B": B, "H": H, "N": N, "d": d, "causal": causal,
                       "step": "fa_fp8_quantize + fa_fwd_fp8_quantized",
                       "l2": "inputs larger than L2"},
            "clocks": clocks, "gpu_launches": args.steps * 3,
            "roofline": add_peak_fracs(
                {"bound": "tensor", "kernel": "fa_fwd_kernel (FP8)",
                 "achieved": flops / t_a / 1e12, "peak": peak, "unit": "TFLOP/s",
                 "frac": flops / t_a / 1e12 / peak, "peak_kind": peak_kind,
                 "traffic": profiled_traffic("fa_fwd_kernel_fp8_" + w["name"])},
                flops / t_a / 1e12, tp, "e4m3"),
            "attention_ms": t_a * 1e3, "quantize_ms": t_q * 1e3,
            "quantize_gbs_inputs_read": in_bytes / t_q / 1e9}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--workload", default=WORKLOAD["name"],
                    help="one of the synthetic workloads (default: the headline one)")
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d,causal: a custom iid N(0,1) workload (small profiling cases)")
    ap.add_argument("--cpu-heads", type=int, default=2,
                    help="heads of the workload the cpu_baseline leg times (GPU arm)")
    ap.add_argument("--ref-heads", type=int, default=1,
                    help="heads of the workload per step of the reference arm")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-sets", type=int, default=3,
                    help="device buffer sets the end-to-end pipeline rotates through (>= 2)")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams per copy direction in the end-to-end run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the d=128 N sweep (1K, 2K, 4K, 16K) reported beside the headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fwd-kernel", choices=["auto", "pair", "one"], default="auto",
                    help="non-causal d=128 forward kernel: the library's choice (one CTA per "
                         "item), or forced CTA pairs / one CTA per item (FA_FWD_PAIR)")
    args = ap.parse_args(argv)
    if args.fwd_kernel != "auto":  # read by the library on its first forward call
        os.environ["FA_FWD_PAIR"] = "1" if args.fwd_kernel == "pair" else "0"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        print("warning: WORLD_SIZE=%d but --gpus %d" % (world, args.gpus), file=sys.stderr)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.shape:
        B, H, N, d, c = (int(x) for x in args.shape.split(","))
        w = dict(name="custom_B%d_H%d_N%d_d%d_%s" % (B, H, N, d, "causal" if c else "full"),
                 B=B, H=H, N=N, d=d, causal=bool(c))
    else:
        from io_aware_exact_02_gb300 import synth
        if args.workload in [g.name for g in synth.GQA_ALL]:
            if args.impl == "reference":
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the reference arm times the square workloads only"}))
                return 0
            return run_gqa(args, synth.gqa_by_name(args.workload), rank, world, local_rank)
        if args.workload == FP8_WORKLOAD["name"]:
            if args.impl == "reference":
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the reference arm times the square workloads only"}))
                return 0
            return run_fp8(args, FP8_WORKLOAD, rank, world, local_rank)
        if args.workload in [b.name for b in synth.BLOCKSPARSE_ALL]:
            if args.impl == "reference":
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the reference arm times the square workloads only"}))
                return 0
            return run_blocksparse(args, synth.blocksparse_by_name(args.workload), rank, world,
                                   local_rank)
        w = workload_dict(args.workload)
    try:
        if args.impl == "reference":
            return run_reference(args, w, rank, world)
        return run_gpu(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
