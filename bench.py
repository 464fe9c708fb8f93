"""Bench of the primitive-op graph hot path on GB300.

One step = one pass of the View-indexed elementwise workload on one batch of
synthetic input, fully resident in HBM:
  * the fused chain y = WHERE(CMPLT(a, b), EXP(a*0.5), LOG(b*b + 1)) over
    a[4096,4096] float32 with b[4096] expanded as a column (stride-0 View);
  * CONTIGUOUS(permute(1,0)) of x[8192,8192] float32 (the tiled transpose).
The metric is fused-op HBM throughput: algorithmic bytes (every operand byte
read once and every result byte written once) per second.  L2 is flushed
(a write of twice the L2 size) before every timed step, outside the events.

Extra rows of the same JSON line time the other hot-path calls on their own
workloads (row reductions, the MUL+SUM contraction, gather/scatter) when their
kernels are present, each against its own roofline.

--impl reference runs the plain CPU oracle (the reference implementation of
the method on these pages) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as SI  # noqa: E402

CHAIN_BYTES = 4096 * 4096 * 4 * 2 + 4096 * 4          # a read + y write + b read once
TRANSPOSE_BYTES = 8192 * 8192 * 4 * 2                  # x read + out write
STEP_BYTES = CHAIN_BYTES + TRANSPOSE_BYTES
METRIC = "fused-op HBM GB/s and MUL+SUM TFLOP/s, % of GB300 roofline, 1 GPU"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d["bf16_tflops_sustained"]), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# ------------------------------------------------------------ distributed ----

def dist_setup(n_gpus):
    if n_gpus <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist
    dist.init_process_group("gloo")
    return dist.get_rank(), dist.get_world_size(), dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks ----

class Clocks:
    """nvidia-smi samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.f is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for k, nm in enumerate(names):
                if len(r) > 5 + k and r[5 + k].strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workloads ----

class Step:
    """The C2 workload on one device, driven through the C ABI."""

    def __init__(self, A, seed=0):
        self.A = A
        a, b = SI.chain(seed)
        x = SI.transpose_input(seed)
        self.host = dict(a=a, b=b, x=x)
        self.a, self.b, self.x = a.cuda(), b.cuda(), x.cuda()
        self.y = torch.empty_like(self.a)
        self.xt = torch.empty((8192, 8192), dtype=torch.float32, device="cuda")
        n = A.node
        self.prog = [n("LOAD", 0), n("LOAD", 1), n("CMPLT", 0, 1), n("CONST", cval=0.5),
                     n("MUL", 0, 3), n("EXP", 4), n("MUL", 1, 1), n("CONST", cval=1.0),
                     n("ADD", 6, 7), n("LOG", 8), n("WHERE", 2, 5, 9)]
        self.bind()

    def bind(self):
        A = self.A
        self.va = A.view_of(self.a)
        self.vb = A.view_of(self.b, shape=(4096, 4096), strides=(1, 0))
        self.vy = A.view_of(self.y)
        self.vx = A.view_of(self.x)
        self.vxt = A.view_of(self.xt)

    def chain(self, stream):
        self.A.psg_elementwise(self.prog, [self.a, self.b], [self.va, self.vb], self.y, self.vy,
                               stream=stream)

    def transpose(self, stream):
        self.A.psg_permute(self.x, self.vx, [1, 0], self.xt, self.vxt, stream=stream)

    def run(self, stream):
        self.chain(stream)
        self.transpose(stream)


def l2_flush_buffer():
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    return torch.empty(int(2 * max(l2, 64 << 20)), dtype=torch.uint8, device="cuda")


def timed_steps(step, K, W, dist):
    """W warm-ups, then K steps each preceded by an L2 flush outside its
    events; returns (total ms over K steps, chain ms avg, transpose ms avg)."""
    s = torch.cuda.current_stream()
    flush = l2_flush_buffer()
    for _ in range(W):
        flush.zero_()
        step.run(s.cuda_stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        flush.zero_()
        ev[k][0].record(s)
        step.chain(s.cuda_stream)
        ev[k][1].record(s)
        step.transpose(s.cuda_stream)
        ev[k][2].record(s)
    torch.cuda.synchronize()
    barrier(dist)
    wall = time.perf_counter() - t0
    ch = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    tr = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    total = sum(c + t for c, t in zip(ch, tr))
    return total, sum(ch) / K, sum(tr) / K, wall


def e2e_steps(step, K, W):
    """The same step through the C ABI with host buffers: pinned host ->
    device copies of a, b, x, the two kernels, device -> host copies of the
    two results; all inside the timed region."""
    s = torch.cuda.current_stream()
    ha, hb, hx = (step.host[k].pin_memory() for k in ("a", "b", "x"))
    hy = torch.empty_like(ha).pin_memory()
    hxt = torch.empty_like(hx).pin_memory()

    def one():
        step.a.copy_(ha, non_blocking=True)
        step.b.copy_(hb, non_blocking=True)
        step.x.copy_(hx, non_blocking=True)
        step.run(s.cuda_stream)
        hy.copy_(step.y, non_blocking=True)
        hxt.copy_(step.xt, non_blocking=True)

    for _ in range(W):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(K):
        one()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    h2d = ha.numel() * 4 + hb.numel() * 4 + hx.numel() * 4
    d2h = hy.numel() * 4 + hxt.numel() * 4
    return ms, h2d, d2h


# ----------------------------------------------------------- CPU oracle ----

def oracle_sample(threads: int, rows: int = 512):
    """The oracle on a bounded sample of the step: the chain on the first
    `rows` rows of a, the transpose of a [rows*2, 8192] slab of x.  Returns
    (seconds, algorithmic bytes of the sample)."""
    import oracle as O
    O.build()
    O.NTHREADS = threads
    a, b = SI.chain(0)
    x = SI.transpose_input(0)
    a_s = O.T(a[:rows].numpy(), "f32")
    b_s = O.T(b[:rows].numpy(), "f32")
    x_s = O.T(x[: rows * 2].numpy(), "f32")
    t0 = time.perf_counter()
    O.chain_where_exp_log(a_s, b_s)
    O.view(x_s, (8192, rows * 2), (1, 8192))  # CONTIGUOUS(permute(1,0)) of the slab
    sec = time.perf_counter() - t0
    nbytes = rows * 4096 * 4 * 2 + rows * 4 + rows * 2 * 8192 * 4 * 2
    return sec, nbytes


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ main ----

def run_reference(args):
    rank, world, dist = dist_setup(args.gpus)
    if rank != 0:
        return
    cores = cpu_cores()
    times, nbytes = [], 0
    for _ in range(args.warmup):
        oracle_sample(cores, rows=64)
    for _ in range(args.steps):
        sec, nbytes = oracle_sample(cores)
        times.append(sec)
    total = sum(times)
    gbs = nbytes * len(times) / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "chain y=WHERE(CMPLT(a,b),EXP(a*0.5),LOG(b*b+1)) a[4096,4096] "
                                   "b[4096] expanded + permute(1,0) of x[8192,8192] f32",
                       "sample": "first 512 rows of the chain, x[:1024,:] transposed"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle",
                             "sample": "512 of 4096 chain rows + a 1024x8192 transpose slab"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    rank, world, dist = dist_setup(args.gpus)
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    from primitive_sm_graph_gb300 import build as B
    B.build()
    from primitive_sm_graph_gb300 import _abi as A

    step = Step(A)
    with Clocks(local) as clk:
        total_ms, chain_ms, tr_ms, wall = timed_steps(step, args.steps, args.warmup, dist)
    clocks = clk.summary()
    total_ms = max_over_ranks(dist, total_ms)
    ms_step = total_ms / args.steps
    value = STEP_BYTES * world / (ms_step * 1e-3) / 1e9
    P = peaks()
    # dominant kernel: the one with the larger share of the step
    dom = ("transpose", TRANSPOSE_BYTES, tr_ms) if tr_ms >= chain_ms else ("chain", CHAIN_BYTES, chain_ms)
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        traffic = json.load(open(tp)).get(dom[0])
    e2e_ms, h2d, d2h = e2e_steps(step, max(3, args.steps // 4), 2)
    e2e_gbs = STEP_BYTES * world / (max_over_ranks(dist, e2e_ms) * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "chain y=WHERE(CMPLT(a,b),EXP(a*0.5),LOG(b*b+1)) a[4096,4096] "
                               "b[4096] expanded + permute(1,0) of x[8192,8192] f32",
                   "bytes_per_step": STEP_BYTES, "l2": "flushed before every step (2x L2 write)",
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "kernel": dom[0], "achieved": round(achieved, 2),
                     "peak": P["hbm"], "peak_source": P["source"] + " burst copy",
                     "unit": "GB/s", "frac": round(achieved / P["hbm"], 4), "traffic": traffic},
        "kernels_ms": {"chain": round(chain_ms, 5), "transpose": round(tr_ms, 5)},
        "kernels_gbs": {"chain": round(CHAIN_BYTES / (chain_ms * 1e-3) / 1e9, 2),
                        "transpose": round(TRANSPOSE_BYTES / (tr_ms * 1e-3) / 1e9, 2)},
        "clocks": clocks,
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
    }
    if rank == 0 and not args.no_cpu_baseline:
        cores = cpu_cores()
        sec, nbytes = oracle_sample(cores)
        line["cpu_baseline"] = {"value": round(nbytes / sec / 1e9, 4), "unit": "GB/s",
                                "cores": cores, "kind": "oracle",
                                "sample": "512 of 4096 chain rows + a 1024x8192 transpose slab"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
