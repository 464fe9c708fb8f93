"""Bench of the primitive-op graph hot path on GB300.

One step = one pass of the View-indexed elementwise workload on one batch of
synthetic input, fully resident in HBM:
  * the fused chain y = WHERE(CMPLT(a, b), EXP(a*0.5), LOG(b*b + 1)) over
    a[4096,4096] float32 with b[4096] expanded as a column (stride-0 View);
  * CONTIGUOUS(permute(1,0)) of x[8192,8192] float32 (the tiled transpose).
The metric is fused-op HBM throughput: algorithmic bytes (every operand byte
read once and every result byte written once) per second.  L2 is flushed
before every timed step, outside the events: a write of twice the L2 size,
then a read of twice the L2 size so no dirty flush lines remain.

The "rows" object of the same JSON line times the other hot-path calls on
their own workloads, each against its own ceiling: softmax over x[4096,1024]
f32 and RMSNorm over x[8192,4096] bf16 (HBM, L2 flushed), the MUL+SUM
contraction in bf16 8192^3 (tensor pipe, measured cuBLAS peak) and f32 4096^3
(FFMA, peak derived from unit counts and clock), the token gather and
scatter-add of the GPT block, the tiny MUL+SUM graph (eager and CUDA Graph
replay) and one GPT block forward + backward through the graph layer.

--profile-case NAME runs one workload a few times and exits, for a profiler.

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


def whole_job_gbs(dist, world: int, bytes_per_rank_step: int, ms_per_step_local: float):
    """Whole-job throughput of N replicas: every rank processes
    bytes_per_rank_step per step, the job takes the slowest rank's time.
    Returns (GB/s over all ranks, max ms per step)."""
    ms = max_over_ranks(dist, ms_per_step_local)
    return bytes_per_rank_step * world / (ms * 1e-3) / 1e9, ms


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


class L2Flush:
    """Empties L2 between timed iterations (outside the events): write a
    buffer of twice the L2 size, then read a second one, so the timed kernel
    starts with no useful lines in L2 and no dirty lines of the flush itself
    left to write back while it runs."""

    def __init__(self):
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
        n = int(2 * max(l2, 64 << 20))
        self.w = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(n // 4, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.max()


def l2_flush_buffer():
    return L2Flush()


def timed_steps(step, K, W, dist):
    """W warm-ups, then K steps each preceded by an L2 flush outside its
    events; returns (total ms over K steps, chain ms avg, transpose ms avg)."""
    s = torch.cuda.current_stream()
    flush = l2_flush_buffer()
    for _ in range(W):
        flush()
        step.run(s.cuda_stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        flush()
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
    """The same step through the C ABI with host buffers: every step copies
    a, b, x from pinned host memory to the device, runs the two kernels and
    copies the two results back to pinned host memory, all inside the timed
    region.  Steps are pipelined over two device buffer sets and three
    streams: step k+1's inputs go in while step k computes and step k's
    results come out (each copy engine direction busy at once), as a stream
    of batches would run.  Returns (ms per step, H2D bytes, D2H bytes)."""
    import copy
    ha, hb, hx = (step.host[k].pin_memory() for k in ("a", "b", "x"))
    hy = torch.empty_like(ha).pin_memory()
    hxt = torch.empty_like(hx).pin_memory()
    other = copy.copy(step)
    other.a, other.b, other.x = step.a.clone(), step.b.clone(), step.x.clone()
    other.y, other.xt = torch.empty_like(step.y), torch.empty_like(step.xt)
    other.bind()
    sets = [step, other]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    out_done = [ev(), ev()]
    for e in out_done:
        e.record(s_out)

    def one(k):
        S = sets[k % 2]
        in_done, cmp_done = ev(), ev()
        s_in.wait_event(out_done[k % 2])        # this set's previous results are out
        with torch.cuda.stream(s_in):
            S.a.copy_(ha, non_blocking=True)
            S.b.copy_(hb, non_blocking=True)
            S.x.copy_(hx, non_blocking=True)
        in_done.record(s_in)
        s_cmp.wait_event(in_done)
        S.run(s_cmp.cuda_stream)
        cmp_done.record(s_cmp)
        s_out.wait_event(cmp_done)
        with torch.cuda.stream(s_out):
            hy.copy_(S.y, non_blocking=True)
            hxt.copy_(S.xt, non_blocking=True)
        out_done[k % 2] = ev()
        out_done[k % 2].record(s_out)

    cur = torch.cuda.current_stream()
    for k in range(W):
        one(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for k in range(K):
        one(k)
    for st in (s_in, s_cmp):
        s_out.wait_stream(st)
    e1.record(s_out)
    torch.cuda.synchronize()
    cur.wait_stream(s_out)
    ms = e0.elapsed_time(e1) / K
    h2d = ha.numel() * 4 + hb.numel() * 4 + hx.numel() * 4
    d2h = hy.numel() * 4 + hxt.numel() * 4
    return ms, h2d, d2h


# ------------------------------------------------------ the other rows ----

FP32_LANES_PER_SM = 128   # FFMA lanes per SM (Blackwell SM: 4 partitions x 32)
IMAD_PER_FFMA = 0.5       # integer multiply-adds issue at half the FFMA rate
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense TF32 / bf16 tensor rates (the fallback when cuBLAS TF32 cannot be timed)


def cublas_tf32_tflops(n=8192, reps=5):
    """Dense TF32 tensor rate of cuBLAS on this GPU: a float32 n^3 matmul with
    TF32 allowed, best of `reps` after warm-up (the ceiling the 3xTF32
    contraction issues its products against)."""
    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn((n, n), device="cuda", generator=g)
        b = torch.randn((n, n), device="cuda", generator=g)
        for _ in range(3):
            a @ b
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            a @ b
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old


def fp32_alu_peak():
    """FFMA peak from unit counts and the maximum SM clock: SMs x 128 lanes x
    2 flop x clock (no measured FFMA figure is on file)."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    mhz = 2070.0
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        mhz = float(json.load(open(p)).get("sm_max_mhz", mhz))
    return props.multi_processor_count * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def time_events(fn, iters, warm=3, flush=None):
    """Median ms of fn() over iters runs, CUDA events on the current stream,
    each run preceded (outside its events) by an L2 flush when given."""
    s = torch.cuda.current_stream()
    for _ in range(warm):
        if flush is not None:
            flush()
        fn(s.cuda_stream)
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        fn(s.cuda_stream)
        e1.record(s)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts)


def _hbm_row(name, nbytes, ms, P, extra=None):
    gbs = nbytes / (ms * 1e-3) / 1e9
    r = {"ms": round(ms, 5), "bytes": nbytes, "achieved": round(gbs, 2), "unit": "GB/s",
         "bound": "hbm", "peak": P["hbm"], "frac": round(gbs / P["hbm"], 4)}
    r.update(extra or {})
    return r


class Rows:
    """One workload per remaining hot-path row, each driven through the C ABI
    on its own inputs and timed against its own ceiling."""

    def __init__(self, A, P, iters=20):
        self.A, self.P, self.iters = A, P, iters
        self.flush = l2_flush_buffer()
        self.launches = 0

    # C3a: softmax over rows of x[4096,1024] f32
    def softmax(self):
        from primitive_sm_graph_gb300 import programs as PR
        A = self.A
        x = SI.softmax_input(0).cuda()
        y = torch.empty_like(x)
        stages, epi = PR.softmax_rows("f32")
        vx, vy = A.view_of(x), A.view_of(y)
        fn = lambda st: A.psg_reduce_rows(stages, epi, [x], [vx], y, vy, stream=st)
        return fn, lambda ms: _hbm_row("softmax", 2 * x.numel() * 4, ms, self.P,
                                       {"workload": "softmax rows x[4096,1024] f32"})

    # C3b: RMSNorm x[8192,4096] bf16, w[4096] bf16, eps 1e-6, f32 accumulate
    def rmsnorm(self):
        from primitive_sm_graph_gb300 import programs as PR
        A = self.A
        xh, wh = SI.rmsnorm_input(0)
        x, w = xh.cuda(), wh.cuda()
        y = torch.empty_like(x)
        R, N = x.shape
        stages, epi = PR.rmsnorm(N, 1e-6, "bf16")
        vx, vw, vy = A.view_of(x), A.view_of(w, shape=(R, N), strides=(0, 1)), A.view_of(y)
        fn = lambda st: A.psg_reduce_rows(stages, epi, [x, w], [vx, vw], y, vy, stream=st)
        nbytes = 2 * x.numel() * 2 + N * 2
        return fn, lambda ms: _hbm_row("rmsnorm", nbytes, ms, self.P,
                                       {"workload": "RMSNorm x[8192,4096] bf16, w[4096], eps 1e-6"})

    def _contract(self, a, b, out_dtype):
        A = self.A
        M, K = a.shape
        N = b.shape[1]
        va = A.view_of(a, shape=(M, N, K), strides=(K, 0, 1))
        vb = A.view_of(b, shape=(M, N, K), strides=(0, 1, N))
        c = torch.empty((M, N), dtype=out_dtype, device="cuda")
        vc = A.view_of(c)
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        fn = lambda s: A.psg_contract(a, va, b, vb, c, vc, st, stream=s)
        return fn, 2.0 * M * N * K

    # The GPT block's MLP backward contraction (8192 x 2048 x 512, bf16) with
    # its ReLU-mask program fused into the epilogue, and without: profile
    # cases only (--profile-case), not bench rows
    def _gemm_epilogue(self, fused):
        A = self.A
        g = SI.gen(41)
        M, N, K = 8192, 2048, 512
        a = SI.normal((M, K), 0, 1, g, torch.bfloat16).cuda()
        b = SI.normal((K, N), 0, 1, g, torch.bfloat16).cuda()
        u = SI.normal((M, N), 0, 1, g, torch.bfloat16).cuda()
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        va = A.view_of(a, shape=(M, N, K), strides=(K, 0, 1))
        vb = A.view_of(b, shape=(M, N, K), strides=(0, 1, N))
        n = lambda op, x=0, y=0, z=0, dt="bf16": A.node(op, x, y, z, dtype=dt)
        prog = [n("CONST"), n("LOAD", 0), n("CMPLT", 0, 1), n("ACC", dt="f32"), n("CAST", 3), n("WHERE", 2, 4, 0)]
        epi = (prog, [u], [A.view_of(u)]) if fused else None
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        fn = lambda s: A.psg_contract(a, va, b, vb, c, A.view_of(c), st, stream=s, epilogue=epi)
        return fn, lambda ms: {"ms": round(ms, 5)}

    def gemm_epilogue_mask(self):
        return self._gemm_epilogue(True)

    def gemm_epilogue_plain(self):
        return self._gemm_epilogue(False)

    # C4a: bf16 A,B [8192,8192] -> bf16, f32 accumulate
    def gemm_bf16(self):
        a, b = SI.contraction_bf16(0)
        fn, flops = self._contract(a.cuda(), b.cuda(), torch.bfloat16)
        pk = self.P["bf16"]

        def fin(ms):
            tf = flops / (ms * 1e-3) / 1e12
            return {"ms": round(ms, 5), "flops": flops, "achieved": round(tf, 2), "unit": "TFLOP/s",
                    "bound": "tensor", "peak": pk, "peak_source": self.P["source"] + " cuBLAS bf16 burst",
                    "frac": round(tf / pk, 4),
                    "workload": "bf16 A[8192,8192] @ B[8192,8192] as MUL+SUM, f32 accumulate, bf16 out"}
        return fn, fin

    # C4b: f32 A,B [4096,4096] -> f32: 3xTF32 on the tensor cores
    def gemm_f32(self):
        a, b = SI.contraction_f32(0)
        fn, flops = self._contract(a.cuda(), b.cuda(), torch.float32)
        try:
            tf32 = cublas_tf32_tflops()
            src = "measured here: cuBLAS float32 8192^3 with TF32 allowed (best of 5)"
        except Exception:
            tf32 = self.P["bf16"] * TF32_PER_BF16
            src = "measured cuBLAS bf16 burst x nominal TF32/bf16 ratio (1.1/2.25)"
        ffma = fp32_alu_peak()

        def fin(ms):
            tf = flops / (ms * 1e-3) / 1e12          # float32 MUL+SUM flops per second
            pipe = 3 * tf                            # TF32 tensor flops issued (three products per term)
            return {"ms": round(ms, 5), "flops": flops, "achieved": round(tf, 2), "unit": "TFLOP/s",
                    "bound": "tensor", "peak": round(tf32 / 3, 2),
                    "peak_source": src + ", divided by the 3 TF32 products per float32 term",
                    "tf32_ceiling_tflops": round(tf32, 2),
                    "frac": round(pipe / tf32, 4),
                    "tf32_pipe_tflops": round(pipe, 2),
                    "ffma_ceiling": round(ffma, 2), "vs_ffma_ceiling": round(tf / ffma, 3),
                    "workload": "f32 A[4096,4096] @ B[4096,4096] as MUL+SUM (3xTF32, f32 accumulate)"}
        return fn, fin

    # integer MUL+SUM on the integer pipes: int8 operands, wrapping int32 total
    def gemm_i8(self):
        a, b = SI.contraction_i8(0)
        fn, ops = self._contract(a.cuda(), b.cuda(), torch.int32)
        pk = fp32_alu_peak() * IMAD_PER_FFMA

        def fin(ms):
            t = ops / (ms * 1e-3) / 1e12
            return {"ms": round(ms, 5), "ops": ops, "achieved": round(t, 2), "unit": "TOP/s", "bound": "alu",
                    "peak": round(pk, 2),
                    "peak_source": "derived: SMs x 64 IMAD lanes (half the FFMA lanes) x 2 ops x max SM clock",
                    "frac": round(t / pk, 4),
                    "workload": "int8 A[2048,2048] @ B[2048,2048] as MUL+SUM, uint32 wraparound total, int32 out"}
        return fn, fin

    # C5 shapes: token embedding gather and its scatter-add backward
    def gather(self):
        A = self.A
        tok, w = SI.gpt_block(0, **SI.GPT_SHAPES)
        E = w["E"].cuda()
        idx = tok.reshape(-1).cuda()
        n = idx.numel()
        out = torch.empty((n, E.shape[1]), dtype=E.dtype, device="cuda")
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        vE, vo = A.view_of(E), A.view_of(out)
        fn = lambda s: A.psg_gather(E, vE, idx, n, out, vo, st, stream=s)
        nbytes = out.numel() * 2 * 2 + n * 4   # rows read + written, indices
        return fn, lambda ms: _hbm_row("gather", nbytes, ms, self.P,
                                       {"workload": "E[256,512] bf16 gathered by 8192 int32 tokens"})

    def scatter(self):
        A = self.A
        tok, _ = SI.gpt_block(0, **SI.GPT_SHAPES)
        idx = tok.reshape(-1).cuda()
        n = idx.numel()
        g = SI.gen(1)
        upd = SI.normal((n, 512), 0.0, 1.0, g, torch.bfloat16).cuda()
        dst = torch.zeros((256, 512), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty((max(1, A.psg_scatter_workspace(n)),), dtype=torch.uint8, device="cuda")
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        vd, vu = A.view_of(dst), A.view_of(upd)
        fn = lambda s: A.psg_scatter_add(dst, vd, idx, n, upd, vu, ws, ws.numel(), st, stream=s)
        nbytes = upd.numel() * 2 + n * 4 + 2 * dst.numel() * 2
        return fn, lambda ms: _hbm_row("scatter", nbytes, ms, self.P,
                                       {"workload": "scatter-add of [8192,512] bf16 rows into [256,512]"})

    def copy_ms(self, nbytes):
        """A device-to-device copy moving the same bytes (half read, half
        written) in the same harness: the practical ceiling at this size,
        where launch and ramp costs weigh against the peak copy rate."""
        src = torch.empty(max(1, nbytes // 2), dtype=torch.uint8, device="cuda")
        dst = torch.empty_like(src)
        ms = time_events(lambda s: dst.copy_(src), self.iters, flush=self.flush)
        del src, dst
        return ms

    # C5 shapes: the fused attention forward + backward (B32, T256, H8, head dim 64)
    def attention(self):
        A = self.A
        B_, T, H = 32, 256, 8
        g = SI.gen(5)
        qkv = SI.normal((B_, T, 3, H, 64), 0, 1, g, torch.bfloat16).cuda()
        do = SI.normal((B_, T, H, 64), 0, 1, g, torch.bfloat16).cuda()
        vs = [A.view_of(qkv, shape=(B_, T, H, 64), strides=qkv[:, :, 0].stride(), offset=i * H * 64)
              for i in range(3)]
        o = torch.empty((B_, T, H, 64), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B_, H, T), dtype=torch.float32, device="cuda")
        delta = torch.empty_like(lse)
        dqkv = torch.empty_like(qkv)
        dvs = [A.view_of(dqkv, shape=(B_, T, H, 64), strides=dqkv[:, :, 0].stride(), offset=i * H * 64)
               for i in range(3)]
        vo, vdo = A.view_of(o), A.view_of(do)

        def fn(s):
            A.psg_attention_fwd(qkv, vs[0], qkv, vs[1], qkv, vs[2], o, vo, lse, 0.125, True, stream=s)
            A.psg_attention_bwd(qkv, vs[0], qkv, vs[1], qkv, vs[2], o, vo, do, vdo, lse, delta, dqkv, dvs[0],
                                dqkv, dvs[1], dqkv, dvs[2], 0.125, True, stream=s)
        return fn, self._attn_fin(B_, T, H, "fused attention fwd+bwd B32 T256 H8 hd64 causal bf16 (4 launches)")

    def _attn_fin(self, B_, T, H, workload):
        # the products' visible cells only: a causal row i has i + 1 keys
        per = 2.0 * B_ * H * 64 * (T * (T + 1) / 2)
        flops = 7 * per                       # forward: S, O; backward: S, dP, dV, dK, dQ
        pk = self.P["bf16"]

        def fin(ms):
            tf = flops / (ms * 1e-3) / 1e12
            return {"ms": round(ms, 5), "flops": flops, "achieved": round(tf, 2), "unit": "TFLOP/s",
                    "bound": "tensor", "peak": pk, "frac": round(tf / pk, 4),
                    "note": "FLOPs of the causal products' visible cells (T(T+1)/2 per head), 7 products",
                    "workload": workload}
        return fin

    # fused attention past one key block: the running softmax over 128-key blocks
    def attention_long(self):
        A = self.A
        B_, T, H = 2, 4096, 8
        g = SI.gen(6)
        qkv = SI.normal((B_, T, 3, H, 64), 0, 1, g, torch.bfloat16).cuda()
        do = SI.normal((B_, T, H, 64), 0, 1, g, torch.bfloat16).cuda()
        vs = [A.view_of(qkv, shape=(B_, T, H, 64), strides=qkv[:, :, 0].stride(), offset=i * H * 64)
              for i in range(3)]
        o = torch.empty((B_, T, H, 64), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B_, H, T), dtype=torch.float32, device="cuda")
        delta = torch.empty_like(lse)
        dqkv = torch.empty_like(qkv)
        dvs = [A.view_of(dqkv, shape=(B_, T, H, 64), strides=dqkv[:, :, 0].stride(), offset=i * H * 64)
               for i in range(3)]
        vo, vdo = A.view_of(o), A.view_of(do)

        def fn(s):
            A.psg_attention_fwd(qkv, vs[0], qkv, vs[1], qkv, vs[2], o, vo, lse, 0.125, True, stream=s)
            A.psg_attention_bwd(qkv, vs[0], qkv, vs[1], qkv, vs[2], o, vo, do, vdo, lse, delta, dqkv, dvs[0],
                                dqkv, dvs[1], dqkv, dvs[2], 0.125, True, stream=s)
        return fn, self._attn_fin(B_, T, H, "fused attention fwd+bwd B2 T4096 H8 hd64 causal bf16, "
                                            "32 key blocks (4 launches)")

    def stream_ms(self, nm, pairs=8, rounds=4):
        """Device ms per launch of row nm in steady state: a CUDA Graph of
        pairs x rounds back-to-back launches cycling through `pairs` distinct
        input/output sets (together more than twice the L2), so no launch finds
        its input in L2; timed with events around the replay."""
        from primitive_sm_graph_gb300 import programs as PR
        A = self.A
        if nm == "softmax":
            x0 = SI.softmax_input(0).cuda()
            xs = [x0.clone() for _ in range(pairs)]
            ys = [torch.empty_like(x0) for _ in range(pairs)]
            stages, epi = PR.softmax_rows("f32")
            calls = [(lambda st, x=x, y=y: A.psg_reduce_rows(stages, epi, [x], [A.view_of(x)], y, A.view_of(y),
                                                             stream=st)) for x, y in zip(xs, ys)]
        else:
            xh, wh = SI.rmsnorm_input(0)
            x0, w = xh.cuda(), wh.cuda()
            xs = [x0.clone() for _ in range(pairs)]
            ys = [torch.empty_like(x0) for _ in range(pairs)]
            R, N = x0.shape
            stages, epi = PR.rmsnorm(N, 1e-6, "bf16")
            vw = A.view_of(w, shape=(R, N), strides=(0, 1))
            calls = [(lambda st, x=x, y=y: A.psg_reduce_rows(stages, epi, [x, w], [A.view_of(x), vw], y,
                                                             A.view_of(y), stream=st)) for x, y in zip(xs, ys)]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for c in calls:
                c(side.cuda_stream)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            s = torch.cuda.current_stream().cuda_stream
            for _ in range(rounds):
                for c in calls:
                    c(s)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / (pairs * rounds))
        self.launches += 8 * pairs * rounds
        del g, xs, ys, calls
        torch.cuda.empty_cache()
        return statistics.median(ts)

    def run_kernel_rows(self, names):
        out = {}
        for nm in names:
            fn, fin = getattr(self, nm)()
            ms = time_events(fn, self.iters, flush=self.flush)
            self.launches += self.iters
            out[nm] = fin(ms)
            del fn
            torch.cuda.empty_cache()
            if out[nm].get("bound") == "hbm":
                cms = self.copy_ms(out[nm]["bytes"])
                out[nm]["copy_same_bytes_ms"] = round(cms, 5)
                out[nm]["frac_of_copy_same_bytes"] = round(cms / ms, 4)
            if nm in ("softmax", "rmsnorm"):
                sms = self.stream_ms(nm)
                gbs = out[nm]["bytes"] / (sms * 1e-3) / 1e9
                out[nm]["stream"] = {
                    "ms": round(sms, 5), "achieved": round(gbs, 2), "frac": round(gbs / self.P["hbm"], 4),
                    "how": "per launch over 32 back-to-back launches (one CUDA Graph) cycling through 8 distinct "
                           "input/output sets, more than twice the L2 together, so no launch finds its input "
                           "in L2; ms above is one launch after an L2 flush"}
        return out

    # C1: the tiny graph, eager realize and CUDA Graph replay
    def tiny_graph(self):
        from primitive_sm_graph_gb300 import graph as G
        from primitive_sm_graph_gb300.workloads import tiny_graph
        a, b = SI.tiny_graph(0)
        da, db = a.cuda(), b.cuda()

        def once():
            return tiny_graph(G.Tensor.from_torch(da), G.Tensor.from_torch(db)).realize()
        for _ in range(5):
            once()
        torch.cuda.synchronize()
        ex = G._executor()
        ex.log.clear()
        once()
        kernels = len(ex.log)
        n = 200
        t0 = time.perf_counter()
        for _ in range(n):
            once()
        torch.cuda.synchronize()
        eager_us = (time.perf_counter() - t0) / n * 1e6
        # the same with the plan cache off: every realize schedules afresh
        G.PLAN_CACHE = False
        try:
            t0 = time.perf_counter()
            for _ in range(n):
                once()
            torch.cuda.synchronize()
            fresh_us = (time.perf_counter() - t0) / n * 1e6
        finally:
            G.PLAN_CACHE = True
        r = {"eager_us_per_realize": round(eager_us, 2), "eager_unplanned_us_per_realize": round(fresh_us, 2),
             "kernels": kernels, "workload": "SUM(relu(A[64,32] @ B[32,48])^2) f32"}
        rep = G.Replay(lambda x, y: tiny_graph(G.Tensor.from_torch(x), G.Tensor.from_torch(y)).realize(), da, db)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            rep.replay()
        e1.record()
        torch.cuda.synchronize()
        r["graph_replay_us"] = round(e0.elapsed_time(e1) / n * 1e3, 3)
        # device time per realize: 20 realizes recorded in one CUDA Graph, so
        # the host's graph-launch call is paid once per 20 (one replay above is
        # bounded by that call)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            once()
        torch.cuda.current_stream().wait_stream(side)
        g20 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g20):
            for _ in range(20):
                once()
        g20.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(10):
            g20.replay()
        e1.record()
        torch.cuda.synchronize()
        r["graph_device_us"] = round(e0.elapsed_time(e1) / 200 * 1e3, 3)
        return r

    # C5: one forward + backward of the GPT block through the graph layer
    def gpt(self, steps=10):
        from primitive_sm_graph_gb300.workloads import gpt_step
        tok, w = SI.gpt_block(0, **SI.GPT_SHAPES)
        dtok = tok.cuda()
        dw = {k: v.cuda() for k, v in w.items()}
        H = SI.GPT_SHAPES["H"]
        gpt_step(dtok, dw, H)          # first call compiles the specialised kernels
        torch.cuda.synchronize()
        from primitive_sm_graph_gb300 import graph as G
        ex = G._executor()
        ts, kernels = [], 0
        for _ in range(steps):
            ex.log.clear()
            t0 = time.perf_counter()
            gpt_step(dtok, dw, H)
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
            kernels = len(ex.log)
        ms = statistics.median(ts) * 1e3
        # the same with the plan cache off: the step scheduled afresh
        G.PLAN_CACHE = False
        try:
            t0 = time.perf_counter()
            gpt_step(dtok, dw, H)
            torch.cuda.synchronize()
            fresh_ms = (time.perf_counter() - t0) * 1e3
        finally:
            G.PLAN_CACHE = True
        # the same step recorded once and replayed (device time, CUDA events)
        from primitive_sm_graph_gb300.workloads import GPT_WEIGHTS

        def fwd_bwd(t, *ws):
            loss, grads = gpt_step(t, dict(zip(GPT_WEIGHTS, ws)), H)
            return (loss,) + tuple(grads[k] for k in GPT_WEIGHTS)
        rep = G.Replay(fwd_bwd, dtok, *[dw[k] for k in GPT_WEIGHTS])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        e0.record()
        for _ in range(reps):
            rep.replay()
        e1.record()
        torch.cuda.synchronize()
        rms = e0.elapsed_time(e1) / reps
        # a training step: the same plus one AdamW step over the seven weights
        from primitive_sm_graph_gb300.workloads import AdamW, gpt_train_step
        tw = {k: v.clone() for k, v in dw.items()}
        opt = AdamW([tw[k] for k in GPT_WEIGHTS])
        trep = G.Replay(lambda t: gpt_train_step(t, tw, H, opt), dtok)
        e0.record()
        for _ in range(reps):
            trep.replay()
        e1.record()
        torch.cuda.synchronize()
        tms = e0.elapsed_time(e1) / reps
        # algorithmic flops of the contractions: 8192 tokens x 6,553,600 linear
        # + 2 x B*H*T*T*hd attention (QK^T and PV), times 3 for fwd + bwd
        Bn, T, V, D, Hh, F = (SI.GPT_SHAPES[k] for k in ("B", "T", "V", "D", "H", "F"))
        lin = 2 * Bn * T * (D * 3 * D + D * D + 2 * D * F + D * V)
        att = 2 * 2 * Bn * Hh * T * T * (D // Hh)
        flops = 3 * (lin + att)
        return {"ms_per_step": round(ms, 3), "unplanned_ms_per_step": round(fresh_ms, 3),
                "kernels_per_step": kernels, "flops": flops,
                "achieved": round(flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "replay_ms_per_step": round(rms, 4),
                "train_replay_ms_per_step": round(tms, 4),
                "replay_achieved": round(flops / (rms * 1e-3) / 1e12, 3),
                "note": "ms_per_step: host wall clock, graph building included, the schedule replayed "
                        "from the plan cache (unplanned_ms_per_step: scheduled afresh); "
                        "replay: the recorded step relaunched (CUDA Graph), device time; "
                        "train_replay: forward, backward and one AdamW step (one launch for all weights)",
                "workload": "1-layer byte GPT fwd+bwd B32 T256 V256 d512 H8 MLP2048 bf16"}


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


def oracle_rows(threads: int):
    """The oracle on a bounded sample of each other row's workload (the
    first rows of each input), OpenMP over output rows: {row: (seconds,
    units of the row's metric, unit, sample)}."""
    import oracle as O
    O.build()
    O.NTHREADS = threads
    out = {}
    x = SI.softmax_input(0)[:256]
    xs = O.T(x.numpy(), "f32")
    t0 = time.perf_counter()
    O.softmax_rows(xs)
    out["softmax"] = (time.perf_counter() - t0, 256 * 1024 * 8, "GB/s", "256 of 4096 rows")
    xr, wr = SI.rmsnorm_input(0)
    xo, wo = O.T(SI.bits(xr[:128]), "bf16"), O.T(SI.bits(wr), "bf16")
    t0 = time.perf_counter()
    O.rmsnorm(xo, wo)
    out["rmsnorm"] = (time.perf_counter() - t0, 128 * 4096 * 4, "GB/s", "128 of 8192 rows")
    a, b = SI.contraction_bf16(0)
    ao, bt = O.T(SI.bits(a[:32]), "bf16"), O.transpose(O.T(SI.bits(b), "bf16"))
    t0 = time.perf_counter()
    O.matmul_bt(ao, bt, "bf16")
    out["gemm_bf16"] = (time.perf_counter() - t0, 2 * 32 * 8192 * 8192, "TFLOP/s", "32 of 8192 rows of C")
    a, b = SI.contraction_f32(0)
    ao, bt = O.T(a[:32].numpy(), "f32"), O.transpose(O.T(b.numpy(), "f32"))
    t0 = time.perf_counter()
    O.matmul_bt(ao, bt, "f32")
    out["gemm_f32"] = (time.perf_counter() - t0, 2 * 32 * 4096 * 4096, "TFLOP/s", "32 of 4096 rows of C")
    return out


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


KERNEL_ROWS = ["softmax", "rmsnorm", "gemm_bf16", "gemm_f32", "gemm_i8", "gather", "scatter", "attention",
               "attention_long"]
ROW_NAMES = KERNEL_ROWS + ["tiny_graph", "gpt"]


def profile_case(A, name, iters):
    """One workload, iters launches, nothing timed: the command a profiler
    wraps to capture that kernel."""
    if name in ("chain", "transpose"):
        step = Step(A)
        fn = getattr(step, name)
    elif name == "gpt":
        from primitive_sm_graph_gb300.workloads import gpt_step
        tok, w = SI.gpt_block(0, **SI.GPT_SHAPES)
        dtok, dw = tok.cuda(), {k: v.cuda() for k, v in w.items()}

        def fn(_s):
            gpt_step(dtok, dw, SI.GPT_SHAPES["H"])
    else:
        fn, _ = getattr(Rows(A, peaks()), name)()
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(iters):
        fn(s)
    torch.cuda.synchronize()
    print("profile case", name, "x", iters, "ok", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", default="all",
                    help="comma list of extra rows to time (softmax,rmsnorm,gemm_bf16,gemm_f32,gemm_i8,"
                         "gather,scatter,attention,attention_long,tiny_graph,gpt), 'all' or 'none'")
    ap.add_argument("--profile-case", default=None,
                    help="run one workload --iters times and exit (for a profiler capture); "
                         "chain, transpose, gpt (one eager forward + backward) or a row name")
    ap.add_argument("--iters", type=int, default=3)
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

    if args.profile_case:
        return profile_case(A, args.profile_case, args.iters)
    step = Step(A)
    with Clocks(local) as clk:
        total_ms, chain_ms, tr_ms, wall = timed_steps(step, args.steps, args.warmup, dist)
    clocks = clk.summary()
    value, ms_step = whole_job_gbs(dist, world, STEP_BYTES, total_ms / args.steps)
    P = peaks()
    # dominant kernel: the one with the larger share of the step
    dom = ("transpose", TRANSPOSE_BYTES, tr_ms) if tr_ms >= chain_ms else ("chain", CHAIN_BYTES, chain_ms)
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        traffic = json.load(open(tp)).get(dom[0])
    e2e_ms, h2d, d2h = e2e_steps(step, max(8, args.steps // 2), 2)
    e2e_gbs, _ = whole_job_gbs(dist, world, STEP_BYTES, e2e_ms)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "chain y=WHERE(CMPLT(a,b),EXP(a*0.5),LOG(b*b+1)) a[4096,4096] "
                               "b[4096] expanded + permute(1,0) of x[8192,8192] f32",
                   "bytes_per_step": STEP_BYTES, "l2": "flushed before every step: 2x L2 write then 2x L2 read, outside the events",
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
    names = ROW_NAMES if args.rows == "all" else [r for r in args.rows.split(",") if r and r != "none"]
    if names:
        rows = Rows(A, P)
        kr = [n for n in names if n in KERNEL_ROWS]
        line["rows"] = rows.run_kernel_rows(kr)
        if "tiny_graph" in names:
            line["rows"]["tiny_graph"] = rows.tiny_graph()
        if "gpt" in names:
            line["rows"]["gpt"] = rows.gpt()
        if "gemm_bf16" in line["rows"]:
            line["mul_sum_tflops"] = line["rows"]["gemm_bf16"]["achieved"]
    if rank == 0 and not args.no_cpu_baseline:
        cores = cpu_cores()
        sec, nbytes = oracle_sample(cores)
        sec1, nbytes1 = oracle_sample(1, rows=64)  # one thread: the serial loops the team splits
        rows_cpu = {}
        for name, (s, units, unit, sample) in oracle_rows(cores).items():
            scale = 1e9 if unit == "GB/s" else 1e12
            rows_cpu[name] = {"value": round(units / s / scale, 6), "unit": unit, "sample": sample}
        line["cpu_baseline"] = {"value": round(nbytes / sec / 1e9, 4), "unit": "GB/s",
                                "cores": cores, "kind": "oracle",
                                "sample": "512 of 4096 chain rows + a 1024x8192 transpose slab",
                                "serial": {"value": round(nbytes1 / sec1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                                           "sample": "64 of 4096 chain rows + a 128x8192 transpose slab"},
                                "rows": rows_cpu}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
