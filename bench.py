#!/usr/bin/env python3
"""Benchmark of the NVFP4 router hot path on GB300.

One step = one pass of the whole path over one decode batch of T tokens:
  1. nvfp4_quantize               X [T, 7168] bf16 -> NVFP4 (one launch: a cluster
                                  meets on the global maximum in shared memory)
  2. nvfp4_gemm_topk              gate GEMM vs 256 NVFP4 experts, sqrt(softplus) + bias, top-8
  3. nvfp4_deinterleave_quantize  SwiGLU output [T, 2*2048] (granularity 8) -> NVFP4,
                                  on a side stream beside 1-2
Three kernel launches per step (the library counts its own launches; the
JSON line's gpu_launches is that count).  Inputs rotate over enough
independent sets (activations, weights, biases) that the working set is more
than twice the L2 cache, so every step reads HBM.  Steps are replayed from
CUDA graphs.  Detail lines time the other shapes of the pages (quantize
sweep, RMSNorm producer, prefill router, indexer, router variant, grouped MoE
projection).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle (the
only reference this path has) on a bounded sample instead.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_BYTES = 126 * 1024 * 1024
HIDDEN, EXPERTS, TOPK, INTER, GRAN = workloads.HIDDEN, workloads.EXPERTS, workloads.ROUTER_TOPK, \
    workloads.MOE_INTER, 8
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense NVFP4 / BF16 tensor ratio on GB300


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


# ---------------------------------------------------------------- algorithmic bytes

def quantize_bytes(rows, cols):
    """Read bf16 once, write codes + scale bytes + gs."""
    return rows * cols * 2 + rows * cols // 2 + rows * cols // 16 + 4


def gemm_bytes(M, N, K, k, bias=True):
    """A and B codes + scales, global scales, bias, top-k outputs (idx, score, weight)."""
    return (M + N) * (K // 2 + K // 16) + 8 + (N * 4 if bias else 0) + M * k * 12


def gemm_flops(M, N, K):
    return 2.0 * M * N * K


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.samples = []

    def __enter__(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def mark(self):
        return time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        for line in self.tmp.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                self.samples.append(dict(t=ts + frac, sm=float(parts[2]), sm_max=float(parts[3]),
                                         reasons=parts[5], hw=parts[6], hwt=parts[7], swt=parts[8],
                                         pcap=parts[9]))
            except (ValueError, IndexError):
                continue
        self.tmp.close()
        os.unlink(self.tmp.name)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s["t"] <= t1]
        window = "timed"
        if not inside:
            inside, window = self.samples, "run"
        if not inside:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"], window="none")
        reasons = set()
        for s in inside:
            if s["hw"] == "Active":
                reasons.add("hw_slowdown")
            if s["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if s["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if s["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return dict(sm_mhz=statistics.median(s["sm"] for s in inside),
                    sm_max_mhz=max(s["sm_max"] for s in inside), reasons=sorted(reasons),
                    samples=len(inside), window=window)


# ---------------------------------------------------------------- distributed helpers

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (identity for one process)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def throughput(rows_per_rank: int, steps: int, max_seconds: float, world: int) -> float:
    """Whole-job rows/s: rows of all ranks over the slowest rank's time."""
    return rows_per_rank * steps * world / max_seconds


# ---------------------------------------------------------------- the GPU arm

class RouterSets:
    """R rotating input sets of the router decode step, all on the device."""

    def __init__(self, nv, tokens, n_sets, ws, seed=1234):
        import torch
        self.tokens, self.n = tokens, n_sets
        rng = np.random.default_rng(seed)
        dev = "cuda"
        T = tokens
        # Each set's inputs sit in one arena ([x | h], bf16) and its outputs in
        # another, so the end-to-end run moves one buffer each way per step.
        self.xin = [torch.empty(T * HIDDEN + T * 2 * INTER, dtype=torch.int16, device=dev) for _ in range(n_sets)]
        self.x = [a[:T * HIDDEN].view(T, HIDDEN) for a in self.xin]
        self.h = [a[T * HIDDEN:].view(T, 2 * INTER) for a in self.xin]
        for i in range(n_sets):
            self.x[i].copy_(torch.from_numpy(workloads.bf16_bits(rng.standard_normal((T, HIDDEN), np.float32))
                                             .view(np.int16)))
            self.h[i].copy_(torch.from_numpy(workloads.bf16_bits(rng.standard_normal((T, 2 * INTER), np.float32))
                                             .view(np.int16)))
        self.bias = [torch.from_numpy((rng.standard_normal(EXPERTS) * 0.01).astype(np.float32)).to(dev)
                     for _ in range(n_sets)]
        # gate weights: drawn as bf16 N(0, 0.02) and quantized once by the library (static per layer)
        self.qb, self.sfb, self.gsb = [], [], []
        for _ in range(n_sets):
            w = torch.from_numpy(workloads.bf16_bits(rng.standard_normal((EXPERTS, HIDDEN), np.float32)
                                                     * np.float32(0.02)).view(np.int16)).to(dev)
            q, sf, gs = nv.quantize(w, ws)
            self.qb.append(q)
            self.sfb.append(sf)
            self.gsb.append(gs)
        e = lambda *s, dt=torch.uint8: [torch.empty(*s, dtype=dt, device=dev) for _ in range(n_sets)]
        self.qa, self.sfa, self.gsa = e(T, HIDDEN // 2), e(T, HIDDEN // 16), e(1, dt=torch.float32)
        # output arena: idx | score | weight | qh | sfh | gsh (16-byte aligned pieces)
        sizes = [T * TOPK * 4, T * TOPK * 4, T * TOPK * 4, T * INTER, T * INTER // 8, 4]
        offs = np.concatenate([[0], np.cumsum([(z + 15) // 16 * 16 for z in sizes])])
        self.out = [torch.empty(int(offs[-1]), dtype=torch.uint8, device=dev) for _ in range(n_sets)]
        piece = lambda a, j, dt, shape: a[int(offs[j]):int(offs[j]) + sizes[j]].view(dt).view(*shape)
        self.idx = [piece(a, 0, torch.int32, (T, TOPK)) for a in self.out]
        self.score = [piece(a, 1, torch.float32, (T, TOPK)) for a in self.out]
        self.weight = [piece(a, 2, torch.float32, (T, TOPK)) for a in self.out]
        self.qh = [piece(a, 3, torch.uint8, (T, INTER)) for a in self.out]
        self.sfh = [piece(a, 4, torch.uint8, (T, INTER // 8)) for a in self.out]
        self.gsh = [piece(a, 5, torch.float32, (1,)) for a in self.out]
        # The SwiGLU-output quantize does not depend on the router: it runs on a
        # second stream (with its own workspace) beside quantize -> GEMM.
        self.side = torch.cuda.Stream()
        self.ws2 = nv.workspace()
        torch.cuda.synchronize()

    def footprint(self):
        per = sum(t[0].numel() * t[0].element_size() for t in (
            self.x, self.h, self.bias, self.qb, self.sfb, self.qa, self.sfa, self.idx, self.score,
            self.weight, self.qh, self.sfh))
        return per * self.n

    # the three calls of one step on set i
    def op_quantize(self, nv, ws, i):
        nv.nvfp4_quantize(self.x[i], self.qa[i], self.sfa[i], self.gsa[i], ws)

    def op_gemm(self, nv, ws, i):
        nv.nvfp4_gemm_topk(self.qa[i], self.sfa[i], self.gsa[i], self.qb[i], self.sfb[i], self.gsb[i],
                           nv.EPILOGUE_SQRT_SOFTPLUS_BIAS, self.bias[i], TOPK, self.idx[i],
                           self.score[i], self.weight[i], None, ws)

    def op_deinterleave(self, nv, ws, i):
        nv.nvfp4_deinterleave_quantize(self.h[i], GRAN, self.qh[i], self.sfh[i], self.gsh[i], ws)

    def steps(self, nv, ws, indices, ready=None, done=None):
        """Steps on sets `indices`: quantize -> GEMM + top-k on the current
        stream, the SwiGLU-output quantize of each step on the side stream
        (forked once, joined once, so consecutive router kernels stay adjacent
        on their stream).  ready(i) may return an event that step i's inputs
        wait for, and done(i, main, side) is called once step i's work is
        enqueued on both streams (end-to-end copies)."""
        import torch
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        for i in indices:
            ev = ready(i) if ready is not None else None
            with torch.cuda.stream(self.side):
                if ev is not None:
                    self.side.wait_event(ev)
                self.op_deinterleave(nv, self.ws2, i)
            if ev is not None:
                main.wait_event(ev)
            self.op_quantize(nv, ws, i)
            self.op_gemm(nv, ws, i)
            if done is not None:
                done(i, main, self.side)
        main.wait_stream(self.side)

    def step(self, nv, ws, i):
        self.steps(nv, ws, [i])


def capture_runs(run, n_sets, chunk):
    """CUDA graphs of run(indices) for chunk-sized runs of consecutive sets,
    and of single sets (for a remainder)."""
    import torch
    run(range(n_sets))  # eager warm-up of every set (kernel attributes, tensor maps)
    torch.cuda.synchronize()
    graphs = []
    for c0 in range(0, n_sets, chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(range(c0, min(c0 + chunk, n_sets)))
        graphs.append(g)
    singles = []
    for i in range(chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run([i])
        singles.append(g)
    torch.cuda.synchronize()
    return graphs, singles


def capture_chunks(fn, n_sets, chunk):
    """CUDA graphs replaying fn(i) for chunk-sized runs of consecutive sets."""
    import torch
    graphs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(n_sets):  # eager warm-up of every set (kernel attributes, tensor maps)
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for c0 in range(0, n_sets, chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(c0, min(c0 + chunk, n_sets)):
                fn(i)
        graphs.append(g)
    singles = []
    for i in range(chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(i)
        singles.append(g)
    torch.cuda.synchronize()
    return graphs, singles


def replay_steps(graphs, singles, chunk, steps):
    """Replay exactly `steps` calls of fn (whole chunks, then single steps)."""
    full, rest = divmod(steps, chunk)
    for j in range(full):
        graphs[j % len(graphs)].replay()
    for j in range(rest):
        singles[j].replay()


def time_graphs(graphs, singles, chunk, steps, world):
    import torch
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    replay_steps(graphs, singles, chunk, steps)
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    return start.elapsed_time(end) / 1e3, t_wall0, t_wall1


def load_traffic(kernel_file: str, workload: str):
    """ncu DRAM bytes per launch recorded for a kernel source, if the source is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, "quantize_block_scaled_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for r in rec.get("records", []):
        if r.get("source") == kernel_file and r.get("sha") == sha and r.get("workload") == workload:
            return r.get("dram_bytes_per_launch")
    return None


def flush_l2(buf):
    """Evict L2: write one buffer larger than L2, then read another, so the
    timed call starts with clean (not dirty) lines of unrelated data."""
    half = buf.numel() // 2
    buf[:half].zero_()
    buf[half:].max()


def time_op_flushed(fn, iters, flush):
    """Average device time of fn() with an L2 flush before each call (flush not timed)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    fn()
    torch.cuda.synchronize()
    for a, b in evs:
        flush_l2(flush)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / iters / 1e3


class MoeL1:
    """The MoE first projection of one layer: 256 experts' [2I, 7168] gate/up
    weights (N(0, 0.02), drawn on the device per expert and quantized by the
    library, each with its own global scale), and the grouped activations of
    T tokens routed top-8 (the token rows gathered by expert, then quantized
    together).  Set-up only; the timed call is nvfp4_grouped_swiglu_gemm."""

    LIMIT = 10.0

    def __init__(self, nv, ws, seed=2048, experts=EXPERTS):
        import torch
        self.E = E = experts
        I, K = INTER, HIDDEN
        self.qb = torch.empty(E * 2 * I, K // 2, dtype=torch.uint8, device="cuda")
        self.sfb = torch.empty(E * 2 * I, K // 16, dtype=torch.uint8, device="cuda")
        self.gsb = torch.empty(E, dtype=torch.float32, device="cuda")
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        for e in range(E):
            w = (torch.randn(2 * I, K, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
            r = slice(e * 2 * I, (e + 1) * 2 * I)
            nv.nvfp4_quantize(w, self.qb[r], self.sfb[r], self.gsb[e:e + 1], ws)
        torch.cuda.synchronize()

    def batch(self, nv, ws, tokens, seed):
        import torch
        tok, offs = workloads.moe_routing(tokens, self.E, TOPK, seed)
        x = torch.from_numpy(workloads.quantize_input(tokens, seed=seed + 1).view(np.int16)).cuda()
        xg = x[torch.from_numpy(tok).cuda()].contiguous()
        qa, sfa, gsa = nv.quantize(xg, ws)
        out = torch.empty(xg.shape[0], INTER, dtype=torch.bfloat16, device="cuda")
        active = int((offs[1:] > offs[:-1]).sum())
        return dict(qa=qa, sfa=sfa, gsa=gsa, offs=torch.from_numpy(offs).cuda(), out=out, M=xg.shape[0],
                    active=active)

    def call(self, nv, ws, b):
        nv.nvfp4_grouped_swiglu_gemm(b["qa"], b["sfa"], b["gsa"], self.qb, self.sfb, self.gsb, b["offs"], INTER,
                                     GRAN, self.LIMIT, 0, b["out"], ws)

    def bytes(self, b):
        """A codes + scales, the used experts' weights (codes + scales), the
        global scales and offsets, the bf16 output."""
        K = HIDDEN
        return (b["M"] * (K // 2 + K // 16) + b["active"] * 2 * INTER * (K // 2 + K // 16)
                + self.E * 4 * 2 + 8 + b["M"] * INTER * 2)

    @staticmethod
    def flops(b):
        return 2.0 * b["M"] * 2 * INTER * HIDDEN


ROTATE_BYTES = int(2.2 * L2_BYTES)  # inputs rotated per timed pass: more than twice the L2 cache
ROTATE_MAX_SETS = 2048


def rotating_sets(bytes_per_call):
    """Input copies a rotation needs so that one pass reads more than 2.2x L2, or
    None when that takes more than ROTATE_MAX_SETS copies (then L2 is flushed)."""
    n = -(-ROTATE_BYTES // max(1, bytes_per_call))
    return max(2, n) if n <= ROTATE_MAX_SETS else None


def time_rotating(fn, n_sets, reps=3):
    """Average device time of fn(i) over one pass of i = 0 .. n_sets - 1 (each
    call on its own input copy, so the inputs come from HBM while the
    kernels' code stays in L2), replayed from a CUDA graph; eager replays if
    the calls cannot be captured."""
    import torch
    cur = torch.cuda.current_stream()
    s = torch.cuda.Stream()
    s.wait_stream(cur)
    with torch.cuda.stream(s):
        for i in range(n_sets):  # eager warm-up (kernel attributes, tensor maps)
            fn(i)
    cur.wait_stream(s)
    torch.cuda.synchronize()
    g = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_sets):
                fn(i)
        g.replay()
        torch.cuda.synchronize()
    except RuntimeError:
        g = None
        torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        if g is not None:
            g.replay()
        else:
            for i in range(n_sets):
                fn(i)
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / (reps * n_sets), ("graph" if g is not None else "eager")


def time_op(make_inputs, call, bytes_per_call, flush, iters=30):
    """(seconds per call, how): rotating input copies when a pass over them can
    exceed 2.2x L2 (make_inputs(i) builds copy i), else an L2 flush before each
    call on copy 0."""
    n = rotating_sets(bytes_per_call)
    if n is None:
        inp = make_inputs(0)
        return time_op_flushed(lambda: call(inp), iters, flush), "l2 flushed before each call"
    sets = [make_inputs(i) for i in range(n)]
    t, how = time_rotating(lambda i: call(sets[i]), n)
    return t, f"{n} rotating input copies ({n * bytes_per_call / 2**20:.0f} MiB), {how} replay"


def secondary(nv, ws, pk, flush):
    """Per-kernel figures on the other pages' shapes: inputs rotated over more
    than twice the L2 cache where that is possible, else L2 flushed per call."""
    import torch
    out = {}
    hbm = pk["hbm_gbs"] * 1e9
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16 * 1e12
    # quantize sweep
    sweep = {}
    for T in (1, 128, 2048, 16384):
        x0 = torch.from_numpy(workloads.quantize_input(T).view(np.int16)).cuda()
        q, sf, gs = nv.quantize(x0, ws)
        t, how = time_op(lambda i: x0 if i == 0 else x0.clone(), lambda x: nv.nvfp4_quantize(x, q, sf, gs, ws),
                         T * HIDDEN * 2, flush, 10 if T > 2048 else 30)
        b = quantize_bytes(T, HIDDEN)
        sweep[f"T{T}"] = dict(us=round(t * 1e6, 2), gbs=round(b / t / 1e9, 1), hbm_frac=round(b / t / hbm, 3), l2=how)
        del x0, q, sf, gs
        torch.cuda.empty_cache()
    hh = torch.from_numpy(workloads.swiglu_interleaved(2048).view(np.int16)).cuda()
    q, sf, gs = nv.deinterleave_quantize(hh, GRAN, ws)
    t, how = time_op(lambda i: hh if i == 0 else hh.clone(),
                     lambda h: nv.nvfp4_deinterleave_quantize(h, GRAN, q, sf, gs, ws), hh.numel() * 2, flush)
    b = quantize_bytes(2048, 2 * INTER)
    sweep["deinterleave_T2048_g8"] = dict(us=round(t * 1e6, 2), gbs=round(b / t / 1e9, 1),
                                          hbm_frac=round(b / t / hbm, 3), l2=how)
    del hh, q, sf, gs
    # NEXT-2: RMSNorm fused into the quantize (the norm output never reaches HBM)
    rng = np.random.default_rng(7)
    wn = torch.from_numpy(workloads.bf16_bits((1.0 + 0.1 * rng.standard_normal(HIDDEN)).astype(np.float32))
                          .view(np.int16)).cuda()
    for T in (32, 2048):
        x0 = torch.from_numpy(workloads.quantize_input(T).view(np.int16)).cuda()
        q, sf, gs = nv.rmsnorm_quantize(x0, wn, 1e-6, ws)
        t, how = time_op(lambda i: x0 if i == 0 else x0.clone(),
                         lambda x: nv.nvfp4_rmsnorm_quantize(x, wn, 1e-6, q, sf, gs, ws), T * HIDDEN * 2, flush)
        b = quantize_bytes(T, HIDDEN) + HIDDEN * 2
        sweep[f"rmsnorm_T{T}"] = dict(us=round(t * 1e6, 2), gbs=round(b / t / 1e9, 1), hbm_frac=round(b / t / hbm, 3),
                                      l2=how)
        del x0, q, sf, gs
    torch.cuda.empty_cache()
    out["quantize"] = sweep
    # router prefill T = 8192 (Student-t activations with outliers)
    d = workloads.router_prefill()
    x = torch.from_numpy(d["x"].view(np.int16)).cuda()
    w = torch.from_numpy(d["w"].view(np.int16)).cuda()
    bias = torch.from_numpy(d["bias"]).cuda()
    qa, sfa, gsa = nv.quantize(x, ws)
    qb, sfb, gsb = nv.quantize(w, ws)
    M = x.shape[0]
    idx = torch.empty(M, TOPK, dtype=torch.int32, device="cuda")
    sc = torch.empty(M, TOPK, dtype=torch.float32, device="cuda")
    wt = torch.empty(M, TOPK, dtype=torch.float32, device="cuda")
    tq, how_q = time_op(lambda i: x if i == 0 else x.clone(), lambda xx: nv.nvfp4_quantize(xx, qa, sfa, gsa, ws),
                        x.numel() * 2, flush, 10)
    nv.nvfp4_quantize(x, qa, sfa, gsa, ws)
    tg, how_g = time_op(lambda i: (qa, sfa) if i == 0 else (qa.clone(), sfa.clone()),
                        lambda a: nv.nvfp4_gemm_topk(a[0], a[1], gsa, qb, sfb, gsb, 1, bias, TOPK, idx, sc, wt,
                                                     None, ws),
                        qa.numel() + sfa.numel(), flush, 10)
    fl, by = gemm_flops(M, EXPERTS, HIDDEN), gemm_bytes(M, EXPERTS, HIDDEN, TOPK)
    out["router_prefill_T8192"] = dict(
        quantize_us=round(tq * 1e6, 2), gemm_topk_us=round(tg * 1e6, 2),
        gemm_tflops=round(fl / tg / 1e12, 1), fp4_tensor_frac=round(fl / tg / fp4_peak, 3),
        gemm_hbm_frac=round(by / tg / hbm, 3), rows_per_s=round(M / (tq + tg), 1), l2_quantize=how_q, l2_gemm=how_g)
    torch.cuda.empty_cache()
    del x, w, qa, sfa, qb, sfb, idx, sc, wt
    # indexer-shaped scoring
    d = workloads.indexer()
    qa, sfa, gsa = nv.quantize(torch.from_numpy(d["x"].view(np.int16)).cuda(), ws)
    qb, sfb, gsb = nv.quantize(torch.from_numpy(d["w"].view(np.int16)).cuda(), ws)
    M, N, K, k = 64, workloads.INDEXER_KEYS, workloads.INDEXER_DIM, workloads.INDEXER_TOPK
    idx = torch.empty(M, k, dtype=torch.int32, device="cuda")
    sc = torch.empty(M, k, dtype=torch.float32, device="cuda")
    keys = lambda i: (qb, sfb) if i == 0 else (qb.clone(), sfb.clone())  # the keys stream from HBM per call
    ti, how = time_op(keys, lambda kk: nv.nvfp4_gemm_topk(qa, sfa, gsa, kk[0], kk[1], gsb, 0, None, k, idx, sc, None,
                                                         None, ws), qb.numel() + sfb.numel(), flush)
    by = gemm_bytes(M, N, K, k, bias=False) - M * k * 4
    out["indexer_M64_N2048_k512"] = dict(us=round(ti * 1e6, 2), hbm_frac=round(by / ti / hbm, 4),
                                         rows_per_s=round(M / ti, 1), l2=how)
    # NEXT-1: the indexer's weighted ReLU head sum fused in (one token, 64 heads x 128 dims)
    hw = torch.from_numpy((np.random.default_rng(64).standard_normal((1, 64)) / 8).astype(np.float32)).cuda()
    qa, sfa, gsa = nv.quantize(torch.from_numpy(d["x"].view(np.int16)).cuda(), ws)
    qb, sfb, gsb = nv.quantize(torch.from_numpy(d["w"].view(np.int16)).cuda(), ws)
    idx1 = torch.empty(1, k, dtype=torch.int32, device="cuda")
    sc1 = torch.empty(1, k, dtype=torch.float32, device="cuda")
    th, how = time_op(lambda i: (qb, sfb) if i == 0 else (qb.clone(), sfb.clone()),
                      lambda kk: nv.nvfp4_indexer_topk(qa, sfa, gsa, kk[0], kk[1], gsb, 64, hw, k, idx1, sc1, None, ws),
                      qb.numel() + sfb.numel(), flush)
    by = gemm_bytes(64, N, K, k, bias=False) - 64 * k * 12 + k * 8 + 64 * 4
    out["indexer_heads64_T1_N2048_k512"] = dict(us=round(th * 1e6, 2), hbm_frac=round(by / th / hbm, 4),
                                                tokens_per_s=round(1 / th, 1), l2=how)
    torch.cuda.empty_cache()
    # router variant: 384 experts, top-6, normalised gating weights (decode, T = 32)
    rng = np.random.default_rng(384)
    E, kv = 384, 6
    xv = torch.from_numpy(workloads.bf16_bits(rng.standard_normal((32, HIDDEN), np.float32))
                          .view(np.int16)).cuda()
    wv = torch.from_numpy(workloads.bf16_bits(rng.standard_normal((E, HIDDEN), np.float32) * np.float32(0.02))
                          .view(np.int16)).cuda()
    bv = torch.from_numpy((rng.standard_normal(E) * 0.01).astype(np.float32)).cuda()
    qa, sfa, gsa = nv.quantize(xv, ws)
    qb, sfb, gsb = nv.quantize(wv, ws)
    idx = torch.empty(32, kv, dtype=torch.int32, device="cuda")
    sc = torch.empty(32, kv, dtype=torch.float32, device="cuda")
    wt = torch.empty(32, kv, dtype=torch.float32, device="cuda")
    tv, how = time_op(lambda i: (qb, sfb) if i == 0 else (qb.clone(), sfb.clone()),
                      lambda w_: nv.nvfp4_gemm_topk(qa, sfa, gsa, w_[0], w_[1], gsb, nv.EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM,
                                                    bv, kv, idx, sc, wt, None, ws),
                      qb.numel() + sfb.numel(), flush)
    by = gemm_bytes(32, E, HIDDEN, kv)
    out["router_E384_k6_norm_decode_T32"] = dict(us=round(tv * 1e6, 2), hbm_frac=round(by / tv / hbm, 4),
                                                 rows_per_s=round(32 / tv, 1), l2=how)
    # NEXT-4: grouped NVFP4 GEMM + SwiGLU, MoE first projection (256 experts,
    # I = 2048, granularity 8, limit 10): decode (32 tokens x top-8) and
    # prefill (8192 tokens x top-8)
    moe = MoeL1(nv, ws)
    for T, seed in ((32, 90), (8192, 91)):
        b = moe.batch(nv, ws, T, seed)
        tm = time_op_flushed(lambda: moe.call(nv, ws, b), 10 if T > 32 else 20, flush)
        by, fl = moe.bytes(b), MoeL1.flops(b)
        out[f"moe_l1_T{T}_E256_I2048"] = dict(
            us=round(tm * 1e6, 2), rows=b["M"], active_experts=b["active"], gbs=round(by / tm / 1e9, 1),
            hbm_frac=round(by / tm / hbm, 3), tflops=round(fl / tm / 1e12, 1),
            fp4_tensor_frac=round(fl / tm / fp4_peak, 3), tokens_per_s=round(T / tm, 1))
        del b
    del moe
    torch.cuda.synchronize()
    return out


def run_gpu(args, rank, world, local):
    import torch
    import quantize_block_scaled_gb300 as nv
    torch.cuda.set_device(local)
    pk = peaks()
    ws = nv.workspace()
    T = args.tokens
    per_set = (T * HIDDEN * 2 + T * 2 * INTER * 2 + EXPERTS * (HIDDEN // 2 + HIDDEN // 16) + EXPERTS * 4
               + T * (HIDDEN // 2 + HIDDEN // 16) + T * (INTER + INTER // 8) + T * TOPK * 12)
    n_sets = max(16, int(np.ceil(2.2 * L2_BYTES / per_set)))
    chunk = 16
    n_sets = int(np.ceil(n_sets / chunk) * chunk)
    sets = RouterSets(nv, T, n_sets, ws)
    # kernels one step launches (counted by the library itself)
    torch.cuda.synchronize()
    before = nv.kernel_launches()
    sets.step(nv, ws, 0)
    kernels_per_step = nv.kernel_launches() - before
    torch.cuda.synchronize()

    graphs, singles = capture_runs(lambda idx: sets.steps(nv, ws, idx), n_sets, chunk)
    with ClockSampler(local) as clk:
        replay_steps(graphs, singles, chunk, args.warmup)
        secs, t0, t1 = time_graphs(graphs, singles, chunk, args.steps, world)
    secs_max = reduce_max(secs, world)
    value = throughput(T, args.steps, secs_max, world)

    # per-op average launch durations (same sets, back-to-back graph replays)
    op_times = {}
    for name, fn in (("quantize", sets.op_quantize), ("gemm_topk", sets.op_gemm),
                     ("deinterleave_quantize", sets.op_deinterleave)):
        g, s1 = capture_chunks(lambda i, fn=fn: fn(nv, ws, i), n_sets, chunk)
        replay_steps(g, s1, chunk, n_sets)
        n_ops = max(args.steps, n_sets)
        t_op, _, _ = time_graphs(g, s1, chunk, n_ops, 1)
        op_times[name] = t_op / n_ops
        del g, s1
    op_bytes = dict(quantize=quantize_bytes(T, HIDDEN),
                    gemm_topk=gemm_bytes(T, EXPERTS, HIDDEN, TOPK),
                    deinterleave_quantize=quantize_bytes(T, 2 * INTER))
    dominant = max(op_times, key=op_times.get)
    achieved = op_bytes[dominant] / op_times[dominant] / 1e9
    kernel_file = dict(quantize="quantize.cu", gemm_topk="gemm_topk.cu",
                       deinterleave_quantize="quantize.cu")[dominant]
    traffic = load_traffic(kernel_file, f"{dominant}_router_decode_T{T}")
    roofline = dict(bound="hbm", achieved=round(achieved, 1), peak=pk["hbm_gbs"], unit="GB/s",
                    frac=round(achieved / pk["hbm_gbs"], 4), traffic=traffic, kernel=dominant,
                    algorithmic_bytes=op_bytes[dominant], launch_us=round(op_times[dominant] * 1e6, 3),
                    peak_source=pk["source"])

    # End to end through the public API with host buffers (pinned), copies
    # inside the timed region: every step copies its own inputs in (one
    # arena, [x | h]) and its results out (one arena: router top-k and the
    # SwiGLU-output codes, scales and global scale).  The copies run on
    # their own streams, so step i + 1's inputs travel while step i computes
    # and step i's results travel while step i + 1 computes; the timed region
    # ends after the last step's results are on the host.
    hin = [torch.empty(a.numel(), dtype=torch.int16, pin_memory=True) for a in sets.xin]
    hout = [torch.empty(a.numel(), dtype=torch.uint8, pin_memory=True) for a in sets.out]
    for i in range(n_sets):
        hin[i].copy_(sets.xin[i].cpu())
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_steps(indices):
        main = torch.cuda.current_stream()
        h2d_s.wait_stream(main)
        landed = {}
        for i in indices:  # every step's inputs, in order, on the copy-in stream
            with torch.cuda.stream(h2d_s):
                sets.xin[i].copy_(hin[i], non_blocking=True)
                landed[i] = torch.cuda.Event()
                landed[i].record(h2d_s)
        d2h_s.wait_stream(main)

        def results_out(i, m, side):  # step i's results leave once both its streams are done with it
            for st in (m, side):
                ev = torch.cuda.Event()
                ev.record(st)
                d2h_s.wait_event(ev)
            with torch.cuda.stream(d2h_s):
                hout[i].copy_(sets.out[i], non_blocking=True)

        sets.steps(nv, ws, indices, ready=lambda i: landed[i], done=results_out)
        main.wait_stream(h2d_s)
        main.wait_stream(d2h_s)

    ge, se = capture_runs(e2e_steps, n_sets, chunk)
    replay_steps(ge, se, chunk, min(args.warmup, n_sets))
    e2e_secs, _, _ = time_graphs(ge, se, chunk, args.steps, world)
    e2e_secs = reduce_max(e2e_secs, world)
    h2d = sets.xin[0].numel() * 2
    d2h = sets.out[0].numel()
    e2e = dict(value=round(throughput(T, args.steps, e2e_secs, world), 1), unit="rows/s",
               h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h)
    # the copies really ran: every set's host results equal its device results
    torch.cuda.synchronize()
    for i in range(n_sets):
        assert torch.equal(hout[i], sets.out[i].cpu()), "end-to-end results differ from the device results"

    status = nv.read_device_status(ws)
    detail = None
    if not args.quick and rank == 0:
        flush = torch.zeros(4 * L2_BYTES, dtype=torch.uint8, device="cuda")
        detail = secondary(nv, ws, pk, flush)
        del flush
    clocks = clk.summary(t0, t1)
    return dict(value=value, secs=secs_max, kernels_per_step=kernels_per_step, roofline=roofline, e2e=e2e, op_us={k: round(v * 1e6, 3)
                for k, v in op_times.items()}, clocks=clocks, detail=detail, n_sets=n_sets,
                footprint=sets.footprint(), device_status=status)


# ---------------------------------------------------------------- the CPU oracle

def oracle_step(orc, x, h, w_q, bias, rows, threads):
    """The oracle's pass over the sample rows of one step (gs over the whole batch)."""
    gsa = orc.global_scale(x)
    qa, sfa = orc.quantize_rows(x, gsa, 0, rows)
    qb, sfb, gsb = w_q
    orc.gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 1, bias, TOPK, threads=threads)
    orc.deinterleave_quantize(h[:rows], GRAN)


def run_oracle(T, sample_rows, steps, budget_s=None, threads=None):
    import oracle as orc
    orc.build()
    rng = np.random.default_rng(1234)
    x = workloads.bf16_bits(rng.standard_normal((T, HIDDEN), np.float32))
    h = workloads.bf16_bits(rng.standard_normal((T, 2 * INTER), np.float32))
    bias = (rng.standard_normal(EXPERTS) * 0.01).astype(np.float32)
    w = workloads.bf16_bits(rng.standard_normal((EXPERTS, HIDDEN), np.float32) * np.float32(0.02))
    w_q = orc.quantize(w)  # static weight quantization, outside the timed steps
    threads = threads or min(os.cpu_count() or 1, sample_rows)
    done = 0
    t0 = time.perf_counter()
    while done < steps:
        oracle_step(orc, x, h, w_q, bias, sample_rows, threads)
        done += 1
        if budget_s is not None and time.perf_counter() - t0 > budget_s and done >= 3:
            break
    secs = time.perf_counter() - t0
    return dict(value=sample_rows * done / secs, steps=done, secs=secs, cores=threads)


# ---------------------------------------------------------------- profiling hook

def run_profile(kind: str, iters: int):
    """Eager runs of one workload inside an NVTX range named "profile" (for ncu --nvtx)."""
    import torch
    import quantize_block_scaled_gb300 as nv
    ws = nv.workspace()
    if kind == "decode":
        sets = RouterSets(nv, 32, 4, ws)
        fns = [lambda i=i: sets.step(nv, ws, i) for i in range(4)]
    elif kind == "prefill":
        d = workloads.router_prefill()
        x = torch.from_numpy(d["x"].view(np.int16)).cuda()
        w = torch.from_numpy(d["w"].view(np.int16)).cuda()
        bias = torch.from_numpy(d["bias"]).cuda()
        qb, sfb, gsb = nv.quantize(w, ws)
        M = x.shape[0]
        qa = torch.empty(M, HIDDEN // 2, dtype=torch.uint8, device="cuda")
        sfa = torch.empty(M, HIDDEN // 16, dtype=torch.uint8, device="cuda")
        gsa = torch.empty(1, dtype=torch.float32, device="cuda")
        out = [torch.empty(M, TOPK, dtype=dt, device="cuda") for dt in (torch.int32, torch.float32, torch.float32)]

        def f():
            nv.nvfp4_quantize(x, qa, sfa, gsa, ws)
            nv.nvfp4_gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 1, bias, TOPK, *out, None, ws)
        fns = [f]
    elif kind in ("quantize", "quantize2048"):
        x = torch.from_numpy(workloads.quantize_input(16384 if kind == "quantize" else 2048)
                             .view(np.int16)).cuda()
        q, sf, gs = nv.quantize(x, ws)
        fns = [lambda: nv.nvfp4_quantize(x, q, sf, gs, ws)]
    elif kind == "rmsnorm2048":
        x = torch.from_numpy(workloads.quantize_input(2048).view(np.int16)).cuda()
        wn = torch.ones(HIDDEN, dtype=torch.bfloat16, device="cuda")
        q, sf, gs = nv.rmsnorm_quantize(x, wn, 1e-6, ws)
        fns = [lambda: nv.nvfp4_rmsnorm_quantize(x, wn, 1e-6, q, sf, gs, ws)]
    elif kind == "indexer_heads":
        d = workloads.indexer()
        qa, sfa, gsa = nv.quantize(torch.from_numpy(d["x"].view(np.int16)).cuda(), ws)
        qb, sfb, gsb = nv.quantize(torch.from_numpy(d["w"].view(np.int16)).cuda(), ws)
        hw = torch.full((1, 64), 0.125, dtype=torch.float32, device="cuda")
        idx = torch.empty(1, 512, dtype=torch.int32, device="cuda")
        sc = torch.empty(1, 512, dtype=torch.float32, device="cuda")
        fns = [lambda: nv.nvfp4_indexer_topk(qa, sfa, gsa, qb, sfb, gsb, 64, hw, 512, idx, sc, None, ws)]
    elif kind in ("moe_decode", "moe_prefill", "moe_small"):
        # moe_small: 32 experts (0.5 GB of weights), 1024 tokens: a capture-sized
        # case with full 128-row tiles
        moe = MoeL1(nv, ws, experts=32 if kind == "moe_small" else EXPERTS)
        b = moe.batch(nv, ws, {"moe_decode": 32, "moe_prefill": 8192, "moe_small": 1024}[kind], 90)
        fns = [lambda: moe.call(nv, ws, b)]
    elif kind == "indexer":
        d = workloads.indexer()
        qa, sfa, gsa = nv.quantize(torch.from_numpy(d["x"].view(np.int16)).cuda(), ws)
        qb, sfb, gsb = nv.quantize(torch.from_numpy(d["w"].view(np.int16)).cuda(), ws)
        idx = torch.empty(64, 512, dtype=torch.int32, device="cuda")
        sc = torch.empty(64, 512, dtype=torch.float32, device="cuda")
        fns = [lambda: nv.nvfp4_gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 0, None, 512, idx, sc, None, None, ws)]
    else:
        raise ValueError(kind)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("profile")
    for i in range(iters):
        fns[i % len(fns)]()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    assert nv.read_device_status(ws) == 0
    print(f"profile {kind}: {iters} iterations", flush=True)


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--tokens", type=int, default=32, choices=(1, 32))
    ap.add_argument("--quick", action="store_true", help="skip the secondary per-config figures")
    ap.add_argument("--profile", choices=("decode", "prefill", "quantize", "quantize2048", "indexer",
                                          "indexer_heads", "rmsnorm2048", "moe_decode", "moe_prefill", "moe_small"),
                    help="run --warmup eager iterations of one workload in an NVTX range and exit")
    args = ap.parse_args()
    if args.profile:
        run_profile(args.profile, args.warmup)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_setup(args.gpus)
    T = args.tokens
    config = dict(workload="router_decode", tokens=T, hidden=HIDDEN, experts=EXPERTS, top_k=TOPK,
                  swiglu_inter=INTER, interleave_granularity=GRAN, parallelism=f"replicas{world}")
    metric = f"router_decode_T{T}_rows_per_s"

    if args.impl == "reference":
        if rank != 0:
            return
        r = run_oracle(T, 1, args.steps)
        line = dict(impl="reference", metric=metric, value=round(r["value"], 3), unit="rows/s",
                    n_gpus=world, steps=args.steps, warmup=args.warmup,
                    ms_per_step=round(r["secs"] / r["steps"] * 1e3, 3), higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="f32/f64", data="synthetic",
                    config=dict(config, sample="1 token row per step (gs over the full batch)"),
                    cpu_baseline=dict(value=round(r["value"], 3), unit="rows/s", cores=r["cores"],
                                      kind="oracle", sample="1 token row per step"),
                    e2e=dict(value=round(r["value"], 3), unit="rows/s", h2d_bytes_per_step=0,
                             d2h_bytes_per_step=0))
        print(json.dumps(line), flush=True)
        return

    res = run_gpu(args, rank, world, local)
    cpu = None
    if rank == 0 and world == 1:
        c = run_oracle(T, T, 10 ** 6, budget_s=12.0)
        cpu = dict(value=round(c["value"], 2), unit="rows/s", cores=c["cores"], kind="oracle",
                   sample=f"{c['steps']} full steps of T={T} rows ({c['secs']:.1f} s)")
    if rank != 0:
        return
    config["l2"] = (f"{res['n_sets']} rotating input sets, {res['footprint'] / 2**20:.0f} MiB "
                    f"(> 2x L2); no flush inside the timed region")
    line = dict(metric=metric, value=round(res["value"], 1), unit="rows/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup,
                ms_per_step=round(res["secs"] / args.steps * 1e3, 5), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="nvfp4-e2m1/f32", data="synthetic",
                config=config, roofline=res["roofline"], cpu_baseline=cpu, e2e=res["e2e"],
                gpu_launches=res["kernels_per_step"] * args.steps, clocks=res["clocks"],
                op_us=res["op_us"], device_status=res["device_status"], detail=res["detail"])
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
