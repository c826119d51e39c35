#!/usr/bin/env python3
"""Benchmark of the NVFP4 router hot path on GB300.

Headline step (router prefill, the largest single-GPU workload): one pass of
the whole path over one batch of T = 8192 tokens of hidden size 7168
(Student-t(3) activations with 0.01% of the entries set to +-U(500, 2000)):
  1. nvfp4_quantize    X [8192, 7168] bf16 -> NVFP4 (grid-wide amax -> global
                       scale, E4M3 block scales, E2M1 codes)
  2. nvfp4_gemm_topk   block-scaled FP4 GEMM against 256 NVFP4 gate rows,
                       sqrt(softplus) + bias, top-8 per token
Two kernel launches per step (the library counts its own launches; the JSON
line's gpu_launches is that count over the timed region).  Three input sets
(activations, gate weights, biases: 352 MB) rotate, so every step reads its
activations from HBM.  Steps are replayed from CUDA graphs; the timed region
is many back-to-back windows of --steps steps each, and the headline is the
median window.  Detail lines give the router decode step (T = 32 and T = 1)
with the same fields, and per-kernel figures on the pages' other shapes
(quantize sweep, deinterleave, RMSNorm producer, indexer, router variant,
grouped MoE projection).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle (the
only reference this path has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import shutil
import signal
import statistics
import subprocess
import sys
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
PREFILL_TOKENS = 8192
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense NVFP4 / BF16 tensor ratio on GB300


def peaks():
    """HBM copy bandwidth and the dense FP4 tensor peak (the measured bf16
    GEMM rate times the nominal FP4/BF16 ratio of 6)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        pk = dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]), source="measured")
    else:
        pk = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")
    pk["fp4_tflops"] = pk["bf16_tflops"] * FP4_OVER_BF16
    return pk


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

SMI_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_smi_line(line: str):
    """One `nvidia-smi --query-gpu=SMI_FIELDS --format=csv,noheader,nounits`
    line -> a sample dict, or None for a line that is not a sample."""
    parts = [p.strip() for p in line.split(",")]
    if len(parts) < 10:
        return None
    try:
        stamp = parts[0]
        ts = time.mktime(time.strptime(stamp.split(".")[0], "%Y/%m/%d %H:%M:%S"))
        frac = float("0." + stamp.split(".")[1]) if "." in stamp else 0.0
        return dict(t=ts + frac, sm=float(parts[2]), sm_max=float(parts[3]), reasons=parts[5], hw=parts[6],
                    hwt=parts[7], swt=parts[8], pcap=parts[9])
    except (ValueError, IndexError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background: lines are read
    from a pipe as nvidia-smi prints them (line-buffered through stdbuf when
    it is there), and it is stopped with SIGINT, so no sample is lost in a
    buffer when it stops."""

    def __init__(self, index: int, period_ms: int = 20):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.samples = []
        self.reader = None

    def _read(self):
        for line in self.proc.stdout:
            s = parse_smi_line(line)
            if s is not None:
                self.samples.append(s)

    def __enter__(self):
        cmd = ["nvidia-smi", f"--id={self.index}", f"--query-gpu={SMI_FIELDS}",
               "--format=csv,noheader,nounits", f"-lms={self.period_ms}"]
        if shutil.which("stdbuf"):
            cmd = ["stdbuf", "-oL"] + cmd
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.send_signal(signal.SIGINT)
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.reader.join(timeout=5)

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


# ---------------------------------------------------------------- inputs on the device

def device_student_t(gen, rows, cols, nu=3, frac=1e-4, lo=500.0, hi=2000.0):
    """bf16 [rows, cols] Student-t(nu) (= Z / sqrt(chi2_nu / nu)) with `frac`
    of the entries replaced by +-U(lo, hi): the prefill activations of the
    router workload, drawn on the device from a seeded generator."""
    import torch
    z = torch.randn(rows, cols, generator=gen, device="cuda")
    chi2 = torch.zeros(rows, cols, device="cuda")
    for _ in range(nu):
        t = torch.randn(rows, cols, generator=gen, device="cuda")
        chi2.addcmul_(t, t)
        del t
    x = z / torch.sqrt(chi2 / nu)
    del chi2
    flat = x.view(-1)
    n = max(1, int(round(frac * flat.numel())))
    idx = torch.randint(0, flat.numel(), (n,), generator=gen, device="cuda")
    mag = lo + (hi - lo) * torch.rand(n, generator=gen, device="cuda")
    sign = torch.where(torch.rand(n, generator=gen, device="cuda") < 0.5, -1.0, 1.0)
    flat[idx] = mag * sign
    return x.to(torch.bfloat16)


def device_normal(gen, rows, cols, std=1.0):
    import torch
    return (torch.randn(rows, cols, generator=gen, device="cuda") * std).to(torch.bfloat16)


class RouterSets:
    """n rotating input sets of the router step (quantize -> GEMM + top-k),
    all on the device: activations X [T, 7168] bf16 (Student-t with outliers
    for prefill, N(0,1) for decode), gate weights [256, 7168] drawn
    N(0, 0.02) in bf16 and quantized once by the library (static per layer),
    bias N(0, 0.01).  Each set's input is one arena and its results (top-k
    indices, scores, weights) another, so the end-to-end run moves one
    buffer each way per step."""

    def __init__(self, nv, ws, tokens, n_sets, prefill, seed=1234):
        import torch
        self.T, self.n, self.prefill = tokens, n_sets, prefill
        T = tokens
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        self.xin = []
        for _ in range(n_sets):
            x = device_student_t(gen, T, HIDDEN) if prefill else device_normal(gen, T, HIDDEN)
            self.xin.append(x.view(torch.int16).reshape(-1))
            del x
        self.x = [a.view(T, HIDDEN) for a in self.xin]
        self.bias = [(torch.randn(EXPERTS, generator=gen, device="cuda") * 0.01).float() for _ in range(n_sets)]
        self.qb, self.sfb, self.gsb = [], [], []
        for _ in range(n_sets):
            q, sf, gs = nv.quantize(device_normal(gen, EXPERTS, HIDDEN, 0.02), ws)
            self.qb.append(q)
            self.sfb.append(sf)
            self.gsb.append(gs)
        e = lambda *s, dt=torch.uint8: [torch.empty(*s, dtype=dt, device="cuda") for _ in range(n_sets)]
        self.qa, self.sfa, self.gsa = e(T, HIDDEN // 2), e(T, HIDDEN // 16), e(1, dt=torch.float32)
        self.out = e(3 * T * TOPK * 4)
        self.idx = [a[:T * TOPK * 4].view(torch.int32).view(T, TOPK) for a in self.out]
        self.score = [a[T * TOPK * 4:2 * T * TOPK * 4].view(torch.float32).view(T, TOPK) for a in self.out]
        self.weight = [a[2 * T * TOPK * 4:].view(torch.float32).view(T, TOPK) for a in self.out]
        torch.cuda.synchronize()

    def footprint(self):
        per = sum(t[0].numel() * t[0].element_size() for t in (
            self.xin, self.bias, self.qb, self.sfb, self.qa, self.sfa, self.out))
        return per * self.n

    def op_quantize(self, nv, ws, i):
        nv.nvfp4_quantize(self.x[i], self.qa[i], self.sfa[i], self.gsa[i], ws)

    def op_gemm(self, nv, ws, i):
        nv.nvfp4_gemm_topk(self.qa[i], self.sfa[i], self.gsa[i], self.qb[i], self.sfb[i], self.gsb[i],
                           nv.EPILOGUE_SQRT_SOFTPLUS_BIAS, self.bias[i], TOPK, self.idx[i],
                           self.score[i], self.weight[i], None, ws)

    def steps(self, nv, ws, indices, ready=None, done=None):
        """Steps on sets `indices`, in order on the current stream.  ready(i)
        may return an event that step i's inputs wait for; done(i) is called
        once step i is enqueued (end-to-end copies)."""
        import torch
        main = torch.cuda.current_stream()
        for i in indices:
            ev = ready(i) if ready is not None else None
            if ev is not None:
                main.wait_event(ev)
            self.op_quantize(nv, ws, i)
            self.op_gemm(nv, ws, i)
            if done is not None:
                done(i, main)


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


def time_windows(replay_window, world, min_secs=2.0, min_windows=20, max_windows=20000):
    """Back-to-back timed windows of replay_window() (each one window of
    --steps steps), bracketed by a barrier and a synchronize on both sides:
    CUDA events between consecutive windows give each window's device time.
    Windows keep being enqueued until `min_secs` of wall time have passed (the
    host waits on the event of a window several behind, so the queue stays
    short and the GPU never idles), so that clock sampling sees the region.
    Returns (window seconds, wall start, wall end)."""
    import torch
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    evs = [torch.cuda.Event(enable_timing=True)]
    evs[0].record()
    lag = 8
    while True:
        replay_window()
        ev = torch.cuda.Event(enable_timing=True)
        ev.record()
        evs.append(ev)
        n = len(evs) - 1
        if n > lag:
            evs[n - lag].synchronize()
        if n >= max_windows or (n >= min_windows and time.time() - t_wall0 >= min_secs):
            break
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    secs = [evs[j].elapsed_time(evs[j + 1]) / 1e3 for j in range(len(evs) - 1)]
    return secs, t_wall0, t_wall1


def time_graphs(graphs, singles, chunk, steps):
    """Average device seconds per call over `steps` replayed calls (one window)."""
    import torch
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    replay_steps(graphs, singles, chunk, steps)
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3 / steps


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
    # RMSNorm fused into the quantize (the norm output never reaches HBM)
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
    # mHC pre-mix of the 4 residual streams + RMSNorm + quantize (x_in and the
    # normalised rows never reach HBM)
    for T in (1, 32, 2048):
        n_hc = 4
        x0 = torch.from_numpy(workloads.quantize_input(T * n_hc).view(np.int16)).cuda().view(T, n_hc, HIDDEN)
        a0 = torch.from_numpy(workloads.bf16_bits(rng.uniform(0.05, 1.0, (T, n_hc)).astype(np.float32))
                              .view(np.int16)).cuda()
        q, sf, gs = nv.mhc_rmsnorm_quantize(x0, a0, wn, 1e-6, ws)
        t, how = time_op(lambda i: x0 if i == 0 else x0.clone(),
                         lambda x: nv.nvfp4_mhc_rmsnorm_quantize(x, a0, wn, 1e-6, q, sf, gs, ws),
                         T * n_hc * HIDDEN * 2, flush)
        b = T * n_hc * HIDDEN * 2 + T * n_hc * 2 + HIDDEN * 2 + T * HIDDEN // 2 + T * HIDDEN // 16 + 4
        sweep[f"mhc_rmsnorm_T{T}_nhc4"] = dict(us=round(t * 1e6, 2), gbs=round(b / t / 1e9, 1),
                                               hbm_frac=round(b / t / hbm, 3), l2=how)
        del x0, a0, q, sf, gs
    torch.cuda.empty_cache()
    out["quantize"] = sweep
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
    # the indexer's weighted ReLU head sum fused in (one token, 64 heads x 128 dims)
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
    # grouped NVFP4 GEMM + SwiGLU, MoE first projection (256 experts,
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


def run_workload(nv, ws, pk, tokens, prefill, steps, warmup, world, min_secs):
    """The router step on T tokens: headline figures, per-kernel times and
    rooflines, and the end-to-end figure with host buffers."""
    import torch
    T = tokens
    hbm = pk["hbm_gbs"]
    per_set = (T * HIDDEN * 2 + EXPERTS * (HIDDEN // 2 + HIDDEN // 16) + EXPERTS * 4
               + T * (HIDDEN // 2 + HIDDEN // 16) + 3 * T * TOPK * 4)
    n_sets = max(3, int(np.ceil(2.2 * L2_BYTES / per_set)))
    chunk = min(n_sets, 16)
    n_sets = int(np.ceil(n_sets / chunk) * chunk)
    sets = RouterSets(nv, ws, T, n_sets, prefill)
    torch.cuda.synchronize()
    before = nv.kernel_launches()
    sets.steps(nv, ws, [0])
    kernels_per_step = nv.kernel_launches() - before
    torch.cuda.synchronize()

    graphs, singles = capture_runs(lambda idx: sets.steps(nv, ws, idx), n_sets, chunk)
    replay_steps(graphs, singles, chunk, warmup)
    secs, t0, t1 = time_windows(lambda: replay_steps(graphs, singles, chunk, steps), world, min_secs)
    med = reduce_max(statistics.median(secs), world)
    value = throughput(T, steps, med, world)

    # per-kernel average launch durations (same sets, graph replays of one op)
    op_times = {}
    for name, fn in (("quantize", sets.op_quantize), ("gemm_topk", sets.op_gemm)):
        g, s1 = capture_chunks(lambda i, fn=fn: fn(nv, ws, i), n_sets, chunk)
        replay_steps(g, s1, chunk, n_sets)
        op_times[name] = min(time_graphs(g, s1, chunk, max(steps, n_sets)) for _ in range(3))
        del g, s1
    qb = quantize_bytes(T, HIDDEN)
    gb = gemm_bytes(T, EXPERTS, HIDDEN, TOPK)
    gf = gemm_flops(T, EXPERTS, HIDDEN)
    tag = "router_prefill" if prefill else f"router_decode_T{T}"
    tq, tg = op_times["quantize"], op_times["gemm_topk"]
    roof = dict(
        quantize=dict(bound="hbm", achieved=round(qb / tq / 1e9, 1), peak=hbm, unit="GB/s",
                      frac=round(qb / tq / 1e9 / hbm, 4), traffic=load_traffic("quantize.cu", f"quantize_{tag}"),
                      kernel="quantize", algorithmic_bytes=qb, launch_us=round(tq * 1e6, 3),
                      peak_source=pk["source"]),
        gemm_topk=dict(bound="tensor" if prefill else "hbm",
                       achieved=round(gf / tg / 1e12, 1) if prefill else round(gb / tg / 1e9, 1),
                       peak=round(pk["fp4_tflops"], 1) if prefill else hbm,
                       unit="TFLOP/s" if prefill else "GB/s",
                       frac=round(gf / tg / 1e12 / pk["fp4_tflops"], 4) if prefill else round(gb / tg / 1e9 / hbm, 4),
                       hbm_frac=round(gb / tg / 1e9 / hbm, 4),
                       traffic=load_traffic("gemm_topk.cu", f"gemm_topk_{tag}"), kernel="gemm_topk",
                       algorithmic_bytes=gb, flops=gf, launch_us=round(tg * 1e6, 3),
                       peak_source=(f"dense FP4 = {pk['source']} bf16 GEMM {pk['bf16_tflops']} TFLOP/s x "
                                    f"{FP4_OVER_BF16:g} (nominal FP4/BF16 ratio)" if prefill else pk["source"])))
    dominant = max(op_times, key=op_times.get)

    # End to end through the public API with host buffers (pinned), copies
    # inside the timed region: every step copies its own activations in and
    # its results (indices, scores, weights) out, on two copy streams, so
    # step i + 1's inputs and step i's results travel while the neighbouring
    # step computes; a window ends when its last results are on the host.
    hin = [torch.empty(a.numel(), dtype=torch.int16, pin_memory=True) for a in sets.xin]
    hout = [torch.empty(a.numel(), dtype=torch.uint8, pin_memory=True) for a in sets.out]
    for i in range(n_sets):
        hin[i].copy_(sets.xin[i].cpu())
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_steps(indices):
        main = torch.cuda.current_stream()
        h2d_s.wait_stream(main)
        d2h_s.wait_stream(main)
        landed = {}
        for i in indices:
            with torch.cuda.stream(h2d_s):
                sets.xin[i].copy_(hin[i], non_blocking=True)
                landed[i] = torch.cuda.Event()
                landed[i].record(h2d_s)

        def results_out(i, m):
            ev = torch.cuda.Event()
            ev.record(m)
            d2h_s.wait_event(ev)
            with torch.cuda.stream(d2h_s):
                hout[i].copy_(sets.out[i], non_blocking=True)

        sets.steps(nv, ws, indices, ready=lambda i: landed[i], done=results_out)
        main.wait_stream(h2d_s)
        main.wait_stream(d2h_s)

    ge, se = capture_runs(e2e_steps, n_sets, chunk)
    replay_steps(ge, se, chunk, min(warmup, n_sets))
    e_secs, _, _ = time_windows(lambda: replay_steps(ge, se, chunk, steps), world, min_secs / 2, min_windows=5)
    e_med = reduce_max(statistics.median(e_secs), world)
    e2e = dict(value=round(throughput(T, steps, e_med, world), 1), unit="rows/s",
               h2d_bytes_per_step=sets.xin[0].numel() * 2, d2h_bytes_per_step=sets.out[0].numel(),
               windows=len(e_secs))
    torch.cuda.synchronize()
    for i in range(n_sets):  # the copies really ran: host results equal the device results
        assert torch.equal(hout[i], sets.out[i].cpu()), "end-to-end results differ from the device results"
    status = nv.read_device_status(ws)
    fp = sets.footprint()
    del sets, graphs, singles, ge, se, hin, hout
    torch.cuda.empty_cache()
    return dict(value=value, secs=med, windows=len(secs), t0=t0, t1=t1, kernels_per_step=kernels_per_step,
                roofline=roof[dominant], roofline_kernels=roof,
                op_us={k: round(v * 1e6, 3) for k, v in op_times.items()}, e2e=e2e, n_sets=n_sets,
                footprint=fp, device_status=status)


def run_gpu(args, rank, world, local):
    import torch
    import quantize_block_scaled_gb300 as nv
    torch.cuda.set_device(local)
    pk = peaks()
    ws = nv.workspace()
    with ClockSampler(local) as clk:
        head = run_workload(nv, ws, pk, PREFILL_TOKENS, True, args.steps, args.warmup, world, args.min_secs)
        decode = {}
        if not args.quick:
            for T in (32, 1):
                d = run_workload(nv, ws, pk, T, False, args.steps, args.warmup, world, args.min_secs / 2)
                d["clocks"] = clk.summary(d["t0"], d["t1"])
                decode[T] = d
    head["clocks"] = clk.summary(head["t0"], head["t1"])
    detail = None
    if not args.quick and rank == 0:
        flush = torch.zeros(4 * L2_BYTES, dtype=torch.uint8, device="cuda")
        detail = secondary(nv, ws, pk, flush)
        del flush
    return head, decode, detail


# ---------------------------------------------------------------- the CPU oracle

def oracle_data(T, prefill):
    """The router workload on the host (numpy, seeded): activations, gate
    weights quantized by the oracle, bias."""
    import oracle as orc
    orc.build()
    d = workloads.router_prefill(tokens=T) if prefill else workloads.router_decode(T, seed=1)
    return dict(x=d["x"], w_q=orc.quantize(d["w"]), bias=d["bias"])


def run_oracle(d, sample_rows, budget_s, threads, max_reps=None):
    """The oracle's router step on a bounded sample: the global scale over the
    whole batch (every row), then quantize + GEMM + epilogue + top-8 of the
    first `sample_rows` rows on `threads` host threads, repeated while the
    budget lasts.  A full step is estimated as t_gs + (T / sample_rows) *
    t_rows, so the rate is in rows of the whole step per second."""
    import oracle as orc
    x, (qb, sfb, gsb), bias = d["x"], d["w_q"], d["bias"]
    T = x.shape[0]
    t_gs, t_rows, reps = 0.0, 0.0, 0
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        gsa = orc.global_scale(x)
        t1 = time.perf_counter()
        qa, sfa = orc.quantize_rows(x, gsa, 0, sample_rows)
        orc.gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 1, bias, TOPK, threads=threads)
        t2 = time.perf_counter()
        t_gs += t1 - t0
        t_rows += t2 - t1
        reps += 1
        if (max_reps is not None and reps >= max_reps) or (max_reps is None and time.perf_counter() - t_start > budget_s
                                                         and reps >= 2):
            break
    step_s = t_gs / reps + (T / sample_rows) * (t_rows / reps)
    return dict(value=T / step_s, step_s=step_s, reps=reps, secs=time.perf_counter() - t_start,
                sample=(f"{reps} reps of: global scale over all {T} rows, then quantize + GEMM + top-{TOPK} of "
                        f"{sample_rows} rows on {threads} threads; full step = t_gs + {T}/{sample_rows} x t_rows"))


def cpu_baseline(T, prefill, budget_s):
    threads = os.cpu_count() or 1
    d = oracle_data(T, prefill)
    r = run_oracle(d, min(T, 512), budget_s, threads)
    return dict(value=round(r["value"], 2), unit="rows/s", cores=threads, kind="oracle", sample=r["sample"])


# ---------------------------------------------------------------- profiling hook

def run_profile(kind: str, iters: int):
    """Eager runs of one workload inside an NVTX range named "profile" (for ncu --nvtx)."""
    import torch
    import quantize_block_scaled_gb300 as nv
    ws = nv.workspace()
    if kind == "decode":
        sets = RouterSets(nv, ws, 32, 4, False)
        fns = [lambda i=i: sets.steps(nv, ws, [i]) for i in range(4)]
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
    elif kind == "deinterleave2048":
        hh = torch.from_numpy(workloads.swiglu_interleaved(2048).view(np.int16)).cuda()
        q, sf, gs = nv.deinterleave_quantize(hh, GRAN, ws)
        fns = [lambda: nv.nvfp4_deinterleave_quantize(hh, GRAN, q, sf, gs, ws)]
    elif kind in ("mhc32", "mhc2048"):
        T = 32 if kind == "mhc32" else 2048
        x = torch.from_numpy(workloads.quantize_input(T * 4).view(np.int16)).cuda().view(T, 4, HIDDEN)
        a = torch.full((T, 4), 0.5, dtype=torch.bfloat16, device="cuda")
        wn = torch.ones(HIDDEN, dtype=torch.bfloat16, device="cuda")
        q, sf, gs = nv.mhc_rmsnorm_quantize(x, a, wn, 1e-6, ws)
        fns = [lambda: nv.nvfp4_mhc_rmsnorm_quantize(x, a, wn, 1e-6, q, sf, gs, ws)]
    elif kind == "router384":
        rng = np.random.default_rng(384)
        xv = torch.from_numpy(workloads.bf16_bits(rng.standard_normal((32, HIDDEN), np.float32)).view(np.int16)).cuda()
        wv = torch.from_numpy(workloads.bf16_bits(rng.standard_normal((384, HIDDEN), np.float32) * np.float32(0.02))
                              .view(np.int16)).cuda()
        bv = torch.from_numpy((rng.standard_normal(384) * 0.01).astype(np.float32)).cuda()
        qa, sfa, gsa = nv.quantize(xv, ws)
        qb, sfb, gsb = nv.quantize(wv, ws)
        out = [torch.empty(32, 6, dtype=dt, device="cuda") for dt in (torch.int32, torch.float32, torch.float32)]
        fns = [lambda: nv.nvfp4_gemm_topk(qa, sfa, gsa, qb, sfb, gsb, nv.EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM, bv, 6,
                                          *out, None, ws)]
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

def workload_config(world):
    return dict(workload="router_prefill", tokens=PREFILL_TOKENS, hidden=HIDDEN, experts=EXPERTS, top_k=TOPK,
                activations="Student-t(3), 0.01% of entries +-U(500, 2000)", parallelism=f"replicas{world}")


METRIC = f"router_prefill_T{PREFILL_TOKENS}_rows_per_s"


def decode_line(d, T, cpu):
    return dict(metric=f"router_decode_T{T}_rows_per_s", value=round(d["value"], 1), unit="rows/s",
                ms_per_step=round(d["secs"] / max(1, d.get("steps", 1)) * 1e3, 6), windows=d["windows"],
                config=dict(workload="router_decode", tokens=T, hidden=HIDDEN, experts=EXPERTS, top_k=TOPK,
                            l2=f"{d['n_sets']} rotating input sets, {d['footprint'] / 2**20:.0f} MiB (> 2x L2)"),
                roofline=d["roofline"], roofline_kernels=d["roofline_kernels"], op_us=d["op_us"], e2e=d["e2e"],
                cpu_baseline=cpu, clocks=d["clocks"], device_status=d["device_status"])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20, help="steps per timed window")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--min-secs", type=float, default=3.0,
                    help="wall time the repeated timed windows of the headline last at least")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only (no decode or per-shape detail)")
    ap.add_argument("--profile", choices=("decode", "prefill", "quantize", "quantize2048", "indexer",
                                          "indexer_heads", "rmsnorm2048", "moe_decode", "moe_prefill", "moe_small",
                                          "deinterleave2048", "mhc32", "mhc2048", "router384"),
                    help="run --warmup eager iterations of one workload in an NVTX range and exit")
    args = ap.parse_args()
    if args.profile:
        run_profile(args.profile, args.warmup)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_setup(args.gpus)
    config = workload_config(world)

    if args.impl == "reference":
        if rank != 0:
            return
        threads = os.cpu_count() or 1
        d = oracle_data(PREFILL_TOKENS, True)
        rows = 64
        run_oracle(d, rows, 0, threads, max_reps=args.warmup)  # warm-up steps, untimed
        r = run_oracle(d, rows, 0, threads, max_reps=args.steps)
        line = dict(impl="reference", metric=METRIC, value=round(r["value"], 3), unit="rows/s",
                    n_gpus=world, steps=args.steps, warmup=args.warmup,
                    ms_per_step=round(r["step_s"] * 1e3, 3), higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="f32/f64", data="synthetic",
                    config=dict(config, sample=r["sample"]),
                    cpu_baseline=dict(value=round(r["value"], 3), unit="rows/s", cores=threads,
                                      kind="oracle", sample=r["sample"]),
                    e2e=dict(value=round(r["value"], 3), unit="rows/s", h2d_bytes_per_step=0,
                             d2h_bytes_per_step=0))
        print(json.dumps(line), flush=True)
        return

    head, decode, detail = run_gpu(args, rank, world, local)
    cpu, cpu_dec = None, {}
    if rank == 0 and world == 1:
        cpu = cpu_baseline(PREFILL_TOKENS, True, 12.0)
        for T in decode:
            cpu_dec[T] = cpu_baseline(T, False, 4.0)
    if rank != 0:
        return
    config["l2"] = (f"{head['n_sets']} rotating input sets, {head['footprint'] / 2**20:.0f} MiB (> 2x L2); "
                    f"no flush inside the timed region")
    config["timing"] = (f"median of {head['windows']} back-to-back windows of {args.steps} graph-replayed "
                        f"steps (max over ranks)")
    for T, d in decode.items():
        d["steps"] = args.steps
    line = dict(metric=METRIC, value=round(head["value"], 1), unit="rows/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup,
                ms_per_step=round(head["secs"] / args.steps * 1e3, 5), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="nvfp4-e2m1/f32", data="synthetic",
                config=config, roofline=head["roofline"], roofline_kernels=head["roofline_kernels"],
                cpu_baseline=cpu, e2e=head["e2e"],
                gpu_launches=head["kernels_per_step"] * args.steps * head["windows"],
                clocks=head["clocks"], op_us=head["op_us"], device_status=head["device_status"],
                decode={f"T{T}": decode_line(d, T, cpu_dec.get(T)) for T, d in decode.items()},
                detail=detail)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
