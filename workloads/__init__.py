"""Seeded synthetic inputs shaped like the DeepSeek-V4-Pro decode workloads.

This module only draws random numbers and lays them out as the byte
formats the library consumes (bf16 bit patterns as ``uint16``, FP32 bias
vectors).  It holds none of the NVFP4 arithmetic: no amax, no scales, no
codes, no GEMM, no top-k.  Both the CUDA path and the CPU oracle read the
arrays produced here; neither side's code lives here.

Shapes follow the pages:

* hidden size 7168 and 256 routed-gate experts with top-8 selection
  ("Router decode" / "Router prefill"),
* 128-dim indexer keys, 2048 compressed blocks at 8192 context
  (compression ratio 4), top-512 ("Indexer-shaped scoring"),
* the MoE SwiGLU output of width 2 * 2048 with gate/up columns interleaved
  ("Quantize sweep", deinterleave variant).

Random draws use numpy's PCG64 generator (``numpy.random.default_rng``),
one seed per workload, so every run sees the same bytes.
"""
from __future__ import annotations

import numpy as np

HIDDEN = 7168          # model hidden size
EXPERTS = 256          # routed experts scored by the gate
ROUTER_TOPK = 8
INDEXER_DIM = 128      # indexer head dim (one shared key per compressed block)
INDEXER_KEYS = 2048    # 8192 context / compression ratio 4
INDEXER_ROWS = 64      # query rows of one decode step (indexer heads flattened)
INDEXER_TOPK = 512
MOE_INTER = 2048       # SwiGLU intermediate size I; the interleaved output is 2*I wide


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Store float32 values as bf16 bit patterns (round to nearest, ties to even).

    This is the storage conversion of the synthetic input, done once when the
    input is made; it is not part of the quantizer.  Inputs here are finite.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = u >> np.uint32(16)
    lsb &= np.uint32(1)
    lsb += np.uint32(0x7FFF)
    lsb += u                      # finite inputs never overflow 32 bits here
    lsb >>= np.uint32(16)
    return lsb.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact), for building test cases."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)


def _plant(rng: np.random.Generator, flat: np.ndarray, frac: float) -> np.ndarray:
    """Indices of about ``frac`` of the entries (drawn with replacement)."""
    count = max(1, int(round(frac * flat.size)))
    return rng.integers(0, flat.size, size=count)


def router_tiny(seed: int = 0) -> dict:
    """Tiny router: X 4x512 N(0,1); gate weight 64x512 N(0,0.02); bias 64 N(0,0.01); top-6."""
    rng = np.random.default_rng(seed)
    x = bf16_bits(_normal(rng, (4, 512)))
    w = bf16_bits(_normal(rng, (64, 512), 0.02))
    bias = _normal(rng, (64,), 0.01)
    return dict(name="router_tiny", x=x, w=w, bias=bias, k=6, epilogue=1)


def router_weights(seed: int, experts: int = EXPERTS, hidden: int = HIDDEN) -> dict:
    """Gate weight (experts x hidden) N(0,0.02) as bf16 and FP32 bias N(0,0.01)."""
    rng = np.random.default_rng(seed)
    w = bf16_bits(_normal(rng, (experts, hidden), 0.02))
    bias = _normal(rng, (experts,), 0.01)
    return dict(w=w, bias=bias)


def router_decode(tokens: int, seed: int) -> dict:
    """Router decode: T x 7168 bf16 N(0,1) activations, 256 experts, top-8."""
    rng = np.random.default_rng(seed)
    x = bf16_bits(_normal(rng, (tokens, HIDDEN)))
    wb = router_weights(seed + 1000)
    return dict(name=f"router_decode_T{tokens}", x=x, k=ROUTER_TOPK, epilogue=1, **wb)


def student_t_with_outliers(rng: np.random.Generator, shape, nu: float = 3.0,
                            frac: float = 1e-4, lo: float = 500.0, hi: float = 2000.0) -> np.ndarray:
    """Student-t(nu) entries with ``frac`` of them replaced by +-U(lo, hi)."""
    a = rng.standard_t(nu, size=shape).astype(np.float32)
    flat = a.reshape(-1)
    idx = _plant(rng, flat, frac)
    mag = rng.uniform(lo, hi, size=idx.size).astype(np.float32)
    sign = np.where(rng.integers(0, 2, size=idx.size) == 1, np.float32(1), np.float32(-1))
    flat[idx] = mag * sign
    return a


def router_prefill(tokens: int = 8192, seed: int = 3) -> dict:
    """Router prefill with outliers: T x 7168 Student-t(3), 0.01% entries +-U(500,2000)."""
    rng = np.random.default_rng(seed)
    x = bf16_bits(student_t_with_outliers(rng, (tokens, HIDDEN)))
    wb = router_weights(seed + 1000)
    return dict(name=f"router_prefill_T{tokens}", x=x, k=ROUTER_TOPK, epilogue=1, **wb)


def indexer(seed: int = 4, rows: int = INDEXER_ROWS, keys: int = INDEXER_KEYS,
            dim: int = INDEXER_DIM, k: int = INDEXER_TOPK) -> dict:
    """Indexer-shaped scoring: Q rows x 128 N(0,1), keys 2048 x 128 N(0,1), identity, top-512."""
    rng = np.random.default_rng(seed)
    q = bf16_bits(_normal(rng, (rows, dim)))
    keys_ = bf16_bits(_normal(rng, (keys, dim)))
    return dict(name="indexer", x=q, w=keys_, bias=None, k=k, epilogue=0)


def quantize_input(tokens: int, seed: int = 5, cols: int = HIDDEN) -> np.ndarray:
    """T x 7168 bf16 N(0,1) with 0.1% of the entries multiplied by 100."""
    rng = np.random.default_rng(seed)
    a = _normal(rng, (tokens, cols))
    if a.size:
        flat = a.reshape(-1)
        flat[_plant(rng, flat, 1e-3)] *= np.float32(100.0)
    return bf16_bits(a)


def swiglu_interleaved(tokens: int, inter: int = MOE_INTER, seed: int = 6) -> np.ndarray:
    """T x 2I bf16 N(0,1) (0.1% x100): a SwiGLU output with gate/up columns interleaved.

    The values are i.i.d., so the interleave granularity is a property of how
    the consumer reads the row, not of how it was drawn.
    """
    return quantize_input(tokens, seed=seed, cols=2 * inter)


def moe_routing(tokens: int, experts: int, topk: int, seed: int):
    """Token-to-expert routing of one MoE layer: each token picks ``topk``
    distinct experts uniformly at random.  Returns (token_of_row, offsets):
    the (token, expert) pairs sorted by expert (then token), as the source
    token of each grouped row, and the int32 [experts + 1] group offsets."""
    rng = np.random.default_rng(seed)
    picks = np.stack([rng.choice(experts, size=topk, replace=False) for _ in range(tokens)]) \
        if tokens else np.zeros((0, topk), np.int64)
    tok = np.repeat(np.arange(tokens), topk)
    exp_ = picks.reshape(-1)
    order = np.lexsort((tok, exp_))
    counts = np.bincount(exp_, minlength=experts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return tok[order].astype(np.int64), offsets


def moe_l1_weights(experts: int, inter: int, hidden: int, seed: int, std: float = 0.02) -> np.ndarray:
    """The experts' first-projection weights, [experts * 2I, hidden] bf16 N(0, std):
    rows e*2I .. e*2I + 2I - 1 are expert e's gate/up rows (interleaved layout
    is a matter of how they are read; the draws are i.i.d.)."""
    rng = np.random.default_rng(seed)
    return bf16_bits(_normal(rng, (experts * 2 * inter, hidden), std))
