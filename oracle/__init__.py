"""CPU oracle for the NVFP4 quantize and GEMM + top-k path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only callers.  The library's product path
never imports this package.

The arithmetic lives in ``nvfp4_oracle.cpp`` (plain C++, one IEEE operation
per FP32 step, double accumulation in the GEMM); this module compiles it with
the host compiler and wraps each function for numpy arrays.  ``ctypes``
releases the GIL during each call, so callers may run disjoint row ranges in
threads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

# Host flags: no FMA contraction, no fast-math, IEEE single for every FP32 op.
CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libnvfp4_oracle.so``; return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["g++", *CXXFLAGS, _SRC, "-o", tmp], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        F = ctypes.c_float
        sigs = {
            "orc_bf16_to_f32": (F, [ctypes.c_uint16]),
            "orc_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e2m1_encode": (ctypes.c_uint8, [F]),
            "orc_e4m3_decode": (F, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [F]),
            "orc_global_scale": (F, [P, I64, I64, I64]),
            "orc_quantize_rows": (None, [P, I64, I64, F, I64, I64, P, P]),
            "orc_quantize": (None, [P, I64, I64, I64, P, P, P]),
            "orc_deinterleave": (None, [P, I64, I64, I64, P]),
            "orc_deinterleave_quantize": (None, [P, I64, I64, I64, P, P, P]),
            "orc_dequantize": (None, [P, P, F, I64, I64, P]),
            "orc_gemm_logits": (None, [P, P, F, P, P, F, I64, I64, I64, I64, P]),
            "orc_epilogue": (None, [P, I64, I64, ctypes.c_int, P, P, P]),
            "orc_topk": (None, [P, P, I64, I64, ctypes.c_int, P, P, P]),
            "orc_normalize_topk_weights": (None, [P, P, I64, ctypes.c_int]),
            "orc_rmsnorm": (None, [P, I64, I64, I64, P, F, P]),
            "orc_rms_sum_of_squares": (None, [P, I64, I64, I64, P]),
            "orc_mhc_mix": (None, [P, I64, I64, I64, I64, P, P]),
            "orc_mhc_rmsnorm_quantize": (None, [P, I64, I64, I64, I64, P, P, F, P, P, P]),
            "orc_indexer_scores": (None, [P, P, F, P, P, F, I64, I64, I64, I64, P, P]),
            "orc_rmsnorm_quantize": (None, [P, I64, I64, I64, P, F, P, P, P]),
            "orc_gemm_topk_rows": (None, [P, P, F, P, P, F, I64, I64, ctypes.c_int, P,
                                          ctypes.c_int, I64, I64, P, P, P]),
            "orc_grouped_swiglu": (None, [P, P, F, P, P, P, P, I64, I64, I64, I64,
                                          ctypes.c_double, P, P]),
            "orc_to_bf16": (None, [P, I64, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar codecs ------------------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return _load().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return int(_load().orc_e2m1_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


def bf16_to_f32(bits: int) -> float:
    return _load().orc_bf16_to_f32(int(bits))


# ---- quantize -----------------------------------------------------------------------

def global_scale(x: np.ndarray) -> np.float32:
    """gs = max(max|x|, 1e-8) / 2688 for a 2-D bf16-bits array."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    return np.float32(_load().orc_global_scale(_ptr(x), rows, cols, cols))


def quantize(x: np.ndarray):
    """Quantize a 2-D bf16-bits array; returns (q [rows, cols/2] u8, sf [rows, cols/16] u8, gs f32)."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    q = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    gs = np.zeros(1, np.float32)
    _load().orc_quantize(_ptr(x), rows, cols, cols, _ptr(q), _ptr(sf), _ptr(gs))
    return q, sf, gs[0]


def quantize_rows(x: np.ndarray, gs: float, row_begin: int, row_end: int):
    """Quantize rows [row_begin, row_end) of x with a given gs (for sampled parity checks)."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    assert 0 <= row_begin <= row_end <= rows
    n = row_end - row_begin
    q = np.zeros((n, cols // 2), np.uint8)
    sf = np.zeros((n, cols // 16), np.uint8)
    _load().orc_quantize_rows(_ptr(x), cols, cols, float(gs), row_begin, row_end, _ptr(q), _ptr(sf))
    return q, sf


def deinterleave(x: np.ndarray, granularity: int) -> np.ndarray:
    x = _c(x, np.uint16)
    rows, width = x.shape
    out = np.zeros_like(x)
    _load().orc_deinterleave(_ptr(x), rows, width // 2, granularity, _ptr(out))
    return out


def deinterleave_quantize(x: np.ndarray, granularity: int):
    x = _c(x, np.uint16)
    rows, width = x.shape
    q = np.zeros((rows, width // 2), np.uint8)
    sf = np.zeros((rows, width // 16), np.uint8)
    gs = np.zeros(1, np.float32)
    _load().orc_deinterleave_quantize(_ptr(x), rows, width // 2, granularity, _ptr(q), _ptr(sf),
                                      _ptr(gs))
    return q, sf, gs[0]


def dequantize(q: np.ndarray, sf: np.ndarray, gs: float) -> np.ndarray:
    q = _c(q, np.uint8)
    sf = _c(sf, np.uint8)
    rows, half = q.shape
    out = np.zeros((rows, 2 * half), np.float64)
    _load().orc_dequantize(_ptr(q), _ptr(sf), float(gs), rows, 2 * half, _ptr(out))
    return out


# ---- GEMM + epilogue + top-k --------------------------------------------------------

def gemm_logits(qa, sfa, gsa, qb, sfb, gsb, row_begin: int = 0, row_end: int | None = None):
    qa, sfa, qb, sfb = (_c(a, np.uint8) for a in (qa, sfa, qb, sfb))
    M, K = qa.shape[0], qa.shape[1] * 2
    N = qb.shape[0]
    row_end = M if row_end is None else row_end
    out = np.zeros((row_end - row_begin, N), np.float32)
    _load().orc_gemm_logits(_ptr(qa), _ptr(sfa), float(gsa), _ptr(qb), _ptr(sfb), float(gsb),
                            N, K, row_begin, row_end, _ptr(out))
    return out


def epilogue(logits: np.ndarray, kind: int, bias=None):
    """Returns (score, weight) for epilogue 0 (identity) or 1 (sqrt-softplus + bias)."""
    logits = _c(logits, np.float32)
    rows, N = logits.shape
    bias_c = None if bias is None else _c(bias, np.float32)
    if kind == 1 and bias_c is None:
        bias_c = np.zeros(N, np.float32)
    score = np.zeros_like(logits)
    weight = np.zeros_like(logits)
    _load().orc_epilogue(_ptr(logits), rows, N, int(kind), _ptr(bias_c), _ptr(score), _ptr(weight))
    return score, weight


def topk(score: np.ndarray, k: int, weight=None):
    score = _c(score, np.float32)
    rows, N = score.shape
    w = None if weight is None else _c(weight, np.float32)
    idx = np.zeros((rows, k), np.int32)
    val = np.zeros((rows, k), np.float32)
    wout = np.zeros((rows, k), np.float32)
    _load().orc_topk(_ptr(score), _ptr(w), rows, N, int(k), _ptr(idx), _ptr(val), _ptr(wout))
    return idx, val, wout


def indexer_scores(qa, sfa, gsa, qb, sfb, gsb, heads: int, head_w: np.ndarray) -> np.ndarray:
    """I[t, s] = sum_h w[t, h] * ReLU(q[t, h] . K[s]); A rows are t * heads + h."""
    qa, sfa, qb, sfb = (_c(a, np.uint8) for a in (qa, sfa, qb, sfb))
    M, K = qa.shape[0], qa.shape[1] * 2
    N = qb.shape[0]
    T = M // heads
    w = _c(head_w, np.float32)
    out = np.zeros((T, N), np.float32)
    _load().orc_indexer_scores(_ptr(qa), _ptr(sfa), float(gsa), _ptr(qb), _ptr(sfb), float(gsb), T, heads, N, K,
                               _ptr(w), _ptr(out))
    return out


def rms_sum_of_squares(x: np.ndarray) -> np.ndarray:
    """Per row of bf16 bits: the exact sum of squares rounded once to FP32."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    out = np.zeros(rows, np.float32)
    _load().orc_rms_sum_of_squares(_ptr(x), rows, cols, cols, _ptr(out))
    return out


def rmsnorm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """bf16 bits of RMSNorm(x) * weight (x, weight: bf16 bits), the oracle's op order."""
    x = _c(x, np.uint16)
    w = _c(weight, np.uint16)
    rows, cols = x.shape
    out = np.zeros((rows, cols), np.uint16)
    _load().orc_rmsnorm(_ptr(x), rows, cols, cols, _ptr(w), float(eps), _ptr(out))
    return out


def rmsnorm_quantize(x: np.ndarray, weight: np.ndarray, eps: float):
    """RMSNorm to bf16, then NVFP4 quantize: (codes, scales, gs)."""
    x = _c(x, np.uint16)
    w = _c(weight, np.uint16)
    rows, cols = x.shape
    q = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    gs = np.zeros(1, np.float32)
    _load().orc_rmsnorm_quantize(_ptr(x), rows, cols, cols, _ptr(w), float(eps), _ptr(q), _ptr(sf), _ptr(gs))
    return q, sf, gs[0]


def mhc_mix(x: np.ndarray, a: np.ndarray) -> np.ndarray:
    """bf16 bits of the mHC layer input: x [T, n_hc, d] bf16 bits, a [T, n_hc] bf16 bits."""
    x = _c(x, np.uint16)
    a = _c(a, np.uint16)
    T, n, d = x.shape
    out = np.zeros((T, d), np.uint16)
    _load().orc_mhc_mix(_ptr(x), T, n, d, n * d, _ptr(a), _ptr(out))
    return out


def mhc_rmsnorm_quantize(x: np.ndarray, a: np.ndarray, weight: np.ndarray, eps: float):
    """The fused op: mHC pre-mix, RMSNorm * weight, NVFP4 quantize -> (codes, scales, gs)."""
    x = _c(x, np.uint16)
    a = _c(a, np.uint16)
    w = _c(weight, np.uint16)
    T, n, d = x.shape
    q = np.zeros((T, d // 2), np.uint8)
    sf = np.zeros((T, d // 16), np.uint8)
    gs = np.zeros(1, np.float32)
    _load().orc_mhc_rmsnorm_quantize(_ptr(x), T, n, d, n * d, _ptr(a), _ptr(w), float(eps), _ptr(q), _ptr(sf),
                                     _ptr(gs))
    return q, sf, gs[0]


def normalize_topk_weights(idx: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """Router gating normalisation (epilogue 2): each row's selected weights over their sum."""
    idx = _c(idx, np.int32)
    w = _c(weight, np.float32).copy()
    rows, k = idx.shape
    _load().orc_normalize_topk_weights(_ptr(idx), _ptr(w), rows, int(k))
    return w


def gemm_topk(qa, sfa, gsa, qb, sfb, gsb, kind: int, bias, k: int,
              row_begin: int = 0, row_end: int | None = None, threads: int = 1):
    """GEMM + epilogue + top-k over rows [row_begin, row_end); optional row-parallel threads."""
    qa, sfa, qb, sfb = (_c(a, np.uint8) for a in (qa, sfa, qb, sfb))
    M, K = qa.shape[0], qa.shape[1] * 2
    N = qb.shape[0]
    row_end = M if row_end is None else row_end
    rows = row_end - row_begin
    bias_c = None if bias is None else _c(bias, np.float32)
    if kind in (1, 2) and bias_c is None:
        bias_c = np.zeros(N, np.float32)
    idx = np.zeros((rows, k), np.int32)
    val = np.zeros((rows, k), np.float32)
    wout = np.zeros((rows, k), np.float32)
    lib = _load()

    def run(r0, r1):
        off = r0 - row_begin
        lib.orc_gemm_topk_rows(_ptr(qa), _ptr(sfa), float(gsa), _ptr(qb), _ptr(sfb), float(gsb),
                               N, K, int(kind), _ptr(bias_c), int(k), r0, r1,
                               _ptr(idx[off:]), _ptr(val[off:]), _ptr(wout[off:]))

    threads = max(1, min(int(threads), rows)) if rows else 1
    if threads == 1:
        if rows:
            run(row_begin, row_end)
    else:
        bounds = np.linspace(row_begin, row_end, threads + 1).astype(np.int64)
        ts = [threading.Thread(target=run, args=(int(bounds[i]), int(bounds[i + 1])))
              for i in range(threads) if bounds[i + 1] > bounds[i]]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    return idx, val, wout


# ---- grouped GEMM + SwiGLU (MoE first projection) -----------------------------------

def grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, offsets, inter: int, granularity: int,
                   limit: float = float("inf")):
    """SwiGLU of a grouped NVFP4 GEMM, in double: returns (h, a), each [M, I].

    qb/sfb hold E experts' [2I, K] weights stacked as [E*2I, K/2] / [E*2I, K/16];
    gsb has E entries; offsets (E + 1 int32) give each expert's rows of A.
    h = silu(min(gate, limit)) * clip(up, -limit, limit); a = silu(min(gate, limit)).
    Rows outside every group stay 0.
    """
    qa, sfa, qb, sfb = (_c(a, np.uint8) for a in (qa, sfa, qb, sfb))
    gsb = _c(np.atleast_1d(gsb), np.float32)
    offs = _c(offsets, np.int32)
    M, K = qa.shape[0], qa.shape[1] * 2
    E = offs.size - 1
    assert gsb.size == E and qb.shape[0] == E * 2 * inter
    h = np.zeros((M, inter), np.float64)
    a = np.zeros((M, inter), np.float64)
    _load().orc_grouped_swiglu(_ptr(qa), _ptr(sfa), float(gsa), _ptr(qb), _ptr(sfb), _ptr(gsb), _ptr(offs),
                               E, inter, K, granularity, float(limit), _ptr(h), _ptr(a))
    return h, a


def to_bf16(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of doubles (rounded to float, then to bf16, nearest even)."""
    v = _c(v, np.float64)
    out = np.zeros(v.shape, np.uint16)
    _load().orc_to_bf16(_ptr(v), v.size, _ptr(out))
    return out


def grouped_swiglu_bf16(qa, sfa, gsa, qb, sfb, gsb, offsets, inter: int, granularity: int,
                        limit: float = float("inf"), layout: int = 0) -> np.ndarray:
    """The stored bf16 output: layout 0 = h [M, I]; layout 1 = [M, 2I] with the
    gate columns of the weights' interleave holding a and the up columns h."""
    h, a = grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, offsets, inter, granularity, limit)
    if layout == 0:
        return to_bf16(h)
    M = h.shape[0]
    g = granularity
    out = np.zeros((M, 2 * inter), np.float64)
    for j0 in range(0, inter, g):
        base = 2 * j0
        out[:, base:base + g] = a[:, j0:j0 + g]
        out[:, base + g:base + 2 * g] = h[:, j0:j0 + g]
    return to_bf16(out)
