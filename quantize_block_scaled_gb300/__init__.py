"""Python binding of libnvfp4 (GB300 / sm_103a NVFP4 quantize and GEMM + top-k).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels, reached through its C ABI (``include/nvfp4.h``) with ``ctypes``.
PyTorch supplies device memory and streams.  There is no fallback: if
``libnvfp4.so`` has not been built (``quantize_block_scaled_gb300.build``) or
cannot be loaded, every call raises.

The three entry points keep the C names:

* ``nvfp4_quantize(x, q, sf, gs, ws, stream=None)``
* ``nvfp4_deinterleave_quantize(x, granularity, q, sf, gs, ws, stream=None)``
* ``nvfp4_gemm_topk(qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, k, idx, score,
  weight=None, logits=None, ws=..., stream=None)``
* ``nvfp4_grouped_swiglu_gemm(qa, sfa, gsa, qb, sfb, gsb, offsets, inter,
  granularity, limit, layout, out, ws, stream=None)``

plus allocating conveniences (``quantize``, ``deinterleave_quantize``,
``gemm_topk``, ``workspace``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4.so")

EPILOGUE_IDENTITY = 0
EPILOGUE_SQRT_SOFTPLUS_BIAS = 1
EPILOGUE_SQRT_SOFTPLUS_BIAS_NORM = 2
DEVICE_TIMEOUT = 0x1
DEVICE_BAD_GROUPS = 0x2

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape or alignment",
           3: "workspace missing or too small", 4: "CUDA error"}

_lock = threading.Lock()
_lib = None


class NVFP4Error(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        msg = f"{fn}: {_STATUS.get(status, 'unknown status')} (status {status})"
        if status == 4:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libnvfp4.so (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run quantize_block_scaled_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.nvfp4_workspace_bytes.restype = SZ
        L.nvfp4_workspace_bytes.argtypes = [I, I64, I64, I64, I]
        L.nvfp4_workspace_init.restype = I
        L.nvfp4_workspace_init.argtypes = [P, SZ, P]
        L.nvfp4_quantize.restype = I
        L.nvfp4_quantize.argtypes = [P, I64, I64, I64, P, P, P, P, SZ, P]
        L.nvfp4_deinterleave_quantize.restype = I
        L.nvfp4_deinterleave_quantize.argtypes = [P, I64, I64, I, P, P, P, P, SZ, P]
        L.nvfp4_gemm_topk.restype = I
        L.nvfp4_gemm_topk.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, P, I, P, P, P, P, P, SZ, P]
        L.nvfp4_read_device_status.restype = I
        L.nvfp4_read_device_status.argtypes = [P, SZ, ctypes.POINTER(ctypes.c_uint32), P]
        L.nvfp4_status_string.restype = ctypes.c_char_p
        L.nvfp4_status_string.argtypes = [I]
        L.nvfp4_last_cuda_error.restype = I
        L.nvfp4_last_cuda_error.argtypes = []
        L.nvfp4_indexer_topk.restype = I
        L.nvfp4_indexer_topk.argtypes = [P, P, P, P, P, P, I64, I, I64, I64, P, I, P, P, P, P, SZ, P]
        L.nvfp4_mhc_rmsnorm_quantize.restype = I
        L.nvfp4_mhc_rmsnorm_quantize.argtypes = [P, I64, I, I64, I64, P, P, ctypes.c_float, P, P, P, P, SZ, P]
        L.nvfp4_rmsnorm_quantize.restype = I
        L.nvfp4_rmsnorm_quantize.argtypes = [P, I64, I64, I64, P, ctypes.c_float, P, P, P, P, SZ, P]
        L.nvfp4_kernel_launches.restype = ctypes.c_uint64
        L.nvfp4_kernel_launches.argtypes = []
        L.nvfp4_quantize_noalloc.restype = I
        L.nvfp4_quantize_noalloc.argtypes = [P, I64, I64, I64, P, P, P, P]
        L.nvfp4_grouped_swiglu_gemm.restype = I
        L.nvfp4_grouped_swiglu_gemm.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, ctypes.c_float, I,
                                                P, I64, P, SZ, P]
        _lib = L
        return L


EXPORTED_SYMBOLS = ("nvfp4_workspace_bytes", "nvfp4_workspace_init", "nvfp4_quantize",
                    "nvfp4_deinterleave_quantize", "nvfp4_gemm_topk", "nvfp4_read_device_status",
                    "nvfp4_status_string", "nvfp4_last_cuda_error", "nvfp4_quantize_noalloc",
                    "nvfp4_kernel_launches", "nvfp4_rmsnorm_quantize", "nvfp4_indexer_topk",
                    "nvfp4_grouped_swiglu_gemm", "nvfp4_mhc_rmsnorm_quantize")


def _check(fn: str, status: int):
    if status != 0:
        raise NVFP4Error(fn, status, lib().nvfp4_last_cuda_error() if status == 4 else 0)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libnvfp4 must be CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _bf16_bits(x: torch.Tensor) -> torch.Tensor:
    if x.dtype == torch.bfloat16:
        return x
    if x.dtype in (torch.int16, torch.uint16):
        return x
    raise TypeError("x must be bfloat16 (or its bit patterns as int16/uint16)")


# ---------------------------------------------------------------- raw entry points

OP_QUANTIZE, OP_DEINTERLEAVE_QUANTIZE, OP_GEMM_TOPK, OP_RMSNORM_QUANTIZE, OP_INDEXER_TOPK, \
    OP_GROUPED_SWIGLU_GEMM, OP_MHC_RMSNORM_QUANTIZE = range(7)


def workspace_bytes(op: int = OP_QUANTIZE, rows: int = 0, cols: int = 0, n: int = 0, k: int = 0) -> int:
    return int(lib().nvfp4_workspace_bytes(op, rows, cols, n, k))


def workspace(device=None, stream=None) -> torch.Tensor:
    """A zeroed workspace buffer for the calls below (one per stream)."""
    ws = torch.empty(workspace_bytes(), dtype=torch.uint8, device=device or "cuda")
    _check("nvfp4_workspace_init", lib().nvfp4_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))
    return ws


def nvfp4_quantize(x, q, sf, gs, ws, stream=None):
    x = _bf16_bits(x)
    rows, cols = x.shape
    _check("nvfp4_quantize", lib().nvfp4_quantize(
        _ptr(x), rows, cols, x.stride(0), _ptr(q), _ptr(sf), _ptr(gs), _ptr(ws), ws.numel(),
        _stream(stream)))


def nvfp4_rmsnorm_quantize(x, weight, eps, q, sf, gs, ws, stream=None):
    x = _bf16_bits(x)
    weight = _bf16_bits(weight)
    rows, cols = x.shape
    _check("nvfp4_rmsnorm_quantize", lib().nvfp4_rmsnorm_quantize(
        _ptr(x), rows, cols, x.stride(0), _ptr(weight), float(eps), _ptr(q), _ptr(sf), _ptr(gs), _ptr(ws),
        ws.numel(), _stream(stream)))


def rmsnorm_quantize(x, weight, eps, ws, stream=None):
    """Allocating convenience: (q, sf, gs) of RMSNorm(x) * weight."""
    rows, cols = x.shape
    q = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device=x.device)
    gs = torch.empty(1, dtype=torch.float32, device=x.device)
    nvfp4_rmsnorm_quantize(x, weight, eps, q, sf, gs, ws, stream)
    return q, sf, gs


def nvfp4_mhc_rmsnorm_quantize(x, a, weight, eps, q, sf, gs, ws, stream=None):
    """x: bf16 [rows, n_hc, cols] (the token's streams contiguous; any token
    stride), a: bf16 [rows, n_hc]; the mixed, normalised rows are quantized."""
    x = _bf16_bits(x)
    a = _bf16_bits(a)
    weight = _bf16_bits(weight)
    rows, n_hc, cols = x.shape
    if x.stride(2) != 1 or x.stride(1) != cols or not a.is_contiguous():
        raise ValueError("x must have contiguous streams of cols elements and a must be contiguous")
    _check("nvfp4_mhc_rmsnorm_quantize", lib().nvfp4_mhc_rmsnorm_quantize(
        _ptr(x), rows, int(n_hc), cols, x.stride(0), _ptr(a), _ptr(weight), float(eps), _ptr(q), _ptr(sf),
        _ptr(gs), _ptr(ws), ws.numel(), _stream(stream)))


def mhc_rmsnorm_quantize(x, a, weight, eps, ws, stream=None):
    """Allocating convenience: (q, sf, gs) of RMSNorm(sum_i a[:, i] x[:, i]) * weight."""
    rows, _, cols = x.shape
    q = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device=x.device)
    gs = torch.empty(1, dtype=torch.float32, device=x.device)
    nvfp4_mhc_rmsnorm_quantize(x, a, weight, eps, q, sf, gs, ws, stream)
    return q, sf, gs


def nvfp4_indexer_topk(qa, sfa, gsa, qb, sfb, gsb, heads, head_w, k, idx, score, scores=None, ws=None,
                       stream=None):
    rows = qa.shape[0]
    K = qa.shape[1] * 2
    N = qb.shape[0]
    _check("nvfp4_indexer_topk", lib().nvfp4_indexer_topk(
        _ptr(qa), _ptr(sfa), _ptr(gsa), _ptr(qb), _ptr(sfb), _ptr(gsb), rows // heads, int(heads), N, K,
        _ptr(head_w), int(k), _ptr(idx), _ptr(score), _ptr(scores), _ptr(ws), 0 if ws is None else ws.numel(),
        _stream(stream)))


def indexer_topk(qa, sfa, gsa, qb, sfb, gsb, heads, head_w, k, ws, want_scores=False, stream=None):
    """Allocating convenience: (idx, score, I or None) per token."""
    T = qa.shape[0] // heads
    dev = qa.device
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    score = torch.empty(T, k, dtype=torch.float32, device=dev)
    scores = torch.empty(T, qb.shape[0], dtype=torch.float32, device=dev) if want_scores else None
    nvfp4_indexer_topk(qa, sfa, gsa, qb, sfb, gsb, heads, head_w, k, idx, score, scores, ws, stream)
    return idx, score, scores


def kernel_launches() -> int:
    """Kernels the library has launched in this process (graph captures count once)."""
    return int(lib().nvfp4_kernel_launches())


def nvfp4_quantize_noalloc(x, q, sf, gs, stream=None):
    """nvfp4_quantize without a workspace: the library's static scratch is used
    (for callers that cannot allocate device memory; overlapping calls race)."""
    x = _bf16_bits(x)
    rows, cols = x.shape
    _check("nvfp4_quantize_noalloc", lib().nvfp4_quantize_noalloc(
        _ptr(x), rows, cols, x.stride(0), _ptr(q), _ptr(sf), _ptr(gs), _stream(stream)))


def nvfp4_deinterleave_quantize(x, granularity, q, sf, gs, ws, stream=None):
    x = _bf16_bits(x)
    rows, width = x.shape
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    _check("nvfp4_deinterleave_quantize", lib().nvfp4_deinterleave_quantize(
        _ptr(x), rows, width // 2, int(granularity), _ptr(q), _ptr(sf), _ptr(gs), _ptr(ws),
        ws.numel(), _stream(stream)))


def nvfp4_gemm_topk(qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, k, idx, score, weight=None,
                    logits=None, ws=None, stream=None):
    M = qa.shape[0]
    K = qa.shape[1] * 2
    N = qb.shape[0]
    _check("nvfp4_gemm_topk", lib().nvfp4_gemm_topk(
        _ptr(qa), _ptr(sfa), _ptr(gsa), _ptr(qb), _ptr(sfb), _ptr(gsb), M, N, K, int(epilogue),
        _ptr(bias), int(k), _ptr(idx), _ptr(score), _ptr(weight), _ptr(logits), _ptr(ws),
        ws.numel(), _stream(stream)))


def nvfp4_grouped_swiglu_gemm(qa, sfa, gsa, qb, sfb, gsb, offsets, inter, granularity, limit, layout, out,
                              ws, stream=None):
    """Grouped GEMM + SwiGLU: qb/sfb hold E experts' [2I, K] weights stacked, offsets
    (int32 [E+1], device) the groups' row ranges of A; out is bf16 [M, I] or [M, 2I]."""
    M = qa.shape[0]
    K = qa.shape[1] * 2
    E = offsets.numel() - 1
    if offsets.dtype != torch.int32:
        raise TypeError("offsets must be int32")
    _check("nvfp4_grouped_swiglu_gemm", lib().nvfp4_grouped_swiglu_gemm(
        _ptr(qa), _ptr(sfa), _ptr(gsa), _ptr(qb), _ptr(sfb), _ptr(gsb), _ptr(offsets), M, E, int(inter), K,
        int(granularity), float(limit), int(layout), _ptr(out), out.stride(0), _ptr(ws), ws.numel(),
        _stream(stream)))


def grouped_swiglu_gemm(qa, sfa, gsa, qb, sfb, gsb, offsets, inter, granularity, ws,
                        limit=float("inf"), layout=0, stream=None):
    """Allocating convenience: the bf16 output (rows outside every group are left as zeros)."""
    M = qa.shape[0]
    out = torch.zeros(M, inter if layout == 0 else 2 * inter, dtype=torch.bfloat16, device=qa.device)
    nvfp4_grouped_swiglu_gemm(qa, sfa, gsa, qb, sfb, gsb, offsets, inter, granularity, limit, layout, out,
                              ws, stream)
    return out


def read_device_status(ws, stream=None) -> int:
    """Synchronising diagnostic: device status bits recorded in ws (then cleared)."""
    out = ctypes.c_uint32(0)
    _check("nvfp4_read_device_status", lib().nvfp4_read_device_status(
        _ptr(ws), ws.numel(), ctypes.byref(out), _stream(stream)))
    return int(out.value)


# ---------------------------------------------------------------- allocating helpers

def quantize(x: torch.Tensor, ws: torch.Tensor, stream=None):
    """(q [rows, cols/2] u8, sf [rows, cols/16] u8, gs [1] f32) of a bf16 [rows, cols] tensor."""
    rows, cols = x.shape
    q = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device=x.device)
    gs = torch.empty(1, dtype=torch.float32, device=x.device)
    nvfp4_quantize(x, q, sf, gs, ws, stream)
    return q, sf, gs


def deinterleave_quantize(x: torch.Tensor, granularity: int, ws: torch.Tensor, stream=None):
    rows, width = x.shape
    q = torch.empty(rows, width // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(rows, width // 16, dtype=torch.uint8, device=x.device)
    gs = torch.empty(1, dtype=torch.float32, device=x.device)
    nvfp4_deinterleave_quantize(x, granularity, q, sf, gs, ws, stream)
    return q, sf, gs


def gemm_topk(qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, k, ws, want_weight=True,
              want_logits=False, stream=None):
    M, N = qa.shape[0], qb.shape[0]
    dev = qa.device
    idx = torch.empty(M, k, dtype=torch.int32, device=dev)
    score = torch.empty(M, k, dtype=torch.float32, device=dev)
    weight = torch.empty(M, k, dtype=torch.float32, device=dev) if want_weight else None
    logits = torch.empty(M, N, dtype=torch.float32, device=dev) if want_logits else None
    nvfp4_gemm_topk(qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, k, idx, score, weight, logits,
                    ws, stream)
    return idx, score, weight, logits
