"""Host-side checks of the C ABI that need no GPU.

The library must build, load, and export every function include/nvfp4.h
declares.  Argument validation runs on the host before any CUDA call, so
invalid calls can be exercised here with fake (never dereferenced) pointers.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from quantize_block_scaled_gb300 import build as b
    b.build()
    import quantize_block_scaled_gb300 as q
    return q.lib()


def test_header_declares_the_three_entry_points():
    fns = _declared_functions()
    for name in ("nvfp4_quantize", "nvfp4_deinterleave_quantize", "nvfp4_gemm_topk"):
        assert name in fns


def test_library_exports_every_declared_symbol(L):
    import quantize_block_scaled_gb300 as q
    for name in _declared_functions():
        assert hasattr(L, name), name
    assert set(_declared_functions()) == set(q.EXPORTED_SYMBOLS)


def test_status_strings_and_workspace_size(L):
    assert L.nvfp4_status_string(0) == b"ok"
    assert L.nvfp4_status_string(2) == b"unsupported shape or alignment"
    import quantize_block_scaled_gb300 as q
    # one constant for every operation and shape (the kernels keep counters only)
    for op in range(7):
        assert L.nvfp4_workspace_bytes(op, 8192, 7168, 256, 8) == 256
        assert q.workspace_bytes(op, 1, 16, 0, 0) == 256
    assert L.nvfp4_workspace_bytes(7, 1, 16, 0, 0) == 0     # unknown operation
    assert L.nvfp4_workspace_bytes(-1, 1, 16, 0, 0) == 0
    assert L.nvfp4_workspace_bytes(0, -1, 16, 0, 0) == 0    # negative size


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: validation fails first


def _p(v):
    return ctypes.c_void_p(v)


def test_quantize_validation(L):
    ws = _p(FAKE)
    # null input (allowed only when there are no rows), null gs
    assert L.nvfp4_quantize(None, 4, 32, 32, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 1
    assert L.nvfp4_quantize(_p(FAKE), 4, 32, 32, _p(FAKE), _p(FAKE), None, ws, 256, None) == 1
    # negative rows, ld < cols
    assert L.nvfp4_quantize(_p(FAKE), -1, 32, 32, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 1
    assert L.nvfp4_quantize(_p(FAKE), 4, 32, 16, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 1
    # cols not a multiple of 16, misaligned x, ld not a multiple of 8
    assert L.nvfp4_quantize(_p(FAKE), 4, 40, 40, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 2
    assert L.nvfp4_quantize(_p(FAKE + 2), 4, 32, 32, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 2
    assert L.nvfp4_quantize(_p(FAKE), 4, 32, 36, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 2
    # workspace missing or short
    assert L.nvfp4_quantize(_p(FAKE), 4, 32, 32, _p(FAKE), _p(FAKE), _p(FAKE), None, 256, None) == 3
    assert L.nvfp4_quantize(_p(FAKE), 4, 32, 32, _p(FAKE), _p(FAKE), _p(FAKE), ws, 64, None) == 3


def test_deinterleave_validation(L):
    ws = _p(FAKE)
    assert L.nvfp4_deinterleave_quantize(_p(FAKE), 2, 64, 3, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 2
    assert L.nvfp4_deinterleave_quantize(_p(FAKE), 2, 40, 8, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 2
    assert L.nvfp4_deinterleave_quantize(_p(FAKE), 2, 0, 8, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 1
    assert L.nvfp4_deinterleave_quantize(None, 2, 64, 8, _p(FAKE), _p(FAKE), _p(FAKE), ws, 256, None) == 1


def _gemm(L, M=4, N=64, K=512, epilogue=1, bias=FAKE, k=6, qa=FAKE, sfa=FAKE, ws=FAKE, ws_bytes=256):
    P = _p
    return L.nvfp4_gemm_topk(P(qa), P(sfa), P(FAKE), P(FAKE), P(FAKE), P(FAKE), M, N, K, epilogue,
                             P(bias) if bias else None, k, P(FAKE), P(FAKE), None, None,
                             P(ws) if ws else None, ws_bytes, None)


def test_gemm_validation(L):
    assert _gemm(L, k=0) == 1
    assert _gemm(L, k=1025) == 1
    assert _gemm(L, epilogue=3) == 1
    assert _gemm(L, epilogue=1, bias=0) == 1       # router epilogues need a bias
    assert _gemm(L, epilogue=2, bias=0) == 1
    assert _gemm(L, epilogue=2, k=40) == 2         # normalised weights: k <= 32
    assert _gemm(L, M=-1) == 1
    assert _gemm(L, N=0) == 1
    assert _gemm(L, K=480) == 2                    # K must be a multiple of 64
    assert _gemm(L, k=512, N=8192) == 2            # large k needs N <= 4096
    assert _gemm(L, qa=FAKE + 8) == 2              # codes must be 16-byte aligned
    assert _gemm(L, sfa=FAKE + 2) == 2             # scales 4-byte aligned
    assert _gemm(L, ws=0) == 3
    assert _gemm(L, ws_bytes=16) == 3


def test_rmsnorm_quantize_validation(L):
    P, ws = _p, _p(FAKE)
    f = ctypes.c_float
    call = lambda x=FAKE, rows=4, cols=64, ld=64, w=FAKE, eps=1e-6: L.nvfp4_rmsnorm_quantize(
        P(x) if x else None, rows, cols, ld, P(w) if w else None, f(eps), P(FAKE), P(FAKE), P(FAKE), ws, 256, None)
    assert call(w=0) == 1                 # weight required
    assert call(eps=-1.0) == 1            # eps must be >= 0
    assert call(cols=40, ld=40) == 2      # cols multiple of 16
    assert call(cols=16400, ld=16400) == 2  # at most 16384 columns
    assert call(w=FAKE + 8) == 2          # weight 16-byte aligned


def test_indexer_topk_validation(L):
    P, ws = _p, _p(FAKE)
    call = lambda heads=64, N=2048, K=128, k=512, hw=FAKE: L.nvfp4_indexer_topk(
        P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 2, heads, N, K, P(hw) if hw else None, k,
        P(FAKE), P(FAKE), None, ws, 256, None)
    assert call(heads=48) == 2            # 32, 64 or 128 heads
    assert call(hw=0) == 1                # head weights required
    assert call(k=0) == 1
    assert call(N=5000) == 2              # keys on chip: N <= 4096
    assert call(K=100) == 2               # K a multiple of 64
    too_many = L.nvfp4_indexer_topk(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1 << 60, 64, 2048, 128,
                                    P(FAKE), 512, P(FAKE), P(FAKE), None, ws, 256, None)
    assert too_many == 1                  # tokens bounded before tokens * heads


def test_grouped_swiglu_validation(L):
    P, f = _p, ctypes.c_float

    def call(qa=FAKE, sfa=FAKE, offs=FAKE, out=FAKE, M=256, E=8, inter=2048, K=7168, g=8, limit=10.0,
             layout=0, ld=2048, ws=FAKE, ws_bytes=256, gsb=FAKE):
        return L.nvfp4_grouped_swiglu_gemm(P(qa) if qa else None, P(sfa) if sfa else None, P(FAKE), P(FAKE),
                                           P(FAKE), P(gsb) if gsb else None, P(offs) if offs else None, M, E,
                                           inter, K, g, f(limit), layout, P(out) if out else None, ld,
                                           P(ws) if ws else None, ws_bytes, None)

    assert call(offs=0) == 1                      # device offsets required when M > 0
    assert call(out=0) == 1
    assert call(gsb=0) == 1
    assert call(E=0) == 1
    assert call(E=1025) == 2                      # at most 1024 groups
    assert call(layout=2) == 1
    assert call(limit=0.0) == 1                   # limit > 0 (infinity allowed)
    assert call(limit=float("nan")) == 1
    assert call(g=3) == 2                         # granularity 1, 2, 4, 8, 16
    assert call(inter=200) == 2                   # I a multiple of 128
    assert call(inter=1 << 62) == 1               # sizes are checked before any product of them
    assert call(K=7168 + 64) == 2                 # K a multiple of 256
    assert call(ld=2040) == 2                     # ld >= I and a multiple of 8
    assert call(layout=1, ld=2048) == 2           # layout 1 rows hold 2I values
    assert call(ld=2052) == 2
    assert call(qa=FAKE + 8) == 2                 # codes 16-byte aligned
    assert call(sfa=FAKE + 4) == 2                # scales 16-byte aligned (TMA boxes)
    assert call(out=FAKE + 2) == 2                # bf16 rows stored 16 bytes at a time
    assert call(offs=FAKE + 2) == 2
    assert call(ws=0) == 3
    assert call(ws_bytes=64) == 3
    # M == 0 launches nothing and accepts NULL activations, offsets and output
    assert call(M=0, qa=0, sfa=0, offs=0, out=0) == 0


def test_mhc_rmsnorm_quantize_validation(L):
    P = _p(FAKE)
    ws = _p(FAKE)
    args = lambda rows, n, cols, ld: (P, rows, n, cols, ld, P, P, ctypes.c_float(1e-6), P, P, P, ws, 256, None)
    assert L.nvfp4_mhc_rmsnorm_quantize(*args(4, 0, 64, 64)) == 1       # no streams
    assert L.nvfp4_mhc_rmsnorm_quantize(*args(4, 9, 64, 9 * 64)) == 1   # more than 8 streams
    assert L.nvfp4_mhc_rmsnorm_quantize(*args(4, 4, 64, 200)) == 1      # token stride shorter than the streams
    assert L.nvfp4_mhc_rmsnorm_quantize(*args(4, 4, 24, 96)) == 2       # cols not a multiple of 16
    assert L.nvfp4_mhc_rmsnorm_quantize(*args(4, 1, 8208, 8208)) == 2   # cols beyond 8192
    assert L.nvfp4_mhc_rmsnorm_quantize(*args(4, 4, 64, 260)) == 2      # token stride not a multiple of 8
