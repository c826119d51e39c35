"""GPU parity of nvfp4_quantize / nvfp4_deinterleave_quantize with the oracle.

Bit-exact: packed codes, E4M3 scale bytes and the FP32 global scale.  The
sizes cover all three kernel paths: one cluster (up to 512 KB of input), one
cooperative grid (up to ~30 MB), and the amax + quantize kernel pair beyond.
Inputs are the seeded workloads (N(0,1) with 0.1% x100 outliers, the
Student-t prefill activations with +-U(500,2000) outliers) plus edge cases.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantize_block_scaled_gb300 import build as b
    b.build()
    import quantize_block_scaled_gb300 as nv
    nv.lib()
    return nv


@pytest.fixture(scope="module")
def ws(nv):
    return nv.workspace()


def gpu_quantize(nv, ws, x_bits: np.ndarray, ld=None):
    rows, cols = x_bits.shape
    if ld is None or ld == cols:
        xd = torch.from_numpy(x_bits.view(np.int16)).cuda()
    else:
        wide = np.zeros((rows, ld), np.uint16)
        wide[:, :cols] = x_bits
        xd = torch.from_numpy(wide.view(np.int16)).cuda()[:, :cols]
    q, sf, gs = nv.quantize(xd, ws)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), gs.cpu().numpy()[0]


def assert_quant_equal(got, ref, what):
    q, sf, gs = got
    rq, rsf, rgs = ref
    assert np.float32(gs).view(np.uint32) == np.float32(rgs).view(np.uint32), f"{what}: gs {gs} vs {rgs}"
    if not np.array_equal(sf, rsf):
        i = np.argwhere(sf != rsf)[0]
        raise AssertionError(f"{what}: {int((sf != rsf).sum())} scale bytes differ; first {tuple(i)}: "
                             f"gpu {sf[tuple(i)]:#x} oracle {rsf[tuple(i)]:#x}")
    if not np.array_equal(q, rq):
        i = np.argwhere(q != rq)[0]
        raise AssertionError(f"{what}: {int((q != rq).sum())} code bytes differ; first {tuple(i)}: "
                             f"gpu {q[tuple(i)]:#04x} oracle {rq[tuple(i)]:#04x}")


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (5, 7168), (300, 512), (129, 4096), (7, 2064)])
def test_quantize_small_shapes(nv, ws, rows, cols):
    x = workloads.quantize_input(rows, seed=100 + rows, cols=cols)
    assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), f"{rows}x{cols}")


@pytest.mark.parametrize("tokens", [1, 128, 2048, 16384])
def test_quantize_sweep(nv, ws, tokens):
    x = workloads.quantize_input(tokens)
    assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), f"sweep T={tokens}")


def test_quantize_prefill_outliers(nv, ws):
    x = workloads.router_prefill()["x"]
    assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), "prefill Student-t outliers")


def test_quantize_strided_rows(nv, ws):
    x = workloads.quantize_input(37, seed=7, cols=1024)
    assert_quant_equal(gpu_quantize(nv, ws, x, ld=1040), oracle.quantize(x), "ld 1040")


def test_quantize_strided_two_pass(nv, ws):
    # 2200 x 7168 bf16 = 31.5 MB: beyond what the one-pass kernel holds on chip
    # (about 30 MB), so the amax + quantize kernels run, on strided rows.
    x = workloads.quantize_input(2200, seed=8)
    assert_quant_equal(gpu_quantize(nv, ws, x, ld=7184), oracle.quantize(x), "two-pass ld 7184")


def test_quantize_edge_values(nv, ws):
    f = np.zeros((4, 64), np.float32)
    f[1, :] = -1e-30                      # all tiny negatives: one far-below-max block
    f[2, 5] = 3.0e38 / 1e30               # single large value
    f[2, 6:22] = np.linspace(-7, 7, 16)
    f[3, :16] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0]
    f[3, 16:32] = -0.01
    x = workloads.bf16_bits(f)
    assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), "edge values")
    z = np.zeros((3, 32), np.uint16)
    assert_quant_equal(gpu_quantize(nv, ws, z), oracle.quantize(z), "all zero")


def test_quantize_wide_scale_range(nv, ws):
    # Block maxima spread over 2^-30 .. 2^21, so the E4M3 scales run through
    # zero, the subnormal steps of 2^-9, every normal binade and saturation.
    rng = np.random.default_rng(12)
    rows, cols = 96, 1024
    f = rng.standard_normal((rows, cols)).astype(np.float32)
    e = rng.integers(-30, 21, size=(rows, cols // 16)).astype(np.float32)
    f *= np.repeat(np.exp2(e), 16, axis=1)
    x = workloads.bf16_bits(f)
    assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), "wide scale range")


def test_quantize_signed_zero_inputs(nv, ws):
    # -0.0 and +0.0 inputs next to normal values: codes 0x8 and 0x0
    x = workloads.quantize_input(8, seed=31, cols=512)
    x[:, ::7] = 0x8000
    x[:, 3::11] = 0x0000
    assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), "signed zeros")


def test_quantize_midpoint_quotients(nv, ws):
    # Blocks whose quotients x/den sit exactly on E2M1 rounding midpoints
    # (gs = 1 from a 2688 entry, block max 6 * 2^e so den = 2^e).
    rng = np.random.default_rng(9)
    f = np.zeros((64, 256), np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    for r in range(64):
        for b in range(16):
            e = rng.integers(-6, 8)
            blk = rng.choice(np.concatenate([mids, -mids]), 16)
            blk[0] = 6.0
            f[r, b * 16:(b + 1) * 16] = blk * np.float32(2.0 ** e)
    f[0, 0] = 2688.0
    x = workloads.bf16_bits(f)
    assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), "midpoints")


def test_quantize_zero_rows_writes_floor_scale(nv, ws):
    xd = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    q, sf, gs = nv.quantize(xd, ws)
    torch.cuda.synchronize()
    assert gs.item() == float(np.float32(1e-8) / np.float32(2688.0))


def test_quantize_repeated_calls_reuse_workspace(nv, ws):
    x1 = workloads.quantize_input(64, seed=21)
    x2 = workloads.quantize_input(64, seed=22) // 4  # different bit patterns, smaller values
    for x in (x1, x2, x1):
        assert_quant_equal(gpu_quantize(nv, ws, x), oracle.quantize(x), "repeat")
    w = ws.cpu().numpy().view(np.uint32)
    assert (w[:2] == 0).all()  # amax slot and block counter are left zeroed
    assert nv.read_device_status(ws) == 0


def gpu_deinterleave(nv, ws, x_bits, g):
    xd = torch.from_numpy(x_bits.view(np.int16)).cuda()
    q, sf, gs = nv.deinterleave_quantize(xd, g, ws)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), gs.cpu().numpy()[0]


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("tokens", [1, 7, 128])
def test_deinterleave_quantize(nv, ws, tokens, g):
    x = workloads.swiglu_interleaved(tokens)
    assert_quant_equal(gpu_deinterleave(nv, ws, x, g), oracle.deinterleave_quantize(x, g),
                       f"deinterleave T={tokens} g={g}")


@pytest.mark.parametrize("g", [1, 8])
def test_deinterleave_quantize_large(nv, ws, g):
    x = workloads.swiglu_interleaved(2048)
    assert_quant_equal(gpu_deinterleave(nv, ws, x, g), oracle.deinterleave_quantize(x, g),
                       f"deinterleave T=2048 g={g}")


def test_deinterleave_quantize_two_pass(nv, ws):
    # 4096 x 4096 bf16 = 33.5 MB: the amax + deinterleave kernels, not the one-pass kernel
    x = workloads.swiglu_interleaved(4096, seed=11)
    assert_quant_equal(gpu_deinterleave(nv, ws, x, 1), oracle.deinterleave_quantize(x, 1),
                       "deinterleave T=4096 g=1")


def test_deinterleave_small_width(nv, ws):
    x = workloads.swiglu_interleaved(5, inter=16, seed=3)
    for g in (1, 8, 16):
        assert_quant_equal(gpu_deinterleave(nv, ws, x, g), oracle.deinterleave_quantize(x, g),
                           f"deinterleave I=16 g={g}")
