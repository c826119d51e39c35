"""GPU parity of nvfp4_rmsnorm_quantize (RMSNorm fused into the quantize)
with the oracle: bit-exact codes, scales and global scale.  Sizes cover the
three kernel paths: one cluster (up to 512 KB of input), one cooperative
grid (rows that fit in the SMs' shared memory), and the two row-parallel
passes beyond.  The sum of squares is the exact sum rounded once, so rows
of very wide range (bf16 subnormals, squares below FP32's normal range, a
row whose low-order terms decide the rounding) are compared too.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

EPS = 1e-6


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


def norm_weight(cols, seed):
    rng = np.random.default_rng(seed)
    return workloads.bf16_bits((1.0 + 0.1 * rng.standard_normal(cols)).astype(np.float32))


def run(nv, ws, x, w, ld=None):
    rows, cols = x.shape
    if ld is None or ld == cols:
        xd = torch.from_numpy(x.view(np.int16)).cuda()
    else:
        wide = np.zeros((rows, ld), np.uint16)
        wide[:, :cols] = x
        xd = torch.from_numpy(wide.view(np.int16)).cuda()[:, :cols]
    wd = torch.from_numpy(w.view(np.int16)).cuda()
    q, sf, gs = nv.rmsnorm_quantize(xd, wd, EPS, ws)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), gs.cpu().numpy()[0]


def check(got, ref, what):
    q, sf, gs = got
    rq, rsf, rgs = ref
    assert np.float32(gs).view(np.uint32) == np.float32(rgs).view(np.uint32), f"{what}: gs {gs} vs {rgs}"
    assert np.array_equal(sf, rsf), f"{what}: {int((sf != rsf).sum())} scale bytes differ"
    assert np.array_equal(q, rq), f"{what}: {int((q != rq).sum())} code bytes differ"


# (2600, 7168), (4000, 4096) and (1100, 16384) exceed the SMs' shared memory:
# the two passes, with 512 threads of one block, 256 of one, 512 of two
@pytest.mark.parametrize("rows,cols", [(1, 7168), (32, 7168), (5, 16), (40, 16384), (300, 4096),
                                       (1500, 7168), (2600, 7168), (4000, 4096), (1100, 16384)])
def test_rmsnorm_quantize_shapes(nv, ws, rows, cols):
    x = workloads.quantize_input(rows, seed=rows + cols, cols=cols)
    w = norm_weight(cols, cols)
    check(run(nv, ws, x, w), oracle.rmsnorm_quantize(x, w, EPS), f"{rows}x{cols}")


def test_rmsnorm_quantize_strided_and_outliers(nv, ws):
    d = workloads.router_prefill(tokens=64)
    x = d["x"]
    w = norm_weight(x.shape[1], 3)
    check(run(nv, ws, x, w, ld=7168 + 64), oracle.rmsnorm_quantize(x, w, EPS), "prefill rows, ld 7232")


def test_rmsnorm_quantize_two_calls_and_zero_rows(nv, ws):
    x1 = workloads.quantize_input(16, seed=91)
    # smaller values (scaled as floats): a stale maximum from the first call would show
    x2 = workloads.bf16_bits(workloads.bf16_to_f32(workloads.quantize_input(16, seed=92)) * np.float32(0.25))
    w = norm_weight(7168, 5)
    for x in (x1, x2):
        check(run(nv, ws, x, w), oracle.rmsnorm_quantize(x, w, EPS), "repeat")
    assert nv.read_device_status(ws) == 0
    xd = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    wd = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    q, sf, gs = nv.rmsnorm_quantize(xd, wd, EPS, ws)
    torch.cuda.synchronize()
    assert gs.item() == float(np.float32(1e-8) / np.float32(2688.0))


def _bits(e, m):
    """bf16 bit pattern with exponent field e and the 7 stored mantissa bits of m."""
    return (e << 7) | (m & 0x7F)


def wide_range_rows(cols):
    """Rows whose sum of squares needs more than the two windows the kernel
    sums by default: magnitudes over ~2^100 in one row, bf16 subnormals,
    squares below FP32's normal range, and a crafted row whose window sums
    sit right below a carry with a tiny term under them (the kernel then
    sums every window)."""
    rng = np.random.default_rng(77)
    rows = []
    for lo, hi in ((-50, 50), (-120, -60), (-133, -126), (0, 100)):
        f = rng.standard_normal(cols) * np.exp2(rng.integers(lo, hi, cols).astype(np.float64))
        rows.append(workloads.bf16_bits(f.astype(np.float32)))
    crafted = [_bits(127, 128)] + [_bits(109, 129)] * 3 + [_bits(107, 129)] * 15 + [_bits(87, 128)]
    crafted = np.array(crafted + [0] * (cols - len(crafted)), np.uint16)
    rows.append(crafted)
    rows.append(np.where(np.arange(cols) % 2 == 0, crafted[np.arange(cols) % 20], 0).astype(np.uint16))
    tie = np.zeros(cols, np.uint16)  # 4096^2 + 1 = 2^24 + 1: halfway, ties to even
    tie[0], tie[1] = _bits(139, 128), _bits(127, 128)
    rows.append(tie)
    return np.stack(rows)


@pytest.mark.parametrize("rows_rep", [1, 300])
def test_rmsnorm_quantize_exact_sum_wide_range(nv, ws, rows_rep):
    # rows_rep = 1: one cluster; 300 (2100 rows x 16 KB): the cooperative grid
    x = np.tile(wide_range_rows(7168), (rows_rep, 1))
    w = norm_weight(7168, 11)
    check(run(nv, ws, x, w), oracle.rmsnorm_quantize(x, w, EPS), f"wide-range rows x{rows_rep}")


def test_rmsnorm_quantize_exact_sum_wide_range_two_pass(nv, ws):
    # enough rows that the row-parallel two-pass kernels run
    x = np.tile(wide_range_rows(7168), (400, 1))
    w = norm_weight(7168, 12)
    check(run(nv, ws, x, w), oracle.rmsnorm_quantize(x, w, EPS), "wide-range rows, two passes")
