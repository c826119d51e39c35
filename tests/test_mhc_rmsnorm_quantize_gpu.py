"""GPU parity of nvfp4_mhc_rmsnorm_quantize (the mHC pre-mix of the residual
streams, RMSNorm and the NVFP4 quantize in one op) with the oracle:
bit-exact codes, scales and global scale.  Sizes cover the kernel paths:
one cluster (the tokens' streams up to 512 KB), one cooperative grid (up to
the SMs' shared memory) and the two row-parallel passes beyond; stream
counts 1 to 4 and a token stride wider than the streams.
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


def case(T, n, d, seed):
    """Residual streams ~ N(0, 1) with 0.1% outliers x100 (the residual grows
    large in places), input mapping sigmoid(N(0,1)) + 1e-6 as bf16, norm
    weight 1 + N(0, 0.1)."""
    rng = np.random.default_rng(seed)
    x = workloads.quantize_input(T * n, seed=seed, cols=d).reshape(T, n, d)
    a = workloads.bf16_bits((1.0 / (1.0 + np.exp(-rng.standard_normal((T, n)))) + 1e-6).astype(np.float32))
    w = workloads.bf16_bits((1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32))
    return x, a, w


def run(nv, ws, x, a, w, pad=0):
    T, n, d = x.shape
    if pad:
        wide = np.zeros((T, n * d + pad), np.uint16)
        wide[:, :n * d] = x.reshape(T, n * d)
        xd = torch.from_numpy(wide.view(np.int16)).cuda()[:, :n * d].view(T, n, d)
    else:
        xd = torch.from_numpy(x.view(np.int16)).cuda()
    q, sf, gs = nv.mhc_rmsnorm_quantize(xd, torch.from_numpy(a.view(np.int16)).cuda(),
                                        torch.from_numpy(w.view(np.int16)).cuda(), EPS, ws)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), gs.cpu().numpy()[0]


def check(got, ref, what):
    q, sf, gs = got
    rq, rsf, rgs = ref
    assert np.float32(gs).view(np.uint32) == np.float32(rgs).view(np.uint32), f"{what}: gs {gs} vs {rgs}"
    assert np.array_equal(sf, rsf), f"{what}: {int((sf != rsf).sum())} scale bytes differ"
    assert np.array_equal(q, rq), f"{what}: {int((q != rq).sum())} code bytes differ"


# (600, 4, 7168) and (1200, 4, 4096) exceed the SMs' shared memory: the two passes
@pytest.mark.parametrize("T,n,d", [(1, 4, 7168), (8, 4, 7168), (32, 4, 7168), (3, 1, 512), (5, 2, 2048),
                                   (300, 3, 4096), (600, 4, 7168), (1200, 4, 4096)])
def test_mhc_rmsnorm_quantize_shapes(nv, ws, T, n, d):
    x, a, w = case(T, n, d, seed=T + 10 * n + d)
    check(run(nv, ws, x, a, w), oracle.mhc_rmsnorm_quantize(x, a, w, EPS), f"{T}x{n}x{d}")


def test_mhc_rmsnorm_quantize_token_stride_and_repeat(nv, ws):
    x, a, w = case(40, 4, 1024, seed=3)
    ref = oracle.mhc_rmsnorm_quantize(x, a, w, EPS)
    check(run(nv, ws, x, a, w, pad=64), ref, "token stride 4160")
    # a second call with smaller streams: nothing of the first one remains
    x2 = workloads.bf16_bits(workloads.bf16_to_f32(x) * np.float32(0.25))
    check(run(nv, ws, x2, a, w), oracle.mhc_rmsnorm_quantize(x2, a, w, EPS), "repeat, smaller")
    assert nv.read_device_status(ws) == 0
