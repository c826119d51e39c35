"""GPU parity of nvfp4_indexer_topk (the full indexer score with the head sum):
I[t, s] = sum_h w[t, h] * ReLU(q[t, h] . K[s]) fused in the GEMM epilogue,
then the top-k per token.  Scores within 1e-3 relative / 1e-4 absolute,
index sets equal up to near-ties (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close, assert_topk

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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


CASES = [
    # tokens, heads, N, K, k
    (1, 64, 2048, 128, 512),   # one decode token, 64 heads, 2048 compressed keys
    (4, 64, 2048, 128, 512),   # two tokens per row tile
    (5, 32, 1000, 256, 100),   # four tokens per tile, ragged keys and tokens
    (3, 128, 640, 128, 64),    # one token per tile
    (3, 64, 300, 128, 16),     # short rows: warp-per-row selection
]


@pytest.mark.parametrize("T,H,N,K,k", CASES)
def test_indexer_topk(nv, ws, T, H, N, K, k):
    rng = np.random.default_rng(T * 7 + H + N + K)
    q = workloads.bf16_bits(rng.standard_normal((T * H, K)).astype(np.float32))
    keys = workloads.bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    w = (rng.standard_normal((T, H)) / 8).astype(np.float32)
    qa, sfa, gsa = oracle.quantize(q)
    qb, sfb, gsb = oracle.quantize(keys)
    idx, score, I = nv.indexer_topk(dev(qa), dev(sfa), dev(np.float32([gsa])), dev(qb), dev(sfb),
                                    dev(np.float32([gsb])), H, dev(w), k, ws, want_scores=True)
    torch.cuda.synchronize()
    ref = oracle.indexer_scores(qa, sfa, gsa, qb, sfb, gsb, H, w)
    assert_close(I.cpu().numpy(), ref, f"indexer I {T}x{H}x{N}")
    assert_topk(idx.cpu().numpy(), score.cpu().numpy(), None, ref, None, k, f"indexer {T}x{H}x{N} k={k}")
    assert nv.read_device_status(ws) == 0


def test_indexer_no_tokens(nv, ws):
    z8 = torch.zeros(0, 64, dtype=torch.uint8, device="cuda")
    zs = torch.zeros(0, 8, dtype=torch.uint8, device="cuda")
    kb = torch.zeros(32, 64, dtype=torch.uint8, device="cuda")
    sk = torch.zeros(32, 8, dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    hw = torch.zeros(0, 64, dtype=torch.float32, device="cuda")
    idx, score, _ = nv.indexer_topk(z8, zs, g, kb, sk, g, 64, hw, 8, ws)
    torch.cuda.synchronize()
    assert idx.shape == (0, 8)
