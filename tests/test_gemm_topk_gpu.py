"""GPU parity of nvfp4_gemm_topk with the oracle.

Logits and scores within 1e-3 relative / 1e-4 absolute (FP32); top-k index
sets identical up to near-ties at the k-th score (tests/parity.py).  B
operands are quantized by the oracle's quantizer; A operands either by the
oracle (GEMM-stage checks) or by the GPU quantizer (end-to-end checks, after
checking those bytes equal the oracle's).
"""
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


def run_gpu(nv, ws, qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, k, logits=True):
    out = nv.gemm_topk(dev(qa), dev(sfa), dev(np.float32([gsa])), dev(qb), dev(sfb),
                       dev(np.float32([gsb])), epilogue,
                       None if bias is None else dev(np.asarray(bias, np.float32)), k, ws,
                       want_weight=True, want_logits=logits)
    torch.cuda.synchronize()
    idx, score, weight, lg = out
    return (idx.cpu().numpy(), score.cpu().numpy(), weight.cpu().numpy(),
            None if lg is None else lg.cpu().numpy())


def oracle_rows(qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, rows):
    """Oracle logits / scores / weights for a list of row indices."""
    lg = np.concatenate([oracle.gemm_logits(qa, sfa, gsa, qb, sfb, gsb, r, r + 1) for r in rows])
    score, weight = oracle.epilogue(lg, 1 if epilogue == 2 else epilogue, bias)
    return lg, score, weight


def check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, k, rows=None, what=""):
    M = qa.shape[0]
    rows = list(range(M)) if rows is None else list(rows)
    idx, score, weight, lg = run_gpu(nv, ws, qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, k)
    rlg, rscore, rweight = oracle_rows(qa, sfa, gsa, qb, sfb, gsb, epilogue, bias, rows)
    assert_close(lg[rows], rlg, f"{what} logits")
    assert_topk(idx[rows], score[rows], weight[rows], rscore, rweight, k, what, normalized=epilogue == 2)
    assert nv.read_device_status(ws) == 0
    return idx, score


def quantized(x):
    return oracle.quantize(x)


def test_tiny_router_end_to_end(nv, ws):
    d = workloads.router_tiny(0)
    xd = dev(d["x"].view(np.int16))
    qa, sfa, gsa = nv.quantize(xd, ws)
    torch.cuda.synchronize()
    rqa, rsfa, rgsa = quantized(d["x"])
    assert np.array_equal(qa.cpu().numpy(), rqa) and np.array_equal(sfa.cpu().numpy(), rsfa)
    assert gsa.item() == rgsa
    qb, sfb, gsb = quantized(d["w"])
    check_case(nv, ws, rqa, rsfa, rgsa, qb, sfb, gsb, 1, d["bias"], d["k"], what="tiny router")


@pytest.mark.parametrize("tokens,seed", [(1, 1), (32, 2)])
def test_router_decode(nv, ws, tokens, seed):
    d = workloads.router_decode(tokens, seed)
    qa, sfa, gsa = quantized(d["x"])
    qb, sfb, gsb = quantized(d["w"])
    check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, 1, d["bias"], d["k"], what=f"decode T={tokens}")


def test_router_prefill_sampled_rows(nv, ws):
    d = workloads.router_prefill()
    xd = dev(d["x"].view(np.int16))
    qa_d, sfa_d, gsa_d = nv.quantize(xd, ws)
    torch.cuda.synchronize()
    qa, sfa, gsa = qa_d.cpu().numpy(), sfa_d.cpu().numpy(), gsa_d.cpu().numpy()[0]
    M = qa.shape[0]
    rng = np.random.default_rng(0)
    rows = sorted(set(range(0, 128)) | set(range(M - 128, M)) | set(rng.integers(0, M, 256).tolist()))
    # the GPU-quantized activation must equal the oracle's on the sampled rows
    rgsa = oracle.global_scale(d["x"])
    assert gsa == rgsa
    rq, rsf = oracle.quantize_rows(d["x"], rgsa, 0, 128)
    assert np.array_equal(qa[:128], rq) and np.array_equal(sfa[:128], rsf)
    qb, sfb, gsb = quantized(d["w"])
    check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, 1, d["bias"], d["k"], rows=rows,
               what="prefill T=8192")


def test_indexer_shape(nv, ws):
    d = workloads.indexer()
    qa, sfa, gsa = quantized(d["x"])
    qb, sfb, gsb = quantized(d["w"])
    check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, 0, None, d["k"], what="indexer")


EDGE = [
    # M, N, K, k, epilogue
    (1, 16, 64, 1, 0),
    (130, 200, 320, 8, 1),      # ragged M and N tiles, K not a multiple of 256
    (257, 384, 1024, 32, 0),
    (5, 10, 64, 16, 1),         # k > N: padded slots
    (3, 100, 192, 64, 1),       # select path with the router epilogue
    (33, 1000, 256, 100, 0),    # select path, ragged
    (200, 4096, 128, 1024, 0),  # largest k, largest N for the select path
    (9, 4000, 64, 1024, 1),
    (300, 256, 512, 20, 1),     # split K, warp arg-max rounds (8 < k <= 32)
    (64, 128, 7168, 8, 1),      # split K over many slices, butterfly top-8
]


@pytest.mark.parametrize("M,N,K,k,epi", EDGE)
def test_edge_shapes(nv, ws, M, N, K, k, epi):
    rng = np.random.default_rng(M * 7 + N)
    xa = workloads.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    xb = workloads.bf16_bits((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    bias = (rng.standard_normal(N) * 0.01).astype(np.float32) if epi == 1 else None
    qa, sfa, gsa = quantized(xa)
    qb, sfb, gsb = quantized(xb)
    check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, epi, bias, k, what=f"edge {M}x{N}x{K} k={k}")


# Many row tiles: two 128-column CTAs per tile, per-thread register lists of
# 16 / 32 entries merged across the pair (checked on sampled rows).
WIDE = [
    (5000, 256, 256, 12, 1),
    (5000, 200, 512, 24, 0),
    (4900, 256, 768, 32, 1),
]


@pytest.mark.parametrize("M,N,K,k,epi", WIDE)
def test_many_row_tiles(nv, ws, M, N, K, k, epi):
    rng = np.random.default_rng(M + N + K)
    xa = workloads.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    xb = workloads.bf16_bits((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    bias = (rng.standard_normal(N) * 0.01).astype(np.float32) if epi == 1 else None
    qa, sfa, gsa = quantized(xa)
    qb, sfb, gsb = quantized(xb)
    rows = sorted(set(range(0, 130)) | set(range(M - 70, M)) | set(rng.integers(0, M, 200).tolist()))
    check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, epi, bias, k, rows=rows,
               what=f"wide {M}x{N}x{K} k={k}")


# Router variant with normalised gating weights (epilogue 2): 384 experts,
# top-6, on the decode and prefill paths, plus wider rows and k > 8.
VARIANTS = [
    # M, N, K, k
    (1, 384, 7168, 6),       # decode: K split, 16 columns per lane
    (32, 384, 7168, 6),
    (2048, 384, 1024, 6),    # direct epilogue, two 256-column CTAs per tile
    (64, 400, 512, 20),      # K split, arg-max rounds over 16 columns per lane
    (40, 640, 256, 6),       # N > 512: block-wide selection
]


@pytest.mark.parametrize("M,N,K,k", VARIANTS)
def test_router_variant_normalised(nv, ws, M, N, K, k):
    rng = np.random.default_rng(M * 3 + N + K)
    xa = workloads.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    xb = workloads.bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    bias = (rng.standard_normal(N) * 0.01).astype(np.float32)
    qa, sfa, gsa = quantized(xa)
    qb, sfb, gsb = quantized(xb)
    rows = None if M <= 64 else sorted(set(range(0, 96)) | set(range(M - 32, M)))
    idx, _ = check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, 2, bias, k, rows=rows,
                        what=f"variant {M}x{N}x{K} k={k}")


@pytest.mark.parametrize("k", [4, 40])
def test_exact_ties_ordered_by_index(nv, ws, k):
    # Duplicate B rows give bit-identical logits; ties must come out by lower index.
    rng = np.random.default_rng(5)
    M, K = 6, 256
    base = workloads.bf16_bits((rng.standard_normal((8, K)) * 0.05).astype(np.float32))
    xb = np.concatenate([base] * 8)  # N = 64, each row repeated 8 times
    xa = workloads.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    qa, sfa, gsa = quantized(xa)
    qb, sfb, gsb = quantized(xb)
    idx, score = check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, 0, None, k, what="ties")
    for r in range(M):
        s = score[r]
        same = np.diff(s) == 0
        assert same.any()
        assert (np.diff(idx[r])[same] > 0).all()


def test_empty_rows_is_a_no_op(nv, ws):
    z8 = torch.zeros(0, 32, dtype=torch.uint8, device="cuda")
    zs = torch.zeros(0, 4, dtype=torch.uint8, device="cuda")
    qb = torch.zeros(16, 32, dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(16, 4, dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    idx, score, _, _ = nv.gemm_topk(z8, zs, g, qb, sfb, g, 0, None, 4, ws)
    torch.cuda.synchronize()
    assert idx.shape == (0, 4)


# The router epilogue of the direct path scores only the columns whose logit
# can still reach the top 8 (a threshold from the logits and the spread of
# the biases).  These cases drive that threshold to its ends: biases wide
# enough that nothing is filtered, biases so narrow that only the top logits
# survive, a ragged last column tile, logits far into both tails of softplus,
# and exact ties (duplicate gate rows with equal biases).
FILTER = [
    # M, N, K, bias_std, weight_std
    (5120, 256, 256, 1.0, 0.05),
    (5120, 256, 256, 1e-4, 0.05),
    (5120, 200, 512, 0.01, 0.05),
    (5120, 256, 256, 0.01, 3.0),
]


@pytest.mark.parametrize("M,N,K,bstd,wstd", FILTER)
def test_router_candidate_filter(nv, ws, M, N, K, bstd, wstd):
    rng = np.random.default_rng(M + N + int(K * wstd))
    xa = workloads.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    xb = workloads.bf16_bits((rng.standard_normal((N, K)) * wstd).astype(np.float32))
    bias = (rng.standard_normal(N) * bstd).astype(np.float32)
    qa, sfa, gsa = quantized(xa)
    qb, sfb, gsb = quantized(xb)
    rows = sorted(set(range(0, 64)) | set(range(M - 64, M)) | set(rng.integers(0, M, 128).tolist()))
    check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, 1, bias, 8, rows=rows,
               what=f"filter {M}x{N}x{K} bias {bstd} w {wstd}")


def test_router_candidate_filter_exact_ties(nv, ws):
    rng = np.random.default_rng(17)
    M, K = 5120, 256
    base = workloads.bf16_bits((rng.standard_normal((32, K)) * 0.05).astype(np.float32))
    xb = np.concatenate([base] * 8)  # N = 256: each gate row 8 times
    bias = np.tile((rng.standard_normal(32) * 0.01).astype(np.float32), 8)
    xa = workloads.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    qa, sfa, gsa = quantized(xa)
    qb, sfb, gsb = quantized(xb)
    rows = list(range(0, 48)) + list(range(M - 16, M))
    idx, score = check_case(nv, ws, qa, sfa, gsa, qb, sfb, gsb, 1, bias, 8, rows=rows, what="router ties")
    for r in rows:
        same = np.diff(score[r]) == 0
        assert same.any()
        assert (np.diff(idx[r])[same] > 0).all()
