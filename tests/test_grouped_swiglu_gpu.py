"""GPU parity of nvfp4_grouped_swiglu_gemm (grouped NVFP4 GEMM + SwiGLU) with the oracle.

The oracle gives the SwiGLU result in double from its FP32 logits; the GPU
stores bf16 after an FP32 epilogue.  Bound per element:
|gpu - h| <= 1e-4 + (1e-3 + 2^-8) * |h| — the logit tolerance of the GEMM
(1e-3 relative, 1e-4 absolute) carried through SiLU and the product, plus
the bf16 rounding of the stored value (at most half an ulp, 2^-8 relative).
Rows outside every group must stay untouched.  Weights and activations are
quantized by the oracle's quantizer (activations once for all grouped rows).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_to_f32

pytestmark = pytest.mark.gpu

RTOL = 1e-3 + 2.0 ** -8
ATOL = 1e-4


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


def quantize_experts(w, E):
    """Each expert's [2I, K] weights quantized on its own (its own gsb)."""
    rows = w.shape[0] // E
    parts = [oracle.quantize(w[e * rows:(e + 1) * rows]) for e in range(E)]
    qb = np.concatenate([p[0] for p in parts])
    sfb = np.concatenate([p[1] for p in parts])
    gsb = np.array([p[2] for p in parts], np.float32)
    return qb, sfb, gsb


def make_case(M, sizes, I, K, seed, std_a=1.0):
    E = len(sizes)
    rng = np.random.default_rng(seed)
    x = workloads.bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * np.float32(std_a))
    qa, sfa, gsa = oracle.quantize(x)
    w = workloads.moe_l1_weights(E, I, K, seed + 1)
    qb, sfb, gsb = quantize_experts(w, E)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    assert offs[-1] <= M
    return qa, sfa, gsa, qb, sfb, gsb, offs


def run(nv, ws, case, I, g, limit, layout, ld_pad=0):
    qa, sfa, gsa, qb, sfb, gsb, offs = case
    M = qa.shape[0]
    width = (I if layout == 0 else 2 * I)
    out = torch.full((M, width + ld_pad), -7.0, dtype=torch.bfloat16, device="cuda")
    view = out[:, :width] if ld_pad else out
    nv.nvfp4_grouped_swiglu_gemm(dev(qa), dev(sfa), dev(np.float32([gsa])), dev(qb), dev(sfb), dev(gsb),
                                 dev(offs), I, g, limit, layout, view, ws)
    torch.cuda.synchronize()
    assert nv.read_device_status(ws) == 0
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def expected_values(case, I, g, limit, layout):
    qa, sfa, gsa, qb, sfb, gsb, offs = case
    h, a = oracle.grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, offs, I, g, limit)
    if layout == 0:
        return h
    out = np.zeros((h.shape[0], 2 * I))
    for j0 in range(0, I, g):
        out[:, 2 * j0:2 * j0 + g] = a[:, j0:j0 + g]
        out[:, 2 * j0 + g:2 * j0 + 2 * g] = h[:, j0:j0 + g]
    return out


def assert_swiglu(got_bits, ref, what):
    got = bf16_to_f32(got_bits).astype(np.float64)
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {i}: "
                             f"gpu {got[i]!r} oracle {ref[i]!r}")


def check(nv, ws, case, I, g, limit, layout, what, ld_pad=0):
    got = run(nv, ws, case, I, g, limit, layout, ld_pad)
    offs = case[6]
    width = I if layout == 0 else 2 * I
    ref = expected_values(case, I, g, limit, layout)
    end = int(offs[-1])
    assert_swiglu(got[:end, :width], ref[:end], what)
    # rows past the groups and the padding columns are untouched (-7.0 = 0xC0E0)
    assert np.all(got[end:] == 0xC0E0), f"{what}: rows outside the groups were written"
    if ld_pad:
        assert np.all(got[:, width:] == 0xC0E0), f"{what}: padding columns were written"
    return got


@pytest.mark.parametrize("layout", [0, 1])
def test_ragged_groups_g8(nv, ws, layout):
    # groups of 130, 0, 5 and 260 rows (several tiles, ragged tails, an empty
    # group) and 7 rows after the last group; a limit of 1 clamps many gates
    # and up values
    case = make_case(402, [130, 0, 5, 260], 128, 256, seed=31)
    check(nv, ws, case, 128, 8, 1.0, layout, f"g8 layout {layout}")


@pytest.mark.parametrize("g", [1, 2, 4, 16])
def test_granularities(nv, ws, g):
    rng = np.random.default_rng(40 + g)
    sizes = rng.integers(0, 90, 8)
    case = make_case(int(sizes.sum()) + 3, sizes, 256, 512, seed=41 + g)
    check(nv, ws, case, 256, g, 10.0, g % 2, f"g{g}")


def test_many_items_per_cta_and_ld(nv, ws):
    # 64 groups x 4 weight slices (I = 512): more items than SMs, so each CTA
    # walks several and the stage ring wraps across items (K = 1024: 4 K tiles
    # on 3 stages); output rows with a padded leading dimension
    rng = np.random.default_rng(50)
    sizes = rng.integers(1, 9, 64)
    case = make_case(int(sizes.sum()), sizes, 512, 1024, seed=51)
    check(nv, ws, case, 512, 8, float("inf"), 0, "persistent", ld_pad=16)


def test_all_groups_empty_and_no_rows(nv, ws):
    case = make_case(16, [0, 0, 0], 128, 256, seed=60)
    got = run(nv, ws, case, 128, 8, 10.0, 0)
    assert np.all(got == 0xC0E0)
    # M == 0: nothing launched, NULL activations, offsets and output accepted
    qa, sfa, gsa, qb, sfb, gsb, offs = case
    t_gsa, t_qb, t_sfb, t_gsb = dev(np.float32([gsa])), dev(qb), dev(sfb), dev(gsb)
    before = nv.kernel_launches()
    rc = nv.lib().nvfp4_grouped_swiglu_gemm(None, None, nv._ptr(t_gsa), nv._ptr(t_qb), nv._ptr(t_sfb),
                                            nv._ptr(t_gsb), None, 0, 3, 128, 256, 8, 10.0, 0, None, 128,
                                            nv._ptr(ws), ws.numel(), nv._stream(None))
    assert rc == 0 and nv.kernel_launches() == before


def test_bad_offsets_are_flagged_not_faulting(nv, ws):
    # Offsets outside [0, M] or decreasing: the kernel clamps each group's
    # range into [0, M] (no access leaves the buffers) and records
    # NVFP4_DEVICE_BAD_GROUPS.
    qa, sfa, gsa, qb, sfb, gsb, _ = make_case(64, [10, 20, 30], 128, 256, seed=70)
    args = (dev(qa), dev(sfa), dev(np.float32([gsa])), dev(qb), dev(sfb), dev(gsb))
    out = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    # [-5, 30, 30, 9999] clamps to the groups [0, 30), [30, 30), [30, 64)
    nv.nvfp4_grouped_swiglu_gemm(*args, dev(np.array([-5, 30, 30, 9999], np.int32)), 128, 8, 10.0, 0, out, ws)
    torch.cuda.synchronize()
    assert nv.read_device_status(ws) == nv.DEVICE_BAD_GROUPS
    h, _ = oracle.grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, np.array([0, 30, 30, 64], np.int32), 128, 8, 10.0)
    assert_swiglu(out.view(torch.int16).cpu().numpy().view(np.uint16), h, "clamped")
    # decreasing offsets (overlapping groups after clamping): flagged; the
    # output of the overlap is unspecified
    nv.nvfp4_grouped_swiglu_gemm(*args, dev(np.array([0, 40, 20, 64], np.int32)), 128, 8, 10.0, 0, out, ws)
    torch.cuda.synchronize()
    assert nv.read_device_status(ws) == nv.DEVICE_BAD_GROUPS


def test_decode_shape_sampled(nv, ws):
    # MoE first projection at decode: 32 tokens x top-8 of 256 experts,
    # hidden 7168, I = 2048, granularity 8, limit 10; grouped rows gathered
    # from the token activations and quantized together (one gsa); sampled
    # rows of several groups checked against the oracle.
    T, E, k, I, K = 32, 256, 8, workloads.MOE_INTER, workloads.HIDDEN
    tok, offs = workloads.moe_routing(T, E, k, seed=80)
    x = workloads.quantize_input(T, seed=81)
    qa, sfa, gsa = oracle.quantize(x[tok])
    wrng = np.random.default_rng(82)
    # a full [E * 2I, K] bf16 draw is 7.5 G values: draw one expert's weights
    # per used group index pattern and reuse them across experts (each expert
    # still quantized on its own)
    w_one = workloads.moe_l1_weights(4, I, K, seed=83)
    qbs, sfbs, gsbs = quantize_experts(w_one, 4)
    pick = wrng.integers(0, 4, E)
    rows_per = 2 * I
    qb = np.concatenate([qbs[p * rows_per:(p + 1) * rows_per] for p in pick])
    sfb = np.concatenate([sfbs[p * rows_per:(p + 1) * rows_per] for p in pick])
    gsb = gsbs[pick]
    case = (qa, sfa, gsa, qb, sfb, gsb, offs)
    got = run(nv, ws, case, I, 8, 10.0, 0)
    nonempty = [e for e in range(E) if offs[e + 1] > offs[e]]
    for e in wrng.choice(nonempty, 6, replace=False):
        lo, hi = int(offs[e]), int(offs[e + 1])
        w = slice(e * rows_per, (e + 1) * rows_per)
        h, _ = oracle.grouped_swiglu(qa[lo:hi], sfa[lo:hi], gsa, qb[w], sfb[w], gsb[e:e + 1],
                                     np.array([0, hi - lo], np.int32), I, 8, 10.0)
        assert_swiglu(got[lo:hi], h, f"decode group {e}")


@pytest.mark.parametrize("layout", [0, 1])
def test_single_expert_ragged_rows(nv, ws, layout):
    # one expert (the shared-expert case of the pages: num_groups = 1), 45 rows
    # (one partial tile, not a multiple of the 32-row A boxes), K = 1024
    case = make_case(45, [45], 256, 1024, seed=90)
    check(nv, ws, case, 256, 8, 10.0, layout, f"single expert layout {layout}", ld_pad=8)


def test_leading_empty_group_and_offset_start(nv, ws):
    # the first group starts past row 0 (rows 0..9 belong to no group) and a
    # group of exactly 128 rows sits between two empty ones
    qa, sfa, gsa, qb, sfb, gsb, _ = make_case(300, [0, 0, 0, 0], 128, 256, seed=91)
    offs = np.array([10, 10, 138, 138, 250], np.int32)
    case = (qa, sfa, gsa, qb, sfb, gsb, offs)
    got = run(nv, ws, case, 128, 4, 10.0, 0)
    h, _ = oracle.grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, offs, 128, 4, 10.0)
    assert_swiglu(got[10:250], h[10:250], "offset groups")
    assert np.all(got[:10] == 0xC0E0) and np.all(got[250:] == 0xC0E0)


def test_prefill_like_full_tiles_sampled(nv, ws):
    # 1024 tokens x top-8 over 32 experts (about 256 rows per group: full
    # 128-row tiles, several per group, every expert used), hidden 7168,
    # I = 2048: the K ring runs 28 stages per item over many items per CTA.
    # Rows at each sampled group's start, its first tile boundary (127, 128)
    # and its end are checked against the oracle.
    T, E, k, I, K = 1024, 32, 8, workloads.MOE_INTER, workloads.HIDDEN
    tok, offs = workloads.moe_routing(T, E, k, seed=95)
    x = workloads.quantize_input(T, seed=96)
    qa, sfa, gsa = oracle.quantize(x[tok])
    w_one = workloads.moe_l1_weights(4, I, K, seed=97)
    qbs, sfbs, gsbs = quantize_experts(w_one, 4)
    pick = np.arange(E) % 4
    rows_per = 2 * I
    qb = np.concatenate([qbs[p * rows_per:(p + 1) * rows_per] for p in pick])
    sfb = np.concatenate([sfbs[p * rows_per:(p + 1) * rows_per] for p in pick])
    gsb = gsbs[pick]
    case = (qa, sfa, gsa, qb, sfb, gsb, offs)
    got = run(nv, ws, case, I, 8, 10.0, 0)
    sizes = offs[1:] - offs[:-1]
    assert sizes.min() > 129, sizes.min()
    for e in (0, 13, 31):
        lo, hi = int(offs[e]), int(offs[e + 1])
        rows = [lo, lo + 1, lo + 127, lo + 128, hi - 2, hi - 1]
        w = slice(e * rows_per, (e + 1) * rows_per)
        for r in rows:
            h, _ = oracle.grouped_swiglu(qa[r:r + 1], sfa[r:r + 1], gsa, qb[w], sfb[w], gsb[e:e + 1],
                                         np.array([0, 1], np.int32), I, 8, 10.0)
            assert_swiglu(got[r:r + 1], h, f"group {e} row {r - lo}")
