"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed independently: the
pages' E2M1 table and scale constants (tests/golden), PyTorch's own
float8_e4m3fn conversion (a library routine), numpy matmul / logaddexp,
closed forms, inputs built exactly on the NVFP4 grid, and brute force on
tiny inputs.  They are chosen so that a dropped term, a wrong sign or index,
a swapped nibble or a transposed operand in the oracle fails at least one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
import workloads
from workloads import bf16_bits, bf16_to_f32

E2M1_TABLE = {int(c, 2): float(v) for c, v in read_golden("e2m1_table.txt")}
CONST = {k: float(v) for k, v in read_golden("scale_constants.txt")}
E2M1_VALUES = [E2M1_TABLE[c] for c in range(8)]


# ---------------------------------------------------------------- E2M1 codec

def test_e2m1_table_from_page():
    assert len(E2M1_TABLE) == 8
    for code, value in E2M1_TABLE.items():
        assert oracle.e2m1_decode(code) == value
        assert oracle.e2m1_decode(code | 8) == -value
    # the two codes the pages single out
    assert oracle.e2m1_decode(0b101) == 3.0 and oracle.e2m1_decode(0b110) == 4.0
    # the bug the pages fixed: magnitude bits are not an integer
    assert any(oracle.e2m1_decode(c) != float(c) for c in range(8))


def test_e2m1_encode_inverts_decode():
    for code in range(8):
        assert oracle.e2m1_encode(E2M1_TABLE[code]) == code
        assert oracle.e2m1_encode(-E2M1_TABLE[code]) == code | 8


def test_e2m1_encode_midpoints_round_to_even():
    # Exact midpoints between neighbouring magnitudes go to the even code.
    expected = {0.25: 0b000, 0.75: 0b010, 1.25: 0b010, 1.75: 0b100,
                2.5: 0b100, 3.5: 0b110, 5.0: 0b110}
    for v, code in expected.items():
        assert oracle.e2m1_encode(v) == code, v
        assert oracle.e2m1_encode(-v) == code | 8, v
        lo = np.nextafter(np.float32(v), np.float32(0))
        hi = np.nextafter(np.float32(v), np.float32(10))
        # just below / above the midpoint: the nearer neighbour
        below = max(c for c in range(8) if E2M1_VALUES[c] < v)
        above = min(c for c in range(8) if E2M1_VALUES[c] > v)
        assert oracle.e2m1_encode(float(lo)) == below
        assert oracle.e2m1_encode(float(hi)) == above


def test_e2m1_encode_nearest_and_saturating():
    grid = np.array(E2M1_VALUES)
    for v in np.linspace(0.0, 9.0, 4001, dtype=np.float32):
        code = oracle.e2m1_encode(float(v))
        d = abs(float(v) - E2M1_VALUES[code])
        assert d <= np.min(np.abs(grid - float(v))) + 1e-12
        if v > 6.0:
            assert code == 7
    for v in (6.0, 7.5, 1e6, 1e30, 3.4e38):
        assert oracle.e2m1_encode(v) == 7 and oracle.e2m1_encode(-v) == 15
    # sign of values that round to zero is kept
    assert oracle.e2m1_encode(-0.1) == 0b1000
    assert oracle.e2m1_encode(-0.0) == 0b1000
    assert oracle.e2m1_encode(0.1) == 0


# ---------------------------------------------------------------- E4M3 codec

def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v)
        else:
            assert v == ref[c], c
    assert oracle.e4m3_decode(0x7E) == CONST["e4m3_max"]
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    vals = [oracle.e4m3_decode(c) for c in range(127)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    sweep = np.concatenate([
        np.float32(vals), np.float32(mids),
        np.nextafter(np.float32(mids), np.float32(0)), np.nextafter(np.float32(mids), np.float32(1e9)),
        np.random.default_rng(11).uniform(0, 464, 20000).astype(np.float32),
        np.float32([0.0, 1e-30, 2.0 ** -10, 448.0, 460.0, 464.0]),
    ]).astype(np.float32)
    ref = torch.from_numpy(sweep).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in sweep], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_inverts_decode_and_saturates():
    for c in range(127):
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c
    for v in (448.0, 464.0, 465.0, 1000.0, 1e30):
        assert oracle.e4m3_encode(v) == 0x7E


# ---------------------------------------------------------------- global scale

def _bf16(a):
    return bf16_bits(np.asarray(a, np.float32))


def test_global_scale_closed_form():
    assert CONST["gs_divisor"] == CONST["fp4_max"] * CONST["e4m3_max"]
    x = np.zeros((3, 32), np.float32)
    x[1, 7] = -2688.0
    assert oracle.global_scale(_bf16(x)) == np.float32(1.0)
    x[1, 7] = 1.0
    assert oracle.global_scale(_bf16(x)) == np.float32(1.0) / np.float32(2688.0)
    # all zero: amax clamps to 1e-8
    z = np.zeros((2, 16), np.float32)
    assert oracle.global_scale(_bf16(z)) == np.float32(1e-8) / np.float32(2688.0)


# ---------------------------------------------------------------- quantize

def _grid_tensor(rng, rows, cols):
    """x on the NVFP4 grid with gs = 1: block b has scale 2^e_b, entries code * 2^e_b."""
    x = np.zeros((rows, cols), np.float32)
    exps = rng.integers(-6, 9, size=(rows, cols // 16))  # 2^-6 .. 2^8: normal E4M3 scales
    vals = rng.choice(np.array(E2M1_VALUES + [-v for v in E2M1_VALUES[1:]], np.float32),
                      size=(rows, cols))
    for r in range(rows):
        for b in range(cols // 16):
            blk = vals[r, b * 16:(b + 1) * 16].copy()
            blk[rng.integers(0, 16)] = 6.0 * rng.choice([-1, 1])  # block max exactly 6 * 2^e
            x[r, b * 16:(b + 1) * 16] = blk * np.float32(2.0 ** exps[r, b])
    # one block at the top scale 448 holds the tensor max 2688 = 6 * 448 -> gs = 1
    x[0, :16] = np.float32(448.0) * vals[0, :16]
    x[0, 3] = 2688.0
    return x


def test_quantize_exact_on_grid_and_nibble_order():
    rng = np.random.default_rng(1)
    x = _grid_tensor(rng, 5, 64)
    xb = _bf16(x)
    assert np.array_equal(bf16_to_f32(xb), x)  # the grid is exact in bf16
    q, sf, gs = oracle.quantize(xb)
    assert gs == np.float32(1.0)
    # scale bytes: 448 for block 0 of row 0, 2^e elsewhere (from torch's E4M3 encoder)
    assert sf[0, 0] == 0x7E
    # codes: the even element sits in the low nibble; values from the page's table
    sign = lambda v: 8 if v < 0 else 0
    val_to_code = {v: c for c, v in E2M1_TABLE.items()}
    for r in range(5):
        for b in range(4):
            s = float(torch.tensor([float(sf[r, b])]).to(torch.uint8).view(torch.float8_e4m3fn).float())
            for j in range(16):
                v = x[r, b * 16 + j] / s
                code = sign(v) | val_to_code[abs(float(v))]
                byte = q[r, (b * 16 + j) // 2]
                got = (byte & 0xF) if j % 2 == 0 else (byte >> 4)
                assert got == code, (r, b, j)
    deq = oracle.dequantize(q, sf, gs)
    np.testing.assert_array_equal(deq, x.astype(np.float64))


def _half_gap(v):
    a = abs(v)
    if a <= 2.0:
        return 0.25
    if a <= 4.0:
        return 0.5
    return 1.0


def test_quantize_roundtrip_error_bound():
    rng = np.random.default_rng(2)
    x32 = rng.standard_normal((16, 256)).astype(np.float32)
    x32.reshape(-1)[rng.integers(0, x32.size, 40)] *= 100.0
    xb = _bf16(x32)
    x = bf16_to_f32(xb).astype(np.float64)
    q, sf, gs = oracle.quantize(xb)
    assert gs == np.float32(np.abs(x).max()) / np.float32(2688.0)
    deq = oracle.dequantize(q, sf, gs)
    e4 = torch.from_numpy(sf.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert sf.max() <= 0x7E  # no block scale above 448
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 16):
            den = e4[r, b] * float(gs)
            blk = x[r, b * 16:(b + 1) * 16]
            for j in range(16):
                v = blk[j] / den
                bound = den * (_half_gap(v) + max(0.0, abs(v) - 6.0)) * (1 + 1e-6) + 1e-30
                assert abs(blk[j] - deq[r, b * 16 + j]) <= bound
            if e4[r, b] >= 2.0 ** -6:  # normal scale: the block max lands on magnitude 6
                jmax = int(np.argmax(np.abs(blk)))
                byte = q[r, (b * 16 + jmax) // 2]
                code = (byte & 0xF) if jmax % 2 == 0 else (byte >> 4)
                assert code & 7 == 7
    # the block holding the tensor max gets scale 448 (x/gsa <= 2688 exactly reached)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sf[r, c // 16] == 0x7E


def test_quantize_zero_and_tiny_blocks():
    z = np.zeros((2, 32), np.float32)
    q, sf, gs = oracle.quantize(_bf16(z))
    assert not q.any() and not sf.any()
    # a block far below the tensor max gets scale byte 0: all codes are signed zeros
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 1000.0
    x[0, 16:] = -1e-4
    q, sf, gs = oracle.quantize(_bf16(x))
    assert sf[0, 1] == 0
    assert (q[0, 8:] == 0x88).all()


# ---------------------------------------------------------------- deinterleave

@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_deinterleave_layout(g):
    inter = 32
    gate = np.arange(inter, dtype=np.uint16) + 100
    up = np.arange(inter, dtype=np.uint16) + 1000
    # interleave: groups of g gate columns alternate with groups of g up columns
    row = np.stack([gate.reshape(-1, g), up.reshape(-1, g)], axis=1).reshape(-1)
    x = np.stack([row, row + 1]).astype(np.uint16)
    out = oracle.deinterleave(x, g)
    np.testing.assert_array_equal(out[0], np.concatenate([gate, up]))
    np.testing.assert_array_equal(out[1], np.concatenate([gate, up]) + 1)


def test_deinterleave_quantize_is_quantize_of_deinterleaved():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((3, 128)).astype(np.float32))
    q1, sf1, gs1 = oracle.deinterleave_quantize(x, 8)
    q2, sf2, gs2 = oracle.quantize(oracle.deinterleave(x, 8))
    assert gs1 == gs2 and np.array_equal(q1, q2) and np.array_equal(sf1, sf2)


# ---------------------------------------------------------------- GEMM

def test_gemm_textbook_case():
    # Unit scales (E4M3 1.0 = 0x38) and unit global scales: logits are plain dot
    # products of table values, unpacked here by hand (low nibble = even element).
    rng = np.random.default_rng(4)
    M, N, K = 3, 5, 64
    qa = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    qb = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    sfa = np.full((M, K // 16), 0x38, np.uint8)
    sfb = np.full((N, K // 16), 0x38, np.uint8)

    def val(nib):
        return (-1 if nib & 8 else 1) * E2M1_TABLE[nib & 7]

    def row_vals(q):
        out = []
        for byte in q:
            out += [val(byte & 0xF), val(byte >> 4)]
        return out

    got = oracle.gemm_logits(qa, sfa, 1.0, qb, sfb, 1.0)
    for m in range(M):
        a = row_vals(qa[m])
        for n in range(N):
            b = row_vals(qb[n])
            assert got[m, n] == np.float32(sum(x * y for x, y in zip(a, b)))


def test_gemm_matches_dequant_matmul():
    rng = np.random.default_rng(5)
    xa = _bf16(rng.standard_normal((7, 512)).astype(np.float32))
    xb = _bf16((rng.standard_normal((9, 512)) * 0.02).astype(np.float32))
    qa, sfa, gsa = oracle.quantize(xa)
    qb, sfb, gsb = oracle.quantize(xb)
    A = oracle.dequantize(qa, sfa, 1.0) * np.float64(gsa)
    B = oracle.dequantize(qb, sfb, 1.0) * np.float64(gsb)
    ref = A @ B.T
    got = oracle.gemm_logits(qa, sfa, gsa, qb, sfb, gsb).astype(np.float64)
    scale = np.abs(A) @ np.abs(B).T
    assert np.all(np.abs(got - ref) <= 2 ** -23 * np.abs(ref) + 1e-12 * scale)
    # operand order matters: the transposed product is a different matrix
    assert got.shape == (7, 9)
    # row range selects the same rows
    np.testing.assert_array_equal(oracle.gemm_logits(qa, sfa, gsa, qb, sfb, gsb, 2, 5), got[2:5])
    # dequant formula: lut[q] * sf * gs on one element by hand
    byte = qb[4, 10]
    code = byte >> 4  # element 21 (odd) -> high nibble
    e4 = float(torch.tensor([int(sfb[4, 21 // 16])], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
    by_hand = (-1 if code & 8 else 1) * E2M1_TABLE[code & 7] * e4 * float(gsb)
    assert oracle.dequantize(qb, sfb, gsb)[4, 21] == by_hand


# ---------------------------------------------------------------- epilogue + top-k

def test_epilogue_closed_forms():
    logits = np.array([[0.0, 30.0, -30.0, 2.0, -3.5]], np.float32)
    bias = np.array([0.1, -0.2, 0.0, 0.5, 0.25], np.float32)
    s, w = oracle.epilogue(logits, 1, bias)
    assert w[0, 0] == np.float32(math.sqrt(math.log(2.0)))
    ref_w = np.sqrt(np.logaddexp(0.0, logits[0].astype(np.float64)))
    np.testing.assert_allclose(w[0], ref_w, rtol=1e-6)
    np.testing.assert_allclose(s[0], ref_w + bias, rtol=1e-6, atol=1e-7)
    assert abs(w[0, 2] - math.exp(-15.0)) < 1e-9
    s0, w0 = oracle.epilogue(logits, 0, None)
    np.testing.assert_array_equal(s0, logits)
    np.testing.assert_array_equal(w0, logits)


def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda i: (-float(row[i]), i))[:k]
    return order


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(6)
    for trial in range(50):
        rows, N = 4, int(rng.integers(1, 65))
        k = int(rng.integers(1, 12))
        s = rng.integers(-5, 6, (rows, N)).astype(np.float32)  # many exact ties
        idx, val, _ = oracle.topk(s, k)
        for r in range(rows):
            ref = _brute_topk(s[r], k)
            take = min(k, N)
            assert list(idx[r, :take]) == ref
            np.testing.assert_array_equal(val[r, :take], s[r, ref])
            assert (idx[r, take:] == -1).all() and np.isneginf(val[r, take:]).all()


def test_gemm_topk_composes_steps():
    d = __import__("workloads").router_tiny(0)
    qa, sfa, gsa = oracle.quantize(d["x"])
    qb, sfb, gsb = oracle.quantize(d["w"])
    logits = oracle.gemm_logits(qa, sfa, gsa, qb, sfb, gsb)
    score, weight = oracle.epilogue(logits, 1, d["bias"])
    idx, val, wt = oracle.gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 1, d["bias"], d["k"])
    for r in range(logits.shape[0]):
        ref = _brute_topk(score[r], d["k"])
        assert list(idx[r]) == ref
        np.testing.assert_array_equal(val[r], score[r, ref])
        np.testing.assert_array_equal(wt[r], weight[r, ref])
    idx2, _, _ = oracle.gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 1, d["bias"], d["k"], threads=3)
    np.testing.assert_array_equal(idx, idx2)


def test_router_weight_normalisation():
    # Epilogue 2: the selected weights of a row divided by their sum.  Worked
    # by hand: weights 1, 3, 4 (plus an empty slot) -> 1/8, 3/8, 4/8, 0.
    idx = np.array([[5, 2, 9, -1]], np.int32)
    w = np.array([[1.0, 3.0, 4.0, 0.0]], np.float32)
    out = oracle.normalize_topk_weights(idx, w)
    assert out.tolist() == [[0.125, 0.375, 0.5, 0.0]]
    # a row of one: weight 1; an all-empty row stays as it is
    idx = np.array([[7, -1], [-1, -1]], np.int32)
    w = np.array([[0.3, 0.0], [0.0, 0.0]], np.float32)
    assert oracle.normalize_topk_weights(idx, w).tolist() == [[1.0, 0.0], [0.0, 0.0]]


def test_gemm_topk_epilogue2_is_epilogue1_then_normalised():
    rng = np.random.default_rng(77)
    xa = workloads.bf16_bits(rng.standard_normal((3, 128)).astype(np.float32))
    xb = workloads.bf16_bits((rng.standard_normal((40, 128)) * 0.05).astype(np.float32))
    bias = (rng.standard_normal(40) * 0.01).astype(np.float32)
    qa, sfa, gsa = oracle.quantize(xa)
    qb, sfb, gsb = oracle.quantize(xb)
    i1, s1, w1 = oracle.gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 1, bias, 6)
    i2, s2, w2 = oracle.gemm_topk(qa, sfa, gsa, qb, sfb, gsb, 2, bias, 6)
    assert np.array_equal(i1, i2) and np.array_equal(s1, s2)
    np.testing.assert_allclose(w2, w1 / w1.sum(axis=1, keepdims=True), rtol=1e-6)
    np.testing.assert_allclose(w2.sum(axis=1), 1.0, rtol=1e-6)


# ---- RMSNorm producer of the quantize input (fused RMSNorm + quantize)

def _bf16(vals):
    return bf16_bits(np.asarray(vals, np.float32))


def _nearest_f32(frac):
    """The float32 nearest a non-negative Fraction (ties to the even
    significand), found by comparing the exact value with its float32
    neighbours; inf beyond float32's range."""
    from fractions import Fraction
    big = Fraction(np.finfo(np.float32).max.item()) + Fraction(2) ** 103  # max + half its step
    if frac >= big:
        return np.float32(np.inf)
    c = np.float32(float(frac))  # within one step of the answer
    best = None
    for cand in (np.nextafter(c, np.float32(0)), c, np.nextafter(c, np.float32(np.inf))):
        if not np.isfinite(cand) or cand < 0:
            continue
        d = abs(Fraction(cand.item()) - frac)
        key = (d, int(np.float32(cand).view(np.uint32)) & 1)  # tie: even significand bit
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def _exact_sum_sq(row_bits):
    from fractions import Fraction
    return sum((Fraction(v.item()) ** 2 for v in bf16_to_f32(row_bits).astype(np.float64)), Fraction(0))


def test_rms_sum_of_squares_is_nearest_float_of_exact_sum():
    # rows over a wide range of magnitudes, with bf16 subnormals, zeros and
    # negative values; the reference is Python's exact rational arithmetic
    rng = np.random.default_rng(33)
    rows = [rng.standard_normal(300) * 2.0 ** rng.integers(-30, 30) for _ in range(6)]
    rows.append(np.concatenate([rng.standard_normal(150) * 1e3, rng.standard_normal(150) * 1e-30]))
    rows.append(np.concatenate([rng.standard_normal(10) * 2.0 ** -128, np.zeros(290)]))  # bf16 subnormals
    rows.append(rng.standard_normal(300) * 2.0 ** -70)  # squares below FP32's normal range
    x = bf16_bits(np.array(rows, np.float32))
    got = oracle.rms_sum_of_squares(x)
    for r in range(x.shape[0]):
        want = _nearest_f32(_exact_sum_sq(x[r]))
        assert got[r].view(np.uint32) == want.view(np.uint32), (r, got[r], want)


def test_rms_sum_of_squares_ties_and_limits():
    # 2^24 + 1 is halfway between 2^24 and 2^24 + 2: ties to even (2^24);
    # any positive term below it breaks the tie upwards; 2^24 + 9 -> 2^24 + 8
    cases = [([4096.0, 1.0], 2.0 ** 24), ([4096.0, 1.0, 2.0 ** -20], 2.0 ** 24 + 2),
             ([4096.0, 3.0], 2.0 ** 24 + 8), ([2.0 ** 100], np.inf), ([2.0 ** -80], 0.0),
             ([2.0 ** -70, 2.0 ** -70], 2.0 ** -139), ([], 0.0)]
    for vals, want in cases:
        x = _bf16([list(vals) + [0.0] * (16 - len(vals))])
        assert oracle.rms_sum_of_squares(x)[0] == np.float32(want), (vals, want)


def test_rms_sum_of_squares_is_order_free():
    # the reading has no summation order: any permutation of a row gives the same FP32 sum
    rng = np.random.default_rng(34)
    x = bf16_bits((rng.standard_normal((4, 7168)) * 2.0 ** rng.integers(-20, 20, (4, 7168))).astype(np.float32))
    s0 = oracle.rms_sum_of_squares(x)
    for seed in range(3):
        perm = np.random.default_rng(seed).permutation(7168)
        assert np.array_equal(oracle.rms_sum_of_squares(x[:, perm]), s0)


def test_rmsnorm_worked_row():
    # x = [3, 4, 0 x 14], weight 1, eps 0: sum 25, mean 25/16, rms 1.25,
    # y = [2.4, 3.2, 0 ...] -> bf16 2.40625, 3.203125 (round to nearest even)
    x = _bf16([[3.0, 4.0] + [0.0] * 14])
    w = _bf16(np.ones(16))
    y = bf16_to_f32(oracle.rmsnorm(x, w, 0.0))
    assert y[0, 0] == 2.40625 and y[0, 1] == 3.203125 and (y[0, 2:] == 0).all()


def test_rmsnorm_constant_row_and_weight_scaling():
    # a constant row normalises to ~1 (eps 1e-6 makes it 0.99999988 -> bf16 1.0);
    # a weight of 2 (a power of two) doubles every output exactly
    x = _bf16(np.full((2, 64), 2.0))
    y1 = bf16_to_f32(oracle.rmsnorm(x, _bf16(np.ones(64)), 1e-6))
    y2 = bf16_to_f32(oracle.rmsnorm(x, _bf16(np.full(64, 2.0)), 1e-6))
    assert (y1 == 1.0).all() and (y2 == 2.0).all()


def test_rmsnorm_matches_double_precision_textbook():
    # against sqrt(mean(x^2) + eps) in double on wide-range rows: within one
    # bf16 rounding of the exact value (relative 2^-8), every element
    rng = np.random.default_rng(31)
    f = (rng.standard_normal((6, 7168)) * np.exp2(rng.integers(-8, 8, (6, 1)))).astype(np.float32)
    x = bf16_bits(f)
    wf = (1.0 + 0.2 * rng.standard_normal(7168)).astype(np.float32)
    w = bf16_bits(wf)
    xd = bf16_to_f32(x).astype(np.float64)
    wd = bf16_to_f32(w).astype(np.float64)
    ref = xd / np.sqrt((xd ** 2).mean(axis=1, keepdims=True) + 1e-6) * wd
    y = bf16_to_f32(oracle.rmsnorm(x, w, 1e-6)).astype(np.float64)
    assert (np.abs(y - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30).all()


def test_rmsnorm_quantize_is_rmsnorm_then_quantize():
    rng = np.random.default_rng(32)
    x = bf16_bits(rng.standard_normal((5, 256)).astype(np.float32))
    w = bf16_bits((1.0 + 0.1 * rng.standard_normal(256)).astype(np.float32))
    q, sf, gs = oracle.rmsnorm_quantize(x, w, 1e-6)
    rq, rsf, rgs = oracle.quantize(oracle.rmsnorm(x, w, 1e-6))
    assert np.array_equal(q, rq) and np.array_equal(sf, rsf) and gs == rgs


# ---- full indexer score (head reduction), I[t,s] = sum_h w[t,h] ReLU(q[t,h] . K[s])

def _indexer_case(T, H, N, K, seed):
    rng = np.random.default_rng(seed)
    qa, sfa, gsa = oracle.quantize(bf16_bits(rng.standard_normal((T * H, K)).astype(np.float32)))
    qb, sfb, gsb = oracle.quantize(bf16_bits(rng.standard_normal((N, K)).astype(np.float32)))
    return qa, sfa, gsa, qb, sfb, gsb


def test_indexer_single_head_unit_weight_is_relu_of_logits():
    qa, sfa, gsa, qb, sfb, gsb = _indexer_case(3, 1, 40, 64, 41)
    I = oracle.indexer_scores(qa, sfa, gsa, qb, sfb, gsb, 1, np.ones((3, 1), np.float32))
    lg = oracle.gemm_logits(qa, sfa, gsa, qb, sfb, gsb)
    assert np.array_equal(I, np.maximum(lg, 0))


def test_indexer_scores_against_dequantized_einsum():
    # the textbook: dequantize both operands, einsum 'thd,sd->ths' in double,
    # ReLU, weighted head sum (the row order t * H + h is what is pinned)
    T, H, N, K = 2, 4, 24, 128
    qa, sfa, gsa, qb, sfb, gsb = _indexer_case(T, H, N, K, 42)
    rng = np.random.default_rng(43)
    w = rng.standard_normal((T, H)).astype(np.float32)
    A = oracle.dequantize(qa, sfa, gsa).astype(np.float64).reshape(T, H, K)
    B = oracle.dequantize(qb, sfb, gsb).astype(np.float64)
    ref = (np.maximum(np.einsum("thd,sd->ths", A, B), 0) * w[:, :, None].astype(np.float64)).sum(axis=1)
    I = oracle.indexer_scores(qa, sfa, gsa, qb, sfb, gsb, H, w)
    np.testing.assert_allclose(I, ref, rtol=1e-5, atol=1e-6)


def test_indexer_scores_linear_in_head_weights():
    qa, sfa, gsa, qb, sfb, gsb = _indexer_case(1, 8, 16, 64, 44)
    w = np.arange(1, 9, dtype=np.float32).reshape(1, 8)
    I1 = oracle.indexer_scores(qa, sfa, gsa, qb, sfb, gsb, 8, w)
    I2 = oracle.indexer_scores(qa, sfa, gsa, qb, sfb, gsb, 8, 2 * w)
    np.testing.assert_allclose(I2, 2 * I1, rtol=1e-6)


# ---------------------------------------------------------------- grouped GEMM + SwiGLU

def _decode_by_table(q, sf):
    """NVFP4 values without the global scale, decoded with the page's table and
    torch's E4M3 conversion (no oracle code): [rows, 2 * bytes]."""
    lo, hi = q & 0xF, q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
    mag = np.array(E2M1_VALUES)[codes & 7]
    vals = np.where(codes & 8, -mag, mag)
    s = torch.from_numpy(np.ascontiguousarray(sf)).view(torch.float8_e4m3fn).double().numpy()
    return vals * np.repeat(s, 16, axis=1)


def _swiglu_case(rng, M, E, I, K, g, sizes):
    qa = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    qb = rng.integers(0, 256, (E * 2 * I, K // 2)).astype(np.uint8)
    # power-of-two block scales (E4M3 bytes 0x30 = 0.5, 0x38 = 1, 0x40 = 2)
    sfa = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), (M, K // 16))
    sfb = rng.choice(np.array([0x28, 0x30, 0x38], np.uint8), (E * 2 * I, K // 16))
    gsb = (2.0 ** rng.integers(-8, -4, E)).astype(np.float32)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    assert offs[-1] <= M
    return qa, sfa, qb, sfb, gsb, offs


@pytest.mark.parametrize("g", [1, 8])
def test_grouped_swiglu_against_library_math(g):
    # Expected values from the page's E2M1 table, torch's E4M3, numpy matmul,
    # a reshape-based split of the interleaved weight rows and scipy's
    # logistic function; groups of size 5, 0, 3 and 4 over 12 of 14 rows.
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(21)
    M, E, I, K = 14, 4, 16, 128
    qa, sfa, qb, sfb, gsb, offs = _swiglu_case(rng, M, E, I, K, g, [5, 0, 3, 4])
    gsa = np.float32(2.0)
    limit = 1.0
    h, a = oracle.grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, offs, I, g, limit)
    clamped = {"gate": 0, "up_hi": 0, "up_lo": 0}
    A = _decode_by_table(qa, sfa)
    B = _decode_by_table(qb, sfb)
    for e in range(E):
        rows = slice(offs[e], offs[e + 1])
        We = B[e * 2 * I:(e + 1) * 2 * I].reshape(I // g, 2, g, K)
        gate_w, up_w = We[:, 0].reshape(I, K), We[:, 1].reshape(I, K)
        s = float(gsa) * float(gsb[e])
        gate = (A[rows] @ gate_w.T * s).astype(np.float32).astype(np.float64)
        up = (A[rows] @ up_w.T * s).astype(np.float32).astype(np.float64)
        clamped["gate"] += int(np.sum(gate > limit))
        clamped["up_hi"] += int(np.sum(up > limit))
        clamped["up_lo"] += int(np.sum(up < -limit))
        gate = np.minimum(gate, limit)
        up = np.clip(up, -limit, limit)
        silu = gate * special.expit(gate)
        np.testing.assert_allclose(a[rows], silu, rtol=1e-13, atol=1e-300)
        np.testing.assert_allclose(h[rows], silu * up, rtol=1e-13, atol=1e-300)
    # rows past the last group are not written
    assert np.all(h[offs[-1]:] == 0) and np.all(a[offs[-1]:] == 0)
    # every side of the clamp is exercised, and a clamped gate gives silu(limit)
    assert min(clamped.values()) > 0, clamped
    assert np.max(a) == limit / (1.0 + math.exp(-limit))


def test_grouped_swiglu_closed_forms():
    # Zero up weights give h = 0; zero gate weights give a = silu(0) = 0; an
    # unbounded limit is no clamp; a group equals the same rows run as a
    # one-expert problem with that expert's weights.
    rng = np.random.default_rng(22)
    M, E, I, K, g = 9, 3, 8, 64, 8
    qa, sfa, qb, sfb, gsb, offs = _swiglu_case(rng, M, E, I, K, g, [2, 4, 3])
    gsa = np.float32(1.0)
    qb_up0 = qb.copy()
    for e in range(E):
        for p in range(I // g):
            r0 = e * 2 * I + 2 * g * p + g
            qb_up0[r0:r0 + g] = 0
    h, a = oracle.grouped_swiglu(qa, sfa, gsa, qb_up0, sfb, gsb, offs, I, g)
    assert np.all(h == 0) and np.any(a != 0)
    qb_gate0 = qb.copy()
    for e in range(E):
        for p in range(I // g):
            r0 = e * 2 * I + 2 * g * p
            qb_gate0[r0:r0 + g] = 0
    h, a = oracle.grouped_swiglu(qa, sfa, gsa, qb_gate0, sfb, gsb, offs, I, g)
    assert np.all(a == 0) and np.all(h == 0)
    h_all, a_all = oracle.grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, offs, I, g)
    h_big, _ = oracle.grouped_swiglu(qa, sfa, gsa, qb, sfb, gsb, offs, I, g, limit=1e30)
    np.testing.assert_array_equal(h_all, h_big)
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        w = slice(e * 2 * I, (e + 1) * 2 * I)
        h1, a1 = oracle.grouped_swiglu(qa[lo:hi], sfa[lo:hi], gsa, qb[w], sfb[w], gsb[e:e + 1],
                                       np.array([0, hi - lo], np.int32), I, g)
        np.testing.assert_array_equal(h1, h_all[lo:hi])
        np.testing.assert_array_equal(a1, a_all[lo:hi])
    # swapping two experts' weights and row ranges permutes the output rows
    perm_offs = np.array([0, 4, 6, 9], np.int32)  # expert 1's rows first, then 0, then 2
    rows = np.r_[2:6, 0:2, 6:9]
    wperm = np.r_[2 * I:4 * I, 0:2 * I, 4 * I:6 * I]
    h2, _ = oracle.grouped_swiglu(qa[rows], sfa[rows], gsa, qb[wperm], sfb[wperm], gsb[[1, 0, 2]], perm_offs, I, g)
    np.testing.assert_array_equal(h2, h_all[rows])


def test_grouped_swiglu_interleaved_layout():
    # Layout 1 deinterleaves (with the separately pinned deinterleave) into
    # [bf16(silu(gate)) | bf16(h)]; layout 0 is bf16(h).
    rng = np.random.default_rng(23)
    M, E, I, K, g = 6, 2, 32, 64, 8
    qa, sfa, qb, sfb, gsb, offs = _swiglu_case(rng, M, E, I, K, g, [4, 2])
    h, a = oracle.grouped_swiglu(qa, sfa, 1.0, qb, sfb, gsb, offs, I, g, 10.0)
    out0 = oracle.grouped_swiglu_bf16(qa, sfa, 1.0, qb, sfb, gsb, offs, I, g, 10.0, layout=0)
    out1 = oracle.grouped_swiglu_bf16(qa, sfa, 1.0, qb, sfb, gsb, offs, I, g, 10.0, layout=1)
    assert out0.shape == (M, I) and out1.shape == (M, 2 * I)
    de = oracle.deinterleave(out1, g)
    np.testing.assert_array_equal(de[:, I:], out0)
    # bf16 rounding of the stored values: within half a bf16 ulp of the doubles
    got = bf16_to_f32(out0).astype(np.float64)
    assert np.all(np.abs(got - h) <= 2.0 ** -8 * np.abs(h) + 1e-300)
    got_a = bf16_to_f32(de[:, :I]).astype(np.float64)
    assert np.all(np.abs(got_a - a) <= 2.0 ** -8 * np.abs(a) + 1e-300)


# ---- mHC pre-mix of the residual streams, fused with RMSNorm + quantize

def test_mhc_single_stream_with_unit_mapping_is_rmsnorm_quantize():
    # n_hc = 1 and A = 1: the mix is the stream itself, so the fused op is
    # exactly the pinned RMSNorm + quantize
    rng = np.random.default_rng(51)
    x = bf16_bits(rng.standard_normal((5, 1, 512)).astype(np.float32))
    a = _bf16(np.ones((5, 1)))
    w = bf16_bits((1.0 + 0.1 * rng.standard_normal(512)).astype(np.float32))
    got = oracle.mhc_rmsnorm_quantize(x, a, w, 1e-6)
    want = oracle.rmsnorm_quantize(x[:, 0, :], w, 1e-6)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]) and got[2] == want[2]


def test_mhc_mix_on_an_exact_grid():
    # streams and mapping on a grid where every partial sum is exact: the mix
    # is the exact sum_i A[t, i] X[t, i, c] (numpy float64), for any stream order
    rng = np.random.default_rng(52)
    T, n, d = 6, 4, 64
    xf = rng.integers(-3, 4, (T, n, d)).astype(np.float64)
    af = np.array([0.25, 0.5, 1.0, 2.0])[rng.integers(0, 4, (T, n))]
    mix = bf16_to_f32(oracle.mhc_mix(_bf16(xf), _bf16(af))).astype(np.float64)
    assert np.array_equal(mix, np.einsum("ti,tic->tc", af, xf))
    perm = rng.permutation(n)
    assert np.array_equal(oracle.mhc_mix(_bf16(xf[:, perm]), _bf16(af[:, perm])), oracle.mhc_mix(_bf16(xf), _bf16(af)))


def test_mhc_mix_rounds_in_stream_order():
    # the reading: FP32 accumulation over the streams in index order, then bf16.
    # 2^24 + 1 rounds to 2^24 (ties to even), so the sum of (2^24, 1, -2^24)
    # is 0 in that order, although the exact sum is 1
    x = _bf16(np.array([[[2.0 ** 24] * 16, [1.0] * 16, [-(2.0 ** 24)] * 16]]))
    a = _bf16(np.ones((1, 3)))
    assert (bf16_to_f32(oracle.mhc_mix(x, a)) == 0.0).all()
    a2 = _bf16(np.array([[1.0, 1.0, 0.0]]))  # (2^24 + 1) alone rounds to 2^24 in FP32, stays 2^24 in bf16
    assert (bf16_to_f32(oracle.mhc_mix(x, a2)) == 2.0 ** 24).all()


def test_mhc_mapping_scaled_by_a_power_of_two_gives_the_same_codes():
    # scaling A by 2^k scales the mix exactly; with eps = 0 RMSNorm divides the
    # scale out exactly (the FP32 sum, mean, root and reciprocal all scale
    # exactly), so codes, scales and the global scale are identical
    rng = np.random.default_rng(53)
    x = bf16_bits(rng.standard_normal((7, 4, 256)).astype(np.float32))
    af = rng.uniform(0.2, 1.0, (7, 4))
    w = bf16_bits((1.0 + 0.1 * rng.standard_normal(256)).astype(np.float32))
    base = oracle.mhc_rmsnorm_quantize(x, _bf16(af), w, 0.0)
    for k in (-3, 5):
        got = oracle.mhc_rmsnorm_quantize(x, _bf16(af * 2.0 ** k), w, 0.0)
        assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1]) and got[2] == base[2]
