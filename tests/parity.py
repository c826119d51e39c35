"""Comparison rules between the CUDA path and the oracle.

* Quantize outputs (codes, scale bytes, global scale) must be bit-exact.
* GEMM logits and scores: |gpu - oracle| <= ATOL + RTOL * |oracle| (FP32),
  with RTOL = 1e-3 and ATOL = 1e-4.
* Top-k: the index sets must be identical, except that indices whose oracle
  score lies within the tolerance of the oracle's k-th score (a near-tie at
  the selection boundary) may differ; every reported score must match the
  oracle's score of the reported index; scores are non-increasing along the
  row, and equal reported scores appear in increasing index order; slots
  beyond N hold index -1 and score -inf.
"""
import numpy as np

import oracle

RTOL = 1e-3
ATOL = 1e-4


def tol(ref):
    return ATOL + RTOL * np.abs(ref)


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    bad = np.abs(got - ref) > tol(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu {got[tuple(i)]!r} oracle {ref[tuple(i)]!r}")


def assert_topk(gpu_idx, gpu_score, gpu_weight, ref_score_rows, ref_weight_rows, k, what="",
                normalized=False):
    """Check GPU top-k of each row against the oracle's full score rows.

    normalized: the weights are the router's normalised gating weights, so
    the reference is oracle.normalize_topk_weights applied to the oracle's
    weights of the GPU's picks.
    """
    gpu_idx = np.asarray(gpu_idx)
    gpu_score = np.asarray(gpu_score)
    rows, N = ref_score_rows.shape
    take = min(k, N)
    for r in range(rows):
        S = ref_score_rows[r].astype(np.float64)
        gi = gpu_idx[r]
        gs = gpu_score[r]
        # padding slots
        assert (gi[take:] == -1).all(), f"{what} row {r}: padding indices"
        assert np.isneginf(gs[take:]).all(), f"{what} row {r}: padding scores"
        gi = gi[:take]
        gs = gs[:take].astype(np.float64)
        assert ((gi >= 0) & (gi < N)).all(), f"{what} row {r}: index out of range"
        assert len(set(gi.tolist())) == take, f"{what} row {r}: duplicate indices"
        # reported scores are the oracle's scores of the reported indices
        bad = np.abs(gs - S[gi]) > tol(S[gi])
        assert not bad.any(), (f"{what} row {r}: score mismatch at slot {int(np.argmax(bad))}: "
                               f"gpu {gs[bad][0]} oracle {S[gi][bad][0]}")
        if gpu_weight is not None and ref_weight_rows is not None:
            W = ref_weight_rows[r].astype(np.float64)
            gw = np.asarray(gpu_weight)[r][:take].astype(np.float64)
            # normalised: the oracle's own normalisation of its weights of the GPU's picks
            ref_w = (oracle.normalize_topk_weights(gi[None, :], W[gi][None, :].astype(np.float32))[0]
                     .astype(np.float64) if normalized else W[gi])
            assert (np.abs(gw - ref_w) <= tol(ref_w)).all(), f"{what} row {r}: weight mismatch"
        # order: non-increasing, ties by increasing index
        assert (np.diff(gs) <= 0).all(), f"{what} row {r}: scores not descending"
        same = np.diff(gs) == 0
        assert (np.diff(gi)[same] > 0).all(), f"{what} row {r}: tie order"
        # set equality up to near-ties at the boundary
        order = sorted(range(N), key=lambda i: (-S[i], i))
        ref_set = set(order[:take])
        kth = S[order[take - 1]]
        diff = ref_set.symmetric_difference(gi.tolist())
        for i in diff:
            assert abs(S[i] - kth) <= 2 * tol(kth), (
                f"{what} row {r}: index {i} (score {S[i]}) differs from the oracle's top-{k} "
                f"and is not a near-tie of the k-th score {kth}")
