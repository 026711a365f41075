"""Pins for the oracle's top-k routing and routing weights.

The router "picks the top-k experts" (clip "Mixture-of-Kittens: Cursor
open-sources an MoE training megakernel", key flowchart, Router node); the
weights are the softmax renormalised over the selected experts. Pins used:
brute force over all k-subsets, a rank-counting characterisation of the
selection, crafted ties, the fp32 add of the bias, and the k = E special case
that reduces to a library softmax.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _rank_count_topk(z, k):
    """Expert e is selected at rank r iff exactly r experts beat it, where
    e' beats e when z[e'] > z[e], or z[e'] == z[e] and e' < e."""
    N, E = z.shape
    ids = np.full((N, k), -1)
    for t in range(N):
        for e in range(E):
            beats = np.sum((z[t] > z[t, e]) | ((z[t] == z[t, e]) & (np.arange(E) < e)))
            if beats < k:
                ids[t, beats] = e
    return ids


@pytest.mark.parametrize("N,E,k", [(256, 8, 2), (40, 64, 8), (17, 5, 5), (9, 33, 1)])
def test_topk_matches_rank_counting(N, E, k):
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((N, E)).astype(np.float32)
    ids, w = oracle.route_topk(logits, None, k)
    np.testing.assert_array_equal(ids, _rank_count_topk(logits, k))


def test_topk_set_maximises_sum_over_all_subsets():
    """Tiny workload shape (E=8, top-2): the chosen pair has the largest
    logit sum among all C(8,2) pairs (continuous draws, no ties)."""
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((256, 8)).astype(np.float32)
    ids, _ = oracle.route_topk(logits, None, 2)
    pairs = list(itertools.combinations(range(8), 2))
    for t in range(256):
        best = max(pairs, key=lambda p: float(logits[t, p[0]]) + float(logits[t, p[1]]))
        assert set(best) == set(ids[t].tolist())


def test_ties_prefer_lower_expert_index():
    logits = np.zeros((3, 6), np.float32)
    logits[1] = [1, 3, 3, 0, 3, 1]
    logits[2, 5] = -0.0
    logits[2, 0] = 0.0
    ids, w = oracle.route_topk(logits, None, 3)
    assert ids[0].tolist() == [0, 1, 2]
    assert ids[1].tolist() == [1, 2, 4]
    assert ids[2].tolist() == [0, 1, 2]  # +0 and -0 tie
    np.testing.assert_allclose(w[0], [1 / 3] * 3, rtol=0, atol=1e-15)


def test_bias_is_added_in_fp32():
    """z = fl32(logit + bias): 1 + 2^-30 rounds to 1 in fp32, so expert 1
    ties with expert 0 and loses on index; in fp64 it would win."""
    logits = np.array([[1.0, 1.0, -5.0]], np.float32)
    bias = np.array([0.0, 2.0 ** -30, 0.0], np.float32)
    ids, w = oracle.route_topk(logits, bias, 1)
    assert ids[0, 0] == 0
    bias[1] = 2.0 ** -20  # representable increment: expert 1 now strictly larger
    ids, _ = oracle.route_topk(logits, bias, 1)
    assert ids[0, 0] == 1


def test_bias_shifts_selection_and_weights():
    logits = np.array([[0.0, 0.5, 0.2, 0.1]], np.float32)
    bias = np.array([2.0, 0.0, 0.0, 0.0], np.float32)
    ids, w = oracle.route_topk(logits, bias, 2)
    assert ids[0].tolist() == [0, 1]
    z0, z1 = 2.0, 0.5
    np.testing.assert_allclose(w[0], [1 / (1 + np.exp(z1 - z0)), 1 / (1 + np.exp(z0 - z1))],
                               rtol=1e-15)


@pytest.mark.parametrize("E", [4, 8, 33])
def test_k_equals_E_is_plain_softmax(E):
    rng = np.random.default_rng(E)
    logits = (3 * rng.standard_normal((50, E))).astype(np.float32)
    ids, w = oracle.route_topk(logits, None, E)
    p = softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, axis=1), rtol=1e-13, atol=0)


def test_renormalised_topk_equals_full_softmax_restricted():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((64, 16)).astype(np.float32)
    bias = rng.standard_normal(16).astype(np.float32)
    ids, w = oracle.route_topk(logits, bias, 4)
    z = (logits + bias).astype(np.float64)  # numpy fp32 add, then widen
    p = softmax(z, axis=1)
    sel = np.take_along_axis(p, ids, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # ranks are in descending weight


def test_nan_logit_is_an_error():
    logits = np.zeros((2, 4), np.float32)
    logits[1, 2] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.route_topk(logits, None, 2)
