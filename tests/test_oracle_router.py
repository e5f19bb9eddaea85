"""Pins for the oracle's router step (top-k of per-(token, expert) logits,
softmax renormalized over the selected k: "Prime Flash MoE - Faster MoE
Kernels optimized for Blackwell", sec. 1, the router that selects the top-k
experts with normalized weights).  Each test checks it against something other
than itself: brute force over expert subsets, a library softmax, closed forms
and the tie rule.  CPU only."""
import itertools

import numpy as np
import pytest
import scipy.special

import oracle
from grouped_gemm_gb300 import workloads as wl


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 4), (7, 7)])
def test_selection_is_the_max_sum_subset(E, k):
    # brute force: with distinct logits the selected set is the unique k-subset
    # of largest logit sum, listed in order of decreasing logit
    rng = np.random.default_rng(E * 10 + k)
    lg = rng.standard_normal((40, E)).astype(np.float32)
    ids, w = oracle.router_topk(lg, k)
    for t in range(lg.shape[0]):
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(float(lg[t, e]) for e in c))
        assert sorted(ids[t]) == sorted(best)
        vals = lg[t, ids[t]]
        assert np.all(np.diff(vals) < 0)


@pytest.mark.parametrize("E", [3, 16, 128])
def test_k_equals_E_is_the_full_softmax(E):
    rng = np.random.default_rng(E)
    lg = (rng.standard_normal((25, E)) * 3).astype(np.float32)
    ids, w = oracle.router_topk(lg, E)
    ref = scipy.special.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(ref, ids.astype(np.int64), axis=1), rtol=1e-13, atol=0)
    assert np.array_equal(np.sort(ids, axis=1), np.tile(np.arange(E), (25, 1)))


def test_weights_closed_forms():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((50, 32)).astype(np.float32)
    ids, w = oracle.router_topk(lg, 6)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    # ratio of two weights is exp of the logit difference
    sel = np.take_along_axis(lg.astype(np.float64), ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(w[:, 1:] / w[:, :1], np.exp(sel[:, 1:] - sel[:, :1]), rtol=1e-13)
    # top-1 always has weight 1
    ids1, w1 = oracle.router_topk(lg, 1)
    assert np.all(w1 == 1.0) and np.array_equal(ids1[:, 0], np.argmax(lg, axis=1))


def test_renormalized_softmax_equals_full_softmax_restricted():
    # "top-k + renormalized softmax": softmax over all E, keep the selected k,
    # divide by their sum -- the same numbers as the softmax of the k logits
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((30, 64)).astype(np.float32)
    ids, w = oracle.router_topk(lg, 8)
    full = scipy.special.softmax(lg.astype(np.float64), axis=1)
    kept = np.take_along_axis(full, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, kept / kept.sum(axis=1, keepdims=True), rtol=1e-12)


def test_ties_go_to_the_lower_expert_id():
    lg = np.zeros((3, 10), np.float32)
    lg[1, [2, 5, 7]] = 1.0
    lg[2, :] = np.array([0, 1, 1, 0, 1, 0, 0, 1, 0, 0], np.float32)
    ids, w = oracle.router_topk(lg, 4)
    assert ids[0].tolist() == [0, 1, 2, 3] and np.allclose(w[0], 0.25)
    assert ids[1].tolist() == [2, 5, 7, 0]
    assert ids[2].tolist() == [1, 2, 4, 7] and np.allclose(w[2], 0.25)


def test_nan_is_minus_infinity_and_all_minus_infinity_is_flat():
    lg = np.array([[np.nan, 0.5, -np.inf, 2.0, np.nan],
                   [-np.inf] * 5,
                   [np.nan] * 5], np.float32)
    ids, w = oracle.router_topk(lg, 3)
    assert ids[0].tolist() == [3, 1, 0]          # NaN (read as -inf) ties with -inf; lower id first
    assert w[0, 2] == 0.0 and abs(w[0, 0] + w[0, 1] - 1.0) < 1e-15
    assert ids[1].tolist() == [0, 1, 2] and np.all(w[1] == 1.0 / 3)
    assert ids[2].tolist() == [0, 1, 2] and np.all(w[2] == 1.0 / 3)


def test_matches_the_workload_generator_on_its_own_draws():
    # the seeded topk_logits generator selects by a stable argsort and
    # normalizes with its own softmax: an independent implementation of the
    # same rule, run here on float32 logits
    lg = wl.router_logits(300, 40, seed=9)
    order = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")[:, :5]
    ids, w = oracle.router_topk(lg, 5)
    assert np.array_equal(ids, order)


def test_rejects_k_outside_range():
    lg = np.zeros((2, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.router_topk(lg, 5)
    with pytest.raises(ValueError):
        oracle.router_topk(lg, 0)
