"""Pins for the oracle's router with the extra select_experts arguments
(sigmoid scoring, expert groups, score-correction bias, routed scaling
factor), CPU only.  The pages name these arguments without their arithmetic;
the reading under test is the one stated in ``oracle.topk_route_ex``."""

import itertools
import math

import numpy as np
import pytest
import scipy.special

import oracle


def _logits(T, E, seed):
    return np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32)


def _expit(x):
    return 1.0 / (1.0 + math.exp(-x))


@pytest.mark.parametrize("renorm", [False, True])
def test_defaults_reduce_to_plain_router(renorm):
    lg = _logits(50, 64, seed=5)
    w0, i0 = oracle.topk_route(lg, 6, renorm)
    w1, i1 = oracle.topk_route_ex(lg, 6, renorm)
    assert np.array_equal(i0, i1)
    np.testing.assert_allclose(w1, w0, rtol=1e-15)


@pytest.mark.parametrize("E,k", [(5, 2), (7, 3)])
def test_sigmoid_brute_force_and_library_expit(E, k):
    """Sigmoid scoring picks the k-subset with the largest logit sum (no
    ties); the weights are scipy's expit of the chosen logits."""
    lg = _logits(10, E, seed=E + k)
    w, ids = oracle.topk_route_ex(lg, k, False, scoring_func="sigmoid")
    for t in range(10):
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(float(lg[t, e]) for e in c))
        assert set(ids[t].tolist()) == set(best)
    ref = scipy.special.expit(np.take_along_axis(lg.astype(np.float64), ids, 1))
    np.testing.assert_allclose(w, ref, rtol=1e-13)
    wr, idr = oracle.topk_route_ex(lg, k, True, scoring_func="sigmoid")
    assert np.array_equal(idr, ids)
    np.testing.assert_allclose(wr, ref / ref.sum(1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(wr.sum(1), 1.0, rtol=1e-13)


def test_grouped_hand_example():
    """E = 8 in four groups of two, keep two groups, k = 3, sigmoid,
    renormalised, scaled by 2.5.  Group maxima 3.0, 2.8, 2.9, 1.0 keep groups
    0 and 2, so the third expert is 4 (logit 0.0) where the ungrouped router
    would take expert 2 (logit 2.8)."""
    lg = np.array([[3.0, -1.0, 2.8, 2.7, 0.0, 2.9, -2.0, 1.0]], np.float32)
    w, ids = oracle.topk_route_ex(lg, 3, True, scoring_func="sigmoid", num_expert_group=4,
                                  topk_group=2, routed_scaling_factor=2.5)
    assert ids.tolist() == [[0, 5, 4]]
    s = [_expit(3.0), _expit(float(np.float32(2.9))), 0.5]
    np.testing.assert_allclose(w[0], [2.5 * v / sum(s) for v in s], rtol=1e-12)
    _, ids_flat = oracle.topk_route_ex(lg, 3, True, scoring_func="sigmoid")
    assert ids_flat.tolist() == [[0, 5, 2]]


def test_bias_steers_choice_not_weight():
    """A correction bias lifts expert 2 to the top, but its weight is its own
    unbiased score."""
    lg = np.array([[1.0, 0.5, 0.0, -1.0]], np.float32)
    b = np.array([0.0, 0.0, 0.5, 0.0], np.float32)
    w, ids = oracle.topk_route_ex(lg, 2, False, scoring_func="sigmoid", e_score_correction_bias=b)
    assert ids.tolist() == [[2, 0]]          # keys 1.0, 0.731, 0.622, 0.269
    np.testing.assert_allclose(w[0], [0.5, _expit(1.0)], rtol=1e-12)
    w, ids = oracle.topk_route_ex(lg, 2, True, scoring_func="sigmoid", e_score_correction_bias=b)
    np.testing.assert_allclose(w[0], [0.5 / (0.5 + _expit(1.0)), _expit(1.0) / (0.5 + _expit(1.0))],
                               rtol=1e-12)
    # softmax scoring: p = e^l / sum; the bias on expert 3 puts it first
    lg = np.array([[2.0, 1.0, 0.0, 0.0]], np.float32)
    b = np.array([0.0, 0.0, 0.0, 1.0], np.float32)
    w, ids = oracle.topk_route_ex(lg, 2, False, e_score_correction_bias=b)
    z = math.e ** 2 + math.e + 2
    assert ids.tolist() == [[3, 0]]
    np.testing.assert_allclose(w[0], [1 / z, math.e ** 2 / z], rtol=1e-12)


def test_constant_bias_and_trivial_groups_change_nothing():
    """Logits spaced 0.05 apart: a constant bias keeps the sigmoid order;
    one group per expert with topk_group = k, and topk_group = G, both give
    the ungrouped choice."""
    rng = np.random.default_rng(11)
    lg = np.stack([rng.permutation(32) * 0.05 - 0.8 for _ in range(20)]).astype(np.float32)
    w0, i0 = oracle.topk_route_ex(lg, 4, True, scoring_func="sigmoid")
    w1, i1 = oracle.topk_route_ex(lg, 4, True, scoring_func="sigmoid",
                                  e_score_correction_bias=np.full(32, 0.75, np.float32))
    assert np.array_equal(i0, i1)
    np.testing.assert_allclose(w1, w0, rtol=1e-15)
    for G, tg in [(32, 4), (8, 8), (1, 0)]:
        _, ig = oracle.topk_route_ex(lg, 4, True, scoring_func="sigmoid", num_expert_group=G,
                                     topk_group=tg)
        assert np.array_equal(ig, i0)


def test_grouped_invariants_random():
    """On random logits with a bias: the chosen experts come from at most
    topk_group groups, every kept group scores at least as high as every
    dropped one, and no allowed expert outside the choice has a higher key."""
    E, G, tg, k = 64, 8, 3, 6
    lg = _logits(40, E, seed=3)
    b = np.random.default_rng(4).uniform(-0.2, 0.2, E).astype(np.float32)
    w, ids = oracle.topk_route_ex(lg, k, True, scoring_func="sigmoid", num_expert_group=G,
                                  topk_group=tg, e_score_correction_bias=b)
    key = (1 / (1 + np.exp(-lg.astype(np.float64)))) + b    # float64 restatement of the keys
    gsz = E // G
    for t in range(40):
        gmax = key[t].reshape(G, gsz).max(1)
        chosen_groups = set((ids[t] // gsz).tolist())
        assert len(chosen_groups) <= tg
        kept = np.argsort(-gmax, kind="stable")[:tg]
        assert chosen_groups <= set(kept.tolist())
        allowed = np.isin(np.arange(E) // gsz, kept)
        rest = allowed.copy()
        rest[ids[t]] = False
        assert key[t, rest].max() <= key[t, ids[t]].min() + 1e-6
        assert all(key[t, ids[t, j]] >= key[t, ids[t, j + 1]] - 1e-6 for j in range(k - 1))
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-13)


def test_scaling_factor_is_linear():
    lg = _logits(8, 16, seed=9)
    w1, i1 = oracle.topk_route_ex(lg, 3, False, num_expert_group=4, topk_group=2)
    w16, i16 = oracle.topk_route_ex(lg, 3, False, num_expert_group=4, topk_group=2,
                                    routed_scaling_factor=16.0)
    assert np.array_equal(i1, i16)
    np.testing.assert_allclose(w16, 16.0 * w1, rtol=1e-15)


@pytest.mark.parametrize("kw", [dict(scoring_func="tanh"), dict(num_expert_group=3, topk_group=1),
                                dict(num_expert_group=4, topk_group=5),
                                dict(num_expert_group=4, topk_group=0),
                                dict(num_expert_group=8, topk_group=1)])
def test_rejects_bad_options(kw):
    with pytest.raises(ValueError):
        oracle.topk_route_ex(_logits(2, 16, 0), 3, True, **kw)


def test_group_and_expert_ties_go_to_lower_index():
    lg = np.array([[1.0, 0.0, 0.0, 1.0], [0.0, 0.5, 0.5, 0.5]], np.float32)
    _, ids = oracle.topk_route_ex(lg, 1, True, num_expert_group=2, topk_group=1)
    assert ids.tolist() == [[0], [1]]   # equal group maxima: group 0 stays
    _, ids = oracle.topk_route_ex(lg, 2, True, num_expert_group=2, topk_group=1)
    assert ids.tolist() == [[0, 1], [1, 0]]
