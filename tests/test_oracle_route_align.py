"""Pins for the oracle's router and block alignment (CPU only)."""

import itertools

import numpy as np
import pytest
import scipy.special

import oracle


def _logits(T, E, seed):
    return np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32)


# ------------------------------------------------------------------ route --
@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 3)])
def test_route_brute_force_subsets(E, k):
    """The chosen set is the k-subset with the largest logit sum (no ties)."""
    lg = _logits(12, E, seed=E * 10 + k)
    w, ids = oracle.topk_route(lg, k, renormalize=False)
    for t in range(12):
        best = max(itertools.combinations(range(E), k),
                   key=lambda c: sum(float(lg[t, e]) for e in c))
        assert set(ids[t].tolist()) == set(best)
        # slots run from the largest logit down
        assert all(lg[t, ids[t, j]] > lg[t, ids[t, j + 1]] for j in range(k - 1))


def test_route_weights_match_library_softmax():
    lg = _logits(20, 16, seed=1)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    w, ids = oracle.topk_route(lg, 4, renormalize=False)
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-13)
    wr, idr = oracle.topk_route(lg, 4, renormalize=True)
    assert np.array_equal(idr, ids)
    np.testing.assert_allclose(wr.sum(1), 1.0, rtol=1e-13)
    sel = np.take_along_axis(p, ids, 1)
    np.testing.assert_allclose(wr, sel / sel.sum(1, keepdims=True), rtol=1e-13)


def test_route_constant_logits_and_ties():
    lg = np.full((3, 8), 0.7, dtype=np.float32)
    w, ids = oracle.topk_route(lg, 3, renormalize=False)
    assert ids.tolist() == [[0, 1, 2]] * 3
    np.testing.assert_allclose(w, 1 / 8)
    w, ids = oracle.topk_route(lg, 3, renormalize=True)
    np.testing.assert_allclose(w, 1 / 3)
    lg = np.array([[1.0, 2.0, 2.0, 0.0, -0.0, 0.0]], dtype=np.float32)
    _, ids = oracle.topk_route(lg, 4, renormalize=True)
    assert ids.tolist() == [[1, 2, 0, 3]]     # equal logits: lower index first
    _, ids = oracle.topk_route(lg, 6, renormalize=True)
    assert ids.tolist() == [[1, 2, 0, 3, 4, 5]]  # -0.0 ties with 0.0


def test_route_k_equals_e_and_shift_invariance():
    lg = _logits(5, 6, seed=2)
    w, ids = oracle.topk_route(lg, 6, renormalize=True)
    np.testing.assert_allclose(w, np.take_along_axis(
        scipy.special.softmax(lg.astype(np.float64), 1), ids, 1), rtol=1e-13)
    w2, ids2 = oracle.topk_route(lg + np.float32(3.0), 6, renormalize=True)
    assert np.array_equal(ids, ids2)
    np.testing.assert_allclose(w, w2, rtol=1e-5)


def test_route_rejects_bad_k():
    with pytest.raises(ValueError):
        oracle.topk_route(_logits(2, 4, 0), 5, True)


# ------------------------------------------------------------------ align --
def _brute_align(ids, E, bm):
    flat = ids.reshape(-1).tolist()
    S = len(flat)
    order = sorted((s for s in range(S) if 0 <= flat[s] < E), key=lambda s: (flat[s], s))
    out, blocks, offsets = [], [], [0]
    for e in range(E):
        seg = [s for s in order if flat[s] == e]
        while len(seg) % bm:
            seg.append(S)
        out += seg
        blocks += [e] * (len(seg) // bm)
        offsets.append(len(out))
    return out, blocks, offsets


@pytest.mark.parametrize("T,k,E,bm", [(16, 2, 8, 16), (37, 3, 5, 4), (1, 2, 8, 64),
                                      (64, 8, 128, 16), (5, 1, 3, 1)])
def test_align_matches_stable_sort(T, k, E, bm):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    r = oracle.align_block(ids, E, bm)
    out, blocks, offsets = _brute_align(ids, E, bm)
    assert r.sorted_slot_ids.tolist() == out
    assert r.block_expert.tolist() == blocks
    assert r.expert_offsets.tolist() == offsets
    assert r.num_padded == len(out) <= oracle.align_capacity(T, k, E, bm)
    S = T * k
    real = r.sorted_slot_ids[r.sorted_slot_ids < S]
    assert sorted(real.tolist()) == list(range(S))       # each slot exactly once
    counts = np.bincount(ids.reshape(-1), minlength=E)
    assert np.array_equal(np.diff(r.expert_offsets), -(-counts // bm) * bm)


def test_align_zero_token_experts_and_invalid_ids():
    ids = np.array([[2, 2], [0, 2], [7, -1]], dtype=np.int32)   # E = 4: 7, -1 invalid
    r = oracle.align_block(ids, 4, 2)
    assert r.invalid_slots == 2
    assert r.expert_offsets.tolist() == [0, 2, 2, 6, 6]
    assert r.sorted_slot_ids.tolist() == [2, 6, 0, 1, 3, 6]
    assert r.block_expert.tolist() == [0, 2, 2]


def test_align_capacity_bound_is_tight():
    # every expert gets exactly one slot: each pads to a full block
    T, k, E, bm = 4, 2, 8, 16
    ids = np.arange(T * k, dtype=np.int32).reshape(T, k)
    r = oracle.align_block(ids, E, bm)
    assert r.num_padded == E * bm == oracle.align_capacity(T, k, E, bm)
