"""Pins for the oracle's MoE forward (CPU only).

Brute force with explicit loops, the dense-MLP identity (k = E, identical
experts, equal logits) through torch.nn.functional, token-order
equivariance, x = 0, k = 1, and the per-channel factorisation.
"""

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle


def _int8_layer(E, H, I, seed, identical=False):
    rng = np.random.default_rng(seed)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    if identical:
        w13[:] = w13[0]
        w2[:] = w2[0]
    q13, s13 = oracle.quantize_int8_per_channel(w13.reshape(E * 2 * I, H))
    q2, s2 = oracle.quantize_int8_per_channel(w2.reshape(E * H, I))
    return oracle.Int8Experts(q13.reshape(E, 2 * I, H), s13.reshape(E, 2 * I),
                              q2.reshape(E, H, I), s2.reshape(E, H))


def _uint4_layer(E, H, I, gs, seed):
    rng = np.random.default_rng(seed)
    w13 = (rng.standard_normal((E * 2 * I, H)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((E * H, I)) * 0.05).astype(np.float32)
    q13, s13, z13 = oracle.quantize_uint4_group(w13, gs)
    q2, s2, z2 = oracle.quantize_uint4_group(w2, gs)
    return oracle.Uint4Experts(
        oracle.pack_uint4_along_k(q13).reshape(E, 2 * I, H // 2), s13.reshape(E, 2 * I, H // gs),
        oracle.pack_uint4_along_n(z13.reshape(E, 2 * I, H // gs)),
        oracle.pack_uint4_along_k(q2).reshape(E, H, I // 2), s2.reshape(E, H, I // gs),
        oracle.pack_uint4_along_n(z2.reshape(E, H, I // gs)), gs, True)


def _brute_forward(x, ex, w, ids):
    """Explicit loops over tokens, slots, rows and columns (math.exp silu)."""
    E, H, I = ex.shape
    T, k = ids.shape
    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            W13 = ex.deq13(e)
            W2 = ex.deq2(e)
            h = [sum(W13[n, c] * float(x[t, c]) for c in range(H)) for n in range(2 * I)]
            a = [h[i] / (1.0 + math.exp(-h[i])) * h[I + i] for i in range(I)]
            for c in range(H):
                out[t][c] += float(w[t, j]) * sum(W2[c, i] * a[i] for i in range(I))
    return np.array(out)


def test_forward_brute_force_int8():
    E, H, I, T, k = 4, 8, 6, 5, 2
    ex = _int8_layer(E, H, I, seed=1)
    x = np.random.default_rng(2).standard_normal((T, H)).astype(np.float32)
    w, ids = oracle.topk_route(np.random.default_rng(3).standard_normal((T, E)).astype(np.float32), k, True)
    np.testing.assert_allclose(oracle.moe_forward(x, ex, w, ids), _brute_forward(x, ex, w, ids),
                               rtol=1e-12, atol=1e-13)


def test_forward_brute_force_uint4():
    E, H, I, T, k, gs = 3, 8, 4, 4, 2, 4
    ex = _uint4_layer(E, H, I, gs, seed=4)
    x = np.random.default_rng(5).standard_normal((T, H)).astype(np.float32)
    w, ids = oracle.topk_route(np.random.default_rng(6).standard_normal((T, E)).astype(np.float32), k, False)
    np.testing.assert_allclose(oracle.moe_forward(x, ex, w, ids), _brute_forward(x, ex, w, ids),
                               rtol=1e-12, atol=1e-13)


def test_dense_mlp_identity():
    """k = E, identical experts, equal logits, renormalise -> out = MLP(x)."""
    E, H, I, T = 4, 16, 24, 7
    ex = _int8_layer(E, H, I, seed=7, identical=True)
    x = np.random.default_rng(8).standard_normal((T, H)).astype(np.float32)
    w, ids = oracle.topk_route(np.zeros((T, E), np.float32), E, True)
    out = oracle.moe_forward(x, ex, w, ids)
    W13 = torch.from_numpy(ex.deq13(0))
    W2 = torch.from_numpy(ex.deq2(0))
    h = F.linear(torch.from_numpy(x).double(), W13)
    g, u = h.chunk(2, dim=-1)
    ref = F.linear(F.silu(g) * u, W2).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_token_order_equivariance_and_zero_input():
    E, H, I, T, k = 8, 32, 16, 9, 2
    ex = _int8_layer(E, H, I, seed=9)
    rng = np.random.default_rng(10)
    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    w, ids = oracle.topk_route(lg, k, True)
    out = oracle.moe_forward(x, ex, w, ids)
    perm = rng.permutation(T)
    wp, idp = oracle.topk_route(lg[perm], k, True)
    np.testing.assert_allclose(oracle.moe_forward(x[perm], ex, wp, idp), out[perm], rtol=1e-12, atol=1e-14)
    assert np.all(oracle.moe_forward(np.zeros_like(x), ex, w, ids) == 0)
    # token subset and output-column subset agree with the full result
    np.testing.assert_allclose(oracle.moe_forward(x, ex, w, ids, tokens=[3, 7]), out[[3, 7]], rtol=1e-13)
    np.testing.assert_allclose(oracle.moe_forward(x, ex, w, ids, tokens=[1], out_cols=[0, 5, 31]),
                               out[[1]][:, [0, 5, 31]], rtol=1e-13)


def test_k1_renormalise_is_argmax_expert():
    E, H, I, T = 6, 16, 8, 5
    ex = _int8_layer(E, H, I, seed=11)
    rng = np.random.default_rng(12)
    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    w, ids = oracle.topk_route(lg, 1, True)
    assert np.all(w == 1.0) and np.array_equal(ids[:, 0], lg.argmax(1))
    out = oracle.moe_forward(x, ex, w, ids)
    for t in range(T):
        e = int(lg[t].argmax())
        h = ex.deq13(e) @ x[t].astype(np.float64)
        y = ex.deq2(e) @ (oracle.silu(h[:I]) * h[I:])
        np.testing.assert_allclose(out[t], y, rtol=1e-12)


def test_per_channel_factorisation():
    """sum_k x * (q * s) == s * sum_k x * q: the scale can move to the epilogue."""
    E, H, I = 2, 64, 32
    ex = _int8_layer(E, H, I, seed=13)
    x = np.random.default_rng(14).standard_normal(H)
    lhs = ex.deq13(1) @ x
    rhs = ex.s13[1].astype(np.float64) * (ex.w13[1].astype(np.float64) @ x)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-15)


def test_invalid_expert_ids_contribute_nothing():
    E, H, I, T = 4, 8, 8, 3
    ex = _int8_layer(E, H, I, seed=15)
    x = np.random.default_rng(16).standard_normal((T, H)).astype(np.float32)
    w = np.full((T, 2), 0.5)
    ids = np.array([[0, 1], [2, 9], [-1, 3]], dtype=np.int32)
    out = oracle.moe_forward(x, ex, w, ids)
    ok = np.array([[0, 1], [2, 2], [3, 3]], dtype=np.int32)
    wk = np.array([[0.5, 0.5], [0.5, 0.0], [0.0, 0.5]])
    np.testing.assert_allclose(out, oracle.moe_forward(x, ex, wk, ok), rtol=1e-13)
