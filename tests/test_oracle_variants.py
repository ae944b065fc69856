"""Pins of the oracle's weight-format and routing variants: the moe_wna16
8-bit storage (uint8 codes, per-row scales and zeros), the per-tensor int8
scale, and the router weight applied to the expert input."""

import numpy as np
import pytest

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _int8_layer(seed, E=3, H=16, I=8):
    r = _rng(seed)
    return oracle.Int8Experts(
        r.integers(-127, 128, (E, 2 * I, H)).astype(np.int8),
        r.uniform(1e-3, 2e-2, (E, 2 * I)).astype(np.float32),
        r.integers(-127, 128, (E, H, I)).astype(np.int8),
        r.uniform(1e-3, 2e-2, (E, H)).astype(np.float32))


def _routing(seed, T, E, k, renorm=True):
    lg = _rng(seed).standard_normal((T, E)).astype(np.float32)
    return oracle.topk_route(lg, k, renorm)


def test_uint8_zero_points_hand_values():
    """(q - z) * s on a 2 x 4 example worked out by hand."""
    q = np.array([[0, 255, 100, 128], [10, 20, 30, 40]], np.uint8)
    z = np.array([100, 5], np.uint8)
    s = np.array([0.5, 2.0])
    want = np.array([[-50.0, 77.5, 0.0, 14.0], [10.0, 30.0, 50.0, 70.0]])
    assert np.array_equal(oracle.dequantize_uint8_per_channel(q, s, z), want)
    # no zeros: the zero is 128
    want0 = np.array([[-64.0, 63.5, -14.0, 0.0], [-236.0, -216.0, -196.0, -176.0]])
    assert np.array_equal(oracle.dequantize_uint8_per_channel(q, s), want0)


def test_uint8_storage_of_int8_codes_is_the_same_layer():
    """A symmetric int8 code c stored as c + 128 with zero 128 (implicit or
    explicit) dequantises to the same weights, so the forward is identical."""
    ex = _int8_layer(1)
    E, H, I = ex.shape
    u13 = (ex.w13.astype(np.int16) + 128).astype(np.uint8)
    u2 = (ex.w2.astype(np.int16) + 128).astype(np.uint8)
    for zeros in (False, True):
        z13 = np.full((E, 2 * I), 128, np.uint8) if zeros else None
        z2 = np.full((E, H), 128, np.uint8) if zeros else None
        ux = oracle.Uint8Experts(u13, ex.s13, u2, ex.s2, z13, z2)
        for e in range(E):
            assert np.array_equal(ux.deq13(e), ex.deq13(e))
            assert np.array_equal(ux.deq2(e), ex.deq2(e))
        x = _rng(2).standard_normal((5, H))
        w, ids = _routing(3, 5, E, 2)
        assert np.array_equal(oracle.moe_forward(x, ux, w, ids), oracle.moe_forward(x, ex, w, ids))


def test_uint8_zero_shift_is_an_exact_offset():
    """Raising every code and its row's zero by the same amount changes
    nothing (only q - z enters)."""
    r = _rng(4)
    q = r.integers(0, 200, (6, 10)).astype(np.uint8)
    z = r.integers(0, 200, 6).astype(np.uint8)
    s = r.uniform(0.01, 1.0, 6)
    a = oracle.dequantize_uint8_per_channel(q, s, z)
    b = oracle.dequantize_uint8_per_channel(q + 55, s, z + 55)
    assert np.array_equal(a, b)


def test_per_tensor_scale_equals_constant_per_channel_scale():
    ex = _int8_layer(5)
    E, H, I = ex.shape
    s13 = np.array([0.011, 0.002, 0.007])
    s2 = np.array([0.003, 0.013, 0.005])
    tx = oracle.Int8TensorExperts(ex.w13, s13, ex.w2, s2)
    cx = oracle.Int8Experts(ex.w13, np.repeat(s13[:, None], 2 * I, 1), ex.w2,
                            np.repeat(s2[:, None], H, 1))
    x = _rng(6).standard_normal((7, H))
    w, ids = _routing(7, 7, E, 2)
    assert np.array_equal(oracle.moe_forward(x, tx, w, ids), oracle.moe_forward(x, cx, w, ids))


def test_router_weight_on_input_is_a_no_op_for_unit_weights():
    """top_k = 1 with renormalisation gives weight 1 exactly."""
    ex = _int8_layer(8)
    E, H, _ = ex.shape
    x = _rng(9).standard_normal((6, H))
    w, ids = _routing(10, 6, E, 1, renorm=True)
    assert np.all(w == 1.0)
    a = oracle.moe_forward(x, ex, w, ids, apply_router_weight_on_input=True)
    assert np.array_equal(a, oracle.moe_forward(x, ex, w, ids))


def test_router_weight_on_input_brute_force():
    """Explicit loops over tokens, slots, rows and K for a tiny layer."""
    ex = _int8_layer(11, E=3, H=6, I=4)
    E, H, I = ex.shape
    x = _rng(12).standard_normal((3, H))
    w, ids = _routing(13, 3, E, 2, renorm=False)
    got = oracle.moe_forward(x, ex, w, ids, apply_router_weight_on_input=True)
    want = np.zeros((3, H))
    for t in range(3):
        for j in range(2):
            e = int(ids[t, j])
            xs = [float(w[t, j]) * float(x[t, kk]) for kk in range(H)]
            act = []
            for i in range(I):
                g = sum(float(ex.w13[e, i, kk]) * float(ex.s13[e, i]) * xs[kk] for kk in range(H))
                u = sum(float(ex.w13[e, I + i, kk]) * float(ex.s13[e, I + i]) * xs[kk]
                        for kk in range(H))
                act.append(g / (1.0 + np.exp(-g)) * u)
            for h in range(H):
                want[t, h] += sum(float(ex.w2[e, h, i]) * float(ex.s2[e, h]) * act[i]
                                  for i in range(I))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # and it differs from scaling the output (SiLU is not homogeneous)
    assert not np.allclose(got, oracle.moe_forward(x, ex, w, ids), rtol=1e-6)


def test_round_to_bf16_against_torch_and_hand_values():
    """Ties go to even: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6 (even
    mantissa), -(1 + 2^-9) -> -1; and agreement with torch's conversion on
    random float32 values (the library routine rounds the same way)."""
    import torch
    hand = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -9), 0.0, 3.0, 2.0 ** -120])
    want = np.array([1.0, 1 + 2.0 ** -6, -1.0, 0.0, 3.0, 2.0 ** -120])
    assert np.array_equal(oracle.round_to_bf16(hand), want)
    v = (np.random.default_rng(0).standard_normal(100000) * 10.0 ** np.random.default_rng(1).uniform(-8, 8, 100000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_to_bf16(v), ref)


def test_bf16_intermediate_changes_only_the_intermediate():
    """With intermediate values that are already bfloat16 numbers the two
    forms agree exactly; in general they differ by at most the rounding."""
    ex = _int8_layer(21, E=2, H=8, I=4)
    x = _rng(22).standard_normal((3, 8))
    w, ids = _routing(23, 3, 2, 1, renorm=True)
    a = oracle.moe_forward(x, ex, w, ids)
    b = oracle.moe_forward(x, ex, w, ids, intermediate="bf16")
    assert not np.array_equal(a, b)
    # |delta| <= sum_i |W2| |a_i| 2^-8 per output
    E, H, I = ex.shape
    for t in range(3):
        e = int(ids[t, 0])
        h = ex.deq13(e) @ x[t]
        act = oracle.silu(h[:I]) * h[I:]
        bound = np.abs(ex.deq2(e)) @ np.abs(act) * 2.0 ** -8
        assert np.all(np.abs(a[t] - b[t]) <= bound * (1 + 1e-9))
