"""Pins for the oracle's quantisers (CPU only).

Each check comes from somewhere other than the oracle's own formula: exact
rational brute force over all codes, closed forms, invariants, and the
packing rule printed on the moe_wna16 page (AWQ repack, step 5).
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_values(shape, seed, std=0.02):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).float().numpy()


# ---------------------------------------------------------------- int8 ----
def _nearest_code_exact(w, s, lo, hi, zero=0):
    """Exact rational nearest code c in [lo, hi] minimising |(c - zero) * s - w|.

    Returns (code, near_tie) where near_tie flags inputs whose exact ratio
    w / s lies within float32 rounding of a half-integer, where a float32
    division may legitimately round the other way.
    """
    W, Sf = Fraction(float(w)), Fraction(float(s))
    best, best_err = None, None
    for c in range(lo, hi + 1):
        err = abs((c - zero) * Sf - W)
        if best_err is None or err < best_err or (err == best_err and c % 2 == 0):
            best, best_err = c, err
    ratio = W / Sf
    frac = ratio - (ratio.numerator // ratio.denominator)
    near_tie = abs(frac - Fraction(1, 2)) < Fraction(1, 1 << 16)
    return best, near_tie


def test_int8_brute_force_tiny():
    w = _bf16_values((4, 8), seed=1)
    w[2, 3] = 0.0
    q, s = oracle.quantize_int8_per_channel(w)
    for r in range(4):
        m = max(abs(Fraction(float(v))) for v in w[r])
        # scale is the float32 rounding of max|w| / 127
        assert np.float32(s[r]) == np.float32(float(m / 127))
        for c in range(8):
            code, near_tie = _nearest_code_exact(w[r, c], s[r], -127, 127)
            if near_tie:
                assert abs(int(q[r, c]) - code) <= 1
            else:
                assert int(q[r, c]) == code, (r, c, w[r, c], s[r])


def test_int8_golden_rows():
    """Hand-derived rows (tests/golden/int8_rows.json, derivations inside)."""
    with open(os.path.join(GOLDEN, "int8_rows.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        w = np.array([case["w"]], dtype=np.float32)
        q, s = oracle.quantize_int8_per_channel(w)
        assert q[0].tolist() == case["q"], case["why"]
        assert float(s[0]) == float(np.float32(case["scale"])), case["why"]


def test_int8_error_bound_and_range():
    w = _bf16_values((64, 256), seed=2)
    q, s = oracle.quantize_int8_per_channel(w)
    assert q.min() >= -127 and q.max() <= 127          # symmetric: -128 never used
    err = np.abs(q.astype(np.float64) * s[:, None] - w)
    # |dequant - w| <= s/2, up to the float32 rounding of the division
    assert np.all(err <= s[:, None] * (0.5 + 2.0 ** -16))
    # the row maximum maps to +-127 exactly
    am = np.argmax(np.abs(w), axis=1)
    assert np.all(np.abs(q[np.arange(64), am]) == 127)


def test_int8_zero_row_and_symmetry():
    w = _bf16_values((3, 32), seed=3)
    w[1] = 0.0
    q, s = oracle.quantize_int8_per_channel(w)
    assert s[1] == 0 and np.all(q[1] == 0) and np.all(np.isfinite(s))
    qn, sn = oracle.quantize_int8_per_channel(-w)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)


def test_int8_power_of_two_row_scaling():
    """Scaling a row by 2^j scales its scale by 2^j and leaves the codes."""
    w = _bf16_values((8, 64), seed=4)
    q, s = oracle.quantize_int8_per_channel(w)
    for j in (-3, 5):
        q2, s2 = oracle.quantize_int8_per_channel(w * np.float32(2.0 ** j))
        assert np.array_equal(q2, q)
        assert np.array_equal(s2, (s * np.float32(2.0 ** j)).astype(np.float32))


def test_int8_dequant_is_product():
    q = np.array([[1, -2, 127]], dtype=np.int8)
    s = np.array([0.5], dtype=np.float32)
    assert oracle.dequantize_int8_per_channel(q, s).tolist() == [[0.5, -1.0, 63.5]]


# ---------------------------------------------------------------- uint4 ---
def test_uint4_packing_matches_page_rule():
    """tests/golden/uint4_packing.json: the AWQ repack rule of the page."""
    with open(os.path.join(GOLDEN, "uint4_packing.json")) as f:
        g = json.load(f)
    q = np.array(g["along_k"]["values"], dtype=np.uint8)
    assert oracle.pack_uint4_along_k(q).tolist() == g["along_k"]["packed"]
    z = np.array(g["along_n"]["values"], dtype=np.uint8)
    assert oracle.pack_uint4_along_n(z).tolist() == g["along_n"]["packed"]


def test_uint4_pack_roundtrip():
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(6, 10, 32), dtype=np.uint8)
    assert np.array_equal(oracle.unpack_uint4_along_k(oracle.pack_uint4_along_k(q)), q)
    z = rng.integers(0, 16, size=(3, 8, 5), dtype=np.uint8)
    assert np.array_equal(oracle.unpack_uint4_along_n(oracle.pack_uint4_along_n(z)), z)


def test_uint4_brute_force_group():
    w = _bf16_values((2, 32), seed=6)
    q, s16, z = oracle.quantize_uint4_group(w, 16)
    for r in range(2):
        for g in range(2):
            s = np.float32(s16[r, g])
            lo = min(0.0, float(w[r, 16 * g:16 * g + 16].min()))
            hi = max(0.0, float(w[r, 16 * g:16 * g + 16].max()))
            assert s == np.float32(np.float16(np.float32(hi - lo) / np.float32(15)))
            for c in range(16 * g, 16 * g + 16):
                code, near_tie = _nearest_code_exact(w[r, c], s, 0, 15, zero=int(z[r, g]))
                if near_tie:
                    assert abs(int(q[r, c]) - code) <= 1
                else:
                    assert int(q[r, c]) == code


def test_uint4_error_bound():
    w = _bf16_values((32, 512), seed=7)
    q, s16, z = oracle.quantize_uint4_group(w, 128)
    deq = oracle.dequantize_uint4_group(oracle.pack_uint4_along_k(q), s16,
                                        oracle.pack_uint4_along_n(z), 128)
    s = np.repeat(s16.astype(np.float64), 128, axis=1)
    # half a step, plus the slack from rounding the scale to fp16
    # (the range (hi-lo) may exceed 15*s by one fp16 rounding, i.e. 15*s*2^-11)
    assert np.all(np.abs(deq - w) <= s * (0.5 + 16 * 2.0 ** -11))


def test_uint4_zero_group():
    w = np.zeros((2, 16), dtype=np.float32)
    q, s16, z = oracle.quantize_uint4_group(w, 16)
    assert np.all(q == 0) and np.all(s16 == 0) and np.all(z == 0)
    deq = oracle.dequantize_uint4_group(oracle.pack_uint4_along_k(q), s16,
                                        oracle.pack_uint4_along_n(z), 16)
    assert np.all(deq == 0)


def test_gptq_zero_convention():
    """The loader adds 1 to GPTQ's stored (z - 1); stored zero = true zero.

    Start from known weights, store GPTQ-style zeros minus one, apply the
    page's conversion (unpack nibbles, add 1, repack low = even) and check
    that the oracle's dequantisation reproduces the grid values exactly.
    """
    rng = np.random.default_rng(8)
    N, K, gs = 4, 32, 16
    z_true = rng.integers(1, 16, size=(N, K // gs), dtype=np.uint8)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    s = np.full((N, K // gs), 0.125, dtype=np.float16)
    expect = (q.astype(np.float64) - np.repeat(z_true, gs, axis=1)) * 0.125
    # GPTQ checkpoint side: zeros stored minus one, packed along N
    stored = oracle.pack_uint4_along_n((z_true - 1).astype(np.uint8))
    lo, hi = stored & 0xF, stored >> 4
    converted = ((lo + 1) | ((hi + 1) << 4)).astype(np.uint8)   # the page's +1
    deq = oracle.dequantize_uint4_group(oracle.pack_uint4_along_k(q), s, converted, gs)
    assert np.array_equal(deq, expect)


def test_uint4_symmetric_implicit_zero():
    q = np.array([[0, 8, 15, 7]], dtype=np.uint8)
    s = np.array([[0.5]], dtype=np.float16)
    deq = oracle.dequantize_uint4_group(oracle.pack_uint4_along_k(q), s, None, 4, has_zp=False)
    assert deq.tolist() == [[-4.0, 0.0, 3.5, -0.5]]
