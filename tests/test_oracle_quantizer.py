"""Pins of the CPU oracle's quantizer against closed forms, brute force and numpy.

The quantizer follows the KIVI page ("Makale Bulteni -- KIVI", headline paragraph:
asymmetric 2-bit, keys per channel, values per token) under the readings R1-R4
stated at the top of oracle/kivi_oracle.c.  None of these checks re-types the
oracle's formula: each compares it with something the definition or the
mathematics fixes independently.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

F16_MAX = 65504.0


def f16(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float16)


def levels(s_bits, z_bits):
    s = float(np.uint16(s_bits).view(np.float16))
    z = float(np.uint16(z_bits).view(np.float16))
    return s, z


# --------------------------------------------------------------------------------
# fp16 conversions: pinned to numpy's IEEE binary16 implementation
# --------------------------------------------------------------------------------
def test_h2f_matches_numpy_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.h2f(int(b)) for b in bits[::7]], np.float32)
    r = ref[::7]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), r[~nan].view(np.uint32))


def test_f2h_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(11)
    xs = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10.0,
        rng.standard_normal(2000).astype(np.float32) * 1e-5,   # fp16 subnormals
        np.float32([65504.0, 65519.0, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                    1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -0.0, 0.0]),  # overflow, ties
    ])
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f2h(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------------
# packing (R7): hand-worked words
# --------------------------------------------------------------------------------
def test_pack_row_hand_values():
    codes = np.arange(128) % 4                       # channel c has code c mod 4
    # per byte: 0 | 1<<2 | 2<<4 | 3<<6 = 0xE4
    assert np.all(oracle.pack_row(codes) == 0xE4E4E4E4)
    assert np.all(oracle.pack_row(np.full(128, 3)) == 0xFFFFFFFF)
    for c in [0, 1, 15, 16, 37, 127]:
        one = np.zeros(128, np.uint8)
        one[c] = 2
        words = oracle.pack_row(one)
        expect = np.zeros(8, np.uint32)
        expect[c // 16] = 2 << (2 * (c % 16))
        assert np.array_equal(words, expect)


# --------------------------------------------------------------------------------
# quantizer closed forms
# --------------------------------------------------------------------------------
@pytest.mark.parametrize("mn,s", [(-0.5, 0.125), (1.0, 0.25), (-3.0, 2.0), (0.0, 2.0 ** -10), (-100.0, 32.0)])
def test_grid_round_trip_is_exact(mn, s):
    """Inputs already on the 4-level grid mn + k*s come back exactly, codes == k."""
    rng = np.random.default_rng(3)
    k = rng.integers(0, 4, size=64)
    k[0], k[1] = 0, 3                        # the group's min and max are levels 0 and 3
    x = f16(mn + k * s)
    assert np.all(x.astype(np.float64) == mn + k * s), "test grid must be fp16-exact"
    s_bits, z_bits, codes = oracle.quantize_group(x)
    ss, zz = levels(s_bits, z_bits)
    assert ss == s and zz == mn
    assert np.array_equal(codes, k)
    assert np.array_equal(zz + codes * ss, x.astype(np.float64))


def test_ties_round_half_to_even():
    """u = 0.5, 1.5, 2.5 exactly -> codes 0, 2, 2 (mn = 0, mx = 3, s = 1)."""
    x = f16([0.0, 3.0, 0.5, 1.5, 2.5, 1.0, 2.0])
    s_bits, z_bits, codes = oracle.quantize_group(x)
    assert levels(s_bits, z_bits) == (1.0, 0.0)
    assert codes.tolist() == [0, 3, 0, 2, 2, 1, 2]
    # just off the ties the nearest level wins
    x = f16([0.0, 3.0, 0.5 + 2 ** -10, 1.5 - 2 ** -10, 2.5 + 2 ** -9])
    assert oracle.quantize_group(x)[2].tolist() == [0, 3, 1, 1, 3]


def test_degenerate_group_constant_and_underflow():
    s_bits, z_bits, codes = oracle.quantize_group(f16([1.25] * 32))
    assert levels(s_bits, z_bits) == (0.0, 1.25) and not codes.any()
    # range 2^-24 -> (max-min)/3 rounds to fp16 zero: all codes 0, zero = min
    x = f16([2.0 ** -24, 0.0, 2.0 ** -24, 0.0])
    s_bits, z_bits, codes = oracle.quantize_group(x)
    assert s_bits == 0 and z_bits == 0 and not codes.any()


def test_negative_zero_point_is_stored_as_positive_zero():
    s_bits, z_bits, _ = oracle.quantize_group(f16([-0.0, 1.5, 0.75]))
    assert z_bits == 0x0000
    s_bits, z_bits, _ = oracle.quantize_group(f16([-0.0, -0.0]))
    assert z_bits == 0x0000 and s_bits == 0


def _rand_groups(rng, n_groups, size, outlier=False):
    x = rng.standard_normal((n_groups, size))
    if outlier:
        x *= rng.uniform(30, 100, size=(n_groups, 1))
    return f16(x)


@pytest.mark.parametrize("size,outlier", [(32, False), (64, True), (128, False), (128, True), (3, False)])
def test_error_bound_half_scale(size, outlier):
    """|x - x'| <= s16/2 (+ fp32 rounding of the subtraction and division)."""
    rng = np.random.default_rng(size + outlier)
    for x in _rand_groups(rng, 300, size, outlier):
        s_bits, z_bits, codes = oracle.quantize_group(x)
        s, z = levels(s_bits, z_bits)
        xd = x.astype(np.float64)
        err = np.abs(xd - (z + codes * s))
        rng_ = xd.max() - xd.min()
        # the stored scale is (max - min)/3 to fp16 precision
        assert abs(s - rng_ / 3) <= rng_ / 3 * (2.0 ** -11 + 2.0 ** -22)
        assert np.all(err <= s * (0.5 + 2.0 ** -20)), err.max() / s


# --------------------------------------------------------------------------------
# brute force: every group of size 2..4 over a 12-value alphabet
# --------------------------------------------------------------------------------
ALPHABET = [-2.0, -1.5, -1.0, -0.75, -0.5, 0.0, 0.25, 0.5, 1.0, 1.5, 2.25, 3.0]


def _nearest_even(u: Fraction) -> int:
    """argmin_q |u - q| over q in {0,1,2,3}; an exact tie goes to the even q."""
    best = None
    for q in range(4):
        d = abs(u - q)
        if best is None or d < best[0] or (d == best[0] and q % 2 == 0):
            best = (d, q)
    return best[1]


def test_brute_force_tiny_groups():
    import itertools

    ties = fp32_decided = 0
    for size in (2, 3, 4):
        for tup in itertools.product(ALPHABET, repeat=size):
            x = f16(tup)
            s_bits, z_bits, codes = oracle.quantize_group(x)
            s, z = levels(s_bits, z_bits)
            mn, mx = min(tup), max(tup)
            assert z == mn
            if mx == mn:
                assert s == 0 and not codes.any()
                continue
            S = Fraction(s)
            for xi, c in zip(tup, codes):
                u = (Fraction(xi) - Fraction(mn)) / S
                frac = u - int(u)
                if frac == Fraction(1, 2):
                    ties += 1
                elif abs(frac - Fraction(1, 2)) < Fraction(1, 1 << 20):
                    fp32_decided += 1            # fp32 rounding of u decides: either neighbour
                    assert c in (int(u), int(u) + 1)
                    continue
                assert c == _nearest_even(u), (tup, xi, float(u), c)
                assert abs(Fraction(xi) - (Fraction(mn) + c * S)) <= S / 2
    assert ties > 100, "the alphabet must exercise exact half-step ties"


# --------------------------------------------------------------------------------
# the comparison form of the rounding rule used by the GPU quantizer
# --------------------------------------------------------------------------------
def test_threshold_form_equals_division_rule():
    """For fp32 d = fl(x - min) and an fp16 scale s > 0,
    clamp(rint_even(fl(d / s)), 0, 3) == [d > s/2] + [d >= 3s/2] + [d > 5s/2].
    Checked on random and near-threshold fp16 inputs against the oracle's division."""
    rng = np.random.default_rng(5)
    xs = []
    for _ in range(400):
        mn = np.float16(rng.standard_normal() * rng.choice([1e-3, 1.0, 50.0]))
        s = np.float16(abs(rng.standard_normal()) * rng.choice([1e-4, 1.0, 30.0]) + 1e-6)
        if not np.isfinite(s) or s == 0:
            continue
        base = [mn]
        for t in (0.5, 1.5, 2.5, 3.0):
            c = np.float32(mn) + np.float32(t) * np.float32(s)
            h = np.float16(c)
            for k in range(-3, 4):
                b = h.view(np.uint16).astype(np.int32) + k
                if 0 <= b < 0xFFFF:
                    base.append(np.uint16(b).view(np.float16))
        base.append(np.float16(mn + 3 * s))
        grp = np.array(base, np.float16)
        grp = grp[np.isfinite(grp)]
        xs.append(grp)
    checked = 0
    for grp in xs:
        s_bits, z_bits, codes = oracle.quantize_group(grp)
        s = np.float32(np.uint16(s_bits).view(np.float16))
        if s == 0:
            continue
        mn = np.float32(grp.astype(np.float32).min())
        d = grp.astype(np.float32) - mn                      # fp32 RNE subtraction
        cmp = (d > np.float32(0.5) * s).astype(int) + (d >= np.float32(1.5) * s) + (d > np.float32(2.5) * s)
        assert np.array_equal(cmp, codes), (grp, s)
        checked += grp.size
    assert checked > 5000
