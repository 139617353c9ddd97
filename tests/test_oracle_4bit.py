"""Pins of the oracle's 4-bit code width (reading R10: 15 levels, s = (max - min) / 15,
code = clamp(round_half_even((x - min) / s), 0, 15), 8 codes per word).  Each check
compares with a closed form, exact rational arithmetic, a hand-packed word, or
attention written out in numpy.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle

D = 128


def f16(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float16)


def levels(s_bits, z_bits):
    return float(np.uint16(s_bits).view(np.float16)), float(np.uint16(z_bits).view(np.float16))


def test_sixteen_level_grid_round_trip():
    """Values min + k*s (k = 0..15) with s, min and (max - min)/15 exact come back as k."""
    mn, s = -1.0, 0.125
    ks = np.array([0, 15, 3, 7, 8, 12, 1, 14, 2, 9, 4, 11, 5, 10, 6, 13], np.int64)
    x = f16(mn + ks * s)
    s_bits, z_bits, codes = oracle.quantize_group(x, bits=4)
    assert levels(s_bits, z_bits) == (s, mn)
    assert np.array_equal(codes, ks)


def test_half_step_ties_round_to_even():
    s = 0.125
    x = f16([0.0, 15 * s] + [(k + 0.5) * s for k in range(15)])  # u = k + 1/2 exactly
    _, _, codes = oracle.quantize_group(x, bits=4)
    want = [0, 15] + [k if k % 2 == 0 else k + 1 for k in range(15)]
    assert codes.tolist() == want


def test_pack_row_places_channel_i_at_bits_4i():
    codes = np.tile(np.arange(8, dtype=np.uint8), 16)
    words = oracle.pack_row(codes, bits=4)
    assert words.shape == (16,) and (words == 0x76543210).all()
    codes = np.zeros(D, np.uint8)
    codes[9] = 15  # word 1, channel 1 -> bits 4..7
    words = oracle.pack_row(codes, bits=4)
    assert words[1] == 0xF0 and words.sum() == 0xF0


ALPHABET = [-2.0, -1.25, -0.75, 0.0, 0.125, 0.5, 1.0, 1.375, 2.0, 3.0]


def _nearest_even(u: Fraction) -> int:
    best = None
    for q in range(16):
        d = abs(u - q)
        if best is None or d < best[0] or (d == best[0] and q % 2 == 0):
            best = (d, q)
    return best[1]


def test_brute_force_small_groups():
    ties = 0
    for size in (2, 3):
        for tup in itertools.product(ALPHABET, repeat=size):
            s_bits, z_bits, codes = oracle.quantize_group(f16(tup), bits=4)
            s, z = levels(s_bits, z_bits)
            mn, mx = min(tup), max(tup)
            assert z == mn
            if mx == mn:
                assert s == 0 and not codes.any()
                continue
            assert s == float(np.float16(np.float32(mx - mn) / np.float32(15)))
            S = Fraction(s)
            for xi, c in zip(tup, codes):
                u = (Fraction(xi) - Fraction(mn)) / S
                frac = u - int(u)
                if frac == Fraction(1, 2):
                    ties += 1
                elif abs(frac - Fraction(1, 2)) < Fraction(1, 1 << 18):
                    assert c in (int(u), int(u) + 1)  # the fp32 rounding of u decides
                    continue
                assert c == _nearest_even(u), (tup, xi, float(u), c)
                assert abs(Fraction(xi) - (Fraction(mn) + c * S)) <= S / 2
    assert ties >= 10, "the alphabet must exercise exact half-step ties"


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_error_bound_on_random_and_outlier_rows(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((64, D)).astype(np.float32)
    x[:, :2] *= 80
    x = x.astype(np.float16)
    for row in x:
        s_bits, z_bits, codes = oracle.quantize_group(row, bits=4)
        s, z = levels(s_bits, z_bits)
        xd = z + codes.astype(np.float64) * s
        bound = s / 2 + 2 * np.spacing(np.float32(np.abs(row).max()))
        assert np.abs(row.astype(np.float64) - xd).max() <= bound


@pytest.mark.parametrize("G,n0,m", [(32, 0, 70), (32, 45, 40), (64, 100, 90)])
@pytest.mark.parametrize("value_residual", [False, True])
def test_streaming_equals_batch_4bit(G, n0, m, value_residual):
    rng = np.random.default_rng(G + n0 + m)
    k = rng.standard_normal((2, 2, n0 + m, D)).astype(np.float16)
    v = rng.standard_normal((2, 2, n0 + m, D)).astype(np.float16)
    T = ((n0 + m) // G + 2) * G
    c = oracle.prefill(k[:, :, :n0], v[:, :, :n0], G, T, value_residual, bits=4)
    for t in range(n0, n0 + m):
        oracle.append(c, k[:, :, t].copy(), v[:, :, t].copy())
    b = oracle.prefill(k, v, G, T, value_residual, bits=4)
    n = n0 + m
    nq = (n // G) * G
    nv = nq if value_residual else n
    assert c.k_codes.shape[-1] == 16
    assert np.array_equal(c.k_codes[:, :, :nq], b.k_codes[:, :, :nq])
    assert np.array_equal(c.k_meta[:, :, : n // G], b.k_meta[:, :, : n // G])
    assert np.array_equal(c.v_codes[:, :, :nv], b.v_codes[:, :, :nv])
    assert np.array_equal(c.v_meta[:, :, :nv], b.v_meta[:, :, :nv])
    assert np.array_equal(c.k_res[:, :, : n - nq], b.k_res[:, :, : n - nq])


def test_grid_inputs_attend_exactly():
    """Keys on a 16-level grid per group column and values on one per token quantize
    exactly, so attention over the 4-bit cache equals attention over the inputs."""
    rng = np.random.default_rng(21)
    G, n = 32, 32 * 4 + 7
    k = np.empty((1, 2, n, D))
    for g0 in range(0, n, G):
        k[:, :, g0:g0 + G] = -1.0 + 0.125 * rng.integers(0, 16, size=(1, 2, min(G, n - g0), D))
        k[:, :, g0, :] = -1.0        # every column of a group spans the full grid
        k[:, :, min(g0 + 1, n - 1), :] = -1.0 + 15 * 0.125
    v = -0.5 + 0.0625 * rng.integers(0, 16, size=(1, 2, n, D))
    v[:, :, :, 0] = -0.5
    v[:, :, :, 1] = -0.5 + 15 * 0.0625
    k, v = k.astype(np.float16), v.astype(np.float16)
    q = (rng.standard_normal((1, 4, D)) / np.sqrt(D)).astype(np.float16)
    c = oracle.prefill(k, v, G, 5 * G, bits=4)
    got = oracle.attention(c, q, 1.0)
    for h in range(4):
        K, V = k[0, h // 2].astype(np.float64), v[0, h // 2].astype(np.float64)
        s = K @ q[0, h].astype(np.float64)
        p = np.exp(s - s.max())
        assert np.allclose(got[0, h], (p / p.sum()) @ V, rtol=0, atol=1e-12)
