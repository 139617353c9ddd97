"""Pins of the oracle's fp64 attention over the dequantized cache.

KIVI page ("Makale Bulteni -- KIVI"), section "Iddia ve Gerceklik", 2nd paragraph:
the attention output is a weighted sum of the values.  Reading R8 of
oracle/kivi_oracle.c: score = sigma * q.K', p = softmax(score), out = sum p V',
query head h reads KV head h // (Hq / Hkv).  The checks compare the oracle with
closed forms and with scipy's softmax on inputs the quantizer represents exactly.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _two_level(rng, shape_groups, a_choices, s):
    """Values drawn from {a, a + 3s}: quantization of such a group is exact."""
    a = rng.choice(a_choices)
    pick = rng.integers(0, 2, size=shape_groups)
    return a + 3 * s * pick


def _exact_cache_inputs(rng, B, H, n, G, D=128):
    k = np.zeros((B, H, n, D))
    for b in range(B):
        for h in range(H):
            for g0 in range(0, n, G):
                g1 = min(n, g0 + G)
                for c in range(D):
                    k[b, h, g0:g1, c] = _two_level(rng, g1 - g0, [-1.0, -0.5, 0.25, 2.0], rng.choice([0.125, 0.25, 8.0]))
    v = np.zeros((B, H, n, D))
    for b in range(B):
        for h in range(H):
            for t in range(n):
                v[b, h, t] = _two_level(rng, D, [-1.5, -0.25, 0.5], rng.choice([0.125, 0.5]))
    return k.astype(np.float16), v.astype(np.float16)


@pytest.mark.parametrize("n,G,Hq,Hkv", [(70, 32, 2, 2), (129, 64, 4, 1), (64, 32, 4, 2)])
def test_two_level_inputs_attention_equals_unquantized_attention(n, G, Hq, Hkv):
    rng = np.random.default_rng(n + G)
    B, D = 2, 128
    k, v = _exact_cache_inputs(rng, B, Hkv, n, G)
    c = oracle.prefill(k, v, G, n + G)
    kd, vd = oracle.dequantize(c)
    assert np.array_equal(kd, k.astype(np.float64)) and np.array_equal(vd, v.astype(np.float64))
    q = (rng.standard_normal((B, Hq, D)) / np.sqrt(D)).astype(np.float16)
    sigma = 0.7
    got = oracle.attention(c, q, sigma)
    grp = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            K = k[b, h // grp].astype(np.float64)
            V = v[b, h // grp].astype(np.float64)
            p = softmax(sigma * (K @ q[b, h].astype(np.float64)))
            assert np.allclose(got[b, h], p @ V, rtol=0, atol=1e-12)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    k = rng.standard_normal((1, 1, 1, 128)).astype(np.float16)
    v = rng.standard_normal((1, 1, 1, 128)).astype(np.float16)
    c = oracle.prefill(k, v, 32, 32)
    q = rng.standard_normal((1, 1, 128)).astype(np.float16)
    out = oracle.attention(c, q, 1.0)
    _, vd = oracle.dequantize(c)
    assert np.array_equal(out[0, 0], vd[0, 0, 0])


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(2)
    n = 32 * 5 + 9
    k = (rng.standard_normal((1, 1, n, 128)) * 10).astype(np.float16)
    v = rng.standard_normal((1, 1, n, 128)).astype(np.float16)
    c = oracle.prefill(k, v, 32, 256)
    out = oracle.attention(c, np.zeros((1, 1, 128), np.float16), 1.0)
    _, vd = oracle.dequantize(c)
    assert np.allclose(out[0, 0], vd[0, 0].mean(axis=0), rtol=0, atol=1e-13)


def test_dominant_token_wins():
    rng = np.random.default_rng(3)
    n = 100
    k = rng.standard_normal((1, 1, n, 128)).astype(np.float16)
    k[0, 0, 42, 9] = 60.0
    v = rng.standard_normal((1, 1, n, 128)).astype(np.float16)
    c = oracle.prefill(k, v, 32, 128)
    q = np.zeros((1, 1, 128), np.float16)
    q[0, 0, 9] = 10.0
    out = oracle.attention(c, q, 1.0)
    _, vd = oracle.dequantize(c)
    assert np.allclose(out[0, 0], vd[0, 0, 42], atol=1e-9)


def test_gqa_head_mapping_is_contiguous():
    """KV head j holds constant values j: query head h must return h // (Hq/Hkv)."""
    B, Hq, Hkv, n = 1, 8, 2, 40
    k = np.zeros((B, Hkv, n, 128), np.float16)
    v = np.zeros((B, Hkv, n, 128), np.float16)
    for j in range(Hkv):
        v[0, j] = float(j + 1)
    c = oracle.prefill(k, v, 32, 64)
    out = oracle.attention(c, np.ones((B, Hq, 128), np.float16), 1.0)
    for h in range(Hq):
        assert np.allclose(out[0, h], h // (Hq // Hkv) + 1)


def test_head_entry_point_matches_batch_entry_point():
    rng = np.random.default_rng(8)
    k = rng.standard_normal((2, 2, 77, 128)).astype(np.float16)
    v = rng.standard_normal((2, 2, 77, 128)).astype(np.float16)
    c = oracle.prefill(k, v, 32, 96)
    q = rng.standard_normal((2, 4, 128)).astype(np.float16)
    full = oracle.attention(c, q, 0.5)
    one = oracle.attention_head(c, 1, 1, q[1, 3], 0.5)
    assert np.array_equal(full[1, 3], one)


def test_empty_cache_is_an_error():
    c = oracle.Cache.empty(1, 1, 128, 32, 32)
    with pytest.raises(ValueError):
        oracle.attention(c, np.zeros((1, 1, 128), np.float16), 1.0)


def test_raw_attention_matches_scipy_and_the_quantized_path_on_exact_inputs():
    """fp64 attention over the raw fp16 cache: equal to scipy's softmax attention, and
    equal to the quantized-cache attention when quantization is exact."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, n, G = 2, 4, 2, 70, 32
    k, v = _exact_cache_inputs(rng, B, Hkv, n, G)
    q = (rng.standard_normal((B, Hq, 128)) / np.sqrt(128)).astype(np.float16)
    raw = oracle.attention_raw(k, v, q, 0.9)
    for b in range(B):
        for h in range(Hq):
            K = k[b, h // 2].astype(np.float64)
            V = v[b, h // 2].astype(np.float64)
            p = softmax(0.9 * (K @ q[b, h].astype(np.float64)))
            assert np.allclose(raw[b, h], p @ V, rtol=0, atol=1e-12)
            one = oracle.attention_raw_head(k[b, h // 2], v[b, h // 2], q[b, h], 0.9)
            assert np.array_equal(one, raw[b, h])
    c = oracle.prefill(k, v, G, 128)
    assert np.allclose(oracle.attention(c, q, 0.9), raw, rtol=0, atol=1e-12)
