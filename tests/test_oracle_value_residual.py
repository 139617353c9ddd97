"""Pins of the oracle's value-residual variant (reading R9: the last n mod G values
stay fp16 beside the key residual and are quantized per token when the key group
flushes).  Each check compares with the inputs themselves, with the per-row value
quantizer (pinned on its own in test_oracle_quantizer.py), or with attention written
out in numpy.
"""
import numpy as np
import pytest

import oracle

D = 128


def _kv(rng, B, Hkv, n):
    k = rng.standard_normal((B, Hkv, n, D)).astype(np.float16)
    v = rng.standard_normal((B, Hkv, n, D)).astype(np.float16)
    return k, v


def _row_codes(row):
    s, z, codes = oracle.quantize_group(row)
    return oracle.pack_row(codes), s | (z << 16)


@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("extra", [-1, 0, 1, 17])
def test_prefill_keeps_the_last_values_and_quantizes_the_rest_per_row(G, extra):
    n = 2 * G + extra
    rng = np.random.default_rng(100 + G + extra)
    k, v = _kv(rng, 1, 2, n)
    c = oracle.prefill(k, v, G, 4 * G, value_residual=True)
    nq = (n // G) * G
    vb = v.view(np.uint16)
    assert np.array_equal(c.v_res[:, :, : n - nq], vb[:, :, nq:])
    for h in range(2):
        for t in (0, nq // 2, nq - 1):
            words, meta = _row_codes(v[0, h, t])
            assert np.array_equal(c.v_codes[0, h, t], words)
            assert c.v_meta[0, h, t] == meta
    # rows at or beyond nq hold no codes (they were never written)
    assert not c.v_codes[:, :, nq:].any() and not c.v_meta[:, :, nq:].any()


def test_flush_quantizes_the_group_values_token_by_token():
    G = 32
    rng = np.random.default_rng(7)
    k, v = _kv(rng, 1, 1, G + 5)
    c = oracle.prefill(k[:, :, :G - 1], v[:, :, :G - 1], G, 4 * G, value_residual=True)
    assert not c.v_codes.any()
    oracle.append(c, k[:, :, G - 1].copy(), v[:, :, G - 1].copy())  # fills the first group
    for t in range(G):
        words, meta = _row_codes(v[0, 0, t])
        assert np.array_equal(c.v_codes[0, 0, t], words) and c.v_meta[0, 0, t] == meta
    for t in range(G, G + 5):
        oracle.append(c, k[:, :, t].copy(), v[:, :, t].copy())
    assert np.array_equal(c.v_res[0, 0, :5], v[0, 0, G:G + 5].view(np.uint16))
    assert not c.v_codes[0, 0, G:].any()


@pytest.mark.parametrize("G,n0,m", [(32, 0, 70), (32, 45, 40), (64, 100, 90)])
def test_streaming_equals_batch_with_a_value_residual(G, n0, m):
    rng = np.random.default_rng(G + n0 + m)
    k, v = _kv(rng, 2, 2, n0 + m)
    T = ((n0 + m) // G + 2) * G
    c = oracle.prefill(k[:, :, :n0], v[:, :, :n0], G, T, value_residual=True)
    for t in range(n0, n0 + m):
        oracle.append(c, k[:, :, t].copy(), v[:, :, t].copy())
    b = oracle.prefill(k, v, G, T, value_residual=True)
    n = n0 + m
    nq = (n // G) * G
    assert np.array_equal(c.k_codes[:, :, :nq], b.k_codes[:, :, :nq])
    assert np.array_equal(c.k_meta[:, :, : n // G], b.k_meta[:, :, : n // G])
    assert np.array_equal(c.v_codes[:, :, :nq], b.v_codes[:, :, :nq])
    assert np.array_equal(c.v_meta[:, :, :nq], b.v_meta[:, :, :nq])
    assert np.array_equal(c.k_res[:, :, : n - nq], b.k_res[:, :, : n - nq])
    assert np.array_equal(c.v_res[:, :, : n - nq], b.v_res[:, :, : n - nq])


def test_a_cache_shorter_than_a_group_attends_over_the_raw_inputs():
    """Below one group nothing is quantized: the attention is the plain fp64 softmax
    attention over the fp16 inputs, written out here."""
    G, n = 64, 45
    rng = np.random.default_rng(11)
    k, v = _kv(rng, 1, 2, n)
    q = (rng.standard_normal((1, 4, D)) / np.sqrt(D)).astype(np.float16)
    c = oracle.prefill(k, v, G, 2 * G, value_residual=True)
    got = oracle.attention(c, q, 0.8)
    for h in range(4):
        K = k[0, h // 2].astype(np.float64)
        V = v[0, h // 2].astype(np.float64)
        s = 0.8 * (K @ q[0, h].astype(np.float64))
        p = np.exp(s - s.max())
        assert np.allclose(got[0, h], (p / p.sum()) @ V, rtol=0, atol=1e-12)


def test_dequantized_residual_values_are_exact():
    G, n = 32, 32 * 3 + 9
    rng = np.random.default_rng(12)
    k, v = _kv(rng, 1, 1, n)
    c = oracle.prefill(k, v, G, 4 * G, value_residual=True)
    _, v64 = oracle.dequantize(c)
    _, v32 = oracle.dequantize(c, np.float32)
    nq = 96
    assert np.array_equal(v64[0, 0, nq:], v[0, 0, nq:].astype(np.float64))
    assert np.array_equal(v32[0, 0, nq:], v[0, 0, nq:].astype(np.float32))
    # quantized rows dequantize as without the residual
    plain = oracle.prefill(k, v, G, 4 * G)
    _, p64 = oracle.dequantize(plain)
    assert np.array_equal(v64[0, 0, :nq], p64[0, 0, :nq])
