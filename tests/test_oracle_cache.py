"""Pins of the oracle's cache semantics: residual buffer, streaming, layout.

KIVI page ("Makale Bulteni -- KIVI"), section "Iddia ve Gerceklik", 3rd paragraph:
keys are grouped in G-token groups because a new token's channel min/max is not
known in advance, and the tokens of an unfilled group stay in a full-precision
residual buffer (readings R6, R7 of oracle/kivi_oracle.c).
"""
import numpy as np
import pytest

import oracle


def _kv(rng, B, H, n, D=128, outlier=True):
    k = rng.standard_normal((B, H, n, D))
    if outlier:
        k[..., [5, 77]] *= 50.0
    v = rng.standard_normal((B, H, n, D))
    return k.astype(np.float16), v.astype(np.float16)


@pytest.mark.parametrize("G", [32, 64])
def test_residual_holds_last_n_mod_G_tokens_exactly(G):
    rng = np.random.default_rng(G)
    for n in (G - 1, G, G + 1, 2 * G + 17):
        k, v = _kv(rng, 1, 2, n)
        c = oracle.prefill(k, v, G, max_tokens=4 * G)
        nq = (n // G) * G
        r = n - nq
        assert r == n % G
        for h in range(2):
            assert np.array_equal(c.k_res[0, h, :r], k[0, h, nq:].view(np.uint16))
            # dequantized residual keys are the inputs themselves
        kd, _ = oracle.dequantize(c)
        assert np.array_equal(kd[:, :, nq:], k[:, :, nq:].astype(np.float64))


def test_full_group_codes_do_not_depend_on_residual_tokens():
    rng = np.random.default_rng(7)
    G, n = 32, 2 * 32 + 17
    k, v = _kv(rng, 1, 1, n)
    a = oracle.prefill(k, v, G, 128)
    k2 = k.copy()
    k2[:, :, 64:] = (rng.standard_normal((1, 1, 17, 128)) * 1000).astype(np.float16)
    b = oracle.prefill(k2, v, G, 128)
    assert np.array_equal(a.k_codes[:, :, :64], b.k_codes[:, :, :64])
    assert np.array_equal(a.k_meta[:, :, :2], b.k_meta[:, :, :2])


def test_key_groups_are_per_channel_and_values_per_token():
    """A key outlier channel only changes its own channel's meta; a value outlier
    token only changes its own token's meta (the asymmetry of the headline)."""
    rng = np.random.default_rng(9)
    G, n = 32, 64
    k, v = _kv(rng, 1, 1, n, outlier=False)
    base = oracle.prefill(k, v, G, n)
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, :, 3] *= 100                       # one outlier key channel
    v2[0, 0, 10, :] *= 100                      # one outlier value token
    o = oracle.prefill(k2, v2, G, n)
    changed_k = np.nonzero((o.k_meta != base.k_meta)[0, 0].any(axis=0))[0]
    assert changed_k.tolist() == [3]
    changed_v = np.nonzero(o.v_meta[0, 0] != base.v_meta[0, 0])[0]
    assert changed_v.tolist() == [10]
    # other channels' codes are untouched (channel 3 lives in word 0; scaling a
    # channel by 100 may leave its own codes unchanged, as the levels scale too)
    words_k = np.nonzero((o.k_codes != base.k_codes)[0, 0].any(axis=0))[0]
    assert set(words_k.tolist()) <= {0}
    assert np.array_equal(o.v_codes[0, 0, :10], base.v_codes[0, 0, :10])
    assert np.array_equal(o.v_codes[0, 0, 11:], base.v_codes[0, 0, 11:])


@pytest.mark.parametrize("G,n,m", [(32, 0, 70), (32, 31, 1), (32, 50, 100), (64, 64, 65), (64, 17, 200)])
def test_streaming_equals_batch(G, n, m):
    """prefill(n) followed by m appends == prefill(n + m), bit for bit."""
    rng = np.random.default_rng(G * 1000 + n + m)
    B, H, D = 2, 3, 128
    k, v = _kv(rng, B, H, n + m)
    T = ((n + m + G - 1) // G) * G + G
    batch = oracle.prefill(k, v, G, T)
    stream = oracle.prefill(k[:, :, :n].copy(), v[:, :, :n].copy(), G, T)
    for t in range(n, n + m):
        oracle.append(stream, k[:, :, t].copy(), v[:, :, t].copy())
    N = n + m
    nq = (N // G) * G
    assert stream.n == batch.n == N
    assert np.array_equal(stream.k_codes[:, :, :nq], batch.k_codes[:, :, :nq])
    assert np.array_equal(stream.k_meta[:, :, : N // G], batch.k_meta[:, :, : N // G])
    assert np.array_equal(stream.k_res[:, :, : N - nq], batch.k_res[:, :, : N - nq])
    assert np.array_equal(stream.v_codes[:, :, :N], batch.v_codes[:, :, :N])
    assert np.array_equal(stream.v_meta[:, :, :N], batch.v_meta[:, :, :N])


def test_dequant_f32_is_f64_rounded_once():
    """code*s is exact in fp32, so the fp32 dequant is the exact value rounded once."""
    rng = np.random.default_rng(4)
    k, v = _kv(rng, 1, 2, 32 * 3 + 5)
    c = oracle.prefill(k, v, 32, 128)
    k64, v64 = oracle.dequantize(c, np.float64)
    k32, v32 = oracle.dequantize(c, np.float32)
    assert np.array_equal(k32.view(np.uint32), k64.astype(np.float32).view(np.uint32))
    assert np.array_equal(v32.view(np.uint32), v64.astype(np.float32).view(np.uint32))


def test_prefill_of_a_single_head_matches_the_batch():
    rng = np.random.default_rng(12)
    k, v = _kv(rng, 2, 2, 100)
    full = oracle.prefill(k, v, 32, 128)
    one = oracle.prefill_head(k[1, 0], v[1, 0], 32, 128)
    for a, b in zip(full.head(1, 0), one.head(0, 0)):
        assert np.array_equal(a, b)
