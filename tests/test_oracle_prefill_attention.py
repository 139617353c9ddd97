"""Pins of the oracle's causal prefill attention (reading R12), CPU only.

KIVI page, section "Kod ve Entegrasyon Haritasi": FlashAttention runs the prefill,
and the cache is quantized from the prompt's keys and values.  The plainest reading
(R12) is the standard causal attention of the prompt over its own full-precision
keys and values.  It is pinned here by what that definition fixes, not by
re-deriving it:

- position 0 attends to itself only: out_0 = v_0 exactly;
- a zero query weighs the visible positions equally: out_i = mean(v_0..v_i);
- causality: changing keys or values after position i leaves out_i unchanged;
- a dominant key wins: out_i = v_j when q_i . k_j exceeds every other score by far;
- the last position is the decode attention over the whole prompt (the pinned
  raw-cache oracle), and the GQA mapping is the decode one;
- a uniform-value prompt gives that value at every position.
"""
import numpy as np
import pytest

import oracle

D = 128


def _rand(rng, *shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def test_first_position_is_its_own_value():
    rng = np.random.default_rng(1)
    q, k, v = _rand(rng, 2, 3, 9, D), _rand(rng, 2, 3, 9, D), _rand(rng, 2, 3, 9, D)
    out = oracle.prefill_attention(q, k, v, 0.3)
    assert np.array_equal(out[:, :, 0], v[:, :, 0].astype(np.float64))


def test_zero_query_gives_the_running_mean():
    rng = np.random.default_rng(2)
    n = 17
    k, v = _rand(rng, 1, 1, n, D), _rand(rng, 1, 1, n, D)
    q = np.zeros((1, 1, n, D), np.float16)
    out = oracle.prefill_attention(q, k, v, 1.0)
    vd = v[0, 0].astype(np.float64)
    for i in range(n):
        assert np.allclose(out[0, 0, i], vd[:i + 1].mean(0), rtol=0, atol=1e-12)


def test_later_positions_do_not_change_earlier_outputs():
    rng = np.random.default_rng(3)
    n, cut = 23, 11
    q, k, v = _rand(rng, 1, 2, n, D, scale=0.2), _rand(rng, 1, 2, n, D), _rand(rng, 1, 2, n, D)
    a = oracle.prefill_attention(q, k, v, 1.0)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, cut + 1:] = _rand(rng, 1, 2, n - cut - 1, D, scale=5.0)
    v2[:, :, cut + 1:] = _rand(rng, 1, 2, n - cut - 1, D, scale=5.0)
    b = oracle.prefill_attention(q, k2, v2, 1.0)
    assert np.array_equal(a[:, :, :cut + 1], b[:, :, :cut + 1])
    assert not np.array_equal(a[:, :, cut + 1:], b[:, :, cut + 1:])


def test_a_dominant_key_wins():
    rng = np.random.default_rng(4)
    n, i, j = 12, 9, 4
    k = _rand(rng, 1, 1, n, D, scale=0.01)
    v = _rand(rng, 1, 1, n, D)
    q = np.zeros((1, 1, n, D), np.float16)
    k[0, 0, j] = 1.0
    q[0, 0, i] = 100.0  # score 100 * 128 at j against |score| < 0.2 elsewhere
    out = oracle.prefill_attention(q, k, v, 1.0)
    assert np.allclose(out[0, 0, i], v[0, 0, j].astype(np.float64), rtol=0, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 2), (8, 2)])
def test_last_position_is_the_decode_attention_over_the_prompt(Hq, Hkv):
    rng = np.random.default_rng(Hq + Hkv)
    n = 29
    q = _rand(rng, 2, Hq, n, D, scale=1 / np.sqrt(D))
    k, v = _rand(rng, 2, Hkv, n, D), _rand(rng, 2, Hkv, n, D)
    out = oracle.prefill_attention(q, k, v, 1.0)
    last = oracle.attention_raw(k, v, np.ascontiguousarray(q[:, :, -1]), 1.0)
    assert np.allclose(out[:, :, -1], last, rtol=0, atol=1e-12)
    # and every position i is the decode attention over the first i + 1 tokens
    i = 13
    mid = oracle.attention_raw(np.ascontiguousarray(k[:, :, :i + 1]), np.ascontiguousarray(v[:, :, :i + 1]),
                               np.ascontiguousarray(q[:, :, i]), 1.0)
    assert np.allclose(out[:, :, i], mid, rtol=0, atol=1e-12)


def test_uniform_values_pass_through():
    rng = np.random.default_rng(6)
    n = 15
    q, k = _rand(rng, 1, 2, n, D), _rand(rng, 1, 1, n, D)
    row = _rand(rng, D)
    v = np.broadcast_to(row, (1, 1, n, D)).copy()
    out = oracle.prefill_attention(q, k, v, 0.5)
    assert np.allclose(out, np.broadcast_to(row.astype(np.float64), out.shape), rtol=0, atol=1e-12)


def test_empty_prompt_and_bad_heads_are_errors():
    z = np.zeros((1, 1, 0, D), np.float16)
    with pytest.raises(ValueError):
        oracle.prefill_attention(z, z, z, 1.0)
    q = np.zeros((1, 3, 4, D), np.float16)
    kv = np.zeros((1, 2, 4, D), np.float16)
    with pytest.raises(ValueError):
        oracle.prefill_attention(q, kv, kv, 1.0)


def test_selected_rows_are_the_rows_of_the_whole_prompt():
    """The selected-rows entry (used where the whole prompt is too long for the
    oracle) gives, bit for bit, the rows of the whole-prompt attention, which the
    closed forms above pin; positions outside the prompt are errors."""
    rng = np.random.default_rng(21)
    n = 150
    q, k, v = _rand(rng, 1, 1, n, D, scale=0.2), _rand(rng, 1, 1, n, D), _rand(rng, 1, 1, n, D)
    full = oracle.prefill_attention(q, k, v, 0.8)[0, 0]
    rows = [0, 1, 63, 64, 65, 149, 7]
    got = oracle.prefill_attention_rows(q[0, 0], k[0, 0], v[0, 0], rows, 0.8)
    assert np.array_equal(got, full[rows])
    assert np.array_equal(oracle.prefill_attention_rows(q[0, 0], k[0, 0], v[0, 0], [0], 0.8)[0], v[0, 0, 0])
    with pytest.raises(ValueError):
        oracle.prefill_attention_rows(q[0, 0], k[0, 0], v[0, 0], [n], 0.8)
