"""Pins of the oracle's value channel groups (reading R11), CPU only.

KIVI page "Makale Bulteni -- KIVI", section "Iddia ve Gerceklik", paragraph 2: values
are quantized along the token axis, because the attention output is a weighted sum
of values.  The page leaves the number of channels that share one (scale, zero) open;
R5 takes all D channels of the token, and R11 (a variant) splits the token into D/vg
groups of vg consecutive channels, each quantized by the same rule.  These tests pin
the variant to what the rule fixes:

- vg = D is R5, bit for bit;
- a token whose every channel group lies on its own 4-level (2-bit) or 16-level
  (4-bit) grid {lo + k 2^e} dequantizes exactly, which per-token quantization of the
  same token does not: the groups are really independent;
- each group's scale, zero and codes are those of the pinned single-group quantizer
  on that group's channels, at the group's place in the layout;
- streaming appends give the prefill's cache, with and without a value residual;
- attention uses each channel's own group (closed form over the dequantized keys).
"""
import numpy as np
import pytest

import oracle

D = 128


def _grid_values(rng, n_tokens, vg, levels):
    """[n_tokens, D] fp16: every (token, channel group) on its own grid lo + k 2^e,
    k in 0..levels-1, with both ends present (so min = lo and max = lo + (levels-1) 2^e)."""
    v = np.empty((n_tokens, D), np.float64)
    for t in range(n_tokens):
        for g in range(D // vg):
            e = int(rng.integers(-8, 3))
            lo = float(rng.integers(-64, 64)) * 2.0 ** e
            k = rng.integers(0, levels, size=vg)
            k[0], k[1] = 0, levels - 1
            rng.shuffle(k)
            v[t, g * vg:(g + 1) * vg] = lo + k * 2.0 ** e
    v16 = v.astype(np.float16)
    assert np.array_equal(v16.astype(np.float64), v)  # the grid is exact in fp16
    return v16


def _rand(rng, *shape):
    return (rng.standard_normal(shape) * rng.uniform(0.1, 4, size=shape[:-1] + (1,))).astype(np.float16)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("vres", [False, True])
def test_value_group_of_d_channels_is_the_per_token_rule(bits, vres):
    rng = np.random.default_rng(1)
    k, v = _rand(rng, 2, 2, 77, D), _rand(rng, 2, 2, 77, D)
    a = oracle.prefill(k, v, 32, 96, value_residual=vres, bits=bits)
    b = oracle.prefill(k, v, 32, 96, value_residual=vres, bits=bits, value_group=D)
    for name in ("k_codes", "k_meta", "k_res", "v_codes", "v_meta"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    assert b.v_meta.shape == (2, 2, 96)


@pytest.mark.parametrize("bits,levels", [(2, 4), (4, 16)])
@pytest.mark.parametrize("vg", [16, 32, 64])
def test_grid_groups_dequantize_exactly_and_per_token_does_not(vg, bits, levels):
    rng = np.random.default_rng(vg + bits)
    n = 40
    v = _grid_values(rng, n, vg, levels)[None, None]
    k = _rand(rng, 1, 1, n, D)
    grouped = oracle.prefill(k, v, 32, 64, bits=bits, value_group=vg)
    _, vd = oracle.dequantize(grouped)
    assert np.array_equal(vd[0, 0], v[0, 0].astype(np.float64))
    per_token = oracle.prefill(k, v, 32, 64, bits=bits)
    _, vt = oracle.dequantize(per_token)
    assert not np.array_equal(vt[0, 0], v[0, 0].astype(np.float64))


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("vg", [32, 64])
def test_group_meta_and_codes_are_the_single_group_quantizer_at_their_place(vg, bits):
    rng = np.random.default_rng(3 * vg + bits)
    n = 37
    k, v = _rand(rng, 1, 2, n, D), _rand(rng, 1, 2, n, D)
    c = oracle.prefill(k, v, 32, 64, bits=bits, value_group=vg)
    assert c.v_meta.shape == (1, 2, 64, D // vg)
    per_word = 32 // bits
    for h in range(2):
        for t in range(n):
            row = c.v_codes[0, h, t]
            codes = np.array([(int(row[ch // per_word]) >> (bits * (ch % per_word))) & ((1 << bits) - 1)
                              for ch in range(D)])
            for g in range(D // vg):
                s, z, want = oracle.quantize_group(v[0, h, t, g * vg:(g + 1) * vg], bits=bits)
                assert int(c.v_meta[0, h, t, g]) == (s | (z << 16))
                assert np.array_equal(codes[g * vg:(g + 1) * vg], want)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("vres", [False, True])
@pytest.mark.parametrize("vg", [32, 64])
def test_streaming_appends_give_the_prefill_cache(vg, vres, bits):
    rng = np.random.default_rng(vg + 7 * bits + vres)
    G, n0, steps = 32, 21, 75
    k, v = _rand(rng, 2, 2, n0 + steps, D), _rand(rng, 2, 2, n0 + steps, D)
    T = 128
    c = oracle.prefill(k[:, :, :n0], v[:, :, :n0], G, T, value_residual=vres, bits=bits, value_group=vg)
    for t in range(n0, n0 + steps):
        oracle.append(c, k[:, :, t], v[:, :, t])
    full = oracle.prefill(k, v, G, T, value_residual=vres, bits=bits, value_group=vg)
    n, nq = n0 + steps, ((n0 + steps) // G) * G
    nv = nq if vres else n
    assert np.array_equal(c.k_codes[:, :, :nq], full.k_codes[:, :, :nq])
    assert np.array_equal(c.v_codes[:, :, :nv], full.v_codes[:, :, :nv])
    assert np.array_equal(c.v_meta[:, :, :nv], full.v_meta[:, :, :nv])
    if vres:
        assert np.array_equal(c.v_res[:, :, :n - nq], full.v_res[:, :, :n - nq])


@pytest.mark.parametrize("vg", [32, 64])
def test_attention_uses_each_channels_own_group(vg):
    """Values on exact per-group grids: the oracle's attention equals the softmax over
    the dequantized keys applied to the raw values."""
    rng = np.random.default_rng(vg)
    n, R = 70, 2
    v = _grid_values(rng, n, vg, 4)[None, None]
    k = _rand(rng, 1, 1, n, D)
    q = (rng.standard_normal((1, R, D)) / np.sqrt(D)).astype(np.float16)
    c = oracle.prefill(k, v, 32, 96, value_group=vg)
    kd, _ = oracle.dequantize(c)
    out = oracle.attention(c, q, 1.0)
    for h in range(R):
        s = kd[0, 0] @ q[0, h].astype(np.float64)
        p = np.exp(s - s.max())
        ref = (p / p.sum()) @ v[0, 0].astype(np.float64)
        assert np.allclose(out[0, h], ref, rtol=0, atol=1e-12)


def test_value_group_must_divide_d():
    k = np.zeros((1, 1, 4, D), np.float16)
    with pytest.raises(ValueError):
        oracle.prefill(k, k, 32, 32, value_group=48)
