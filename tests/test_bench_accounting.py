"""The bench's byte accounting against the cache layout itself (CPU only).

`bench.algorithmic_bytes` (one decode-attention call) and `bench.prefill_bytes` (one
prompt quantization) are the numerators of the reported roofline fractions.  Here
they are recomputed from the arrays of an oracle cache: the bytes of every code row,
scale/zero entry and residual slot the cache defines for n tokens (what a decode
reads, what a prefill writes), plus q and out or the fp16 prompt.  A wrong term in
either formula (a dropped residual, a meta row counted per token instead of per
group, the code width) fails here.
"""
import numpy as np
import pytest

import bench
import oracle


def _defined_bytes(c: oracle.Cache) -> int:
    n, G = c.n, c.G
    nq, ng, r = (n // G) * G, n // G, n - (n // G) * G
    nv = nq if c.v_res is not None else n
    parts = [c.k_codes[:, :, :nq], c.k_meta[:, :, :ng], c.k_res[:, :, :r], c.v_codes[:, :, :nv], c.v_meta[:, :, :nv]]
    if c.v_res is not None:
        parts.append(c.v_res[:, :, :r])
    return sum(int(p.nbytes) for p in parts)


CASES = [(2, 2, 32, 32 * 5 + 7), (1, 3, 64, 64 * 2 + 63), (2, 1, 32, 32 * 4), (1, 2, 64, 40)]


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("vres", [False, True])
@pytest.mark.parametrize("B,Hkv,G,n", CASES)
def test_byte_formulas_match_the_cache_layout(B, Hkv, G, n, vres, bits):
    rng = np.random.default_rng(n + G)
    k = rng.standard_normal((B, Hkv, n, 128)).astype(np.float16)
    v = rng.standard_normal((B, Hkv, n, 128)).astype(np.float16)
    c = oracle.prefill(k, v, G, ((n + G) // G) * G, value_residual=vres, bits=bits)
    cache = _defined_bytes(c)
    for R in (1, 2, 4):
        Hq = R * Hkv
        q_out = 2 * B * Hq * 128 * 2
        assert bench.algorithmic_bytes(B, Hq, Hkv, G, n, vres, bits) == cache + q_out
    assert bench.prefill_bytes(B, Hkv, G, n, vres, bits) == cache + k.nbytes + v.nbytes


@pytest.mark.parametrize("vg", [32, 64])
@pytest.mark.parametrize("B,Hkv,G,n", CASES)
def test_byte_formulas_with_value_channel_groups(B, Hkv, G, n, vg):
    """With value channel groups each value token carries 128 / vg {s, z} words."""
    rng = np.random.default_rng(n + G + vg)
    k = rng.standard_normal((B, Hkv, n, 128)).astype(np.float16)
    v = rng.standard_normal((B, Hkv, n, 128)).astype(np.float16)
    c = oracle.prefill(k, v, G, ((n + G) // G) * G, value_group=vg)
    assert c.v_meta.shape[-1] == 128 // vg
    cache = _defined_bytes(c)
    for R in (1, 2, 4):
        Hq = R * Hkv
        assert bench.algorithmic_bytes(B, Hq, Hkv, G, n, value_group=vg) == cache + 2 * B * Hq * 128 * 2
    assert bench.prefill_bytes(B, Hkv, G, n, value_group=vg) == cache + k.nbytes + v.nbytes
