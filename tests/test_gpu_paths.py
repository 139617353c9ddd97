"""Both launch paths of the dense decode attention against the CPU oracle.

Small contexts (at most one CTA per SM, at most 8 units of 64 tokens per (batch, KV
head): one unit per warp) run on one CTA per (batch, KV head) whose warps merge their partials in shared
memory; larger ones on the persistent grid with the workspace and the combine
kernel.  The same shapes just below and just above that boundary, with tails and
residual keys, for every GQA ratio and both group sizes, through
kivi_decode_attention and through kivi_decode_step across key-group flushes: the
outputs within 2e-3 of the oracle's fp64 attention, the cache bit for bit.
"""
import pytest
import torch

import oracle
from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi, synth
from helpers import assert_cache_equal, assert_close, gpu_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


def units(n, G):
    """Units of one (batch, KV head): 64-token blocks of quantized keys, plus the residual."""
    ng = n // G
    return (ng * G + 63) // 64 + (1 if n % G else 0)


# (B, Hq, Hkv, G, n): 8 units (small path) and 9 (persistent grid)
SHAPES = [
    (2, 2, 2, 32, 64 * 7 + 17), (2, 2, 2, 32, 64 * 8 + 17),
    (1, 4, 2, 64, 64 * 7 + 40), (1, 4, 2, 64, 64 * 8 + 40),
    (3, 8, 2, 32, 64 * 8), (3, 8, 2, 32, 64 * 9),
    (2, 4, 1, 32, 64 * 6 + 32 + 5), (2, 4, 1, 32, 64 * 7 + 32 + 5),
]


@pytest.mark.parametrize("B,Hq,Hkv,G,n", SHAPES, ids=[f"b{s[0]}-r{s[1] // s[2]}-g{s[3]}-u{units(s[4], s[3])}"
                                                      for s in SHAPES])
def test_decode_attention_on_both_paths(B, Hq, Hkv, G, n):
    wl = synth.small("paths", B, Hq, Hkv, G, n, seed=61 + n % 97, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity()
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    for sigma in (1.0, 0.61):
        out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), sigma)
        assert_close(out, oracle.attention(orc, pre.q.numpy(), sigma))


@pytest.mark.parametrize("Hq,Hkv,G,n0", [(2, 2, 32, 64 * 7 + 20), (8, 2, 64, 64 * 7 + 50), (4, 1, 32, 64 * 7 + 10)])
def test_decode_step_across_the_boundary(Hq, Hkv, G, n0):
    """A stream that starts on the small path and grows onto the persistent grid
    (the unit count passes 8 as the context grows), with key-group flushes."""
    steps = G + 40
    wl = synth.small("paths-step", 2, Hq, Hkv, G, n0, seed=67, steps=steps, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    ws = kivi.workspace(gpu, Hq, n_tokens=T)
    seen = set()
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        seen.add(units(n0 + step + 1, G) <= 8)
        out = kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        assert_close(out, oracle.attention(orc, q.numpy(), 1.0))
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)
    assert seen == {True, False}, "the stream crosses the boundary"
