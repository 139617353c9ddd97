"""Every launch path of the dense decode attention against the CPU oracle.

Small contexts run without the workspace and the combine kernel: at most 8 units of
64 tokens per (batch, KV head) (with at most one CTA per SM) on one CTA of 8 warps
per (batch, KV head), one unit per warp, whose warps merge their partials in shared
memory; 9 to 16 units on a cluster per (batch, KV head) whose later CTAs write their
partials into the first one's shared memory: 4 CTAs of 4 warps while that many
clusters fit at once (a few dozen pairs), else 2 CTAs of 8 warps (up to about 76
pairs).  Larger contexts, or more (batch, KV head) pairs, take the persistent grid
with the workspace and the combine kernel.  The same shapes on both sides of
each boundary, with tails and residual keys, for every GQA ratio and both group
sizes, 4-bit codes and the value residual on the cluster path, through
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


def path(u):
    """The launch path of u units per (batch, KV head) at a few pairs: CTAs per pair."""
    return 1 if u <= 8 else 2 if u <= 16 else 0


# (B, Hq, Hkv, G, n): 8 units (one CTA), 9 and 16 (a cluster of two), 17 (persistent grid)
SHAPES = [
    (2, 2, 2, 32, 64 * 7 + 17), (2, 2, 2, 32, 64 * 8 + 17),
    (2, 2, 2, 32, 64 * 15 + 17), (2, 2, 2, 32, 64 * 16 + 17),
    (1, 4, 2, 64, 64 * 7 + 40), (1, 4, 2, 64, 64 * 8 + 40),
    (1, 4, 2, 64, 64 * 15 + 40), (1, 4, 2, 64, 64 * 16 + 40),
    (3, 8, 2, 32, 64 * 8), (3, 8, 2, 32, 64 * 9), (3, 8, 2, 32, 64 * 16), (3, 8, 2, 32, 64 * 17),
    (2, 4, 1, 32, 64 * 6 + 32 + 5), (2, 4, 1, 32, 64 * 7 + 32 + 5),
    (2, 4, 1, 32, 64 * 14 + 32 + 5), (2, 4, 1, 32, 64 * 15 + 32 + 5),
    (1, 1, 1, 32, 64 * 12),           # 12 units: the last CTA(s) of the cluster idle
    (32, 2, 2, 32, 64 * 12 + 5),      # 64 pairs at 13 units: 2-CTA clusters
    (16, 8, 4, 64, 64 * 10 + 40),     # 64 pairs, GQA 2, G = 64
    (48, 2, 2, 32, 64 * 12),          # 96 pairs at 12 units: more than fit as clusters
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


@pytest.mark.parametrize("bits,vres", [(4, False), (2, True), (4, True)], ids=["4bit", "vres", "4bit-vres"])
@pytest.mark.parametrize("B,Hq,Hkv,G,n", [(2, 8, 2, 32, 64 * 12 + 9), (1, 2, 1, 64, 64 * 15 + 40)],
                         ids=["r4-g32-u13", "r2-g64-u16"])
def test_cluster_path_variants(B, Hq, Hkv, G, n, bits, vres):
    """The two-CTA cluster path with 4-bit codes and with the value residual."""
    wl = synth.small("paths-var", B, Hq, Hkv, G, n, seed=71 + n % 89, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T, vres, bits=bits)
    gpu = kivi.Cache.allocate(B, Hkv, G, T, value_residual=vres, bits=bits)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    assert path(units(n, G)) == 2
    for sigma in (1.0, 0.61):
        out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), sigma)
        assert_close(out, oracle.attention(orc, pre.q.numpy(), sigma))


@pytest.mark.parametrize("Hq,Hkv,G,n0", [(2, 2, 32, 64 * 7 + 20), (8, 2, 64, 64 * 7 + 50), (4, 1, 32, 64 * 7 + 10),
                                         (2, 2, 32, 64 * 15 + 20), (8, 2, 64, 64 * 15 + 50)])
def test_decode_step_across_the_boundary(Hq, Hkv, G, n0):
    """A stream that grows from one launch path onto the next (the unit count passes
    8, or 16, as the context grows), with key-group flushes."""
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
        seen.add(path(units(n0 + step + 1, G)))
        out = kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        assert_close(out, oracle.attention(orc, q.numpy(), 1.0))
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)
    assert len(seen) == 2, "the stream crosses a boundary"
