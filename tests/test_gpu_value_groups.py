"""Value channel groups on the GPU against the CPU oracle (reading R11: a value token
is quantized in D / vg groups of vg consecutive channels, each by the per-token rule,
its D / vg {s, z} words stored in group order; the KIVI page keeps the value error on
the token axis, section "Iddia ve Gerceklik", paragraph 2, and leaves open how many
channels share a scale).

The variant is built for dense 2-bit caches without a value residual, vg in {32, 64}.
Codes, scales and zeros must equal the oracle's bit for bit (prefill, append with key
flushes, the fused prefill, adversarial fp16 inputs); the dequantized cache must equal
the oracle's fp32 dequantization; attention through kivi_decode_attention and
kivi_decode_step must lie within 2e-3 of the oracle's fp64 attention for every GQA
ratio, both key group sizes, tails, contexts shorter than one key group and one token.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi, synth
from helpers import assert_cache_equal, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


def _prefill(pre, G, T, vg):
    B, Hkv = pre.k.shape[:2]
    gpu = kivi.Cache.allocate(B, Hkv, G, T, value_group=vg)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T, value_group=vg)
    return gpu, orc


# (B, Hq, Hkv, G, n)
SHAPES = [
    (2, 2, 2, 32, 64 * 5 + 17),      # MHA, a residual unit
    (1, 4, 2, 64, 64 * 4 + 40),      # GQA 2, G = 64
    (2, 8, 2, 32, 64 * 6 + 32 + 5),  # GQA 4, a trailing single key group and a residual
    (1, 4, 1, 32, 64 * 20),          # GQA 4, whole units only
    (2, 2, 1, 64, 40),               # shorter than one key group: the residual alone
    (1, 1, 1, 32, 1),                # one token
]


@pytest.mark.parametrize("vg", [32, 64])
@pytest.mark.parametrize("B,Hq,Hkv,G,n", SHAPES, ids=[f"b{s[0]}-r{s[1] // s[2]}-g{s[3]}-n{s[4]}" for s in SHAPES])
def test_prefill_dequant_and_attention(B, Hq, Hkv, G, n, vg):
    wl = synth.small("value-groups", B, Hq, Hkv, G, n, seed=81 + n % 89, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    gpu, orc = _prefill(pre, G, T, vg)
    torch.cuda.synchronize()
    assert tuple(gpu.v_meta.shape) == (B, Hkv, T, 128 // vg)
    assert_cache_equal(gpu, orc)
    # the dequantized cache: the oracle's fp32 dequantization, element for element
    kd, vd = kivi.kivi_dequantize_debug(gpu)
    ko, vo = oracle.dequantize(orc, np.float32)
    assert np.array_equal(kd.cpu().numpy(), ko) and np.array_equal(vd.cpu().numpy(), vo)
    for sigma in (1.0, 0.61):
        out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), sigma)
        assert_close(out, oracle.attention(orc, pre.q.numpy(), sigma))


@pytest.mark.parametrize("vg", [32, 64])
@pytest.mark.parametrize("Hq,Hkv,G,n0", [(2, 2, 32, 64 * 3 + 20), (8, 2, 64, 64 * 2 + 50), (4, 1, 32, 10)])
def test_decode_step_stream(Hq, Hkv, G, n0, vg):
    """Append + attention in one call for G + 24 steps: values quantized per group at
    append, key groups flushed, the cache bit for bit and every output within 2e-3."""
    steps = G + 24
    wl = synth.small("value-groups-step", 2, Hq, Hkv, G, n0, seed=83, steps=steps, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    gpu, orc = _prefill(pre, G, T, vg)
    ws = kivi.workspace(gpu, Hq, n_tokens=T)
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        out = kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        assert_close(out, oracle.attention(orc, q.numpy(), 1.0))
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)


@pytest.mark.parametrize("vg", [32, 64])
def test_append_token_by_token(vg):
    """kivi_append_token from an empty cache: every value row quantized per group at
    append, bit for bit (MHA, G = 32, three flushes and a tail)."""
    wl = synth.small("value-groups-append", 2, 2, 2, 32, 32 * 3 + 7, seed=84)
    pre = synth.make_prefill(wl)
    T = 128
    gpu = kivi.Cache.allocate(2, 2, 32, T, value_group=vg)
    for t in range(wl.n):
        kivi.kivi_append_token(gpu, pre.k[:, :, t].contiguous().cuda(), pre.v[:, :, t].contiguous().cuda())
    torch.cuda.synchronize()
    assert_cache_equal(gpu, oracle.prefill(pre.k.numpy(), pre.v.numpy(), 32, T, value_group=vg))


@pytest.mark.parametrize("vg", [32, 64])
def test_fused_prefill(vg):
    """kivi_prefill_attention quantizes its value tiles per group: the cache bit for
    bit, the prompt's attention within 2e-3 of the oracle's."""
    wl = synth.small("value-groups-fused", 1, 8, 2, 32, 64 * 3 + 9, seed=85, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    q = synth.make_prompt_queries(wl)
    T = wl.capacity(extra=32)
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T, value_group=vg)
    out = kivi.kivi_prefill_attention(gpu, q.cuda(), pre.k.cuda(), pre.v.cuda(), 1.0)
    torch.cuda.synchronize()
    assert_cache_equal(gpu, oracle.prefill(pre.k.numpy(), pre.v.numpy(), wl.G, T, value_group=vg))
    assert_close(out, oracle.prefill_attention(q.numpy(), pre.k.numpy(), pre.v.numpy(), 1.0))


def test_workload_shape_sampled_heads():
    """The Llama-2-7B decode shape (B8, H32, n = 4113, G32) with 32-channel value
    groups: the persistent grid over every head, the cache of sampled KV heads bit for
    bit against a per-head oracle, their query heads within 2e-3."""
    wl = synth.LLAMA2_7B_MHA
    pre = synth.make_prefill(wl)
    T = wl.capacity()
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T, value_group=32)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), 1.0)
    torch.cuda.synchronize()
    vmeta = gpu.v_meta.cpu().numpy().view(np.uint32)
    vcodes = gpu.v_codes.cpu().numpy().view(np.uint32)
    n = wl.n
    for b, h in [(0, 0), (3, 17), (7, 31)]:
        orc = oracle.prefill_head(pre.k[b, h].numpy(), pre.v[b, h].numpy(), wl.G, T, value_group=32)
        assert np.array_equal(vmeta[b, h, :n], orc.v_meta[0, 0, :n])
        assert np.array_equal(vcodes[b, h, :n], orc.v_codes[0, 0, :n])
        ref = oracle.attention_head(orc, 0, 0, pre.q[b, h].numpy(), 1.0)
        assert_close(out[b, h], ref)
