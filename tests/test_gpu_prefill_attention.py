"""The fused prefill against the CPU oracle, through the C ABI.

kivi_prefill_attention computes the prompt's causal attention over its raw fp16 keys
and values (reading R12 of the oracle: KIVI page, section "Kod ve Entegrasyon
Haritasi", FlashAttention in the prefill) and writes the quantized cache from the
same tiles.  The outputs must lie within 2e-3 of the oracle's fp64 attention, the
cache must equal the oracle's prefill bit for bit (the cache kivi_quantize_prefill
writes), and the attention alone (no cache) must give the same outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi, synth
from helpers import assert_cache_equal, assert_close, u16, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


CASES = [
    # name, B, Hq, Hkv, G, n, bits, value_residual
    ("mha-g32-tail", 2, 2, 2, 32, 64 * 3 + 17, 2, 0),
    ("gqa2-g64-tail", 1, 4, 2, 64, 64 * 2 + 40, 2, 0),
    ("gqa4-g32-4bit", 1, 8, 2, 32, 64 * 2 + 31, 4, 0),
    ("mha-g32-value-residual", 2, 2, 2, 32, 100, 2, 1),
    ("below-one-group", 1, 4, 1, 32, 5, 2, 0),
    ("whole-tiles", 1, 2, 1, 64, 128, 2, 0),
    ("one-token", 1, 1, 1, 32, 1, 2, 0),
    ("gqa4-g64-4bit-value-residual", 1, 8, 2, 64, 64 * 3 + 1, 4, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("sigma", [1.0, 0.37])
def test_fused_prefill_matches_the_oracle(case, sigma):
    name, B, Hq, Hkv, G, n, bits, vr = case
    wl = synth.small(name, B, Hq, Hkv, G, n, seed=71, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    q = synth.make_prompt_queries(wl)
    T = wl.capacity(extra=G)
    gpu = kivi.Cache.allocate(B, Hkv, G, T, value_residual=bool(vr), bits=bits)
    out = kivi.kivi_prefill_attention(gpu, q.cuda(), pre.k.cuda(), pre.v.cuda(), sigma)
    torch.cuda.synchronize()
    assert gpu.n_tokens == n
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T, value_residual=bool(vr), bits=bits)
    if vr:
        # values of whole groups quantized, the last n mod G kept in fp16
        ng, nq = n // G, (n // G) * G
        for got, ref, m in [(u32(gpu.k_codes), orc.k_codes, nq), (u32(gpu.k_meta), orc.k_meta, ng),
                            (u16(gpu.k_res), orc.k_res, n - nq), (u32(gpu.v_codes), orc.v_codes, nq),
                            (u32(gpu.v_meta), orc.v_meta, nq), (u16(gpu.v_res), orc.v_res, n - nq)]:
            assert np.array_equal(got[:, :, :m], ref[:, :, :m])
    else:
        assert_cache_equal(gpu, orc)
    assert_close(out, oracle.prefill_attention(q.numpy(), pre.k.numpy(), pre.v.numpy(), sigma))
    alone = kivi.kivi_prefill_attention(None, q.cuda(), pre.k.cuda(), pre.v.cuda(), sigma, dims=gpu.dims)
    torch.cuda.synchronize()
    assert torch.equal(alone, out)


def test_fused_prefill_cache_serves_decode():
    """The fused prefill's cache, appended to and attended by the decode step, gives
    the oracle's decode attention (the two halves of the path meet)."""
    wl = synth.small("fused-then-decode", 2, 8, 2, 32, 64 * 4 + 9, seed=72, steps=40, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    q = synth.make_prompt_queries(wl)
    T = wl.capacity(extra=32)
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T)
    kivi.kivi_prefill_attention(gpu, q.cuda(), pre.k.cuda(), pre.v.cuda(), 1.0)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), wl.G, T)
    ws = kivi.workspace(gpu, wl.Hq, n_tokens=T)
    for step in range(wl.steps):
        k_new, v_new, qd = synth.make_step(wl, pre, step)
        out = kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), qd.cuda(), 1.0, ws=ws)
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        assert_close(out, oracle.attention(orc, qd.numpy(), 1.0))
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)


def _sampled_heads(B, Hkv, k, seed):
    rng = np.random.default_rng(seed)
    heads = {(0, 0), (B - 1, Hkv - 1)}
    while len(heads) < min(k, B * Hkv):
        heads.add((int(rng.integers(B)), int(rng.integers(Hkv))))
    return sorted(heads)


@pytest.mark.parametrize("idx", [0, 1, 2], ids=lambda i: synth.CONFIGS[i].name)
def test_fused_prefill_on_the_workload_prompts(idx):
    """The prompts of the tiny, Llama-2 and Mistral workloads: the cache of sampled KV
    heads bit for bit, and the outputs of every query head reading them within 2e-3
    (all positions for the shorter prompts; positions at tile edges, the middle and
    the end for the 32K-token one)."""
    wl = synth.CONFIGS[idx]
    pre = synth.make_prefill(wl)
    q = synth.make_prompt_queries(wl)
    T = wl.capacity()
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T)
    out = kivi.kivi_prefill_attention(gpu, q.cuda(), pre.k.cuda(), pre.v.cuda(), 1.0)
    torch.cuda.synchronize()
    R = wl.Hq // wl.Hkv
    n = wl.n
    rows = None if n <= 4200 else sorted({0, 1, 63, 64, 65, 4095, 4096, n // 2, n - 2, n - 1})
    for b, kvh in _sampled_heads(wl.B, wl.Hkv, 2, seed=idx + 3):
        k, v = pre.k[b, kvh].numpy(), pre.v[b, kvh].numpy()
        orc = oracle.prefill_head(k, v, wl.G, T)
        nq = (n // wl.G) * wl.G
        assert np.array_equal(u32(gpu.k_codes[b, kvh, :nq]), orc.k_codes[0, 0, :nq])
        assert np.array_equal(u32(gpu.k_meta[b, kvh, :n // wl.G]), orc.k_meta[0, 0, :n // wl.G])
        assert np.array_equal(u16(gpu.k_res[b, kvh, :n - nq]), orc.k_res[0, 0, :n - nq])
        assert np.array_equal(u32(gpu.v_codes[b, kvh, :n]), orc.v_codes[0, 0, :n])
        assert np.array_equal(u32(gpu.v_meta[b, kvh, :n]), orc.v_meta[0, 0, :n])
        for j in range(R) if rows is None else range(0, R, 3):
            h = kvh * R + j
            qh = q[b, h].numpy()
            if rows is None:
                ref = oracle.prefill_attention(qh[None, None], k[None, None], v[None, None], 1.0)[0, 0]
                assert_close(out[b, h], ref)
            else:
                ref = oracle.prefill_attention_rows(qh, k, v, rows, 1.0)
                assert_close(out[b, h, rows], ref)
