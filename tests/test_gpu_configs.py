"""Parity at the five full-size workloads, in the launch configuration the benchmark
uses.  The GPU runs the whole batch; the CPU oracle recomputes sampled (batch, KV
head) pairs one by one: their packed codes, scales, zeros and residual bit for bit,
and the attention output of every query head that reads them within 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi, synth
from helpers import assert_close, u16, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


def sample_heads(wl, k=4, seed=0):
    heads = {(0, 0), (wl.B - 1, wl.Hkv - 1)}
    rng = np.random.default_rng(seed)
    while len(heads) < min(k, wl.B * wl.Hkv):
        heads.add((int(rng.integers(wl.B)), int(rng.integers(wl.Hkv))))
    return sorted(heads)


def check_head(gpu: kivi.Cache, orc: oracle.Cache, b: int, kvh: int) -> None:
    n, G = orc.n, orc.G
    ng, nq = n // G, (n // G) * G
    r = n - nq
    d = gpu.dims
    assert np.array_equal(u32(gpu.k_codes[b, kvh, :nq]), orc.k_codes[0, 0, :nq])
    assert np.array_equal(u32(gpu.k_meta[b, kvh, :ng]), orc.k_meta[0, 0, :ng])
    assert np.array_equal(u16(gpu.k_res[b, kvh, :r]), orc.k_res[0, 0, :r])
    assert np.array_equal(u32(gpu.v_codes[b, kvh, :n]), orc.v_codes[0, 0, :n])
    assert np.array_equal(u32(gpu.v_meta[b, kvh, :n]), orc.v_meta[0, 0, :n])
    assert d.G == G


@pytest.mark.parametrize("idx", [0, 1, 2, 4], ids=lambda i: synth.CONFIGS[i].name)
def test_full_size_decode(idx):
    wl = synth.CONFIGS[idx]
    pre = synth.make_prefill(wl)
    T = wl.capacity()
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), 1.0)
    torch.cuda.synchronize()
    R = wl.Hq // wl.Hkv
    for b, kvh in sample_heads(wl):
        orc = oracle.prefill_head(pre.k[b, kvh].numpy(), pre.v[b, kvh].numpy(), wl.G, T)
        check_head(gpu, orc, b, kvh)
        ref = np.stack([oracle.attention_head(orc, 0, 0, pre.q[b, kvh * R + j].numpy(), 1.0) for j in range(R)])
        assert_close(out[b, kvh * R:(kvh + 1) * R], ref)


def test_full_size_streaming():
    """Prefill 8192 tokens (G=32) for 64 x 32 heads, then 512 append + decode steps."""
    wl = synth.STREAMING
    pre = synth.make_prefill(wl)
    T = wl.capacity()
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    heads = sample_heads(wl, k=3, seed=3)
    orcs = {h: oracle.prefill_head(pre.k[h[0], h[1]].numpy(), pre.v[h[0], h[1]].numpy(), wl.G, T) for h in heads}
    check_steps = {0, 1, 30, 31, 32, 255, wl.steps - 1}
    ws = kivi.workspace(gpu, wl.Hq, n_tokens=wl.n + wl.steps)
    for step in range(wl.steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        kivi.kivi_append_token(gpu, k_new.cuda(), v_new.cuda())
        for (b, kvh), orc in orcs.items():
            oracle.append(orc, k_new[b, kvh][None, None].numpy().copy(), v_new[b, kvh][None, None].numpy().copy())
        if step in check_steps:
            out = kivi.kivi_decode_attention(gpu, q.cuda(), 1.0, ws=ws)
            torch.cuda.synchronize()
            for (b, kvh), orc in orcs.items():
                ref = oracle.attention_head(orc, 0, 0, q[b, kvh].numpy(), 1.0)
                assert_close(out[b, kvh:kvh + 1], ref[None])
    torch.cuda.synchronize()
    for (b, kvh), orc in orcs.items():
        check_head(gpu, orc, b, kvh)
