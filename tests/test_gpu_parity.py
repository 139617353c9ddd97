"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Quantizer (KIVI page "Makale Bulteni -- KIVI", headline paragraph and section
"Iddia ve Gerceklik", paragraphs 2-3): codes, scales, zeros and the residual are
compared bit for bit.  Decode attention: max |out - oracle| <= 2e-3 against the
oracle's fp64 attention over its own dequantized cache.  Sizes span several
16-token tiles, several key groups, several context splits and a ragged tail.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi, synth
from helpers import ATOL, assert_cache_equal, assert_close, gpu_prefill, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


CASES = [
    # name, B, Hq, Hkv, G, n
    ("mha-g32-tail", 2, 3, 3, 32, 32 * 9 + 17),
    ("mha-g64-tail", 2, 2, 2, 64, 64 * 5 + 40),
    ("gqa4-g32", 2, 8, 2, 32, 32 * 12 + 31),
    ("gqa4-g64-even", 1, 8, 2, 64, 64 * 8),
    ("gqa2-g32", 2, 4, 2, 32, 32 * 7 + 5),
    ("one-group", 1, 4, 1, 32, 32),
    ("below-one-group", 2, 2, 1, 64, 63),
    ("single-token", 1, 1, 1, 32, 1),
    ("gqa4-g64-residual-only", 1, 4, 1, 64, 40),
]


def _inputs(name, B, Hq, Hkv, G, n, seed, factor=(30.0, 100.0)):
    wl = synth.small(name, B, Hq, Hkv, G, n, seed, factor_lo=factor[0], factor_hi=factor[1])
    return wl, synth.make_prefill(wl)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_cache_bit_exact(case):
    name, B, Hq, Hkv, G, n = case
    wl, pre = _inputs(*case, seed=11)
    T = wl.capacity(extra=G)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)


@pytest.mark.parametrize("case", CASES[:4], ids=[c[0] for c in CASES[:4]])
def test_dequantize_debug_bit_exact(case):
    name, B, Hq, Hkv, G, n = case
    wl, pre = _inputs(*case, seed=12)
    T = wl.capacity()
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    k32, v32 = oracle.dequantize(orc, np.float32)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    kg, vg = kivi.kivi_dequantize_debug(gpu)
    assert np.array_equal(kg.cpu().numpy().view(np.uint32), k32.view(np.uint32))
    assert np.array_equal(vg.cpu().numpy().view(np.uint32), v32.view(np.uint32))


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("sigma", [1.0, 0.37])
def test_decode_attention_matches_oracle(case, sigma):
    name, B, Hq, Hkv, G, n = case
    wl, pre = _inputs(*case, seed=13)
    T = wl.capacity()
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    ref = oracle.attention(orc, pre.q.numpy(), sigma)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), sigma)
    assert_close(out, ref)


@pytest.mark.parametrize("G,n0,steps", [(32, 0, 70), (32, 45, 40), (64, 100, 90)])
def test_streaming_append_equals_oracle_and_batch(G, n0, steps):
    """prefill(n0) + appends on the GPU == oracle streaming == oracle prefill(n0+steps);
    attention after every few steps within tolerance."""
    wl = synth.small("stream", 2, 8, 2, G, n0, seed=14, steps=steps, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    ks, vs = [pre.k], [pre.v]
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        kivi.kivi_append_token(gpu, k_new.cuda(), v_new.cuda())
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        ks.append(k_new[:, :, None])
        vs.append(v_new[:, :, None])
        if step % 7 == 0 or step == steps - 1:
            torch.cuda.synchronize()
            assert_cache_equal(gpu, orc)
            out = kivi.kivi_decode_attention(gpu, q.cuda(), 1.0, ws=ws)
            assert_close(out, oracle.attention(orc, q.numpy(), 1.0))
    batch = oracle.prefill(torch.cat(ks, 2).numpy(), torch.cat(vs, 2).numpy(), G, T)
    assert_cache_equal(gpu, batch)


def test_many_splits_long_context_small_batch():
    """B=1, one KV head, long context: many context splits merged by the combine."""
    wl = synth.small("long", 1, 4, 1, 32, 32 * 300 + 7, seed=15)
    pre = synth.make_prefill(wl)
    T = wl.capacity()
    d = kivi.make_dims(1, 1, 32, T)
    assert kivi.kivi_decode_splits(d, 4, wl.n) > 8
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), 32, T)
    gpu = gpu_prefill(pre.k, pre.v, 32, T)
    out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), 1.0)
    assert_close(out, oracle.attention(orc, pre.q.numpy(), 1.0))


@pytest.mark.parametrize("B,Hq,Hkv,G,n", [
    (2, 8, 2, 32, 32 * 40 + 9),   # every head split between warps
    (64, 64, 64, 32, 100),        # 4096 heads of 3 units: most heads held whole by one warp
    (1, 4, 1, 32, 32 * 300 + 7),  # one head over many warps
], ids=["split", "whole-heads", "one-long-head"])
def test_workspace_contents_do_not_matter_and_one_workspace_serves_many_calls(B, Hq, Hkv, G, n):
    """The workspace holds the split partials: filled with 0xFF bytes (NaN) beforehand
    and reused by consecutive calls, it gives the oracle's attention every time, and
    every output row is written."""
    wl = synth.small("wsfill", B, Hq, Hkv, G, n, seed=21)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    ref = oracle.attention(orc, pre.q.numpy(), 1.0)
    ws = torch.full((kivi.kivi_decode_workspace_bytes(gpu.dims, Hq, n),), 0xFF, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device="cuda")
        kivi.kivi_decode_attention(gpu, pre.q.cuda(), 1.0, out=out, ws=ws)
        assert_close(out, ref)


def test_decode_step_with_a_garbage_workspace():
    """kivi_decode_step with a workspace of 0xFF bytes (NaN) gives the oracle's result
    on every step."""
    wl = synth.small("stepws", 2, 8, 2, 32, 32 * 20 + 30, seed=22, steps=4, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=32)
    gpu = gpu_prefill(pre.k, pre.v, 32, T)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), 32, T)
    ws = torch.full((kivi.kivi_decode_workspace_bytes(gpu.dims, 8, T),), 0xFF, dtype=torch.uint8, device="cuda")
    for step in range(4):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        out = torch.full((2, 8, 128), float("nan"), dtype=torch.float16, device="cuda")
        kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, out=out, ws=ws)
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        assert_close(out, oracle.attention(orc, q.numpy(), 1.0))


def test_workspace_too_small_is_rejected_and_launches_nothing():
    wl = synth.small("ws", 1, 2, 2, 32, 100, seed=16)
    pre = synth.make_prefill(wl)
    gpu = gpu_prefill(pre.k, pre.v, 32, 128)
    need = kivi.kivi_decode_workspace_bytes(gpu.dims, 2, 100)
    assert need > 0
    ws = torch.empty(need - 4, dtype=torch.uint8, device="cuda")
    out = torch.full((1, 2, 128), 7.0, dtype=torch.float16, device="cuda")
    with pytest.raises(kivi.KiviError) as e:
        kivi.kivi_decode_attention(gpu, pre.q.cuda(), 1.0, out=out, ws=ws)
    assert e.value.status == kivi.KIVI_ERR_WORKSPACE
    assert torch.all(out == 7.0)


def test_append_on_full_cache_is_rejected():
    wl = synth.small("full", 1, 1, 1, 32, 64, seed=17)
    pre = synth.make_prefill(wl)
    gpu = gpu_prefill(pre.k, pre.v, 32, 64)
    k_new, v_new, _ = synth.make_step(wl, pre, 0)
    with pytest.raises(kivi.KiviError) as e:
        kivi.kivi_append_token(gpu, k_new.cuda(), v_new.cuda())
    assert e.value.status == kivi.KIVI_ERR_CAPACITY
    assert gpu.n_tokens == 64


def test_two_level_inputs_give_attention_of_the_raw_cache():
    """Inputs on a 2-level grid per group quantize exactly, so the GPU attention over
    the quantized cache matches fp64 attention over the raw fp16 inputs."""
    rng = np.random.default_rng(18)
    B, Hkv, n, G = 1, 2, 32 * 6 + 9, 32
    k = np.empty((B, Hkv, n, 128))
    for g0 in range(0, n, G):
        k[:, :, g0:g0 + G] = -1.0 + 3 * 0.25 * rng.integers(0, 2, size=(B, Hkv, min(G, n - g0), 128))
    v = -0.5 + 3 * 0.125 * rng.integers(0, 2, size=(B, Hkv, n, 128))
    k, v = k.astype(np.float16), v.astype(np.float16)
    q = (rng.standard_normal((B, 4, 128)) / np.sqrt(128)).astype(np.float16)
    gpu = gpu_prefill(torch.from_numpy(k), torch.from_numpy(v), G, 256)
    out = kivi.kivi_decode_attention(gpu, torch.from_numpy(q).cuda(), 1.0)
    ref = np.zeros((B, 4, 128))
    for h in range(4):
        K, V = k[0, h // 2].astype(np.float64), v[0, h // 2].astype(np.float64)
        s = K @ q[0, h].astype(np.float64)
        p = np.exp(s - s.max())
        ref[0, h] = (p / p.sum()) @ V
    assert_close(out, ref)


@pytest.mark.parametrize("Hq,Hkv,G,n0,steps", [(8, 2, 32, 45, 70), (4, 4, 64, 100, 70), (2, 1, 32, 0, 40)])
def test_decode_step_equals_append_then_attention(Hq, Hkv, G, n0, steps):
    """kivi_decode_step (append + attention, the attention overlapping the append)
    against the oracle's append followed by its attention, every step, across group
    flushes; the cache stays bit-exact."""
    wl = synth.small("step", 2, Hq, Hkv, G, n0, seed=19, steps=steps, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    gpu = gpu_prefill(pre.k, pre.v, G, T)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T)
    ws = kivi.workspace(gpu, Hq, n_tokens=T)
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        out = kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        assert_close(out, oracle.attention(orc, q.numpy(), 1.0))
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)


def test_decode_step_on_a_full_cache_is_rejected_before_any_launch():
    wl = synth.small("stepfull", 1, 2, 2, 32, 64, seed=20)
    pre = synth.make_prefill(wl)
    gpu = gpu_prefill(pre.k, pre.v, 32, 64)
    k_new, v_new, q = synth.make_step(wl, pre, 0)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(kivi.KiviError) as e:
        kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
    assert e.value.status == kivi.KIVI_ERR_CAPACITY
    assert gpu.n_tokens == 64
