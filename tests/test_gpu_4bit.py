"""GPU parity of the 4-bit code width (oracle reading R10: 15 levels, 8 codes per
word), dense and paged, with and without the value residual, through the C ABI:
codes, scales, zeros and residuals bit for bit against the oracle; attention within
2e-3 of the oracle's fp64 attention over its own 4-bit cache.
"""
import math

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


def assert_equal4(gpu: kivi.Cache, orc: oracle.Cache, value_residual: bool) -> None:
    n, G = orc.n, orc.G
    assert gpu.n_tokens == n
    ng, nq = n // G, (n // G) * G
    r = n - nq
    nv = nq if value_residual else n
    pairs = [
        (u32(gpu.k_codes), orc.k_codes, nq, "k_codes"), (u32(gpu.k_meta), orc.k_meta, ng, "k_meta"),
        (u16(gpu.k_res), orc.k_res, r, "k_res"), (u32(gpu.v_codes), orc.v_codes, nv, "v_codes"),
        (u32(gpu.v_meta), orc.v_meta, nv, "v_meta"),
    ]
    if value_residual:
        pairs.append((u16(gpu.v_res), orc.v_res, r, "v_res"))
    for g_arr, o_arr, m, name in pairs:
        a, b = g_arr[:, :, :m], o_arr[:, :, :m]
        assert a.shape == b.shape, (name, a.shape, b.shape)
        if not np.array_equal(a, b):
            raise AssertionError(f"{name}: {int((a != b).sum())} mismatches")


CASES = [
    # name, B, Hq, Hkv, G, n
    ("mha-g32-tail", 2, 3, 3, 32, 32 * 9 + 17),
    ("gqa4-g64-tail", 2, 8, 2, 64, 64 * 5 + 40),
    ("gqa2-g32-even", 1, 4, 2, 32, 32 * 6),
    ("below-one-group", 2, 4, 1, 64, 63),
    ("long-many-splits", 1, 4, 1, 32, 32 * 200 + 31),
]


def _setup(case, seed, value_residual=False):
    _, B, Hq, Hkv, G, n = case
    wl = synth.small("q4", B, Hq, Hkv, G, n, seed, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T, value_residual, bits=4)
    gpu = kivi.Cache.allocate(B, Hkv, G, T, value_residual=value_residual, bits=4)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    return wl, pre, orc, gpu


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("value_residual", [False, True], ids=["plain", "vres"])
def test_4bit_prefill_bit_exact(case, value_residual):
    _, _, orc, gpu = _setup(case, 61, value_residual)
    torch.cuda.synchronize()
    assert_equal4(gpu, orc, value_residual)


def test_4bit_dequantize_debug_bit_exact():
    _, _, orc, gpu = _setup(CASES[0], 62)
    k32, v32 = oracle.dequantize(orc, np.float32)
    kg, vg = kivi.kivi_dequantize_debug(gpu)
    assert np.array_equal(kg.cpu().numpy().view(np.uint32), k32.view(np.uint32))
    assert np.array_equal(vg.cpu().numpy().view(np.uint32), v32.view(np.uint32))


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("value_residual", [False, True], ids=["plain", "vres"])
@pytest.mark.parametrize("sigma", [1.0, 0.37])
def test_4bit_attention_matches_oracle(case, value_residual, sigma):
    _, pre, orc, gpu = _setup(case, 63, value_residual)
    out = kivi.kivi_decode_attention(gpu, pre.q.cuda(), sigma)
    assert_close(out, oracle.attention(orc, pre.q.numpy(), sigma))


@pytest.mark.parametrize("Hq,Hkv,G,n0,steps,vres", [(8, 2, 32, 45, 70, False), (4, 4, 64, 10, 70, True),
                                                     (2, 1, 32, 0, 40, False)])
def test_4bit_decode_step_stream(Hq, Hkv, G, n0, steps, vres):
    wl = synth.small("q4s", 2, Hq, Hkv, G, n0, seed=64, steps=steps, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=G)
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), G, T, vres, bits=4)
    gpu = kivi.Cache.allocate(2, Hkv, G, T, value_residual=vres, bits=4)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    ws = kivi.workspace(gpu, Hq, n_tokens=T)
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        out = kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        assert_close(out, oracle.attention(orc, q.numpy(), 1.0))
    torch.cuda.synchronize()
    assert_equal4(gpu, orc, vres)


@pytest.mark.parametrize("vres", [False, True], ids=["plain", "vres"])
def test_4bit_paged_stream(vres):
    Hq, Hkv, G, P, steps = 4, 2, 32, 64, 50
    lens = [0, 31, 70, 5]
    B = len(lens)
    wl = synth.small("q4p", B, Hq, Hkv, G, max(lens), seed=65, steps=steps, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    maxp = math.ceil((max(lens) + steps + 1) / P)
    num_pages = B * maxp
    gpu = kivi.PagedCache.allocate(B, Hkv, G, P, maxp, num_pages, value_residual=vres, bits=4)
    bt = synth.block_table(B, maxp, num_pages, 65)
    gpu.block_table.copy_(bt)
    bt = bt.numpy()
    T = maxp * P
    orcs = []
    for b, n in enumerate(lens):
        kivi.kivi_paged_prefill(gpu, b, pre.k[b, :, :n].contiguous().cuda(), pre.v[b, :, :n].contiguous().cuda())
        orcs.append(oracle.prefill(pre.k[b:b + 1, :, :n].numpy(), pre.v[b:b + 1, :, :n].numpy(), G, T, vres,
                                   bits=4))
    ws = kivi.paged_workspace(gpu, Hq)
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        out = kivi.kivi_paged_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        ref = np.zeros((B, Hq, 128))
        for b in range(B):
            oracle.append(orcs[b], k_new[b:b + 1].numpy(), v_new[b:b + 1].numpy())
            ref[b] = oracle.attention(orcs[b], q[b:b + 1].numpy(), 1.0)[0]
        assert_close(out, ref)
    torch.cuda.synchronize()
    kc, km, vc, vm = (u32(t) for t in (gpu.k_codes, gpu.k_meta, gpu.v_codes, gpu.v_meta))
    for b, o in enumerate(orcs):
        n = o.n
        ng, nq = n // G, (n // G) * G
        nv = nq if vres else n
        t = np.arange(n)
        pages, rows = bt[b, t // P], t % P
        tg = np.arange(ng) * G
        assert np.array_equal(kc[pages[:nq], :, rows[:nq]].transpose(1, 0, 2), o.k_codes[0, :, :nq])
        assert np.array_equal(km[bt[b, tg // P], :, (tg % P) // G].transpose(1, 0, 2), o.k_meta[0, :, :ng])
        assert np.array_equal(vc[pages[:nv], :, rows[:nv]].transpose(1, 0, 2), o.v_codes[0, :, :nv])
        assert np.array_equal(vm[pages[:nv], :, rows[:nv]].transpose(1, 0), o.v_meta[0, :, :nv])
