"""GPU parity of the quantizers on adversarial fp16 inputs, bit for bit against the
oracle (KIVI page "Makale Bulteni -- KIVI", section "Iddia ve Gerceklik",
paragraphs 2-3: keys per channel over G-token groups, values per token, min/max
zero point and scale).

The key and value quantizers decide 2-bit codes by fp16 comparisons with
thresholds derived from the fp32 parameters, and fall back to the fp32 comparisons
where a threshold cannot be proven.  These inputs aim at every place that can go
wrong: values exactly on a threshold (ties) and one or two fp16 steps either side,
minima far below zero with thresholds that land next to zero among subnormals (the
fallback), constant channels and rows (scale 0), signed zeros, subnormals, +-65504,
and uniformly random finite fp16 bit patterns.  Each key channel of a group and each
value row gets one scenario.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi
from helpers import assert_cache_equal, u16, u32

pytestmark = pytest.mark.gpu

F16_MAX = 65504.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


def _f16(x):
    with np.errstate(over="ignore"):  # beyond 65504: inf, clipped by the callers
        return np.asarray(x, dtype=np.float64).astype(np.float16)


def _neighbours(x16: np.ndarray, steps=2) -> np.ndarray:
    """x and the fp16 values up to `steps` ulps either side of it."""
    out = [x16]
    up, dn = x16.copy(), x16.copy()
    for _ in range(steps):
        up = np.nextafter(up, np.float16(np.inf))
        dn = np.nextafter(dn, np.float16(-np.inf))
        out += [up, dn]
    return np.concatenate([np.atleast_1d(o) for o in out])


def _scenario(rng, L: int, kind: int) -> np.ndarray:
    """One channel (keys, L = G) or one row (values, L = 128) of fp16 values."""
    if kind == 0:  # random finite bit patterns (any exponent, either sign)
        b = rng.integers(0, 0x7C00, size=L).astype(np.uint16) | (rng.integers(0, 2, size=L).astype(np.uint16) << 15)
        return b.view(np.float16)
    if kind in (1, 2):
        if kind == 1:  # thresholds anywhere: values on them and next to them
            e = rng.uniform(-14, 15)
            mn = _f16(rng.uniform(-1, 1) * 2.0 ** e)
            mx = _f16(float(mn) + abs(float(mn)) * rng.uniform(0.01, 4) + 2.0 ** rng.uniform(-20, 3))
        else:  # minimum far below zero, first or second threshold next to zero
            a = rng.uniform(100, 9000)
            mn = _f16(-a)
            mx = _f16(-float(mn) * (5.0 if rng.random() < 0.5 else 1.0) + rng.uniform(0, 1))
        mx = np.float16(min(float(mx), F16_MAX))
        if float(mx) <= float(mn):
            mx = np.nextafter(mn, np.float16(np.inf))
        # the oracle's fp32 parameters, only to place inputs on and near the thresholds
        s32 = np.float32(np.float32(np.float32(mx) - np.float32(mn)) / np.float32(3))
        s = np.float32(np.float16(s32))
        cands = []
        for f in (0.5, 1.5, 2.5):
            y = np.float32(np.float32(mn) + np.float32(f) * s)
            cands.append(_neighbours(_f16(y), steps=2))
        cands.append(_f16(rng.uniform(-1, 1, size=8) * 2.0 ** -24 * 40))  # subnormals and zeros
        cands.append(np.array([0.0, -0.0], dtype=np.float16))
        c = np.concatenate(cands)
        c = c[(c.astype(np.float64) >= float(mn)) & (c.astype(np.float64) <= float(mx))]
        fill = _f16(rng.uniform(float(mn), float(mx), size=L))
        out = np.concatenate([[mn, mx], c, fill])[:L].astype(np.float16)
        rng.shuffle(out)
        return out
    if kind == 3:  # constant: scale 0
        c = rng.choice(np.array([0.0, -0.0, 2.0 ** -24, -3.5, 1000.0, F16_MAX, -F16_MAX], dtype=np.float16))
        return np.full(L, c, dtype=np.float16)
    if kind == 4:  # signed zeros and subnormals only
        b = rng.integers(0, 0x0400, size=L).astype(np.uint16) | (rng.integers(0, 2, size=L).astype(np.uint16) << 15)
        return b.view(np.float16)
    if kind == 5:  # the extremes
        return rng.choice(np.array([-F16_MAX, F16_MAX, 0.0, -0.0, 1.0], dtype=np.float16), size=L)
    # kind 6: two levels, minimum and maximum only
    lo = _f16(rng.uniform(-100, 100))
    hi = _f16(float(lo) + 2.0 ** rng.uniform(-10, 6))
    return np.where(rng.random(L) < 0.5, lo, hi).astype(np.float16)


KINDS = 7


def _adversarial(B, Hkv, n, G, seed):
    rng = np.random.default_rng(seed)
    k = np.empty((B, Hkv, n, 128), dtype=np.float16)
    v = np.empty((B, Hkv, n, 128), dtype=np.float16)
    for b in range(B):
        for h in range(Hkv):
            for g0 in range(0, n, G):
                L = min(G, n - g0)
                for c in range(128):
                    k[b, h, g0:g0 + L, c] = _scenario(rng, L, int(rng.integers(0, KINDS)))
            for t in range(n):
                v[b, h, t] = _scenario(rng, 128, int(rng.integers(0, KINDS)))
    return k, v


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("G,n", [(32, 32 * 12 + 7), (64, 64 * 6 + 33)])
def test_adversarial_prefill_bit_exact(G, n, bits):
    k, v = _adversarial(2, 2, n, G, seed=100 + G + bits)
    T = ((n + G) // G) * G
    orc = oracle.prefill(k, v, G, T, bits=bits)
    gpu = kivi.Cache.allocate(2, 2, G, T, bits=bits)
    kivi.kivi_quantize_prefill(gpu, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)


@pytest.mark.parametrize("bits", [2, 4])
def test_adversarial_append_and_flush_bit_exact(bits):
    """Token by token through kivi_append_token: values quantized at append, key
    groups at each flush."""
    G, n = 32, 32 * 3 + 5
    k, v = _adversarial(1, 2, n, G, seed=200 + bits)
    T = 128
    gpu = kivi.Cache.allocate(1, 2, G, T, bits=bits)
    for t in range(n):
        kivi.kivi_append_token(gpu, torch.from_numpy(np.ascontiguousarray(k[:, :, t])).cuda(),
                               torch.from_numpy(np.ascontiguousarray(v[:, :, t])).cuda())
    torch.cuda.synchronize()
    assert_cache_equal(gpu, oracle.prefill(k, v, G, T, bits=bits))


def _ties_and_far_thresholds(k, n, G):
    """Key elements exactly on a threshold (d == t), and thresholds that lie two or
    more fp16 steps above their round-down estimate (where the fp32 path decides)."""
    ties = far = 0
    for b in range(k.shape[0]):
        for h in range(k.shape[1]):
            for g0 in range(0, n, G):
                x = k[b, h, g0:g0 + G].astype(np.float32)
                mn, mx = x.min(0), x.max(0)
                s = np.float16(np.float32(mx - mn) / np.float32(3)).astype(np.float32)
                d = (x - mn).astype(np.float32)
                for f in (0.5, 1.5, 2.5):
                    t = (np.float32(f) * s).astype(np.float32)
                    ties += int(np.sum((d == t) & (s > 0)))
                    y = (mn + t).astype(np.float32)
                    c = y.astype(np.float16)
                    c = np.where(c.astype(np.float32) > y, np.nextafter(c, np.float16(-np.inf)), c)
                    c2 = np.nextafter(np.nextafter(c, np.float16(np.inf)), np.float16(np.inf))
                    far += int(np.sum((s > 0) & np.isfinite(c2.astype(np.float32))
                                      & ((c2.astype(np.float32) - mn).astype(np.float32) <= t)))
    return ties, far


def test_adversarial_inputs_reach_the_fallback_and_the_ties():
    """The scenarios do exercise what they aim at: key channels with values exactly on
    a threshold, and thresholds the fp16 estimate misses (the fp32 fallback)."""
    G, n = 32, 32 * 12
    k, _ = _adversarial(2, 2, n, G, seed=132)
    with np.errstate(over="ignore", invalid="ignore"):
        ties, far = _ties_and_far_thresholds(k, n, G)
    assert ties >= 20, ties
    assert far >= 1, far


@pytest.mark.parametrize("bits,vr", [(2, 0), (4, 0), (2, 1)])
@pytest.mark.parametrize("G,n", [(32, 32 * 12 + 7), (64, 64 * 6 + 33)])
def test_adversarial_fused_prefill_bit_exact(G, n, bits, vr):
    """The fused prefill (kivi_prefill_attention) quantizes its key and value tiles in
    shared memory with the same rule and fast forms: the same adversarial prompts give
    the oracle's cache bit for bit (GQA 2, so that one CTA per KV head quantizes)."""
    k, v = _adversarial(2, 2, n, G, seed=300 + G + bits + vr)
    T = ((n + G) // G) * G
    q = torch.from_numpy((np.random.default_rng(7).standard_normal((2, 4, n, 128)) * 0.05).astype(np.float16))
    orc = oracle.prefill(k, v, G, T, bits=bits, value_residual=bool(vr))
    gpu = kivi.Cache.allocate(2, 2, G, T, bits=bits, value_residual=bool(vr))
    kivi.kivi_prefill_attention(gpu, q.cuda(), torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 1.0)
    torch.cuda.synchronize()
    assert gpu.n_tokens == n
    if not vr:
        assert_cache_equal(gpu, orc)
        return
    # with a value residual: values of whole groups quantized, the last n mod G in fp16
    ng, nq = n // G, (n // G) * G
    for got, ref, m in [(u32(gpu.k_codes), orc.k_codes, nq), (u32(gpu.k_meta), orc.k_meta, ng),
                        (u16(gpu.k_res), orc.k_res, n - nq), (u32(gpu.v_codes), orc.v_codes, nq),
                        (u32(gpu.v_meta), orc.v_meta, nq), (u16(gpu.v_res), orc.v_res, n - nq)]:
        assert np.array_equal(got[:, :, :m], ref[:, :, :m])


@pytest.mark.parametrize("vg", [32, 64])
def test_adversarial_value_groups_bit_exact(vg):
    """Value channel groups (2-bit, the fp32 comparison form per group) on the same
    adversarial rows, through the prefill, token-by-token appends and the fused
    prefill: the oracle's codes and per-group {s, z} bit for bit."""
    G, n = 32, 32 * 4 + 9
    k, v = _adversarial(1, 2, n, G, seed=400 + vg)
    T = 192
    orc = oracle.prefill(k, v, G, T, value_group=vg)
    gpu = kivi.Cache.allocate(1, 2, G, T, value_group=vg)
    kivi.kivi_quantize_prefill(gpu, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    torch.cuda.synchronize()
    assert_cache_equal(gpu, orc)
    app = kivi.Cache.allocate(1, 2, G, T, value_group=vg)
    for t in range(n):
        kivi.kivi_append_token(app, torch.from_numpy(np.ascontiguousarray(k[:, :, t])).cuda(),
                               torch.from_numpy(np.ascontiguousarray(v[:, :, t])).cuda())
    torch.cuda.synchronize()
    assert_cache_equal(app, orc)
    fused = kivi.Cache.allocate(1, 2, G, T, value_group=vg)
    q = torch.from_numpy((np.random.default_rng(9).standard_normal((1, 2, n, 128)) * 0.05).astype(np.float16))
    kivi.kivi_prefill_attention(fused, q.cuda(), torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 1.0)
    torch.cuda.synchronize()
    assert_cache_equal(fused, orc)
