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
from helpers import assert_cache_equal, assert_close, u16, u32

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
    """Prefill 8192 tokens (G=32) for 64 x 32 heads, then 512 append + decode steps:
    every (batch, head) against the oracle's own stream at steps 0, 1, 30, 31, 32
    (around the first key-group flush), 255 and 511, and the whole final cache bit
    for bit (the oracle's batch entry points run over all 2048 heads)."""
    wl = synth.STREAMING
    pre = synth.make_prefill(wl)
    T = wl.capacity()
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    orc = oracle.prefill(pre.k.numpy(), pre.v.numpy(), wl.G, T)
    check_steps = {0, 1, 30, 31, 32, 255, wl.steps - 1}
    ws = kivi.workspace(gpu, wl.Hq, n_tokens=wl.n + wl.steps)
    checked = 0
    for step in range(wl.steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        kivi.kivi_append_token(gpu, k_new.cuda(), v_new.cuda())
        oracle.append(orc, k_new.numpy(), v_new.numpy())
        if step in check_steps:
            out = kivi.kivi_decode_attention(gpu, q.cuda(), 1.0, ws=ws)
            torch.cuda.synchronize()
            assert_close(out, oracle.attention(orc, q.numpy(), 1.0))
            checked += 1
    torch.cuda.synchronize()
    assert checked == len(check_steps)
    assert_cache_equal(gpu, orc)


def flush_neighbourhood(n0: int, G: int, steps: int, cycles: int = 2) -> set:
    """Steps of a stream that starts at n0 tokens: the first two, and the step
    before, at and after each of the first `cycles` key-group flushes (step i
    appends token n0 + i; it flushes when (n0 + i) mod G == G - 1), and the last."""
    first = (G - 1 - n0 % G) % G
    picked = {0, 1, steps - 1}
    for c in range(cycles):
        f = first + c * G
        picked |= {f - 1, f, f + 1}
    return {s for s in picked if 0 <= s < steps}


@pytest.mark.parametrize("idx,steps", [(1, 2 * 32 + 20), (3, 512)], ids=["llama2-7b-mha", "streaming"])
def test_full_size_decode_step(idx, steps):
    """kivi_decode_step, the call the benchmark times, at full size in the benchmark's
    launch configuration (one workspace sized for the whole run, the attention grid
    launched as a programmatic dependent of the append): every query head of sampled
    KV heads against the oracle's append followed by its attention, on the steps
    around two key-group flushes, and the sampled heads' final cache bit for bit."""
    wl = synth.CONFIGS[idx]
    pre = synth.make_prefill(wl)
    T = wl.capacity(extra=steps)
    gpu = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, T)
    kivi.kivi_quantize_prefill(gpu, pre.k.cuda(), pre.v.cuda())
    R = wl.Hq // wl.Hkv
    heads = sample_heads(wl, k=4, seed=idx + 11)
    orcs = {h: oracle.prefill_head(pre.k[h[0], h[1]].numpy(), pre.v[h[0], h[1]].numpy(), wl.G, T) for h in heads}
    nbytes = max(kivi.kivi_decode_workspace_bytes(gpu.dims, wl.Hq, n) for n in range(wl.n + 1, wl.n + steps + 1))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    check = flush_neighbourhood(wl.n, wl.G, steps)
    checked = 0
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        out = kivi.kivi_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        for (b, kvh), orc in orcs.items():
            oracle.append(orc, k_new[b, kvh][None, None].numpy().copy(), v_new[b, kvh][None, None].numpy().copy())
        if step in check:
            torch.cuda.synchronize()
            for (b, kvh), orc in orcs.items():
                ref = np.stack([oracle.attention_head(orc, 0, 0, q[b, kvh * R + j].numpy(), 1.0) for j in range(R)])
                assert_close(out[b, kvh * R:(kvh + 1) * R], ref)
            checked += 1
    torch.cuda.synchronize()
    assert gpu.n_tokens == wl.n + steps and checked == len(check) >= 8
    for (b, kvh), orc in orcs.items():
        check_head(gpu, orc, b, kvh)


def check_paged_head(gpu: kivi.PagedCache, bt: np.ndarray, orc: oracle.Cache, b: int, kvh: int) -> None:
    """Sequence b, KV head kvh of the paged pool, gathered row by row through the
    block table, against the oracle's dense cache of that head."""
    n, G, P = orc.n, orc.G, gpu.dims.page_tokens
    ng, nq = n // G, (n // G) * G
    t = np.arange(n)
    pages, rows = bt[b, t // P], t % P
    tg = np.arange(ng) * G
    kc = u32(gpu.k_codes[:, kvh])
    km = u32(gpu.k_meta[:, kvh])
    vc = u32(gpu.v_codes[:, kvh])
    vm = u32(gpu.v_meta[:, kvh])
    assert np.array_equal(kc[pages[:nq], rows[:nq]], orc.k_codes[0, 0, :nq])
    assert np.array_equal(km[bt[b, tg // P], (tg % P) // G], orc.k_meta[0, 0, :ng])
    assert np.array_equal(u16(gpu.k_res[b, kvh, :n - nq]), orc.k_res[0, 0, :n - nq])
    assert np.array_equal(vc[pages, rows], orc.v_codes[0, 0, :n])
    assert np.array_equal(vm[pages, rows], orc.v_meta[0, 0, :n])


@pytest.mark.parametrize("idx,P", [(1, 64), (2, 256)], ids=["llama2-p64", "mistral-gqa-p256"])
def test_full_size_paged_decode_steps(idx, P):
    """The full-size workload in the paged pool (scattered pages), in the benchmark's
    launch configuration: paged prefill of every sequence, attention over the prompt,
    then decode steps across a key-group flush; sampled heads against the oracle."""
    wl = synth.CONFIGS[idx]
    pre = synth.make_prefill(wl)
    steps = wl.G + 3
    maxp = -(-(wl.n + steps + 1) // P)
    num_pages = wl.B * maxp
    gpu = kivi.PagedCache.allocate(wl.B, wl.Hkv, wl.G, P, maxp, num_pages)
    bt = synth.block_table(wl.B, maxp, num_pages, wl.seed)
    gpu.block_table.copy_(bt)
    bt = bt.numpy()
    for b in range(wl.B):
        kivi.kivi_paged_prefill(gpu, b, pre.k[b].cuda(), pre.v[b].cuda())
    T = maxp * P
    R = wl.Hq // wl.Hkv
    heads = sample_heads(wl, k=3, seed=5)
    orcs = {h: oracle.prefill_head(pre.k[h[0], h[1]].numpy(), pre.v[h[0], h[1]].numpy(), wl.G, T) for h in heads}
    out = kivi.kivi_paged_decode_attention(gpu, pre.q.cuda(), 1.0)
    torch.cuda.synchronize()
    for (b, kvh), orc in orcs.items():
        check_paged_head(gpu, bt, orc, b, kvh)
        ref = np.stack([oracle.attention_head(orc, 0, 0, pre.q[b, kvh * R + j].numpy(), 1.0) for j in range(R)])
        assert_close(out[b, kvh * R:(kvh + 1) * R], ref)
    ws = kivi.paged_workspace(gpu, wl.Hq)
    for step in range(steps):
        k_new, v_new, q = synth.make_step(wl, pre, step)
        out = kivi.kivi_paged_decode_step(gpu, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        for (b, kvh), orc in orcs.items():
            oracle.append(orc, k_new[b, kvh][None, None].numpy().copy(), v_new[b, kvh][None, None].numpy().copy())
        if step in (0, steps - 4, steps - 3, steps - 1):
            torch.cuda.synchronize()
            for (b, kvh), orc in orcs.items():
                ref = np.stack([oracle.attention_head(orc, 0, 0, q[b, kvh * R + j].numpy(), 1.0) for j in range(R)])
                assert_close(out[b, kvh * R:(kvh + 1) * R], ref)
    torch.cuda.synchronize()
    assert gpu.seq_lens.cpu().tolist() == [wl.n + steps] * wl.B
    for (b, kvh), orc in orcs.items():
        check_paged_head(gpu, bt, orc, b, kvh)
