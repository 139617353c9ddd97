"""GPU parity of the paged cache: the CUDA library against the CPU oracle, through
the C ABI.

The paged layout only moves token rows into pages of a pool; the method is the one
of the KIVI page ("Makale Bulteni -- KIVI", section "Iddia ve Gerceklik",
paragraphs 2-3), and the page's section "Kod ve Entegrasyon Haritasi", paragraph 3
is why a paged form is needed at all.  So every sequence b of a paged batch must
hold, row for row, what the oracle's dense cache holds for that sequence alone
(bit-exact codes, scales, zeros and residual), and its attention must match the
oracle's over its own length within 2e-3.  Sequences have different lengths,
including 0, below one group and across several pages; page ids are scattered.
"""
from __future__ import annotations

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


class Paged:
    """A paged batch on the GPU beside one oracle cache per sequence."""

    def __init__(self, Hq, Hkv, G, P, lens, seed, steps=0, spare_pages=3, unassigned=False):
        self.lens = list(lens)
        B = len(lens)
        self.B, self.Hq, self.Hkv, self.G, self.P = B, Hq, Hkv, G, P
        n_max = max(max(lens), 1)
        self.wl = synth.small("paged", B, Hq, Hkv, G, n_max, seed, steps=steps, factor_lo=30, factor_hi=100)
        self.pre = synth.make_prefill(self.wl)
        self.maxp = math.ceil((n_max + steps + 1) / P)
        num_pages = B * self.maxp + spare_pages
        self.cache = kivi.PagedCache.allocate(B, Hkv, G, P, self.maxp, num_pages)
        bt = synth.block_table(B, self.maxp, num_pages, seed)
        if unassigned:
            # pages beyond what each sequence ever holds are left unassigned (-1)
            for b in range(B):
                need = math.ceil((lens[b] + steps + 1) / P)
                bt[b, need:] = -1
        self.cache.block_table.copy_(bt)
        self.bt = bt.numpy()
        self.T = self.maxp * P
        self.orc = []
        for b, n in enumerate(lens):
            k = self.pre.k[b:b + 1, :, :n].contiguous()
            v = self.pre.v[b:b + 1, :, :n].contiguous()
            kivi.kivi_paged_prefill(self.cache, b, k[0].cuda(), v[0].cuda())
            self.orc.append(oracle.prefill(k.numpy(), v.numpy(), G, self.T))

    def step_inputs(self, step):
        return synth.make_step(self.wl, self.pre, step)

    def oracle_append(self, k_new, v_new, full=()):
        for b in range(self.B):
            if b in full:
                continue
            oracle.append(self.orc[b], k_new[b:b + 1].numpy(), v_new[b:b + 1].numpy())
            self.lens[b] += 1

    def reference(self, q, sigma):
        ref = np.zeros((self.B, self.Hq, 128))
        for b in range(self.B):
            if self.lens[b] > 0:
                ref[b] = oracle.attention(self.orc[b], q[b:b + 1].numpy(), sigma)[0]
        return ref

    def assert_cache_equal(self):
        torch.cuda.synchronize()
        assert self.cache.seq_lens.cpu().tolist() == self.lens
        kc, km, vc, vm = (u32(t) for t in (self.cache.k_codes, self.cache.k_meta, self.cache.v_codes,
                                           self.cache.v_meta))
        kr = u16(self.cache.k_res)
        G, P = self.G, self.P
        for b, n in enumerate(self.lens):
            o = self.orc[b]
            assert o.n == n
            ng = n // G
            nq, r = ng * G, n - ng * G
            t = np.arange(n)
            pages, rows = self.bt[b, t // P], t % P
            tg = np.arange(ng) * G
            gpages, gslots = self.bt[b, tg // P], (tg % P) // G
            got = {
                "k_codes": kc[pages[:nq], :, rows[:nq]].transpose(1, 0, 2),
                "k_meta": km[gpages, :, gslots].transpose(1, 0, 2),
                "k_res": kr[b, :, :r],
                "v_codes": vc[pages, :, rows].transpose(1, 0, 2),
                "v_meta": vm[pages, :, rows].transpose(1, 0),
            }
            want = {
                "k_codes": o.k_codes[0, :, :nq], "k_meta": o.k_meta[0, :, :ng], "k_res": o.k_res[0, :, :r],
                "v_codes": o.v_codes[0, :, :n], "v_meta": o.v_meta[0, :, :n],
            }
            for name in want:
                a, w = got[name].reshape(want[name].shape), want[name]
                if not np.array_equal(a, w):
                    bad = np.argwhere(a != w)
                    raise AssertionError(f"seq {b} (n={n}) {name}: {len(bad)} mismatches, first {bad[:4].tolist()}")


CASES = [
    # name, Hq, Hkv, G, P, lens
    ("mha-g32-p64", 2, 2, 32, 64, [0, 1, 31, 32, 33, 64, 65, 200, 517]),
    ("gqa4-g64-p128", 8, 2, 64, 128, [63, 64, 300, 0, 129, 640]),
    ("gqa2-g32-p256", 4, 2, 32, 256, [777, 5, 256, 257]),
    ("gqa4-g32-p64-short", 4, 1, 32, 64, [10, 20, 3]),
    ("mha-g64-p64", 3, 3, 64, 64, [64 * 7 + 40, 64, 1]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_paged_prefill_bit_exact(case):
    _, Hq, Hkv, G, P, lens = case
    pg = Paged(Hq, Hkv, G, P, lens, seed=31)
    pg.assert_cache_equal()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("sigma", [1.0, 0.37])
def test_paged_attention_matches_oracle(case, sigma):
    _, Hq, Hkv, G, P, lens = case
    pg = Paged(Hq, Hkv, G, P, lens, seed=32)
    q = pg.pre.q
    out = kivi.kivi_paged_decode_attention(pg.cache, q.cuda(), sigma)
    assert_close(out, pg.reference(q, sigma))
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.all(out[b] == 0)


@pytest.mark.parametrize("Hq,Hkv,G,P,lens,steps", [
    (8, 2, 32, 64, [0, 30, 61, 100, 127], 70),
    (4, 4, 64, 128, [50, 63, 190, 1], 80),
    (2, 1, 32, 256, [255, 31], 40),
])
def test_paged_decode_step_streaming(Hq, Hkv, G, P, lens, steps):
    """kivi_paged_decode_step every step: sequences flush their groups and cross page
    boundaries on different steps; attention against the oracle each step, the whole
    cache bit-exact at the end."""
    pg = Paged(Hq, Hkv, G, P, lens, seed=33, steps=steps, unassigned=True)
    ws = kivi.paged_workspace(pg.cache, Hq)
    for step in range(steps):
        k_new, v_new, q = pg.step_inputs(step)
        out = kivi.kivi_paged_decode_step(pg.cache, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0, ws=ws)
        pg.oracle_append(k_new, v_new)
        assert_close(out, pg.reference(q, 1.0))
    pg.assert_cache_equal()


def test_paged_append_token_then_attention():
    pg = Paged(4, 2, 32, 64, [31, 0, 95, 64], seed=34, steps=40)
    for step in range(40):
        k_new, v_new, q = pg.step_inputs(step)
        kivi.kivi_paged_append_token(pg.cache, k_new.cuda(), v_new.cuda())
        pg.oracle_append(k_new, v_new)
        if step % 9 == 0 or step == 39:
            out = kivi.kivi_paged_decode_attention(pg.cache, q.cuda(), 1.0)
            assert_close(out, pg.reference(q, 1.0))
    pg.assert_cache_equal()


def test_paged_full_sequence_drops_the_token_and_keeps_its_length():
    """A sequence at the block table's capacity takes no more tokens; the others go on."""
    pg = Paged(2, 2, 32, 64, [40, 10], seed=35, steps=0, spare_pages=0)
    cap = pg.T  # 64: one page per sequence
    assert cap == 64
    # fill sequence 0 to the capacity by prefilling it again with 64 tokens
    wl = synth.small("full", 1, 2, 2, 32, 64, seed=36)
    pre = synth.make_prefill(wl)
    kivi.kivi_paged_prefill(pg.cache, 0, pre.k[0].cuda(), pre.v[0].cuda())
    pg.orc[0] = oracle.prefill(pre.k.numpy(), pre.v.numpy(), 32, pg.T)
    pg.lens[0] = 64
    for step in range(3):
        k_new, v_new, q = pg.step_inputs(step)
        out = kivi.kivi_paged_decode_step(pg.cache, k_new.cuda(), v_new.cuda(), q.cuda(), 1.0)
        pg.oracle_append(k_new, v_new, full=(0,))
        assert_close(out, pg.reference(q, 1.0))
    pg.assert_cache_equal()


def test_paged_matches_dense_on_uniform_lengths():
    """Same prompts in the dense and the paged layout: identical codes, and both
    attentions within the tolerance of the oracle (the unit split differs)."""
    B, Hq, Hkv, G, n = 3, 8, 2, 32, 32 * 11 + 7
    pg = Paged(Hq, Hkv, G, 128, [n] * B, seed=37)
    dense = kivi.Cache.allocate(B, Hkv, G, pg.T)
    kivi.kivi_quantize_prefill(dense, pg.pre.k.cuda(), pg.pre.v.cuda())
    q = pg.pre.q.cuda()
    ref = pg.reference(pg.pre.q, 1.0)
    assert_close(kivi.kivi_paged_decode_attention(pg.cache, q, 1.0), ref)
    assert_close(kivi.kivi_decode_attention(dense, q, 1.0), ref)
    pg.assert_cache_equal()


def test_paged_many_sequences_few_units_and_large_batch():
    """Fewer 64-token units than warps (one warp per unit) and a batch of 200."""
    pg = Paged(2, 1, 32, 64, [5, 70, 3], seed=38)
    out = kivi.kivi_paged_decode_attention(pg.cache, pg.pre.q.cuda(), 1.0)
    assert_close(out, pg.reference(pg.pre.q, 1.0))
    rng = np.random.default_rng(39)
    lens = rng.integers(0, 400, size=200).tolist()
    pg = Paged(4, 2, 64, 64, lens, seed=39)
    out = kivi.kivi_paged_decode_attention(pg.cache, pg.pre.q.cuda(), 1.0)
    assert_close(out, pg.reference(pg.pre.q, 1.0))


def test_paged_workspace_too_small_is_rejected():
    pg = Paged(2, 2, 32, 64, [70, 3], seed=40)
    need = kivi.kivi_paged_decode_workspace_bytes(pg.cache.dims, 2)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    out = torch.full((2, 2, 128), 7.0, dtype=torch.float16, device="cuda")
    with pytest.raises(kivi.KiviError) as e:
        kivi.kivi_paged_decode_attention(pg.cache, pg.pre.q.cuda(), 1.0, out=out, ws=ws)
    assert e.value.status == kivi.KIVI_ERR_WORKSPACE
    assert torch.all(out == 7.0)


def test_paged_decode_step_replays_as_a_cuda_graph():
    """The paged step keeps its lengths on the device, so one captured step replays
    for every following token: parity with the oracle at each replay."""
    Hq = 8
    pg = Paged(Hq, 2, 32, 64, [30, 61, 100, 0], seed=43, steps=40, unassigned=True)
    ws = kivi.paged_workspace(pg.cache, Hq)
    k0, v0, q0 = pg.step_inputs(0)
    k_buf, v_buf, q_buf = k0.cuda(), v0.cuda(), q0.cuda()
    out = torch.empty_like(q_buf)
    # one call outside the capture: the library's first call on a device queries it
    kivi.kivi_paged_decode_step(pg.cache, k_buf, v_buf, q_buf, 1.0, out=out, ws=ws)
    pg.oracle_append(k0, v0)
    assert_close(out, pg.reference(q0, 1.0))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kivi.kivi_paged_decode_step(pg.cache, k_buf, v_buf, q_buf, 1.0, out=out, ws=ws)
    # capturing records the step without running it: the lengths did not move
    assert pg.cache.seq_lens.cpu().tolist() == pg.lens
    for step in range(1, 40):
        k_new, v_new, q = pg.step_inputs(step)
        k_buf.copy_(k_new)
        v_buf.copy_(v_new)
        q_buf.copy_(q)
        graph.replay()
        pg.oracle_append(k_new, v_new)
        assert_close(out, pg.reference(q, 1.0))
    pg.assert_cache_equal()
