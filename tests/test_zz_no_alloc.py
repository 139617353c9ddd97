"""The decode-attention entry point for callers that cannot allocate device memory.

kivi_decode_attention_noalloc takes its workspace from an array built into the
library (for serving loops that must not call cudaMalloc, or processes whose
device memory is reserved up front).  Its results must equal those of
kivi_decode_attention with a caller-allocated workspace, call after call, since
every call reuses the same array.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


def _cache(wl):
    pre = synth.make_prefill(wl)
    c = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, wl.capacity())
    kivi.kivi_quantize_prefill(c, pre.k.cuda(), pre.v.cuda())
    return c, pre


def test_noalloc_matches_the_workspace_entry_point_on_consecutive_calls():
    # Both entry points run the same kernels with the same split, so their outputs
    # agree bit for bit.  The array keeps the last call's partials: a case with many
    # pieces per head (a long context over one KV head) comes before cases with few,
    # so a piece read from a stale slot would show.
    cases = [synth.small("na-long", 1, 4, 1, 64, 64 * 2000 + 5, seed=43),
             synth.small("na-gqa", 2, 8, 2, 32, 32 * 20 + 9, seed=41, factor_lo=30, factor_hi=100),
             synth.small("na-mha", 3, 4, 4, 64, 64 * 9 + 63, seed=42)]
    for wl in cases:
        c, pre = _cache(wl)
        splits = kivi.kivi_decode_splits(c.dims, wl.Hq, c.n_tokens)
        assert kivi.kivi_decode_workspace_bytes(c.dims, wl.Hq, c.n_tokens) <= \
            kivi.kivi_decode_attention_noalloc_max_workspace()
        for call in range(2):  # two calls in a row share the built-in array
            q = (pre.q if call == 0 else synth.make_step(wl, pre, call)[2]).cuda()
            ref = kivi.kivi_decode_attention(c, q, 1.0)
            got = kivi.kivi_decode_attention_noalloc(c, q, 1.0)
            torch.cuda.synchronize()
            assert torch.isfinite(got.float()).all()
            assert torch.equal(got, ref), (wl.name, splits, call, (got.float() - ref.float()).abs().max().item())


def test_noalloc_rejects_sizes_beyond_its_array():
    # many short sequences: one partial slot pair per query head, 512 * 32 of them
    d = kivi.make_dims(512, 8, 32, 64)
    need = kivi.kivi_decode_workspace_bytes(d, 32, 64)
    assert need > kivi.kivi_decode_attention_noalloc_max_workspace()
    fake = 1 << 20  # never dereferenced: the size check comes first
    cache = kivi.kivi_cache(fake, fake, fake, fake, fake, 0, 64)
    st = kivi.lib().kivi_decode_attention_noalloc(ctypes.byref(d), ctypes.byref(cache), fake, 32, 1.0, fake, None)
    assert st == kivi.KIVI_ERR_WORKSPACE
