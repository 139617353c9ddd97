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
from helpers import ATOL

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
    cases = [synth.small("na-gqa", 2, 8, 2, 32, 32 * 20 + 9, seed=41, factor_lo=30, factor_hi=100),
             synth.small("na-mha", 3, 4, 4, 64, 64 * 9 + 63, seed=42)]
    for wl in cases:
        c, pre = _cache(wl)
        for call in range(2):  # two calls in a row share the built-in array
            q = (pre.q if call == 0 else synth.make_step(wl, pre, call)[2]).cuda()
            ref = kivi.kivi_decode_attention(c, q, 1.0)
            got = kivi.kivi_decode_attention_noalloc(c, q, 1.0)
            torch.cuda.synchronize()
            assert torch.isfinite(got.float()).all()
            err = (got.float() - ref.float()).abs().max().item()
            assert err <= ATOL, (wl.name, call, err)


def test_noalloc_rejects_sizes_beyond_its_array():
    # many short sequences: one partial slot pair per query head, 512 * 32 of them
    d = kivi.make_dims(512, 8, 32, 64)
    need = kivi.kivi_decode_workspace_bytes(d, 32, 64)
    assert need > kivi.kivi_decode_attention_noalloc_max_workspace()
    fake = 1 << 20  # never dereferenced: the size check comes first
    cache = kivi.kivi_cache(fake, fake, fake, fake, fake, 0, 64)
    st = kivi.lib().kivi_decode_attention_noalloc(ctypes.byref(d), ctypes.byref(cache), fake, 32, 1.0, fake, None)
    assert st == kivi.KIVI_ERR_WORKSPACE
