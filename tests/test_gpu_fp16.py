"""GPU parity of the fp16-cache decode kernel (the comparison point of the 2-bit
cache) against the oracle's fp64 attention over the raw fp16 keys and values."""
import numpy as np
import pytest
import torch

import oracle
from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi, synth
from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kivi.lib()


@pytest.mark.parametrize("B,Hq,Hkv,n", [(2, 3, 3, 517), (2, 8, 2, 1000), (1, 4, 2, 33), (1, 4, 1, 1),
                                        (3, 4, 4, 15), (1, 8, 2, 16 * 300 + 5)])
@pytest.mark.parametrize("sigma", [1.0, 0.6])
def test_fp16_decode_matches_oracle(B, Hq, Hkv, n, sigma):
    wl = synth.small("fp16", B, Hq, Hkv, 32, n, seed=31, factor_lo=30, factor_hi=100)
    pre = synth.make_prefill(wl)
    out = kivi.kivi_decode_attention_fp16(pre.k.cuda(), pre.v.cuda(), pre.q.cuda(), sigma)
    assert_close(out, oracle.attention_raw(pre.k.numpy(), pre.v.numpy(), pre.q.numpy(), sigma))


def test_fp16_decode_long_context_gqa_sampled():
    """The long-context GQA shapes (4 x 8 KV heads, 131103 tokens): sampled heads."""
    wl = synth.LONG_GQA
    pre = synth.make_prefill(wl)
    out = kivi.kivi_decode_attention_fp16(pre.k.cuda(), pre.v.cuda(), pre.q.cuda(), 1.0)
    torch.cuda.synchronize()
    R = wl.Hq // wl.Hkv
    for b, kvh in [(0, 0), (3, 7), (1, 4)]:
        ref = np.stack([oracle.attention_raw_head(pre.k[b, kvh].numpy(), pre.v[b, kvh].numpy(),
                                                  pre.q[b, kvh * R + j].numpy(), 1.0) for j in range(R)])
        assert_close(out[b, kvh * R:(kvh + 1) * R], ref)


def test_fp16_workspace_too_small_is_rejected():
    wl = synth.small("fp16ws", 1, 2, 2, 32, 100, seed=32)
    pre = synth.make_prefill(wl)
    need = kivi.kivi_decode_fp16_workspace_bytes(1, 2, 2, 100)
    ws = torch.empty(need - 4, dtype=torch.uint8, device="cuda")
    with pytest.raises(kivi.KiviError) as e:
        kivi.kivi_decode_attention_fp16(pre.k.cuda(), pre.v.cuda(), pre.q.cuda(), 1.0, ws=ws)
    assert e.value.status == kivi.KIVI_ERR_WORKSPACE
