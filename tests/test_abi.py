"""The C-ABI library: it loads on a machine without a GPU, exports every entry point
include/kivi.h declares, and rejects bad arguments on the host, before any launch.
No test here touches device memory: every call fails validation first.
"""
import ctypes
import os
import re

import pytest

from bit_asymmetric_kv_gb300 import build as kbuild
from bit_asymmetric_kv_gb300 import kivi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kivi.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "kivi.h")).read()
    return re.findall(r"KIVI_API\s+[\w\s\*]+?\b(kivi_\w+)\s*\(", src)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    for n in ("kivi_quantize_prefill", "kivi_append_token", "kivi_decode_attention", "kivi_dequantize_debug",
              "kivi_buffer_bytes", "kivi_decode_workspace_bytes", "kivi_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code, name in kivi.STATUS.items():
        assert kivi.kivi_status_string(code) == name


def _dims(**kw):
    d = dict(B=2, Hkv=4, D=128, G=32, bits=2, value_residual=0, value_group=0, max_tokens=256)
    d.update(kw)
    return kivi.kivi_dims(d["B"], d["Hkv"], d["D"], d["G"], d["bits"], d["value_residual"], d["value_group"],
                          d["max_tokens"])


FAKE = 1 << 20  # an aligned, never dereferenced address


def _cache(n=0, align=0, v_res=FAKE):
    return kivi.kivi_cache(FAKE + align, FAKE, FAKE, FAKE, FAKE, v_res, n)


def test_buffer_bytes(L):
    out = kivi.kivi_buffer_bytes(_dims(B=3, Hkv=5, G=64, max_tokens=640))
    heads = 15
    assert out == [heads * 640 * 32, heads * 10 * 128 * 4, heads * 64 * 128 * 2, heads * 640 * 32, heads * 640 * 4, 0]
    out = kivi.kivi_buffer_bytes(_dims(B=3, Hkv=5, G=64, max_tokens=640, value_residual=1))
    assert out[5] == heads * 64 * 128 * 2
    out = kivi.kivi_buffer_bytes(_dims(B=3, Hkv=5, G=64, max_tokens=640, bits=4))
    assert out[0] == out[3] == heads * 640 * 64 and out[1] == heads * 10 * 128 * 4
    # value channel groups: 128 / vg {s, z} words per value token
    for vg, words in ((0, 1), (128, 1), (64, 2), (32, 4)):
        out = kivi.kivi_buffer_bytes(_dims(B=3, Hkv=5, G=64, max_tokens=640, value_group=vg))
        assert out[4] == heads * 640 * 4 * words and out[3] == heads * 640 * 32


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(bits=3), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(bits=8), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(G=16), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(B=0), kivi.KIVI_ERR_ARG),
    (dict(max_tokens=100), kivi.KIVI_ERR_ARG),   # not a multiple of G
    (dict(value_residual=2), kivi.KIVI_ERR_ARG),
    (dict(value_group=-32), kivi.KIVI_ERR_ARG),
    (dict(value_group=16), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(value_group=48), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(value_group=256), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(value_group=32, bits=4), kivi.KIVI_ERR_UNSUPPORTED),        # groups: 2-bit codes only
    (dict(value_group=64, value_residual=1), kivi.KIVI_ERR_UNSUPPORTED),  # groups: no value residual
    (dict(max_tokens=1 << 62), kivi.KIVI_ERR_UNSUPPORTED),                    # beyond 2^40 token rows
    (dict(B=1 << 20, Hkv=1 << 10, max_tokens=1 << 12), kivi.KIVI_ERR_UNSUPPORTED),  # 2^42 rows
    (dict(B=2147483647, Hkv=2147483647, max_tokens=32), kivi.KIVI_ERR_UNSUPPORTED),  # no overflow
])
def test_bad_dims(L, kw, status):
    d = _dims(**kw)
    out = (ctypes.c_size_t * 6)()
    assert L.kivi_buffer_bytes(ctypes.byref(d), out) == status
    c = _cache()
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(c), FAKE, FAKE, 10, None) == status
    assert c.n_tokens == 0


def test_prefill_checks(L):
    d = _dims()
    c = _cache()
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(c), None, FAKE, 10, None) == kivi.KIVI_ERR_ARG
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(c), FAKE + 2, FAKE, 10, None) == kivi.KIVI_ERR_ALIGN
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(c), FAKE, FAKE, 257, None) == kivi.KIVI_ERR_CAPACITY
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(c), FAKE, FAKE, -1, None) == kivi.KIVI_ERR_ARG
    bad = _cache(align=4)
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(bad), FAKE, FAKE, 10, None) == kivi.KIVI_ERR_ALIGN
    null = kivi.kivi_cache(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 0)
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(null), FAKE, FAKE, 10, None) == kivi.KIVI_ERR_ARG
    # a value residual needs its buffer, 16-byte aligned; without the variant it is not read
    dv = _dims(value_residual=1)
    assert L.kivi_quantize_prefill(ctypes.byref(dv), ctypes.byref(_cache(v_res=0)), FAKE, FAKE, 10,
                                   None) == kivi.KIVI_ERR_ARG
    assert L.kivi_quantize_prefill(ctypes.byref(dv), ctypes.byref(_cache(v_res=FAKE + 8)), FAKE, FAKE, 10,
                                   None) == kivi.KIVI_ERR_ALIGN
    c0 = _cache(v_res=0)
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(c0), None, None, 0, None) == kivi.KIVI_OK
    # n == 0 launches nothing and succeeds
    c.n_tokens = 7
    assert L.kivi_quantize_prefill(ctypes.byref(d), ctypes.byref(c), None, None, 0, None) == kivi.KIVI_OK
    assert c.n_tokens == 0


def test_append_capacity_leaves_state(L):
    d = _dims()
    c = _cache(n=256)
    assert L.kivi_append_token(ctypes.byref(d), ctypes.byref(c), FAKE, FAKE, None) == kivi.KIVI_ERR_CAPACITY
    assert c.n_tokens == 256
    c = _cache(n=3)
    assert L.kivi_append_token(ctypes.byref(d), ctypes.byref(c), FAKE + 8, FAKE, None) == kivi.KIVI_ERR_ALIGN
    assert c.n_tokens == 3


def test_decode_argument_checks(L):
    d = _dims()
    c = _cache(n=0)
    call = lambda c, Hq=8, q=FAKE, out=FAKE: L.kivi_decode_attention(  # noqa: E731
        ctypes.byref(d), ctypes.byref(c), q, Hq, 1.0, out, FAKE, 1 << 30, None)
    assert call(c) == kivi.KIVI_ERR_ARG                       # empty cache
    c = _cache(n=10)
    assert call(c, Hq=6) == kivi.KIVI_ERR_UNSUPPORTED         # Hq % Hkv != 0
    assert call(c, Hq=32) == kivi.KIVI_ERR_UNSUPPORTED        # Hq / Hkv = 8
    assert call(c, q=None) == kivi.KIVI_ERR_ARG
    assert call(c, out=FAKE + 6) == kivi.KIVI_ERR_ALIGN
    c = _cache(n=300)                                         # more tokens than capacity
    assert call(c) == kivi.KIVI_ERR_ARG
    assert L.kivi_decode_splits(ctypes.byref(d), 6, 10) == 0
    assert L.kivi_decode_workspace_bytes(ctypes.byref(d), 8, 0) == 0


def test_noalloc_reports_the_workspace_entry_points_statuses(L):
    """Invalid arguments get the same status from the allocation-free entry point as
    from kivi_decode_attention (its size check comes after every argument check)."""
    d = _dims()

    def both(c, Hq=8, q=FAKE, out=FAKE):
        ref = L.kivi_decode_attention(ctypes.byref(d), ctypes.byref(c), q, Hq, 1.0, out, FAKE, 1 << 30, None)
        got = L.kivi_decode_attention_noalloc(ctypes.byref(d), ctypes.byref(c), q, Hq, 1.0, out, None)
        return ref, got

    cases = [(_cache(n=0), {}), (_cache(n=300), {}), (_cache(n=257), {}), (_cache(n=-1), {}),
             (_cache(n=10), dict(Hq=6)), (_cache(n=10), dict(Hq=32)), (_cache(n=10), dict(q=None)),
             (_cache(n=10), dict(out=FAKE + 6)), (_cache(n=10, align=4), {}),
             (kivi.kivi_cache(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 10), {})]
    for c, kw in cases:
        ref, got = both(c, **kw)
        assert ref != kivi.KIVI_OK and got == ref, (c.n_tokens, kw, ref, got)
    assert both(_cache(n=300))[1] == kivi.KIVI_ERR_ARG  # n_tokens > max_tokens


# ---- paged cache: geometry and argument checks on the host --------------------------
def _pdims(**kw):
    d = dict(B=3, Hkv=4, D=128, G=32, bits=2, value_residual=0, page_tokens=64, max_pages_per_seq=5, num_pages=20)
    d.update(kw)
    return kivi.kivi_paged_dims(d["B"], d["Hkv"], d["D"], d["G"], d["bits"], d["value_residual"],
                                d["page_tokens"], d["max_pages_per_seq"], d["num_pages"])


def _pcache(align=0, bt_align=0, v_res=FAKE):
    return kivi.kivi_paged_cache(FAKE + align, FAKE, FAKE, FAKE, FAKE, v_res, FAKE + bt_align, FAKE)


def test_paged_buffer_bytes(L):
    out = kivi.kivi_paged_buffer_bytes(_pdims(B=3, Hkv=5, G=64, page_tokens=128, max_pages_per_seq=7, num_pages=11))
    rows = 11 * 5 * 128
    assert out == [rows * 32, rows // 64 * 128 * 4, rows * 32, rows * 4, 3 * 5 * 64 * 128 * 2, 3 * 7 * 4, 3 * 4, 0]
    out = kivi.kivi_paged_buffer_bytes(_pdims(B=3, Hkv=5, G=64, page_tokens=128, max_pages_per_seq=7, num_pages=11,
                                              value_residual=1))
    assert out[7] == 3 * 5 * 64 * 128 * 2


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(G=16), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(bits=3), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(page_tokens=96), kivi.KIVI_ERR_UNSUPPORTED),       # not a power of two
    (dict(page_tokens=32), kivi.KIVI_ERR_UNSUPPORTED),       # below one 64-token unit
    (dict(B=513), kivi.KIVI_ERR_UNSUPPORTED),
    (dict(max_pages_per_seq=1 << 25), kivi.KIVI_ERR_UNSUPPORTED),  # capacity beyond int32 positions
    (dict(B=0), kivi.KIVI_ERR_ARG),
    (dict(num_pages=0), kivi.KIVI_ERR_ARG),
    (dict(max_pages_per_seq=0), kivi.KIVI_ERR_ARG),
    (dict(value_residual=-1), kivi.KIVI_ERR_ARG),
    (dict(num_pages=1 << 40), kivi.KIVI_ERR_UNSUPPORTED),   # pool beyond 2^40 token rows
    (dict(num_pages=(1 << 62) + 1), kivi.KIVI_ERR_UNSUPPORTED),
])
def test_bad_paged_dims(L, kw, status):
    d = _pdims(**kw)
    out = (ctypes.c_size_t * 8)()
    assert L.kivi_paged_buffer_bytes(ctypes.byref(d), out) == status
    c = _pcache()
    assert L.kivi_paged_prefill(ctypes.byref(d), ctypes.byref(c), 0, FAKE, FAKE, 10, None) == status
    assert L.kivi_paged_append_token(ctypes.byref(d), ctypes.byref(c), FAKE, FAKE, None) == status
    assert L.kivi_paged_decode_workspace_bytes(ctypes.byref(d), 8) == 0


def test_paged_prefill_checks(L):
    d = _pdims()
    c = _pcache()
    pre = lambda seq=0, k=FAKE, n=10, c=c: L.kivi_paged_prefill(  # noqa: E731
        ctypes.byref(d), ctypes.byref(c), seq, k, FAKE, n, None)
    assert pre(seq=3) == kivi.KIVI_ERR_ARG            # sequence out of range
    assert pre(seq=-1) == kivi.KIVI_ERR_ARG
    assert pre(n=-1) == kivi.KIVI_ERR_ARG
    assert pre(n=5 * 64 + 1) == kivi.KIVI_ERR_CAPACITY
    assert pre(k=None) == kivi.KIVI_ERR_ARG
    assert pre(k=FAKE + 2) == kivi.KIVI_ERR_ALIGN
    assert pre(c=_pcache(align=4)) == kivi.KIVI_ERR_ALIGN
    assert pre(c=_pcache(bt_align=2)) == kivi.KIVI_ERR_ALIGN
    null = kivi.kivi_paged_cache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE)
    assert pre(c=null) == kivi.KIVI_ERR_ARG
    dv = _pdims(value_residual=1)
    assert L.kivi_paged_prefill(ctypes.byref(dv), ctypes.byref(_pcache(v_res=0)), 0, FAKE, FAKE, 10,
                                None) == kivi.KIVI_ERR_ARG
    assert L.kivi_paged_prefill(ctypes.byref(dv), ctypes.byref(_pcache(v_res=FAKE + 2)), 0, FAKE, FAKE, 10,
                                None) == kivi.KIVI_ERR_ALIGN


def test_paged_decode_argument_checks(L):
    d = _pdims()
    c = _pcache()
    att = lambda Hq=8, q=FAKE, out=FAKE: L.kivi_paged_decode_attention(  # noqa: E731
        ctypes.byref(d), ctypes.byref(c), q, Hq, 1.0, out, FAKE, 1 << 30, None)
    assert att(Hq=6) == kivi.KIVI_ERR_UNSUPPORTED
    assert att(Hq=32) == kivi.KIVI_ERR_UNSUPPORTED
    assert att(q=None) == kivi.KIVI_ERR_ARG
    assert att(out=FAKE + 6) == kivi.KIVI_ERR_ALIGN
    step = lambda k=FAKE, Hq=8: L.kivi_paged_decode_step(  # noqa: E731
        ctypes.byref(d), ctypes.byref(c), k, FAKE, FAKE, Hq, 1.0, FAKE, FAKE, 1 << 30, None)
    assert step(k=None) == kivi.KIVI_ERR_ARG
    assert step(k=FAKE + 4) == kivi.KIVI_ERR_ALIGN
    assert step(Hq=12) == kivi.KIVI_ERR_UNSUPPORTED
