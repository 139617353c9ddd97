"""CPU oracle for the KIVI asymmetric 2-bit KV cache -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or executes anything here, and this package
imports nothing from the product path.

The arithmetic lives in ``kivi_oracle.c`` (plain C, fp32 quantizer with IEEE
round-to-nearest-even and no FMA contraction, fp64 attention).  This module builds
it with gcc on first use and exposes numpy-level wrappers.  Every function follows
the page "Makale Bulteni -- KIVI" (cmlonder.com radar / paper-to-prod, 2026-11-01):
headline paragraph (keys per channel, values per token, asymmetric 2-bit) and
section "Iddia ve Gerceklik", paragraphs 2-3 (fixed outlier key channels; G-token
key groups with a full-precision residual buffer).  The readings R1-R11 are listed
at the top of ``kivi_oracle.c``; R9 is the variant with a value residual kept in
lock-step with the key residual (``value_residual=True``), R10 the 4-bit code
width (``bits=4``), R11 value channel groups of ``value_group`` < D channels,
R12 the causal full-precision prefill attention (``prefill_attention``).

Parity pins (tests/test_oracle_*.py) check this oracle against closed forms,
brute force and library routines, not against itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkivi_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kivi_oracle.c with gcc into oracle/_build/ (skipped when up to date)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            L.oracle_h2f.argtypes, L.oracle_h2f.restype = [ctypes.c_uint16], ctypes.c_float
            L.oracle_f2h.argtypes, L.oracle_f2h.restype = [ctypes.c_float], ctypes.c_uint16
            L.oracle_max_threads.restype = i32
            L.oracle_set_threads.argtypes, L.oracle_set_threads.restype = [i32], None
            L.oracle_quantize_group.argtypes = [P, i64, i64, i32, P, P, P]
            L.oracle_pack_row.argtypes = [P, i32, i32, P]
            L.oracle_prefill_head.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, P, P, P]
            L.oracle_append_head.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, P, P, P]
            L.oracle_append_head.restype = i64
            L.oracle_dequantize_head_f64.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, P, P, P]
            L.oracle_dequantize_head_f32.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, P, P, P]
            L.oracle_attention_head.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, P, P, f64, P]
            L.oracle_attention_head.restype = i32
            L.oracle_prefill.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, P, P, P, P, P, P, P, P]
            L.oracle_append.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, P, P, P, P, P, P, P, P]
            L.oracle_append.restype = i64
            L.oracle_attention.argtypes = [i32, i32, i32, i32, i32, i32, i32, i64, i64, P, P, P, P, P, P, P, f64,
                                           P]
            L.oracle_attention.restype = i32
            L.oracle_attention_raw_head.argtypes = [i32, i64, P, P, P, f64, P]
            L.oracle_attention_raw_head.restype = i32
            L.oracle_attention_raw.argtypes = [i32, i32, i32, i32, i64, P, P, P, f64, P]
            L.oracle_attention_raw.restype = i32
            L.oracle_prefill_attention_head.argtypes = [i32, i64, P, P, P, f64, P]
            L.oracle_prefill_attention_head.restype = i32
            L.oracle_prefill_attention.argtypes = [i32, i32, i32, i32, i64, P, P, P, f64, P]
            L.oracle_prefill_attention.restype = i32
            L.oracle_prefill_attention_rows.argtypes = [i32, i64, i64, P, P, P, P, f64, P]
            L.oracle_prefill_attention_rows.restype = i32
            _lib = L
        return _lib


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def set_threads(n: int) -> None:
    """Threads of the OpenMP loops over (batch, head); results do not depend on it."""
    lib().oracle_set_threads(int(n))


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _f16_bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 (or its uint16 bit pattern), got {a.dtype}")


# ----------------------------------------------------------------------------------
# scalar helpers
# ----------------------------------------------------------------------------------
def h2f(bits: int) -> float:
    return float(lib().oracle_h2f(int(bits)))


def f2h(x: float) -> int:
    return int(lib().oracle_f2h(float(x)))


def quantize_group(x, bits: int = 2) -> tuple[int, int, np.ndarray]:
    """Quantize one contiguous group of fp16 values -> (s16 bits, z16 bits, codes)."""
    xb = _f16_bits(np.asarray(x, dtype=np.float16) if not isinstance(x, np.ndarray) else x).ravel()
    xb = np.ascontiguousarray(xb)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(xb.size, np.uint8)
    lib().oracle_quantize_group(_ptr(xb), xb.size, 1, bits, _ptr(s), _ptr(z), _ptr(codes))
    return int(s[0]), int(z[0]), codes


def pack_row(codes, bits: int = 2) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    words = np.zeros(codes.size * bits // 32, np.uint32)
    lib().oracle_pack_row(_ptr(codes), codes.size, bits, _ptr(words))
    return words


# ----------------------------------------------------------------------------------
# cache state
# ----------------------------------------------------------------------------------
@dataclass
class Cache:
    """Packed cache in the canonical layout (all arrays C-contiguous numpy).

    k_codes [B,Hkv,T,D*bits/32] u32 | k_meta [B,Hkv,T//G,D] u32 {s | z<<16}
    k_res   [B,Hkv,G,D]   u16 (fp16 bits)
    v_codes [B,Hkv,T,D*bits/32] u32 | v_meta [B,Hkv,T] u32 {s | z<<16}
                                       ([B,Hkv,T,D/vg] with value groups of vg < D, R11)
    v_res   [B,Hkv,G,D]   u16, or None: the value residual of reading R9
    n       tokens held;  T = max_tokens;  bits = 2 (R1-R7) or 4 (R10).
    """

    B: int
    Hkv: int
    D: int
    G: int
    max_tokens: int
    k_codes: np.ndarray
    k_meta: np.ndarray
    k_res: np.ndarray
    v_codes: np.ndarray
    v_meta: np.ndarray
    n: int = 0
    v_res: np.ndarray | None = None
    bits: int = 2
    vg: int = 0  # value channel group (R11); 0 or D: one group per token (R5)

    @classmethod
    def empty(cls, B, Hkv, D, G, max_tokens, value_residual: bool = False, bits: int = 2,
              value_group: int | None = None):
        T = int(max_tokens)
        W = D * bits // 32
        vg = D if not value_group else int(value_group)
        if vg <= 0 or D % vg != 0:
            raise ValueError(f"value_group {value_group} must divide D = {D}")
        v_meta = np.zeros((B, Hkv, T), np.uint32) if vg == D else np.zeros((B, Hkv, T, D // vg), np.uint32)
        return cls(
            B, Hkv, D, G, T,
            np.zeros((B, Hkv, T, W), np.uint32),
            np.zeros((B, Hkv, T // G, D), np.uint32),
            np.zeros((B, Hkv, G, D), np.uint16),
            np.zeros((B, Hkv, T, W), np.uint32),
            v_meta,
            0,
            np.zeros((B, Hkv, G, D), np.uint16) if value_residual else None,
            bits,
            vg,
        )

    @property
    def value_group(self) -> int:
        return self.vg if self.vg else self.D

    def _vres_ptr(self, b=None, h=None):
        if self.v_res is None:
            return ctypes.c_void_p(0)
        return _ptr(self.v_res if b is None else self.v_res[b, h])

    def bufs(self):
        return [_ptr(self.k_codes), _ptr(self.k_meta), _ptr(self.k_res), _ptr(self.v_codes), _ptr(self.v_meta),
                self._vres_ptr()]

    def head(self, b: int, h: int):
        """Views of one (batch, KV head) slice."""
        return (self.k_codes[b, h], self.k_meta[b, h], self.k_res[b, h], self.v_codes[b, h], self.v_meta[b, h])


def prefill(k, v, G: int, max_tokens: int, value_residual: bool = False, bits: int = 2,
            value_group: int | None = None) -> Cache:
    """Quantize a prompt: k, v fp16 [B, Hkv, n, D] -> Cache holding n tokens."""
    kb, vb = _f16_bits(k), _f16_bits(v)
    B, Hkv, n, D = kb.shape
    if max_tokens < n:
        raise ValueError("max_tokens < n")
    c = Cache.empty(B, Hkv, D, G, max_tokens, value_residual, bits, value_group)
    lib().oracle_prefill(B, Hkv, D, G, bits, c.value_group, c.max_tokens, n, _ptr(kb), _ptr(vb), *c.bufs())
    c.n = n
    return c


def append(c: Cache, k_new, v_new) -> Cache:
    """Append one token per (batch, KV head): k_new, v_new fp16 [B, Hkv, D]. In place."""
    kb, vb = _f16_bits(k_new), _f16_bits(v_new)
    if c.n >= c.max_tokens:
        raise ValueError("cache full")
    c.n = int(lib().oracle_append(c.B, c.Hkv, c.D, c.G, c.bits, c.value_group, c.max_tokens, c.n, _ptr(kb),
                                  _ptr(vb), *c.bufs()))
    return c


def dequantize(c: Cache, dtype=np.float64, heads=None):
    """Dequantize the cache -> (K', V') [B, Hkv, n, D] in fp64 (default) or fp32.

    ``heads`` (optional list of (b, h)) restricts the work to those heads; other
    entries are left as NaN.
    """
    shape = (c.B, c.Hkv, c.n, c.D)
    kd = np.full(shape, np.nan, dtype)
    vd = np.full(shape, np.nan, dtype)
    fn = lib().oracle_dequantize_head_f64 if dtype == np.float64 else lib().oracle_dequantize_head_f32
    if dtype not in (np.float64, np.float32):
        raise TypeError("dtype must be float64 or float32")
    todo = heads if heads is not None else [(b, h) for b in range(c.B) for h in range(c.Hkv)]
    for b, h in todo:
        kc, km, kr, vc, vm = c.head(b, h)
        ko, vo = kd[b, h], vd[b, h]
        fn(c.D, c.G, c.bits, c.value_group, c.n, _ptr(kc), _ptr(km), _ptr(kr), _ptr(vc), _ptr(vm),
           c._vres_ptr(b, h), _ptr(ko), _ptr(vo))
    return kd, vd


def attention(c: Cache, q, sigma: float) -> np.ndarray:
    """fp64 attention of q fp16 [B, Hq, D] over the dequantized cache -> [B, Hq, D] fp64."""
    qb = _f16_bits(q)
    B, Hq, D = qb.shape
    out = np.zeros((B, Hq, D), np.float64)
    rc = lib().oracle_attention(B, Hq, c.Hkv, D, c.G, c.bits, c.value_group, c.max_tokens, c.n, *c.bufs(),
                                _ptr(qb), float(sigma), _ptr(out))
    if rc != 0:
        raise ValueError("oracle attention: empty cache or Hq % Hkv != 0")
    return out


def attention_head(c: Cache, b: int, kvh: int, q_row, sigma: float) -> np.ndarray:
    """fp64 attention of one query row (fp16 [D]) over KV head (b, kvh) -> [D] fp64."""
    qb = np.ascontiguousarray(_f16_bits(q_row))
    out = np.zeros(c.D, np.float64)
    kc, km, kr, vc, vm = c.head(b, kvh)
    rc = lib().oracle_attention_head(c.D, c.G, c.bits, c.value_group, c.n, _ptr(kc), _ptr(km), _ptr(kr), _ptr(vc),
                                     _ptr(vm), c._vres_ptr(b, kvh), _ptr(qb), float(sigma), _ptr(out))
    if rc != 0:
        raise ValueError("oracle attention: empty cache")
    return out


def prefill_head(k_head, v_head, G: int, max_tokens: int, value_residual: bool = False, bits: int = 2,
                 value_group: int | None = None):
    """Quantize one (batch, KV head) prompt k_head, v_head fp16 [n, D] -> 1x1 Cache."""
    kb = np.ascontiguousarray(_f16_bits(k_head))[None, None]
    vb = np.ascontiguousarray(_f16_bits(v_head))[None, None]
    return prefill(kb, vb, G, max_tokens, value_residual, bits, value_group)


def attention_raw(k, v, q, sigma: float) -> np.ndarray:
    """fp64 attention over an unquantized fp16 cache: k, v [B, Hkv, n, D], q [B, Hq, D]."""
    kb, vb, qb = _f16_bits(k), _f16_bits(v), _f16_bits(q)
    B, Hkv, n, D = kb.shape
    Hq = qb.shape[1]
    out = np.zeros((B, Hq, D), np.float64)
    if lib().oracle_attention_raw(B, Hq, Hkv, D, n, _ptr(kb), _ptr(vb), _ptr(qb), float(sigma), _ptr(out)) != 0:
        raise ValueError("oracle attention: empty cache or Hq % Hkv != 0")
    return out


def attention_raw_head(k_head, v_head, q_row, sigma: float) -> np.ndarray:
    """fp64 attention of one query row over one head's fp16 [n, D] keys and values."""
    kb = np.ascontiguousarray(_f16_bits(k_head))
    vb = np.ascontiguousarray(_f16_bits(v_head))
    qb = np.ascontiguousarray(_f16_bits(q_row))
    out = np.zeros(kb.shape[1], np.float64)
    if lib().oracle_attention_raw_head(kb.shape[1], kb.shape[0], _ptr(kb), _ptr(vb), _ptr(qb), float(sigma),
                                       _ptr(out)) != 0:
        raise ValueError("oracle attention: empty cache")
    return out


def prefill_attention(q, k, v, sigma: float) -> np.ndarray:
    """R12: causal fp64 attention of the prompt over itself, on the raw fp16 values.
    q [B, Hq, n, D], k, v [B, Hkv, n, D] fp16 -> out [B, Hq, n, D] fp64."""
    qb, kb, vb = _f16_bits(q), _f16_bits(k), _f16_bits(v)
    B, Hq, n, D = qb.shape
    Hkv = kb.shape[1]
    out = np.zeros((B, Hq, n, D), np.float64)
    if lib().oracle_prefill_attention(B, Hq, Hkv, D, n, _ptr(qb), _ptr(kb), _ptr(vb), float(sigma), _ptr(out)) != 0:
        raise ValueError("oracle prefill attention: empty prompt or Hq % Hkv != 0")
    return out


def prefill_attention_rows(q, k, v, rows, sigma: float) -> np.ndarray:
    """R12 at selected positions of one head: q, k, v fp16 [n, D], rows int [nr] ->
    out [nr, D] fp64 (the rows of prefill_attention for this head)."""
    qb, kb, vb = _f16_bits(q), _f16_bits(k), _f16_bits(v)
    n, D = qb.shape
    r = np.ascontiguousarray(np.asarray(rows, np.int64))
    out = np.zeros((len(r), D), np.float64)
    if lib().oracle_prefill_attention_rows(D, n, len(r), _ptr(r), _ptr(qb), _ptr(kb), _ptr(vb), float(sigma),
                                           _ptr(out)) != 0:
        raise ValueError("oracle prefill attention rows: empty prompt or a position outside it")
    return out
