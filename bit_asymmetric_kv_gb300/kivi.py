"""Python binding of the C ABI in include/kivi.h (argument marshalling only).

Every step of the hot path runs in the CUDA library ``lib/libkivi.so``; this
module only converts torch tensors into device pointers and the current CUDA
stream into a ``cudaStream_t``.  PyTorch is used for device memory and streams.
There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libkivi.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "kivi.h")

STATUS = {0: "KIVI_OK", 1: "KIVI_ERR_ARG", 2: "KIVI_ERR_ALIGN", 3: "KIVI_ERR_UNSUPPORTED",
          4: "KIVI_ERR_CAPACITY", 5: "KIVI_ERR_WORKSPACE", 6: "KIVI_ERR_CUDA"}
KIVI_OK, KIVI_ERR_ARG, KIVI_ERR_ALIGN, KIVI_ERR_UNSUPPORTED, KIVI_ERR_CAPACITY, KIVI_ERR_WORKSPACE, KIVI_ERR_CUDA = range(7)


class KiviError(RuntimeError):
    def __init__(self, status: int, call: str):
        super().__init__(f"{call}: {STATUS.get(status, status)}")
        self.status = status


class kivi_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("G", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("value_residual", ctypes.c_int32), ("value_group", ctypes.c_int32),
                ("max_tokens", ctypes.c_int64)]


class kivi_cache(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_meta", ctypes.c_void_p), ("k_res", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("v_meta", ctypes.c_void_p), ("v_res", ctypes.c_void_p),
                ("n_tokens", ctypes.c_int64)]


class kivi_paged_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("G", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("value_residual", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int64)]


class kivi_paged_cache(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_meta", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_meta", ctypes.c_void_p), ("k_res", ctypes.c_void_p), ("v_res", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libkivi.so (built by ``bit_asymmetric_kv_gb300.build``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m bit_asymmetric_kv_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, D, C = ctypes.c_void_p, ctypes.POINTER(kivi_dims), ctypes.POINTER(kivi_cache)
        i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.kivi_buffer_bytes.argtypes = [D, ctypes.POINTER(sz)]
        L.kivi_quantize_prefill.argtypes = [D, C, P, P, i64, P]
        L.kivi_append_token.argtypes = [D, C, P, P, P]
        L.kivi_prefill_attention.argtypes = [D, C, P, i32, P, P, i64, ctypes.c_float, P, P]
        L.kivi_prefill_attention.restype = ctypes.c_int
        L.kivi_decode_splits.argtypes = [D, i32, i64]
        L.kivi_decode_workspace_bytes.argtypes = [D, i32, i64]
        L.kivi_decode_workspace_bytes.restype = sz
        L.kivi_decode_attention.argtypes = [D, C, P, i32, ctypes.c_float, P, P, sz, P]
        L.kivi_dequantize_debug.argtypes = [D, C, P, P, P]
        L.kivi_decode_attention_noalloc.argtypes = [D, C, P, i32, ctypes.c_float, P, P]
        L.kivi_decode_attention_noalloc.restype = ctypes.c_int
        L.kivi_decode_attention_noalloc_max_workspace.argtypes = []
        L.kivi_decode_attention_noalloc_max_workspace.restype = sz
        L.kivi_decode_fp16_workspace_bytes.argtypes = [i32, i32, i32, i32, i64]
        L.kivi_decode_fp16_workspace_bytes.restype = sz
        L.kivi_decode_attention_fp16.argtypes = [i32, i32, i32, i32, i64, P, P, P, ctypes.c_float, P, P, sz, P]
        L.kivi_decode_attention_fp16.restype = ctypes.c_int
        L.kivi_decode_step.argtypes = [D, C, P, P, P, i32, ctypes.c_float, P, P, sz, P]
        L.kivi_decode_step.restype = ctypes.c_int
        PD, PC = ctypes.POINTER(kivi_paged_dims), ctypes.POINTER(kivi_paged_cache)
        L.kivi_paged_buffer_bytes.argtypes = [PD, ctypes.POINTER(sz)]
        L.kivi_paged_prefill.argtypes = [PD, PC, i32, P, P, i64, P]
        L.kivi_paged_append_token.argtypes = [PD, PC, P, P, P]
        L.kivi_paged_decode_workspace_bytes.argtypes = [PD, i32]
        L.kivi_paged_decode_workspace_bytes.restype = sz
        L.kivi_paged_decode_attention.argtypes = [PD, PC, P, i32, ctypes.c_float, P, P, sz, P]
        L.kivi_paged_decode_step.argtypes = [PD, PC, P, P, P, i32, ctypes.c_float, P, P, sz, P]
        for name in ("kivi_paged_buffer_bytes", "kivi_paged_prefill", "kivi_paged_append_token",
                     "kivi_paged_decode_attention", "kivi_paged_decode_step"):
            getattr(L, name).restype = ctypes.c_int
        L.kivi_status_string.argtypes = [ctypes.c_int]
        L.kivi_status_string.restype = ctypes.c_char_p
        for name in ("kivi_buffer_bytes", "kivi_quantize_prefill", "kivi_append_token", "kivi_decode_splits",
                     "kivi_decode_attention", "kivi_dequantize_debug"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, call: str) -> None:
    if status != KIVI_OK:
        raise KiviError(status, call)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _f16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA float16 tensor")
    return t


def make_dims(B: int, Hkv: int, G: int, max_tokens: int, D: int = 128, bits: int = 2,
              value_residual: bool = False, value_group: int = 0) -> kivi_dims:
    return kivi_dims(B, Hkv, D, G, bits, int(value_residual), int(value_group), max_tokens)


def kivi_buffer_bytes(dims: kivi_dims) -> list[int]:
    out = (ctypes.c_size_t * 6)()
    _check(lib().kivi_buffer_bytes(ctypes.byref(dims), out), "kivi_buffer_bytes")
    return list(out)


@dataclass
class Cache:
    """Caller-owned device buffers of one quantized KV cache (layouts in include/kivi.h)."""

    dims: kivi_dims
    k_codes: torch.Tensor  # int32 [B, Hkv, T, D*bits/32]   (uint32 bit patterns)
    k_meta: torch.Tensor   # int32 [B, Hkv, T/G, D]    ({s, z} fp16 pairs)
    k_res: torch.Tensor    # fp16  [B, Hkv, G, D]
    v_codes: torch.Tensor  # int32 [B, Hkv, T, D*bits/32]
    v_meta: torch.Tensor   # int32 [B, Hkv, T], or [B, Hkv, T, D/vg] with value channel groups
    c: kivi_cache
    v_res: torch.Tensor | None = None  # fp16 [B, Hkv, G, D] with a value residual

    @property
    def n_tokens(self) -> int:
        return int(self.c.n_tokens)

    @classmethod
    def allocate(cls, B: int, Hkv: int, G: int, max_tokens: int, device="cuda", D: int = 128,
                 value_residual: bool = False, bits: int = 2, value_group: int = 0) -> "Cache":
        dims = make_dims(B, Hkv, G, max_tokens, D, bits=bits, value_residual=value_residual,
                         value_group=value_group)
        kivi_buffer_bytes(dims)  # validates the geometry
        T = max_tokens
        W = D * bits // 32  # words of a packed token row
        kc = torch.empty((B, Hkv, T, W), dtype=torch.int32, device=device)
        km = torch.empty((B, Hkv, T // G, D), dtype=torch.int32, device=device)
        kr = torch.empty((B, Hkv, G, D), dtype=torch.float16, device=device)
        vc = torch.empty((B, Hkv, T, W), dtype=torch.int32, device=device)
        vg = value_group or D
        vm = torch.empty((B, Hkv, T) if vg == D else (B, Hkv, T, D // vg), dtype=torch.int32, device=device)
        vr = torch.empty((B, Hkv, G, D), dtype=torch.float16, device=device) if value_residual else None
        c = kivi_cache(kc.data_ptr(), km.data_ptr(), kr.data_ptr(), vc.data_ptr(), vm.data_ptr(),
                       0 if vr is None else vr.data_ptr(), 0)
        return cls(dims, kc, km, kr, vc, vm, c, vr)


def kivi_quantize_prefill(cache: Cache, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
    """k, v: fp16 [B, Hkv, n, D] on the device."""
    _f16(k, "k"), _f16(v, "v")
    n = k.shape[2]
    _check(lib().kivi_quantize_prefill(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(k), _ptr(v), n,
                                       _stream(stream)), "kivi_quantize_prefill")


def kivi_prefill_attention(cache: Cache | None, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                           softmax_scale: float, out: torch.Tensor | None = None, dims: kivi_dims | None = None,
                           stream=None) -> torch.Tensor:
    """Causal prompt attention (q fp16 [B, Hq, n, D], k, v fp16 [B, Hkv, n, D] on the
    device) with the cache quantized from the same k, v in the same kernel; with
    cache=None (and the cache geometry in `dims`) the attention alone."""
    _f16(q, "q"), _f16(k, "k"), _f16(v, "v")
    if out is None:
        out = torch.empty_like(q)
    _f16(out, "out")
    B, Hq, n, D = q.shape
    if cache is not None:
        d, c = ctypes.byref(cache.dims), ctypes.byref(cache.c)
    else:
        if dims is None:
            raise ValueError("attention alone needs the geometry in `dims`")
        d, c = ctypes.byref(dims), None
    _check(lib().kivi_prefill_attention(d, c, _ptr(q), Hq, _ptr(k), _ptr(v), n, float(softmax_scale), _ptr(out),
                                        _stream(stream)), "kivi_prefill_attention")
    return out


def kivi_append_token(cache: Cache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """k_new, v_new: fp16 [B, Hkv, D] on the device."""
    _f16(k_new, "k_new"), _f16(v_new, "v_new")
    _check(lib().kivi_append_token(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new),
                                   _stream(stream)), "kivi_append_token")


def kivi_decode_splits(dims: kivi_dims, Hq: int, n_tokens: int) -> int:
    return int(lib().kivi_decode_splits(ctypes.byref(dims), Hq, n_tokens))


def kivi_decode_workspace_bytes(dims: kivi_dims, Hq: int, n_tokens: int) -> int:
    return int(lib().kivi_decode_workspace_bytes(ctypes.byref(dims), Hq, n_tokens))


def workspace(cache: Cache, Hq: int, n_tokens: int | None = None, device="cuda") -> torch.Tensor:
    """Allocate a decode workspace for this cache (uint8 device tensor)."""
    n = cache.n_tokens if n_tokens is None else n_tokens
    nbytes = kivi_decode_workspace_bytes(cache.dims, Hq, n)
    if nbytes == 0:
        raise KiviError(KIVI_ERR_ARG, "kivi_decode_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def kivi_decode_attention(cache: Cache, q: torch.Tensor, softmax_scale: float, out: torch.Tensor | None = None,
                          ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q: fp16 [B, Hq, D] -> out fp16 [B, Hq, D]."""
    _f16(q, "q")
    Hq = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(cache, Hq, device=q.device)
    _check(lib().kivi_decode_attention(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(q), Hq,
                                       float(softmax_scale), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)), "kivi_decode_attention")
    return out


def kivi_decode_attention_noalloc(cache: Cache, q: torch.Tensor, softmax_scale: float,
                                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kivi_decode_attention with the workspace taken from the library's built-in
    array (for callers that cannot allocate device memory); q: fp16 [B, Hq, D]."""
    _f16(q, "q")
    if out is None:
        out = torch.empty_like(q)
    _check(lib().kivi_decode_attention_noalloc(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(q), q.shape[1],
                                               float(softmax_scale), _ptr(out), _stream(stream)),
           "kivi_decode_attention_noalloc")
    return out


def kivi_decode_attention_noalloc_max_workspace() -> int:
    return int(lib().kivi_decode_attention_noalloc_max_workspace())


def kivi_decode_step(cache: Cache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor, softmax_scale: float,
                     out: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Append (k_new, v_new fp16 [B, Hkv, D]) then attend with q fp16 [B, Hq, D]."""
    _f16(k_new, "k_new"), _f16(v_new, "v_new"), _f16(q, "q")
    Hq = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(cache, Hq, n_tokens=cache.n_tokens + 1, device=q.device)
    _check(lib().kivi_decode_step(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new), _ptr(q),
                                  Hq, float(softmax_scale), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "kivi_decode_step")
    return out


def kivi_dequantize_debug(cache: Cache, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Dequantized cache as fp32 [B, Hkv, n_tokens, D] (keys, values)."""
    d = cache.dims
    shape = (d.B, d.Hkv, cache.n_tokens, d.D)
    k = torch.empty(shape, dtype=torch.float32, device=cache.k_codes.device)
    v = torch.empty(shape, dtype=torch.float32, device=cache.k_codes.device)
    _check(lib().kivi_dequantize_debug(ctypes.byref(d), ctypes.byref(cache.c), _ptr(k), _ptr(v), _stream(stream)),
           "kivi_dequantize_debug")
    return k, v


def kivi_decode_fp16_workspace_bytes(B: int, Hq: int, Hkv: int, n: int, D: int = 128) -> int:
    return int(lib().kivi_decode_fp16_workspace_bytes(B, Hq, Hkv, D, n))


def kivi_decode_attention_fp16(k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, softmax_scale: float,
                               out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                               stream=None) -> torch.Tensor:
    """Decode attention over an unquantized fp16 cache: k, v [B, Hkv, n, D], q [B, Hq, D]."""
    _f16(k, "k"), _f16(v, "v"), _f16(q, "q")
    B, Hkv, n, D = k.shape
    Hq = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        nbytes = kivi_decode_fp16_workspace_bytes(B, Hq, Hkv, n, D)
        if nbytes == 0:
            raise KiviError(KIVI_ERR_ARG, "kivi_decode_fp16_workspace_bytes")
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(lib().kivi_decode_attention_fp16(B, Hq, Hkv, D, n, _ptr(k), _ptr(v), _ptr(q), float(softmax_scale),
                                            _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "kivi_decode_attention_fp16")
    return out


def kivi_status_string(status: int) -> str:
    return lib().kivi_status_string(status).decode()


# ---------------------------------------------------------------------------------------
# paged cache
# ---------------------------------------------------------------------------------------
def make_paged_dims(B: int, Hkv: int, G: int, page_tokens: int, max_pages_per_seq: int, num_pages: int,
                    D: int = 128, bits: int = 2, value_residual: bool = False) -> kivi_paged_dims:
    return kivi_paged_dims(B, Hkv, D, G, bits, int(value_residual), page_tokens, max_pages_per_seq, num_pages)


def kivi_paged_buffer_bytes(dims: kivi_paged_dims) -> list[int]:
    out = (ctypes.c_size_t * 8)()
    _check(lib().kivi_paged_buffer_bytes(ctypes.byref(dims), out), "kivi_paged_buffer_bytes")
    return list(out)


@dataclass
class PagedCache:
    """Caller-owned device buffers of a paged cache (layouts in include/kivi.h): a
    page pool, per-sequence residual keys, the block table and the lengths."""

    dims: kivi_paged_dims
    k_codes: torch.Tensor      # int32 [num_pages, Hkv, P, D/16]
    k_meta: torch.Tensor       # int32 [num_pages, Hkv, P/G, D]
    v_codes: torch.Tensor      # int32 [num_pages, Hkv, P, D/16]
    v_meta: torch.Tensor       # int32 [num_pages, Hkv, P]
    k_res: torch.Tensor        # fp16  [B, Hkv, G, D]
    block_table: torch.Tensor  # int32 [B, max_pages_per_seq]
    seq_lens: torch.Tensor     # int32 [B]
    c: kivi_paged_cache
    v_res: torch.Tensor | None = None  # fp16 [B, Hkv, G, D] with a value residual

    @classmethod
    def allocate(cls, B: int, Hkv: int, G: int, page_tokens: int, max_pages_per_seq: int, num_pages: int,
                 device="cuda", D: int = 128, value_residual: bool = False, bits: int = 2) -> "PagedCache":
        dims = make_paged_dims(B, Hkv, G, page_tokens, max_pages_per_seq, num_pages, D, bits=bits,
                               value_residual=value_residual)
        kivi_paged_buffer_bytes(dims)  # validates the geometry
        P = page_tokens
        W = D * bits // 32  # words of a packed token row
        kc = torch.empty((num_pages, Hkv, P, W), dtype=torch.int32, device=device)
        km = torch.empty((num_pages, Hkv, P // G, D), dtype=torch.int32, device=device)
        vc = torch.empty((num_pages, Hkv, P, W), dtype=torch.int32, device=device)
        vm = torch.empty((num_pages, Hkv, P), dtype=torch.int32, device=device)
        kr = torch.empty((B, Hkv, G, D), dtype=torch.float16, device=device)
        vr = torch.empty((B, Hkv, G, D), dtype=torch.float16, device=device) if value_residual else None
        bt = torch.zeros((B, max_pages_per_seq), dtype=torch.int32, device=device)
        sl = torch.zeros((B,), dtype=torch.int32, device=device)
        c = kivi_paged_cache(kc.data_ptr(), km.data_ptr(), vc.data_ptr(), vm.data_ptr(), kr.data_ptr(),
                             0 if vr is None else vr.data_ptr(), bt.data_ptr(), sl.data_ptr())
        return cls(dims, kc, km, vc, vm, kr, bt, sl, c, vr)


def kivi_paged_prefill(cache: PagedCache, seq: int, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
    """Prompt of sequence `seq`: k, v fp16 [Hkv, n, D] on the device."""
    _f16(k, "k"), _f16(v, "v")
    _check(lib().kivi_paged_prefill(ctypes.byref(cache.dims), ctypes.byref(cache.c), seq, _ptr(k), _ptr(v),
                                    k.shape[1], _stream(stream)), "kivi_paged_prefill")


def kivi_paged_append_token(cache: PagedCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """k_new, v_new: fp16 [B, Hkv, D] on the device."""
    _f16(k_new, "k_new"), _f16(v_new, "v_new")
    _check(lib().kivi_paged_append_token(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new),
                                         _stream(stream)), "kivi_paged_append_token")


def kivi_paged_decode_workspace_bytes(dims: kivi_paged_dims, Hq: int) -> int:
    return int(lib().kivi_paged_decode_workspace_bytes(ctypes.byref(dims), Hq))


def paged_workspace(cache: PagedCache, Hq: int, device="cuda") -> torch.Tensor:
    nbytes = kivi_paged_decode_workspace_bytes(cache.dims, Hq)
    if nbytes == 0:
        raise KiviError(KIVI_ERR_ARG, "kivi_paged_decode_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def kivi_paged_decode_attention(cache: PagedCache, q: torch.Tensor, softmax_scale: float,
                                out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                                stream=None) -> torch.Tensor:
    """q: fp16 [B, Hq, D] -> out fp16 [B, Hq, D], each sequence over its own length."""
    _f16(q, "q")
    Hq = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = paged_workspace(cache, Hq, device=q.device)
    _check(lib().kivi_paged_decode_attention(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(q), Hq,
                                             float(softmax_scale), _ptr(out), _ptr(ws),
                                             ws.numel() * ws.element_size(), _stream(stream)),
           "kivi_paged_decode_attention")
    return out


def kivi_paged_decode_step(cache: PagedCache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                           softmax_scale: float, out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Append (k_new, v_new fp16 [B, Hkv, D]) at every sequence's length, attend with
    q fp16 [B, Hq, D], advance the lengths."""
    _f16(k_new, "k_new"), _f16(v_new, "v_new"), _f16(q, "q")
    Hq = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = paged_workspace(cache, Hq, device=q.device)
    _check(lib().kivi_paged_decode_step(ctypes.byref(cache.dims), ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new),
                                        _ptr(q), Hq, float(softmax_scale), _ptr(out), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)), "kivi_paged_decode_step")
    return out
