"""Shared helpers of the GPU parity tests: run the CUDA path and the CPU oracle on
the same seeded fp16 inputs and compare.  Codes, scales and zeros must agree bit
for bit; attention outputs within ATOL of the oracle's fp64 attention over the
same dequantized cache."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_asymmetric_kv_gb300 import kivi

ATOL = 2e-3  # max |out_gpu - out_oracle|, the stated attention tolerance


def u32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def gpu_prefill(k: torch.Tensor, v: torch.Tensor, G: int, max_tokens: int) -> kivi.Cache:
    B, Hkv, n, D = k.shape
    c = kivi.Cache.allocate(B, Hkv, G, max_tokens)
    kivi.kivi_quantize_prefill(c, k.cuda(), v.cuda())
    return c


def assert_cache_equal(gpu: kivi.Cache, orc: oracle.Cache, heads=None) -> None:
    """Bit-exact comparison of every element the cache defines for n tokens."""
    n, G = orc.n, orc.G
    assert gpu.n_tokens == n
    ng, nq = n // G, (n // G) * G
    r = n - nq
    sel = (slice(None), slice(None)) if heads is None else heads
    pairs = [
        (u32(gpu.k_codes), orc.k_codes, nq, "k_codes"),
        (u32(gpu.k_meta), orc.k_meta, ng, "k_meta"),
        (u16(gpu.k_res), orc.k_res, r, "k_res"),
        (u32(gpu.v_codes), orc.v_codes, n, "v_codes"),
        (u32(gpu.v_meta), orc.v_meta, n, "v_meta"),
    ]
    for g_arr, o_arr, m, name in pairs:
        if heads is None:
            a, b = g_arr[:, :, :m], o_arr[:, :, :m]
        else:
            a = np.stack([g_arr[bb, hh, :m] for bb, hh in heads])
            b = np.stack([o_arr[bb, hh, :m] for bb, hh in heads])
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError(f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}")


def assert_close(out_gpu: torch.Tensor, ref: np.ndarray, atol: float = ATOL) -> float:
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= atol, f"max |gpu - oracle| = {worst:.3e} > {atol:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    return worst
