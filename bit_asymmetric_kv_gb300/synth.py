"""Seeded synthetic KV-cache workloads (inputs only: no quantization arithmetic).

The workloads follow the KIVI page ("Makale Bulteni -- KIVI", cmlonder.com radar /
paper-to-prod, 2026-11-01): long-context Llama/Mistral decode (section "Makale
Bulteni", 32K/128K contexts), keys whose outliers sit in about 1% of the channels
and stay fixed over the whole sequence, values without outlier channels (section
"Iddia ve Gerceklik", 2nd paragraph).

Draw order (one CPU ``torch.Generator`` per workload, seed = workload.seed):
K, V, outlier channel indices, outlier factors, q.  Decode step i draws its
k_new, v_new, q from a second generator seeded from (seed, i), so any step can be
regenerated on its own.  Everything is drawn on the host; callers copy to the device.
Both the CUDA tests and the CPU oracle read these same fp16 arrays.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    G: int
    n: int                 # tokens in the cache after prefill (quantized groups + residual)
    steps: int = 0         # streaming decode steps after the prefill
    outliers: int = 2      # fixed outlier key channels per KV head (~1% of 128)
    factor_lo: float = 50.0
    factor_hi: float = 50.0
    seed: int = 0
    max_tokens: int = 0    # 0: n + steps (+ slack for benchmarks that keep appending)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    def capacity(self, extra: int = 0) -> int:
        t = self.max_tokens or (self.n + self.steps)
        t += extra
        return ((t + self.G - 1) // self.G) * self.G


# The five workloads of the hot path's measurement plan.
TINY = Workload("tiny-1head-n1024-G32", B=1, Hq=1, Hkv=1, D=128, G=32, n=1024, seed=0)
LLAMA2_7B_MHA = Workload("llama2-7b-mha-b8-n4113-G32", B=8, Hq=32, Hkv=32, D=128, G=32, n=4096 + 17,
                         factor_lo=30.0, factor_hi=100.0, seed=1)
MISTRAL_7B_GQA = Workload("mistral-7b-gqa-b16-n32808-G64", B=16, Hq=32, Hkv=8, D=128, G=64, n=32768 + 40, seed=2)
STREAMING = Workload("streaming-b64-h32-prefill8192-512steps-G32", B=64, Hq=32, Hkv=32, D=128, G=32, n=8192,
                     steps=512, factor_lo=30.0, factor_hi=100.0, seed=3)
LONG_GQA = Workload("long-gqa-b4-n131103-G32", B=4, Hq=32, Hkv=8, D=128, G=32, n=131072 + 31, seed=4)

CONFIGS = [TINY, LLAMA2_7B_MHA, MISTRAL_7B_GQA, STREAMING, LONG_GQA]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal_f16(shape, gen, chunk_rows: int = 1 << 22) -> torch.Tensor:
    """N(0,1) drawn in fp32 chunk by chunk (bounded host memory), stored as fp16."""
    out = torch.empty(shape, dtype=torch.float16)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, shape[-1]), generator=gen, dtype=torch.float32).to(torch.float16)
    return out


@dataclass
class Prefill:
    k: torch.Tensor            # [B, Hkv, n, D] fp16
    v: torch.Tensor            # [B, Hkv, n, D] fp16
    q: torch.Tensor            # [B, Hq, D] fp16
    outlier_idx: torch.Tensor  # [Hkv, outliers] int64
    outlier_fac: torch.Tensor  # [Hkv, outliers] fp32


def _apply_outliers(k: torch.Tensor, idx: torch.Tensor, fac: torch.Tensor) -> None:
    """Scale the fixed outlier channels of every token of k [B, Hkv, ..., D] in place."""
    for h in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            c = int(idx[h, j])
            col = k[:, h, ..., c].to(torch.float32) * float(fac[h, j])
            k[:, h, ..., c] = col.clamp(-65504.0, 65504.0).to(torch.float16)


def make_prefill(wl: Workload, n: int | None = None) -> Prefill:
    """Prompt K/V and the first query of workload ``wl`` (host fp16 tensors)."""
    n = wl.n if n is None else n
    gen = _gen(wl.seed)
    k = _normal_f16((wl.B, wl.Hkv, n, wl.D), gen)
    v = _normal_f16((wl.B, wl.Hkv, n, wl.D), gen)
    idx = torch.stack([torch.randperm(wl.D, generator=gen)[: wl.outliers] for _ in range(wl.Hkv)])
    u = torch.rand((wl.Hkv, wl.outliers), generator=gen, dtype=torch.float32)
    fac = wl.factor_lo + (wl.factor_hi - wl.factor_lo) * u
    q = (torch.randn((wl.B, wl.Hq, wl.D), generator=gen, dtype=torch.float32) / math.sqrt(wl.D)).to(torch.float16)
    _apply_outliers(k, idx, fac)
    return Prefill(k, v, q, idx, fac)


def make_step(wl: Workload, pre: Prefill, step: int):
    """(k_new [B,Hkv,D], v_new [B,Hkv,D], q [B,Hq,D]) fp16 for decode step ``step``."""
    gen = _gen(wl.seed * 1_000_003 + 7 + step)
    k = torch.randn((wl.B, wl.Hkv, wl.D), generator=gen, dtype=torch.float32).to(torch.float16)
    v = torch.randn((wl.B, wl.Hkv, wl.D), generator=gen, dtype=torch.float32).to(torch.float16)
    q = (torch.randn((wl.B, wl.Hq, wl.D), generator=gen, dtype=torch.float32) / math.sqrt(wl.D)).to(torch.float16)
    _apply_outliers(k, pre.outlier_idx, pre.outlier_fac)
    return k, v, q


def make_prompt_queries(wl: Workload, n: int | None = None) -> torch.Tensor:
    """fp16 [B, Hq, n, D]: the prompt's own queries, N(0,1)/sqrt(D) like the decode
    queries, drawn from a generator of their own (the prompt's K and V draws are
    unchanged)."""
    n = wl.n if n is None else n
    gen = _gen(wl.seed * 1_000_003 + 999_983)
    out = torch.empty((wl.B, wl.Hq, n, wl.D), dtype=torch.float16)
    flat = out.view(-1, wl.D)
    rows = 1 << 22
    for r0 in range(0, flat.shape[0], rows):
        r1 = min(flat.shape[0], r0 + rows)
        flat[r0:r1] = (torch.randn((r1 - r0, wl.D), generator=gen, dtype=torch.float32) / math.sqrt(wl.D)).to(
            torch.float16)
    return out


def small(name: str, B: int, Hq: int, Hkv: int, G: int, n: int, seed: int, steps: int = 0,
          factor_lo: float = 50.0, factor_hi: float = 50.0, outliers: int = 2) -> Workload:
    """A reduced workload with the same distributions, for oracle-sized parity cases."""
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=128, G=G, n=n, steps=steps, outliers=outliers,
                    factor_lo=factor_lo, factor_hi=factor_hi, seed=seed)


def block_table(B: int, max_pages_per_seq: int, num_pages: int, seed: int) -> torch.Tensor:
    """int32 [B, max_pages_per_seq]: distinct pages of a pool of num_pages, drawn in a
    seeded random order, so that consecutive positions of a sequence sit in scattered
    pages as in a serving engine's pool after many allocations and frees."""
    if B * max_pages_per_seq > num_pages:
        raise ValueError("the pool holds fewer pages than the block table needs")
    perm = torch.randperm(num_pages, generator=_gen(seed * 7_919 + 3))
    return perm[: B * max_pages_per_seq].reshape(B, max_pages_per_seq).to(torch.int32)
