#!/usr/bin/env python3
"""Decode-step benchmark of the KIVI 2-bit KV cache on GB300.

Workload (default; --workload picks another of the five): streaming generation,
batch 64, 32 heads, head dim 128, an 8192-token fp16 prompt quantized with key
groups of G = 32 and 2-bit codes, then 512 decode steps, seeded synthetic fp16
K/V with fixed outlier key channels.  The prompt is quantized once (untimed); one
step is the whole hot path for one new token per sequence: append (value
quantization, residual write, group flush every G steps) + fused 2-bit decode
attention + split combine, through kivi_decode_step.  The context grows by one
token per step, as in the workload's schedule; after its 512 steps the schedule
starts again from the prompt (token count reset, residual keys restored, outside
the timed events).  The fixed-context workloads instead roll back every 64 steps,
so their context stays within n .. n + 64 tokens.  The metric is decode tokens/s
(batch / step time) with the attention call's achieved HBM GB/s against the
measured copy bandwidth.  L2 is flushed (256 MiB write) before every step,
outside the timed events.  With no flags the timed steps cover one schedule:
16 warm-up steps and 496 timed ones.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kivi|reference]
                  [--workload NAME] [--layout dense|paged [--page-tokens P] [--graph]]
                  [--value-residual] [--bits 2|4] [--compare-fp16] [--prefill-only] [--prefill-fused]

--layout paged runs the same workload through the paged cache (pages of P tokens
from one pool, scattered by a seeded permutation; lengths on the device); with
--graph each step is replayed from a CUDA graph captured once per input set.

--prefill-only times the prompt quantization alone (a separate JSON line);
--prefill-fused the fused prefill (the prompt's causal attention with the cache
quantized in the same kernel) against the attention alone and the separate
quantization pass (one JSON object).

--impl reference times the CPU oracle (plain C, the host's cores) on a bounded
sample of the same workload.  Under torchrun every rank runs an independent
replica (the path has no cross-GPU step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention tokens/s and achieved HBM GB/s (fraction of peak) on 2-bit KV"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
SHORT_CYCLE = 64  # steps between cache rollbacks of the fixed-context workloads


def cycle_of(wl) -> int:
    """Steps between cache rollbacks: the streaming workload runs its whole schedule
    (prefill, then `wl.steps` append + attend steps, the context growing by one token
    per step) before it starts again from the prompt; the fixed-context workloads
    stay within n .. n + 64 tokens."""
    return wl.steps if wl.steps else SHORT_CYCLE


def algorithmic_bytes(B: int, Hq: int, Hkv: int, G: int, n: int, value_residual: bool = False, bits: int = 2,
                      value_group: int = 0) -> int:
    """Bytes one decode-attention launch must move at context n (D = 128, c = 16*bits
    bytes of codes per token row, e = 4 * 128/vg bytes of value {s, z} per token):
    per (batch, KV head) nq*(c + 512/G) + r*256 + n*(c + e), plus q and out; with a
    value residual the last r values are fp16: nq*(c + e) + r*256 instead of n*(c + e)."""
    c = 16 * bits
    e = 4 * (128 // (value_group or 128))
    nq = (n // G) * G
    r = n - nq
    values = nq * (c + e) + r * 256 if value_residual else n * (c + e)
    per_head = nq * c + (nq // G) * 512 + r * 256 + values
    return B * Hkv * per_head + 2 * B * Hq * 128 * 2


def prefill_bytes(B: int, Hkv: int, G: int, n: int, value_residual: bool = False, bits: int = 2,
                  value_group: int = 0) -> int:
    """Bytes one prompt quantization must move (D = 128, c = 16*bits bytes of codes per
    token row, e = 4 * 128/vg bytes of value {s, z}): fp16 K and V read once
    (2 * n * 256 per (batch, KV head)), then written nq*(c + 512/G) + r*256 for the
    keys and n*(c + e) for the values (with a value residual nq*(c + e) + r*256)."""
    c = 16 * bits
    e = 4 * (128 // (value_group or 128))
    nq = (n // G) * G
    r = n - nq
    values = nq * (c + e) + r * 256 if value_residual else n * (c + e)
    return B * Hkv * (2 * n * 256 + nq * c + (nq // G) * 512 + r * 256 + values)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def profiled_traffic(kernel_sha: str, profile: str, workload: str, variant: str):
    """DRAM bytes per decode launch from the committed ncu summary `profile`, if it
    was taken on the current kernel source, on this workload and cache variant (else
    None)."""
    path = os.path.join(ROOT, "profiles", profile)
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    fields = {}
    for ln in lines:
        if ln.startswith("- ") and ":" in ln:
            k, v = ln[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if (fields.get("kernel_source_sha256") != kernel_sha or fields.get("workload") != workload
            or fields.get("variant") != variant):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def kernel_source_sha() -> str:
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_asymmetric_kv_gb300", "csrc")
    for name in ("kivi_decode.cu", "kivi_device.cuh", "kivi_internal.h"):  # the decode kernels' sources
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in (self.out or "").splitlines():
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"], p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def job_throughput(ms_local: float, tokens_per_step: int, world: int, device=None):
    """Whole-job figures of replicas that each decode `tokens_per_step` tokens per
    step: the step time is the max over ranks (the slowest replica bounds the job),
    throughput = tokens_per_step * world / that time.  Returns (ms, tokens/s)."""
    ms = float(ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, tokens_per_step * world / (ms / 1e3)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ----------------------------------------------------------------------------------------
def oracle_timing(wl, pre, steps: int, sample_heads: int, budget_s: float, value_residual: bool = False,
                  bits: int = 2, value_group: int = 0, single_thread: bool = True):
    """Time the oracle's decode step (append + fp64 attention over the dequantized
    cache) on `sample_heads` of the workload's KV heads; scale to the whole batch.
    Like the GPU loop, the cache is rolled back to the prompt every cycle_of(wl)
    steps (untimed)."""
    import copy

    import oracle
    from bit_asymmetric_kv_gb300 import synth

    sample_heads = min(sample_heads, wl.B * wl.Hkv)
    heads = [(i % wl.B, (i * 7) % wl.Hkv) for i in range(sample_heads)]
    cycle = cycle_of(wl)
    T = wl.capacity(extra=cycle + 64)
    k = np.stack([pre.k[b, h].numpy() for b, h in heads])[None]
    v = np.stack([pre.v[b, h].numpy() for b, h in heads])[None]
    c0 = oracle.prefill(k, v, wl.G, T, value_residual=value_residual, bits=bits,
                        value_group=value_group or None)  # untimed, like the GPU's prefill
    R = wl.Hq // wl.Hkv
    t_total, done = 0.0, 0
    c = c0
    for step in range(steps):
        if step % cycle == 0:
            c = copy.deepcopy(c0)
        k_new, v_new, q = synth.make_step(wl, pre, step % cycle)
        kn = np.stack([k_new[b, h].numpy() for b, h in heads])[None]
        vn = np.stack([v_new[b, h].numpy() for b, h in heads])[None]
        qs = np.stack([q[b, h * R + j].numpy() for b, h in heads for j in range(R)])[None]
        t0 = time.perf_counter()
        oracle.append(c, kn, vn)
        oracle.attention(c, qs, 1.0)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total > budget_s:
            break
    per_step = t_total / done * (wl.B * wl.Hkv / sample_heads)
    line = {"value": wl.B / per_step, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{sample_heads} of {wl.B * wl.Hkv} KV heads x {done} decode steps (append + fp64 attention), "
                      f"scaled to the full batch", "seconds": round(t_total, 3)}
    if single_thread and wl.B * wl.Hkv <= 256:
        # the same steps on one host thread, for the small workloads (a few seconds)
        cores = oracle.max_threads()
        oracle.set_threads(1)
        try:
            one = oracle_timing(wl, pre, steps, sample_heads, min(budget_s, 3.0), value_residual, bits, value_group,
                                single_thread=False)
        finally:
            oracle.set_threads(cores)
        line["single_thread"] = {"value": one["value"], "unit": UNIT, "sample": one["sample"]}
    return line


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from bit_asymmetric_kv_gb300 import synth

    pre = synth.make_prefill(wl)
    for w in range(args.warmup):  # untimed warm-up: the first call builds the oracle
        oracle_timing(wl, pre, 1, 4, 0.0)
    cb = oracle_timing(wl, pre, args.steps, 32, 60.0, args.value_residual, args.bits, args.value_group)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wl.B / cb["value"] * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": f"u{args.bits} codes, f16 inputs, f64 attention (CPU oracle)", "data": "synthetic",
            "config": {**workload_config(wl), **make_layout_config(args)}, "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def context_desc(wl, steps_run: int | None = None) -> str:
    """The contexts the timed steps attend over."""
    cycle = cycle_of(wl)
    if wl.steps:
        return (f"grows from {wl.n}: step i appends token {wl.n} + i and attends over {wl.n} + i + 1 tokens "
                f"(the schedule restarts from the {wl.n}-token prompt every {cycle} steps)")
    return f"{wl.n}..{wl.n + cycle} (cache rolled back every {cycle} steps)"


def workload_config(wl):
    cfg = {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D, "G": wl.G, "bits": 2,
           "context_tokens": context_desc(wl),
           "step": "append_token + decode_attention (one new token per sequence)",
           "l2": "flushed by a 256 MiB write before every step (outside the timed events)",
           "api": "kivi_decode_step (append + decode attention, the attention overlapping the append)",
           "parallelism": "replicas (one independent cache per GPU)", "layout": "dense"}
    return cfg


# ----------------------------------------------------------------------------------------
# cache layouts: the same workload in the dense cache or in a paged pool
# ----------------------------------------------------------------------------------------
class DenseLayout:
    """The dense cache [B][Hkv][max_tokens]: kivi_decode_step / kivi_decode_attention."""

    profile_prefix = "decode_attention_"
    kernel = "kivi_decode_attention (decode_kernel + combine_kernel)"

    def __init__(self, wl, pre, dev, value_residual=False, bits=2, value_group=0):
        from bit_asymmetric_kv_gb300 import kivi

        self.wl, self.kivi = wl, kivi
        self.cache = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, wl.capacity(extra=cycle_of(wl) + 64), device=dev,
                                         value_residual=value_residual, bits=bits, value_group=value_group)
        kivi.kivi_quantize_prefill(self.cache, pre.k.to(dev), pre.v.to(dev))
        self.n0 = self.cache.n_tokens
        self.res0 = self.cache.k_res.clone()
        self.vres0 = None if self.cache.v_res is None else self.cache.v_res.clone()
        self.ws = cycle_workspace(self.cache, wl, self.n0, dev)

    def rollback(self):
        self.cache.k_res.copy_(self.res0)
        if self.vres0 is not None:
            self.cache.v_res.copy_(self.vres0)
        self.cache.c.n_tokens = self.n0

    def step(self, k, v, q, out, stream):
        """Returns the number of kernels the step launched."""
        n = self.cache.n_tokens
        self.kivi.kivi_decode_step(self.cache, k, v, q, 1.0, out=out, ws=self.ws, stream=stream)
        # append (+ key group flush, and value rows with a value residual, every G
        # steps), decode attention, combine
        flush = (n % self.wl.G) + 1 == self.wl.G
        return 1 + (0 if not flush else (2 if self.vres0 is not None else 1)) + 2

    def attention(self, q, out, stream):
        self.kivi.kivi_decode_attention(self.cache, q, 1.0, out=out, ws=self.ws, stream=stream)

    def prepare(self, inputs, out):
        pass


class PagedLayout:
    """The paged pool: pages of P tokens scattered by a seeded permutation, lengths on
    the device: kivi_paged_decode_step / kivi_paged_decode_attention."""

    profile_prefix = "decode_attention_paged_"
    kernel = "kivi_paged_decode_attention (paged decode_kernel + paged_combine_kernel)"

    def __init__(self, wl, pre, dev, page_tokens, graph=False, value_residual=False, bits=2):
        from bit_asymmetric_kv_gb300 import kivi, synth

        self.wl, self.kivi, self.P = wl, kivi, page_tokens
        self.graph, self.graphs = graph, {}
        maxp = math.ceil((wl.n + cycle_of(wl) + 64) / page_tokens)
        num_pages = wl.B * maxp
        self.cache = kivi.PagedCache.allocate(wl.B, wl.Hkv, wl.G, page_tokens, maxp, num_pages, device=dev,
                                              value_residual=value_residual, bits=bits)
        self.cache.block_table.copy_(synth.block_table(wl.B, maxp, num_pages, wl.seed))
        for b in range(wl.B):
            kivi.kivi_paged_prefill(self.cache, b, pre.k[b].to(dev), pre.v[b].to(dev))
        self.n0 = wl.n
        self.lens0 = self.cache.seq_lens.clone()
        self.res0 = self.cache.k_res.clone()
        self.vres0 = None if self.cache.v_res is None else self.cache.v_res.clone()
        self.ws = kivi.paged_workspace(self.cache, wl.Hq, device=dev)
        self.ws.zero_()

    def rollback(self):
        self.cache.k_res.copy_(self.res0)
        if self.vres0 is not None:
            self.cache.v_res.copy_(self.vres0)
        self.cache.seq_lens.copy_(self.lens0)

    def prepare(self, inputs, out):
        """With graph replay: capture one step per input set (k, v, q), after one
        eager step (the library's first call on a device queries it)."""
        if not self.graph:
            return
        import torch

        k, v, q = inputs[0]
        self.kivi.kivi_paged_decode_step(self.cache, k, v, q, 1.0, out=out, ws=self.ws)
        torch.cuda.synchronize()
        self.rollback()
        for k, v, q in inputs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.kivi.kivi_paged_decode_step(self.cache, k, v, q, 1.0, out=out, ws=self.ws)
            self.graphs[k.data_ptr()] = g
        torch.cuda.synchronize()

    def step(self, k, v, q, out, stream):
        if self.graph:
            self.graphs[k.data_ptr()].replay()  # on the current stream
        else:
            self.kivi.kivi_paged_decode_step(self.cache, k, v, q, 1.0, out=out, ws=self.ws, stream=stream)
        return 3  # append (group flush fused), decode attention, combine (advances the lengths)

    def attention(self, q, out, stream):
        self.kivi.kivi_paged_decode_attention(self.cache, q, 1.0, out=out, ws=self.ws, stream=stream)


def make_layout(args, wl, pre, dev):
    if args.layout == "paged":
        return PagedLayout(wl, pre, dev, args.page_tokens, graph=args.graph, value_residual=args.value_residual,
                           bits=args.bits)
    return DenseLayout(wl, pre, dev, value_residual=args.value_residual, bits=args.bits, value_group=args.value_group)


# ----------------------------------------------------------------------------------------
# GPU benchmark
# ----------------------------------------------------------------------------------------
def run_kivi(args, wl):
    import torch

    from bit_asymmetric_kv_gb300 import kivi, synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    kivi.lib()
    pre = synth.make_prefill(wl)
    total = args.warmup + args.steps
    cycle = cycle_of(wl)
    lay = make_layout(args, wl, pre, dev)
    n0 = lay.n0
    # the inputs of the steps that run (at most one rollback cycle), drawn once on
    # the host; resident in HBM before timing
    steps_host = [synth.make_step(wl, pre, s) for s in range(min(cycle, total))]
    dev_in = [tuple(t.to(dev) for t in kvq) for kvq in steps_host]
    out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    lay.prepare(dev_in, out)

    def step_events(i, rec):
        if i % cycle == 0:
            lay.rollback()
        k, v, q = dev_in[i % cycle]
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launches = lay.step(k, v, q, out, stream)
        e1.record(stream)
        rec.append((e0, e1, launches))

    warm = []
    for i in range(args.warmup):
        step_events(i, warm)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    rec = []
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.warmup, total):
            step_events(i, rec)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier()
    launches = sum(x[2] for x in rec)
    step_ms = [e0.elapsed_time(e1) for e0, e1, _ in rec]
    ms_per_step, value = job_throughput(sum(step_ms) / len(step_ms), wl.B, world, dev)
    q50, q99 = np.percentile(step_ms, [50, 99])

    # roofline of the dominant kernel: the decode attention call (decode + combine)
    # alone, on the prompt's cache, timed the same way
    lay.rollback()
    attn_ms = []
    q0 = dev_in[0][2]
    for i in range(args.warmup + max(16, args.steps // 8)):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        lay.attention(q0, out, stream)
        e1.record(stream)
        if i >= args.warmup:
            attn_ms.append((e0, e1))
    torch.cuda.synchronize()
    attn_avg_ms = sum(a0.elapsed_time(a1) for a0, a1 in attn_ms) / len(attn_ms)
    bytes_attn = algorithmic_bytes(wl.B, wl.Hq, wl.Hkv, wl.G, n0, args.value_residual, args.bits, args.value_group)
    achieved = bytes_attn / (attn_avg_ms / 1e3) / 1e9
    peak, peak_src = measured_peak()
    sha = kernel_source_sha()
    # DRAM traffic from the committed ncu summary of this workload (named for it),
    # when it was taken on the current decode sources; never for a changed batch
    traffic = None if args.batch else profiled_traffic(sha, lay.profile_prefix + wl.name + ".md", wl.name,
                               f"bits={args.bits}, value_residual={int(bool(args.value_residual))}"
                               + (f", value_group={args.value_group}" if args.value_group else ""))
    del lay

    prefill = prefill_timing(args, wl, pre, dev, stream, flush)

    # ---- end to end through the public API: host buffers, copies inside the timing
    e2e = e2e_run(args, wl, pre, steps_host, dev, stream, flush)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return 0
    cb = (oracle_timing(wl, pre, 100000, 32, 10.0, args.value_residual, args.bits, args.value_group)
          if world == 1 else None)
    lay_cfg = make_layout_config(args)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "step_ms_p50": float(q50), "step_ms_p99": float(q99), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"u{args.bits} codes, f16 q/out, f32 accumulate", "data": "synthetic (seeded, fixed outlier key channels)",
        "config": {**workload_config(wl), **lay_cfg},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": (PagedLayout if args.layout == "paged" else DenseLayout).kernel,
                     "peak_source": peak_src, "attention_ms": attn_avg_ms,
                     "algorithmic_bytes_per_launch": bytes_attn, "context_tokens": n0,
                     "kernel_source_sha256": sha},
        "e2e": e2e,
        "prefill": prefill,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed_loop": t_wall,
        "cpu_baseline": cb,
    }
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def make_layout_config(args):
    cfg = {"layout": "dense"}
    if args.layout == "paged":
        api = "kivi_paged_decode_step (append + decode attention + length advance)"
        if args.graph:
            api += ", replayed from a CUDA graph captured once per input set"
        cfg = {"layout": f"paged: {args.page_tokens} tokens per page, pages scattered by a seeded permutation",
               "api": api}
    cfg["value_residual"] = bool(args.value_residual)
    cfg["bits"] = args.bits
    if args.value_group:
        cfg["value_group"] = args.value_group
    return cfg


def prefill_timing(args, wl, pre, dev, stream, flush, reps: int = 5, warmup: int = 1):
    """Quantize the whole prompt (kivi_quantize_prefill, dense cache) with L2 flushed
    before each call: the quantizers' throughput over fp16 K and V read once and the
    codes, scales and residual written."""
    import torch

    from bit_asymmetric_kv_gb300 import kivi

    cache = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, wl.capacity(), device=dev, value_group=args.value_group,
                                value_residual=args.value_residual,
                                bits=args.bits)
    k, v = pre.k.to(dev), pre.v.to(dev)
    assert k.shape[2] == wl.n, (k.shape, wl.n)
    ms = []
    for i in range(reps + warmup):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        kivi.kivi_quantize_prefill(cache, k, v, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            ms.append(e0.elapsed_time(e1))
    moved = prefill_bytes(wl.B, wl.Hkv, wl.G, wl.n, args.value_residual, args.bits, args.value_group)
    best = min(ms)
    peak, _ = measured_peak()
    return {"ms": best, "ms_mean": sum(ms) / len(ms), "bytes": moved, "GBps": moved / best / 1e6,
            "frac": moved / best / 1e6 / peak, "reps": reps,
            "note": "best of reps; fp16 K and V read once, codes, scales and residual written"}


def run_prefill(args, wl):
    """--prefill-only: time kivi_quantize_prefill alone on the workload's prompt (W
    untimed calls, then K timed ones, L2 flushed before each) and print one JSON line."""
    import torch

    from bit_asymmetric_kv_gb300 import kivi, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kivi.lib()
    pre = synth.make_prefill(wl)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    p = prefill_timing(args, wl, pre, dev, torch.cuda.current_stream(dev), flush, reps=args.steps,
                       warmup=args.warmup)
    peak, src = measured_peak()
    print(json.dumps({
        "metric": "prefill quantization GB/s (kivi_quantize_prefill: fp16 K and V in, codes, scales, residual out)",
        "value": p["GBps"], "unit": "GB/s", "higher_is_better": True, "steps": args.steps, "warmup": args.warmup,
        "ms_best": p["ms"], "ms_mean": p["ms_mean"], "bytes_per_call": p["bytes"],
        "roofline": {"bound": "hbm", "achieved": p["GBps"], "peak": peak, "unit": "GB/s", "frac": p["frac"],
                     "peak_source": src},
        "dtype": "fp16 in, 2-bit codes out" if args.bits == 2 else "fp16 in, 4-bit codes out", "data": "synthetic",
        "config": {**workload_config(wl), **make_layout_config(args), "layout": "dense",
                   "l2": "flushed by a 256 MiB write before every call (outside the timed events)"}}))
    return 0


def run_prefill_fused(args, wl):
    """--prefill-fused: the prompt's causal attention with the cache quantized in the
    same kernel (kivi_prefill_attention), next to the same attention without the cache
    and the separate quantization pass (kivi_quantize_prefill), L2 flushed before each
    call; prints one JSON object."""
    import torch

    from bit_asymmetric_kv_gb300 import kivi, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kivi.lib()
    pre = synth.make_prefill(wl)
    q = synth.make_prompt_queries(wl).to(dev)
    k, v = pre.k.to(dev), pre.v.to(dev)
    out = torch.empty_like(q)
    cache = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, wl.capacity(), device=dev, value_group=args.value_group,
                                value_residual=args.value_residual,
                                bits=args.bits)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ts = []
        for i in range(args.warmup + args.steps):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        ms = sorted(a.elapsed_time(b) for a, b in ts)
        return ms[len(ms) // 2]

    fused = timed(lambda: kivi.kivi_prefill_attention(cache, q, k, v, 1.0, out=out, stream=stream))
    alone = timed(lambda: kivi.kivi_prefill_attention(None, q, k, v, 1.0, out=out, dims=cache.dims, stream=stream))
    quant = timed(lambda: kivi.kivi_quantize_prefill(cache, k, v, stream=stream))
    n = wl.n
    kv_bytes = 2 * wl.B * wl.Hkv * n * wl.D * 2
    moved = prefill_bytes(wl.B, wl.Hkv, wl.G, n, args.value_residual, args.bits, args.value_group)
    flops = 4.0 * wl.D * (n * (n + 1) / 2) * wl.B * wl.Hq  # q.K and P.V over the causal triangle
    peak, src = measured_peak()
    tpeak, tsrc = measured_tensor_peak()
    extra = fused - alone
    print(json.dumps({
        "mode": "fused prefill", "workload": wl.name, "steps": args.steps, "warmup": args.warmup, "bits": args.bits,
        "value_residual": bool(args.value_residual), "l2": "flushed by a 256 MiB write before every call",
        "fused_ms": fused, "attention_alone_ms": alone, "separate_quantize_ms": quant,
        "quantization_cost_in_fused_ms": extra,
        "separate_path_ms": alone + quant, "fused_saving_ms": alone + quant - fused,
        "attention_tflops": flops / (alone / 1e3) / 1e12, "fused_attention_tflops": flops / (fused / 1e3) / 1e12,
        "separate_quantize_GBps": moved / quant / 1e6, "separate_quantize_frac_of_peak": moved / quant / 1e6 / peak,
        "quantize_bytes": moved, "prompt_kv_bytes": kv_bytes,
        "note": "the fused kernel quantizes the key/value tiles it already holds in shared memory: its quantization "
                "cost is fused_ms - attention_alone_ms against separate_quantize_ms for the second read of the prompt",
        "peak_GBps": peak, "peak_source": src,
        "roofline": {"bound": "tensor", "achieved": flops / (fused / 1e3) / 1e12, "peak": tpeak, "unit": "TFLOP/s",
                     "frac": flops / (fused / 1e3) / 1e12 / tpeak, "traffic": None, "kernel": "prefill_kernel",
                     "flops_per_launch": flops,
                     "peak_source": tsrc + "; fp16 has the bf16 rate, the kernel's MMAs are fp16 mma.sync"}}))
    return 0


def measured_tensor_peak():
    """Dense bf16 tensor peak for a kernel timed alone (burst), from MEASURED_PEAKS.json."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s bf16 burst"


def cycle_workspace(cache, wl, n0, dev):
    """A zero-filled decode workspace large enough for every context of a cycle."""
    import torch

    from bit_asymmetric_kv_gb300 import kivi

    nbytes = max(kivi.kivi_decode_workspace_bytes(cache.dims, wl.Hq, n) for n in range(n0, n0 + cycle_of(wl) + 2))
    return torch.zeros(nbytes, dtype=torch.uint8, device=dev)


def e2e_run(args, wl, pre, steps_in, dev, stream, flush):
    """Same metric through the public API with host inputs: every step copies its new
    k, v, q from pinned host memory (one buffer, one copy), runs append + decode
    attention and copies the output back; every copy is inside the timed region.
    steps_in: the host inputs (k, v, q) of the steps of one rollback cycle.

    Workloads whose steps read more than the 256 MiB L2 flush (each step's own reads
    then evict the L2) run as a serving loop would: the inputs of step i+1 are copied
    on a second stream while step i computes, the output of step i is copied back on
    it, and the whole loop of K steps is timed (no flush).  Smaller workloads, and
    graph replay (whose captured steps read fixed buffers), time each step with its
    copies in order on one stream, the L2 flushed before each step outside the events."""
    import torch

    total = args.warmup + args.steps
    cycle = cycle_of(wl)
    lay = make_layout(args, wl, pre, dev)
    # each step's k, v and q side by side in one pinned buffer: one copy per step
    shapes = [t.shape for t in steps_in[0]]
    sizes = [t.numel() for t in steps_in[0]]
    host = [torch.cat([t.reshape(-1) for t in kvq]).pin_memory() for kvq in steps_in]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    h2d = host[0].numel() * host[0].element_size()
    d2h = wl.B * wl.Hq * wl.D * 2
    step_bytes = algorithmic_bytes(wl.B, wl.Hq, wl.Hkv, wl.G, wl.n, args.value_residual, args.bits, args.value_group)
    pipelined = step_bytes > L2_FLUSH_BYTES and not getattr(lay, "graph", False)
    if not pipelined:
        dbuf = host[0].to(dev)
        dk, dv, dq = (p.view(sh) for p, sh in zip(torch.split(dbuf, sizes), shapes))
        out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float16, device=dev)
        out_h = torch.empty_like(out, device="cpu").pin_memory()
        lay.prepare([(dk, dv, dq)], out)
        times = []
        for i in range(total):
            if i % cycle == 0:
                lay.rollback()
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dbuf.copy_(host[i % cycle], non_blocking=True)
            lay.step(dk, dv, dq, out, stream)
            out_h.copy_(out, non_blocking=True)
            e1.record(stream)
            if i >= args.warmup:
                times.append((e0, e1))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in times) / len(times)
        return {"value": wl.B * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "method": "per step on one stream: H2D copy, step, D2H copy, CUDA events around the three; "
                          "L2 flushed before each step (outside the events)"}

    # serving loop: two input and output buffers, copies on a second stream
    copy = torch.cuda.Stream(dev)
    dbufs = [host[0].to(dev) for _ in range(2)]
    views = [[p.view(sh) for p, sh in zip(torch.split(d, sizes), shapes)] for d in dbufs]
    outs = [torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float16, device=dev) for _ in range(2)]
    outs_h = [torch.empty_like(outs[0], device="cpu").pin_memory() for _ in range(2)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    lay.prepare([tuple(views[0])], outs[0])

    def run(i0, i1):
        copy.wait_stream(stream)
        with torch.cuda.stream(copy):
            dbufs[i0 % 2].copy_(host[i0 % cycle], non_blocking=True)
            ev_in[i0 % 2].record(copy)
        for i in range(i0, i1):
            b, nb = i % 2, (i + 1) % 2
            if i % cycle == 0:
                lay.rollback()
            stream.wait_event(ev_in[b])
            if i - i0 >= 2:
                stream.wait_event(ev_out[b])  # outs[b] has been copied back (step i - 2)
            dk, dv, dq = views[b]
            lay.step(dk, dv, dq, outs[b], stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(copy):
                if i + 1 < i1:
                    if i > i0:
                        copy.wait_event(ev_done[nb])  # step i - 1 has read dbufs[nb]
                    dbufs[nb].copy_(host[(i + 1) % cycle], non_blocking=True)
                    ev_in[nb].record(copy)
                copy.wait_event(ev_done[b])
                outs_h[b].copy_(outs[b], non_blocking=True)
                ev_out[b].record(copy)
        stream.wait_stream(copy)

    run(0, args.warmup)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    run(args.warmup, total)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    return {"value": wl.B * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "method": "serving loop: the H2D copy of step i+1 and the D2H copy of step i on a second stream "
                      "while step i computes; CUDA events around the whole loop of K steps, every copy inside",
            "l2": f"no flush: each step reads {step_bytes / 1e9:.2f} GB, more than the 256 MiB flush and "
                  "twice the 129 MB L2"}


def run_compare(args):
    """The long-context GQA decode step over the 2-bit cache next to the same step
    over an unquantized fp16 cache (the in-build comparison kernel).  Prints one JSON
    object with both timings; the default bench line is not printed in this mode."""
    import torch

    from bit_asymmetric_kv_gb300 import kivi, synth

    wl = synth.LONG_GQA
    dev = torch.device("cuda", 0)
    kivi.lib()
    pre = synth.make_prefill(wl)
    k, v, q = pre.k.to(dev), pre.v.to(dev), pre.q.to(dev)
    cache = kivi.Cache.allocate(wl.B, wl.Hkv, wl.G, wl.capacity(), device=dev)
    kivi.kivi_quantize_prefill(cache, k, v)
    out = torch.empty_like(q)
    ws = kivi.workspace(cache, wl.Hq, device=dev)
    ws16 = torch.empty(kivi.kivi_decode_fp16_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n), dtype=torch.uint8,
                       device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ts = []
        for i in range(args.warmup + args.steps):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ts) / len(ts)

    ms2 = timed(lambda: kivi.kivi_decode_attention(cache, q, 1.0, out=out, ws=ws, stream=stream))
    ms16 = timed(lambda: kivi.kivi_decode_attention_fp16(k, v, q, 1.0, out=out, ws=ws16, stream=stream))
    b2 = algorithmic_bytes(wl.B, wl.Hq, wl.Hkv, wl.G, wl.n)
    b16 = wl.B * wl.Hkv * wl.n * wl.D * 2 * 2 + 2 * wl.B * wl.Hq * wl.D * 2
    peak, src = measured_peak()
    print(json.dumps({
        "mode": "comparison", "workload": wl.name, "steps": args.steps, "warmup": args.warmup,
        "l2": "flushed by a 256 MiB write before every call",
        "kivi_2bit": {"ms": ms2, "tokens_per_s": wl.B / (ms2 / 1e3), "bytes": b2, "GBps": b2 / ms2 / 1e6,
                      "frac_of_peak": b2 / ms2 / 1e6 / peak},
        "fp16_kv": {"ms": ms16, "tokens_per_s": wl.B / (ms16 / 1e3), "bytes": b16, "GBps": b16 / ms16 / 1e6,
                    "frac_of_peak": b16 / ms16 / 1e6 / peak},
        "speedup_2bit_over_fp16": ms16 / ms2, "bytes_ratio_fp16_over_2bit": b16 / b2,
        "peak_GBps": peak, "peak_source": src}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=496)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["kivi", "reference"], default="kivi")
    ap.add_argument("--compare-fp16", action="store_true",
                    help="time the long-context GQA step over the 2-bit and an fp16 cache instead")
    ap.add_argument("--layout", choices=["dense", "paged"], default="dense",
                    help="cache layout of the timed path (default: the dense cache)")
    ap.add_argument("--page-tokens", type=int, default=64, help="tokens per page of --layout paged")
    ap.add_argument("--graph", action="store_true",
                    help="--layout paged: replay each step from a captured CUDA graph")
    ap.add_argument("--value-residual", action="store_true",
                    help="keep the last n mod G values in fp16 beside the key residual (the variant cache)")
    ap.add_argument("--bits", type=int, choices=[2, 4], default=2, help="code width of the cache (default 2)")
    ap.add_argument("--value-group", type=int, choices=[0, 32, 64], default=0,
                    help="channels per value scale: 0 (one per token, default) or value channel groups of 32 / 64 "
                         "(dense 2-bit cache without a value residual)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prompt quantization (kivi_quantize_prefill) of the workload")
    ap.add_argument("--prefill-fused", action="store_true",
                    help="time the fused prefill (causal prompt attention + cache quantization in one kernel) "
                         "against the attention alone and the separate quantization pass")
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload's shape with this batch instead (for small profiling captures; "
                         "the JSON line then names the batch in its config)")
    ap.add_argument("--workload", default="streaming",
                    help="workload name or unique prefix (tiny, llama2, mistral, streaming, long-gqa); "
                         "default: the streaming generation (B64, H32, 8192-token prompt, 512 steps), "
                         "the largest of the five")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.value_group and (args.layout != "dense" or args.bits != 2 or args.value_residual):
        ap.error("--value-group needs the dense 2-bit cache without --value-residual")
    if args.graph and args.layout != "paged":
        ap.error("--graph needs --layout paged (the dense step takes its token count from the host)")
    from bit_asymmetric_kv_gb300 import synth

    hits = [w for w in synth.CONFIGS if w.name.startswith(args.workload)]
    if len(hits) != 1:
        ap.error(f"--workload {args.workload!r}: choose one of {[w.name for w in synth.CONFIGS]}")
    wl = hits[0]
    if args.batch:
        import dataclasses

        wl = dataclasses.replace(wl, B=args.batch)
    if args.compare_fp16:
        return run_compare(args)
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.prefill_only:
        return run_prefill(args, wl)
    if args.prefill_fused:
        return run_prefill_fused(args, wl)
    return run_kivi(args, wl)


if __name__ == "__main__":
    sys.exit(main())
