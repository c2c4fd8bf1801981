#!/usr/bin/env python
"""Benchmark of the fused inference attention library on one GB300 (or N replicas).

Headline step: one fia_decode call (length resolution + split planning on the
host, then one split-KV paged decode kernel that also merges the partials of
the splits with their LSE) on the paged GQA decode
workload -- B=16, Q_N=32, KV_N=8, D=128, bf16, actual_seq_kvlen uniform on
[1, 4096], block_size 128, random physical blocks.  value = KV bytes read per
second (the K and V rows of every sequence, sum(L_b) * KV_N * D * 2 bytes * 2).

The other hot-path workloads are measured in the same run under "sections":
varlen TND causal prefill (TFLOP/s), the same with a 1024-key sliding window
(sparse_mode 4), the same with an explicit causal mask (sparse_mode 1), chunked prefill
against a paged cache (TFLOP/s), MLA prefill
(192 / 128, TFLOP/s), block-sparse
prefill (TFLOP/s), MLA decode
(cache GB/s), the headline decode with 4 new tokens per sequence (KV GB/s) and
the small fp16 prefill.  Inputs are seeded synthetic tensors
of the workloads' shapes (fia_inputs.py).  The L2 is flushed (a 512 MB write)
before every timed call; times are CUDA events on the launching stream.

--impl reference times the fp64 CPU oracle on the host cores instead (the
reference arm: there is no runnable upstream implementation).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attention TFLOP/s & % bf16 peak; paged decode KV GB/s & % HBM BW"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed sections run."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(vals, device=None):
    """Max over ranks of a few host floats (the timed region is the slowest
    rank's); the values themselves with one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


class Timer:
    """Per-call CUDA-event timing with an L2 flush before each call."""

    def __init__(self, torch, device):
        self.torch = torch
        self.flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def flush(self):
        self.flush_buf.zero_()

    def run(self, fn, steps, warmup, kernel_events=False):
        torch = self.torch
        import attention_fia_prefill_gb300 as fia
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        calls, kernels = [], []
        for _ in range(steps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ks, ke = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if kernel_events:
                # torch creates the CUDA event on first record: materialise the
                # handles the library will re-record around its kernel
                ks.record()
                ke.record()
            self.flush()
            s.record()
            if kernel_events:
                fia._binding.profile_next_call(ks, ke)
            fn()
            e.record()
            calls.append((s, e))
            if kernel_events:
                kernels.append((ks, ke))
        torch.cuda.synchronize()
        call_ms = [a.elapsed_time(b) for a, b in calls]
        kern_ms = [a.elapsed_time(b) for a, b in kernels]
        return call_ms, kern_ms


def roofline(bound, achieved, peak, unit, traffic=None):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summaries (None if absent)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


# ------------------------------------------------------------------ workloads
def decode_workload(torch, dev):
    import fia_inputs
    c = fia_inputs.workload_paged_gqa_decode()
    kv_bytes = sum(c.kv_lens) * c.num_key_value_heads * c.q.shape[-1] * 2 * 2
    return c, kv_bytes


def prefill_tnd_flops(case):
    lens = [b - a for a, b in zip([0] + case.actual_seq_qlen[:-1], case.actual_seq_qlen)]
    D = case.q.shape[-1]
    return sum(L * (L + 1) // 2 for L in lens) * case.num_heads * 4 * D


def bsa_flops(case):
    m = case.mask.to(dtype=case.mask.dtype).numpy() != 0
    B, N1, nqb, nkb = m.shape
    S = case.q.shape[2]
    X, Y = case.block_shape
    rows = [min(X, S - i * X) for i in range(nqb)]
    cols = [min(Y, S - j * Y) for j in range(nkb)]
    import numpy as np
    pairs = float((m * np.outer(rows, cols)[None, None]).sum())
    return pairs * 4 * case.q.shape[-1]


def measure_decode(torch, dev, timer, steps, warmup, pk, traffic):
    import attention_fia_prefill_gb300 as fia
    c, kv_bytes = decode_workload(torch, dev)
    q, kp, vp, tb = c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev), c.block_table.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
    kw = dict(block_table=tb, block_size=c.block_size, actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads,
              num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
              softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    def call():
        fia.fia_decode(q, kp, vp, **kw)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    res = {"call_ms": statistics.mean(call_ms), "kernel_ms": statistics.mean(kern_ms), "kv_bytes": kv_bytes,
           "launches_per_step": 1}
    # end to end: pinned host inputs -> device, the call, result -> pinned host
    hq, hk, hv, ht = (t.pin_memory() for t in (c.q, c.k_pool, c.v_pool, c.block_table))
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ht))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    def e2e_call():
        q.copy_(hq, non_blocking=True)
        kp.copy_(hk, non_blocking=True)
        vp.copy_(hv, non_blocking=True)
        tb.copy_(ht, non_blocking=True)
        fia.fia_decode(q, kp, vp, **kw)
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    e2e_ms, _ = timer.run(e2e_call, steps, max(1, warmup // 2))
    res["e2e_ms"] = statistics.mean(e2e_ms)
    res["h2d"] = h2d
    res["d2h"] = d2h
    res["roofline"] = roofline("hbm", kv_bytes / (res["kernel_ms"] * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s",
                               traffic.get("decode_kernel"))
    return res, c


def measure_prefill_tnd(torch, dev, timer, steps, warmup, pk, traffic):
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_tnd_varlen()
    flops = prefill_tnd_flops(c)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="TND", sparse_mode=3, actual_seq_qlen=c.actual_seq_qlen,
                        actual_seq_kvlen=c.actual_seq_kvlen, softmax_lse_flag=True, out=out, softmax_lse=lse,
                        workspace=ws)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "varlen TND causal prefill bf16, 8 seqs U[256,4096], Q_N=32, KV_N=8, D=128, LSE",
            "metric": "prefill attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(flops / (statistics.mean(call_ms) * 1e-3) / 1e12, 2), "ms_per_call": statistics.mean(call_ms),
            "kernel_ms": km, "flops": flops, "seq_lens": c.actual_seq_qlen,
            "roofline": roofline("tensor", flops / (km * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s",
                                 traffic.get("prefill_pair_kernel"))}


def measure_prefill_band(torch, dev, timer, steps, warmup, pk, traffic):
    """The varlen TND workload with a sliding window (sparse_mode 4,
    pre_tokens 1024, next_tokens 0): each row sees its 1025 latest keys."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_tnd_varlen()
    pre = 1024
    lens = [b - a for a, b in zip([0] + c.actual_seq_qlen[:-1], c.actual_seq_qlen)]
    pairs = sum(sum(min(i + 1, pre + 1) for i in range(L)) for L in lens)
    flops = pairs * c.num_heads * 4 * c.q.shape[-1]
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="TND", sparse_mode=4, pre_tokens=pre, next_tokens=0,
                        actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                        softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "varlen TND band prefill bf16 (window 1024 keys back), 8 seqs U[256,4096], "
                        "Q_N=32, KV_N=8, D=128, LSE",
            "metric": "prefill attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(flops / (statistics.mean(call_ms) * 1e-3) / 1e12, 2), "ms_per_call": statistics.mean(call_ms),
            "kernel_ms": km, "flops": flops,
            "roofline": roofline("tensor", flops / (km * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s",
                                 traffic.get("prefill_pair_kernel_band"))}


def measure_prefill_mask(torch, dev, timer, steps, warmup, pk, traffic):
    """The varlen TND workload with an explicit mask (sparse_mode 1): a uint8
    lower-triangular (4096, 4096) mask, i.e. causal attention given as a mask.
    An arbitrary mask cannot skip tiles, so every (row, key) tile of each
    sequence is computed; flops count the allowed pairs only."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_tnd_varlen()
    flops = prefill_tnd_flops(c)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    mask = fia_inputs.atten_mask((4096, 4096), "causal").to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="TND", sparse_mode=1, atten_mask=mask,
                        actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                        softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "varlen TND prefill bf16 with an explicit uint8 causal mask (sparse_mode 1, every tile "
                        "computed), 8 seqs U[256,4096], Q_N=32, KV_N=8, D=128, LSE",
            "metric": "prefill attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(flops / (statistics.mean(call_ms) * 1e-3) / 1e12, 2), "ms_per_call": statistics.mean(call_ms),
            "kernel_ms": km, "flops": flops,
            "roofline": roofline("tensor", flops / (km * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s",
                                 traffic.get("prefill_pair_kernel_mask"))}


def measure_chunked_prefill(torch, dev, timer, steps, warmup, pk, traffic):
    """Chunked prefill against a paged cache: 8 sequences, a 2048-token chunk
    after a cached context U[0, 14336], 256-token blocks, right-down causal."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_chunked_prefill()
    D = c.q.shape[-1]
    pairs = sum(sum(L - ql + i + 1 for i in range(ql)) for ql, L in zip(c.q_lens, c.kv_lens))
    flops = pairs * c.num_heads * 4 * D
    q, kp, vp, tab = c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev), c.block_table.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, q.shape[2], 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill_paged(q, kp, vp, tab, block_size=c.block_size, actual_seq_kvlen=c.kv_lens,
                              actual_seq_qlen=c.actual_seq_qlen, num_heads=c.num_heads,
                              num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
                              sparse_mode=3, softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "chunked prefill bf16 against a paged cache: 8 x 2048-token chunks after cached contexts "
                        "U[0,14336], Q_N=32, KV_N=8, D=128, block 256, sparse_mode 3, LSE",
            "metric": "prefill attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(flops / (statistics.mean(call_ms) * 1e-3) / 1e12, 2), "ms_per_call": statistics.mean(call_ms),
            "kernel_ms": km, "flops": flops, "kv_lens": c.kv_lens,
            "roofline": roofline("tensor", flops / (km * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s",
                                 traffic.get("prefill_pair_kernel_chunked"))}


def measure_mla_prefill(torch, dev, timer, steps, warmup, pk, traffic):
    """MLA prefill, TND: the varlen prefill lengths, 32 heads, query/key D 192
    (128 + 64 rope columns), value D 128, right-down causal."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_mla_prefill()
    starts = [0] + c.actual_seq_qlen[:-1]
    lens = [e - s0 for s0, e in zip(starts, c.actual_seq_qlen)]
    flops = sum(L * (L + 1) // 2 for L in lens) * c.num_heads * 2 * (192 + 128)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    out = torch.empty((q.shape[0], c.num_heads, 128), dtype=q.dtype, device=dev)
    lse = torch.empty((q.shape[0], c.num_heads, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill_mla(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                            scale_value=c.scale, input_layout="TND", sparse_mode=3,
                            actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                            softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "MLA prefill bf16, TND, 8 seqs U[256,4096], 32 heads, query/key D 192 (128 + 64 rope), "
                        "value D 128, causal, LSE",
            "metric": "prefill attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(flops / (statistics.mean(call_ms) * 1e-3) / 1e12, 2), "ms_per_call": statistics.mean(call_ms),
            "kernel_ms": km, "flops": flops,
            "roofline": roofline("tensor", flops / (km * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s",
                                 traffic.get("prefill_pair_kernel_mla"))}


def measure_bsa(torch, dev, timer, steps, warmup, pk, traffic):
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_bsa()
    flops = bsa_flops(c)
    q, k, v, m = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.mask.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, q.shape[2], 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.bsa_forward(q, k, v, m, c.block_shape, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="BNSD", softmax_lse_flag=True, out=out, softmax_lse=lse,
                        workspace=ws)

    call_ms, kern_ms = timer.run(call, max(3, steps // 4), max(3, warmup), kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "block-sparse prefill bf16 B=2, 32/8 heads, S=16384, D=128, 128x128 blocks, diag + 25%",
            "metric": "block-sparse attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(flops / (statistics.mean(call_ms) * 1e-3) / 1e12, 2),
            "ms_per_call": statistics.mean(call_ms), "kernel_ms": km, "flops": flops,
            "roofline": roofline("tensor", flops / (km * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s",
                                 traffic.get("bsa_kernel"))}


def measure_bsa_fp8(torch, dev, timer, steps, warmup, pk, traffic):
    """FP8 block-sparse prefill: the bf16 workload's shapes in e4m3 with
    per-block dequant scales, 128 x 256 blocks (the quantisation blocks).
    Q K^T runs at the fp8 tensor rate (2x bf16, the recipe's nominal ratio),
    P V in bf16, so the peak is the harmonic blend of the two halves of the
    work: 2 / (1 / (2 P) + 1 / P) = 4/3 P."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    f = fia_inputs.workload_bsa_fp8()
    c = f.base
    flops = bsa_flops(c)
    q, k, v, m = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.mask.to(dev)
    qs, ks, vs = f.q_scale.to(dev), f.k_scale.to(dev), f.v_scale.to(dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[0], c.num_heads, q.shape[2], 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.bsa_forward(q, k, v, m, c.block_shape, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="BNSD", softmax_lse_flag=True, out=out, softmax_lse=lse,
                        workspace=ws, q_dequant_scale=qs, k_dequant_scale=ks, v_dequant_scale=vs)

    call_ms, kern_ms = timer.run(call, max(3, steps // 4), max(3, warmup), kernel_events=True)
    km = statistics.mean(kern_ms)
    peak = round(pk["bf16_tflops"] * 4 / 3, 1)
    return {"workload": "block-sparse prefill FP8 e4m3 (per-block dequant scales) B=2, 32/8 heads, S=16384, "
                        "D=128, 128x256 blocks, diag + 25%, bf16 out",
            "metric": "block-sparse attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(flops / (statistics.mean(call_ms) * 1e-3) / 1e12, 2),
            "ms_per_call": statistics.mean(call_ms), "kernel_ms": km, "flops": flops,
            "roofline": dict(roofline("tensor", flops / (km * 1e-3) / 1e12, peak, "TFLOP/s",
                                      traffic.get("bsa_fp8_kernel")),
                             peak_source="measured bf16 x 4/3 (fp8 Q K^T at 2x, bf16 P V)")}


def measure_mla(torch, dev, timer, steps, warmup, pk, traffic):
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_mla_decode()
    cache_bytes = sum(c.kv_lens) * (512 + 64) * 2
    q, qr, lat, rope, tb = (t.to(dev) for t in (c.q, c.q_rope, c.latent, c.rope, c.block_table))
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_decode(q, lat, lat, query_rope=qr, key_rope=rope, block_table=tb, block_size=c.block_size,
                       actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads, num_key_value_heads=1, scale_value=c.scale,
                       input_layout="BSND", softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "MLA decode bf16 B=32, 128 heads, latent 512 + rope 64, kv length 8192, block 128",
            "metric": "latent+rope cache GB/s", "unit": "GB/s",
            "value": round(cache_bytes / (statistics.mean(call_ms) * 1e-3) / 1e9, 2),
            "ms_per_call": statistics.mean(call_ms), "kernel_ms": km, "cache_bytes": cache_bytes,
            "roofline": roofline("hbm", cache_bytes / (km * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s",
                                 traffic.get("mla_kernel"))}


def measure_decode_tokens(torch, dev, timer, steps, warmup, pk, traffic):
    """The headline paged workload with 4 new tokens per sequence (speculative
    decoding), right-down causal: the same cache bytes, 4x the query rows."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    base = fia_inputs.workload_paged_gqa_decode()
    c = fia_inputs.paged_decode_case(16, 32, 8, 128, base.kv_lens, block_size=128, workload=3400, q_tokens=4)
    kv_bytes = sum(c.kv_lens) * c.num_key_value_heads * 128 * 2 * 2
    q, kp, vp, tb = c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev), c.block_table.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, q.shape[2], 1), dtype=torch.float32, device=dev)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_decode(q, kp, vp, block_table=tb, block_size=c.block_size, actual_seq_kvlen=c.kv_lens,
                       num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                       input_layout="BNSD", sparse_mode=3, softmax_lse_flag=True, out=out, softmax_lse=lse,
                       workspace=ws)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    km = statistics.mean(kern_ms)
    return {"workload": "paged GQA decode bf16, 4 query tokens (causal): B=16, Q_N=32, KV_N=8, D=128, "
                        "U[1,4096], block 128",
            "metric": "paged decode KV GB/s", "unit": "GB/s",
            "value": round(kv_bytes / (statistics.mean(call_ms) * 1e-3) / 1e9, 2),
            "ms_per_call": statistics.mean(call_ms), "kernel_ms": km, "kv_bytes": kv_bytes,
            "roofline": roofline("hbm", kv_bytes / (km * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s",
                                 traffic.get("decode_kernel_q4"))}


def measure_small_prefill(torch, dev, timer, steps, warmup, pk):
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_prefill_bnsd_f16_small()
    flops = 2 * (128 * 129 // 2) * 4 * 64
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)

    def call():
        fia.fia_prefill(q, k, v, num_heads=2, scale_value=c.scale, input_layout="BNSD", sparse_mode=2,
                        softmax_lse_flag=True)

    call_ms, kern_ms = timer.run(call, steps, warmup, kernel_events=True)
    return {"workload": "prefill BNSD fp16 B=1 N=2 S=128 D=64 causal", "metric": "latency", "unit": "us",
            "value": round(statistics.mean(call_ms) * 1e3, 2), "kernel_us": round(statistics.mean(kern_ms) * 1e3, 2),
            "flops": flops}


def cpu_baseline_decode(case, kv_bytes, budget_s=20.0):
    """The fp64 oracle as it stands, on the host cores, over a bounded sample
    of the decode workload (whole batches until ~budget_s of CPU work)."""
    from oracle import fia_oracle
    import torch
    B = case.q.shape[0]
    done_bytes, t0 = 0, time.perf_counter()
    nb = 0
    for b in range(B):
        fia_oracle.fia_decode(case.q[b:b + 1], case.k_pool, case.v_pool, num_heads=case.num_heads,
                              num_key_value_heads=case.num_key_value_heads, scale_value=case.scale,
                              input_layout="BNSD", actual_seq_kvlen=[case.kv_lens[b]],
                              block_table=case.block_table[b:b + 1], block_size=case.block_size)
        done_bytes += case.kv_lens[b] * case.num_key_value_heads * case.q.shape[-1] * 4
        nb += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": torch.get_num_threads(),
            "kind": "oracle", "sample": f"{nb} of {B} batches of the paged GQA decode workload, fp64 numpy"}


# ------------------------------------------------------------------ arms
def run_ours(args):
    import torch
    ws_, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from attention_fia_prefill_gb300 import build as b
    b.build()
    pk, pk_src = peaks()
    traffic = load_traffic()
    timer = Timer(torch, dev)
    sampler = ClockSampler(local)
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    dec, case = measure_decode(torch, dev, timer, args.steps, args.warmup, pk, traffic)
    sections = {}
    if not args.headline_only:
        for name, fn in (("prefill_tnd", measure_prefill_tnd), ("prefill_band", measure_prefill_band),
                         ("prefill_mask", measure_prefill_mask),
                         ("chunked_prefill", measure_chunked_prefill), ("mla_prefill", measure_mla_prefill),
                         ("bsa", measure_bsa), ("bsa_fp8", measure_bsa_fp8), ("mla_decode", measure_mla), ("decode_q4", measure_decode_tokens)):
            try:
                sections[name] = fn(torch, dev, timer, args.steps, args.warmup, pk, traffic)
            except Exception as e:  # a section failure is reported, not hidden
                sections[name] = {"error": repr(e)}
        try:
            sections["prefill_small"] = measure_small_prefill(torch, dev, timer, args.steps, args.warmup, pk)
        except Exception as e:
            sections["prefill_small"] = {"error": repr(e)}
    torch.cuda.synchronize()
    clocks = sampler.stop()
    dec["call_ms"], dec["e2e_ms"] = max_over_ranks([dec["call_ms"], dec["e2e_ms"]], device=dev)
    if rank != 0:
        return
    value = ws_ * dec["kv_bytes"] / (dec["call_ms"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dec["call_ms"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "paged GQA decode bf16: B=16, Q_N=32, KV_N=8, Q_S=1, D=128, "
                               "actual_seq_kvlen U[1,4096], block_size=128, random block_table",
                   "kv_lens": case.kv_lens, "kv_bytes_per_step": dec["kv_bytes"],
                   "l2": "flushed (512 MB write) before every timed call", "parallelism": f"replicas x{ws_}"},
        "e2e": {"value": round(ws_ * dec["kv_bytes"] / (dec["e2e_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": dec["h2d"], "d2h_bytes_per_step": dec["d2h"]},
        "gpu_launches": dec["launches_per_step"] * args.steps,
        "roofline": dict(dec["roofline"], peak_source=pk_src),
        "kernel_ms": round(dec["kernel_ms"], 5),
        "clocks": clocks,
        "sections": sections,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(case, dec["kv_bytes"])
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The oracle (fp64, host cores) on the headline workload, K timed steps of a
    bounded sample each."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    import fia_inputs
    from oracle import fia_oracle
    c = fia_inputs.workload_paged_gqa_decode()
    nb = 2          # batches per step: a bounded sample (about a second of CPU work)
    times, done = [], 0
    for step in range(args.warmup + args.steps):
        b0 = (step * nb) % c.q.shape[0]
        sl = slice(b0, b0 + nb)
        t0 = time.perf_counter()
        fia_oracle.fia_decode(c.q[sl], c.k_pool, c.v_pool, num_heads=c.num_heads,
                              num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
                              actual_seq_kvlen=c.kv_lens[sl], block_table=c.block_table[sl],
                              block_size=c.block_size)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            done += sum(c.kv_lens[sl]) * c.num_key_value_heads * c.q.shape[-1] * 4
    total = sum(times)
    value = done / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "paged GQA decode bf16: B=16, Q_N=32, KV_N=8, Q_S=1, D=128, "
                                   "actual_seq_kvlen U[1,4096], block_size=128, random block_table"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": torch.get_num_threads(),
                             "kind": "oracle", "sample": f"{nb} batches per step, cycling over the 16"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_target(args):
    """Plain repeated calls of one workload (warmup + steps), for ncu captures."""
    import torch
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    from attention_fia_prefill_gb300 import build as b
    b.build()
    dev = torch.device("cuda", 0)
    name = args.profile
    if name == "decode":
        c = fia_inputs.workload_paged_gqa_decode()
        q, kp, vp, tb = c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev), c.block_table.to(dev)

        def call():
            fia.fia_decode(q, kp, vp, block_table=tb, block_size=c.block_size, actual_seq_kvlen=c.kv_lens,
                           num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                           input_layout="BNSD", softmax_lse_flag=True)
    elif name == "prefill_tnd":
        c = fia_inputs.workload_tnd_varlen()
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)

        def call():
            fia.fia_prefill(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                            scale_value=c.scale, input_layout="TND", sparse_mode=3,
                            actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                            softmax_lse_flag=True)
    elif name == "bsa":
        c = fia_inputs.workload_bsa()
        q, k, v, m = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.mask.to(dev)

        def call():
            fia.bsa_forward(q, k, v, m, c.block_shape, num_heads=c.num_heads,
                            num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
                            softmax_lse_flag=True)
    elif name == "mla":
        c = fia_inputs.workload_mla_decode()
        q, qr, lat, rope, tb = (t.to(dev) for t in (c.q, c.q_rope, c.latent, c.rope, c.block_table))

        def call():
            fia.fia_decode(q, lat, lat, query_rope=qr, key_rope=rope, block_table=tb, block_size=c.block_size,
                           actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads, num_key_value_heads=1,
                           scale_value=c.scale, input_layout="BSND", softmax_lse_flag=True)
    elif name == "bsa_fp8":
        f = fia_inputs.workload_bsa_fp8()
        c = f.base
        q, k, v, m = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.mask.to(dev)
        qs, ks, vs = f.q_scale.to(dev), f.k_scale.to(dev), f.v_scale.to(dev)

        def call():
            fia.bsa_forward(q, k, v, m, c.block_shape, num_heads=c.num_heads,
                            num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
                            softmax_lse_flag=True, q_dequant_scale=qs, k_dequant_scale=ks, v_dequant_scale=vs)
    elif name == "mla_prefill":
        c = fia_inputs.workload_mla_prefill()
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)

        def call():
            fia.fia_prefill_mla(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                                scale_value=c.scale, input_layout="TND", sparse_mode=3,
                                actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                                softmax_lse_flag=True)
    else:
        raise SystemExit(f"unknown profile target {name}")
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    print(f"profile target {name}: {args.warmup + args.steps} calls done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", default=None, help="only run plain calls of one workload (decode, prefill_tnd, bsa, bsa_fp8, mla, mla_prefill)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--headline-only", action="store_true", help="skip the per-workload sections")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile_target(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
