#!/usr/bin/env python
"""Benchmark of the fused inference attention library on one GB300 (or N replicas).

Headline step: one fia_decode call (length resolution + split planning on the
host, then one split-KV paged decode kernel that also merges the partials of
the splits with their LSE) on the paged GQA decode workload -- B=16, Q_N=32,
KV_N=8, D=128, bf16, actual_seq_kvlen uniform on [1, 4096], block_size 128,
random physical blocks.  value = KV bytes read per second (the K and V rows of
every sequence, sum(L_b) * KV_N * D * 2 bytes * 2), timed on the device over
calls run back to back through the public call, cycling over five copies of
the KV pools so each call reads inputs that are not in L2.

The other hot-path workloads are measured in the same run under "sections"
(least important first, the varlen TND causal prefill last), each with its
roofline and the fp64 CPU oracle timed on the host cores over a bounded sample
of the same workload.  Prefill-type sections flush L2 (a 512 MB write) before
every call and time the kernel with events around it.  Inputs are seeded
synthetic tensors of the workloads' shapes (fia_inputs.py).

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
    """CUDA-event timing on the current stream.

    cold(): every call after an L2 flush (a 512 MB write), events around the
    call and around its main kernel.
    back_to_back(): K calls in a row, call i running fns[i % len(fns)] over
    rotating input copies (so consecutive calls read inputs larger than L2);
    the calls are queued behind GPU work longer than twice their enqueueing
    time, so the GPU runs them back to back whatever the host's pace, and one
    event pair brackets all K.  The host's own time per call is measured
    around the enqueueing loop."""

    def __init__(self, torch, device):
        self.torch = torch
        self.flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def flush(self):
        self.flush_buf.zero_()

    def cold(self, fn, steps, warmup):
        torch = self.torch
        import attention_fia_prefill_gb300 as fia
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        calls, kernels = [], []
        for _ in range(steps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ks, ke = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            # torch creates the CUDA event on first record: materialise the
            # handles the library will re-record around its kernel
            ks.record()
            ke.record()
            self.flush()
            s.record()
            fia._binding.profile_next_call(ks, ke)
            fn()
            e.record()
            calls.append((s, e))
            kernels.append((ks, ke))
        torch.cuda.synchronize()
        return ([a.elapsed_time(b) for a, b in calls], [a.elapsed_time(b) for a, b in kernels])

    def back_to_back(self, fns, steps, warmup):
        torch = self.torch
        n = len(fns)
        t0 = time.perf_counter()
        for i in range(warmup):
            fns[i % n]()
        host_us = (time.perf_counter() - t0) / max(warmup, 1) * 1e6
        torch.cuda.synchronize()
        # queue the K calls behind GPU work that outlasts their enqueueing
        # (each flush is a ~80 us write): the GPU then runs them back to back
        # whatever the host's pace; the flush also leaves L2 cold
        for _ in range(max(3, int(steps * host_us * 2 / 80) + 1)):
            self.flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        t0 = time.perf_counter()
        for i in range(steps):
            fns[i % n]()
        t1 = time.perf_counter()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / steps, (t1 - t0) / steps * 1e6


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


def section(workload, value, unit, ms, roof, cpu=None, **extra):
    d = {"workload": workload, "value": round(value, 2), "unit": unit, "ms": round(ms, 5)}
    d.update(extra)
    d["roofline"] = roof
    if cpu is not None:
        d["cpu_baseline"] = cpu
    return d


# ------------------------------------------------------------------ workloads
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


ROTATE = 5   # decode input copies cycled through (5 x ~114 MB of K/V > L2)


def measure_decode(torch, dev, timer, steps, warmup, pk, traffic):
    """The headline: paged GQA decode through the public call, back to back
    over rotating copies of the KV pools."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_paged_gqa_decode()
    kv_bytes = sum(c.kv_lens) * c.num_key_value_heads * c.q.shape[-1] * 2 * 2
    q, tb = c.q.to(dev), c.block_table.to(dev)
    pools = [(c.k_pool.to(dev), c.v_pool.to(dev)) for _ in range(ROTATE)]
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
    kw = dict(block_table=tb, block_size=c.block_size, actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads,
              num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
              softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)
    fns = [lambda kp=kp, vp=vp: fia.fia_decode(q, kp, vp, **kw) for kp, vp in pools]
    step_ms, host_us = timer.back_to_back(fns, steps, warmup)
    cold_ms, cold_kernel_ms = timer.cold(fns[0], max(3, steps // 2), 3)
    res = {"step_ms": step_ms, "host_us": host_us, "kv_bytes": kv_bytes,
           "cold_call_us": statistics.mean(cold_ms) * 1e3, "cold_kernel_us": statistics.mean(cold_kernel_ms) * 1e3}
    # end to end: pinned host inputs -> device, the call, result -> pinned host
    hq, hk, hv, ht = (t.pin_memory() for t in (c.q, c.k_pool, c.v_pool, c.block_table))
    kp, vp = pools[0]
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    res["h2d"] = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ht))
    res["d2h"] = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    def e2e_call():
        q.copy_(hq, non_blocking=True)
        kp.copy_(hk, non_blocking=True)
        vp.copy_(hv, non_blocking=True)
        tb.copy_(ht, non_blocking=True)
        fia.fia_decode(q, kp, vp, **kw)
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    res["e2e_ms"], _ = timer.back_to_back([e2e_call], steps, max(3, warmup // 2))
    res["roofline"] = roofline("hbm", kv_bytes / (step_ms * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s",
                               traffic.get("decode_gqa_kernel"))
    return res, c


def measure_decode_tokens(torch, dev, timer, steps, warmup, pk, traffic, pool):
    """The headline paged workload with 4 new tokens per sequence (speculative
    decoding), right-down causal: the same cache bytes, 4x the query rows."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    base = fia_inputs.workload_paged_gqa_decode()
    c = fia_inputs.paged_decode_case(16, 32, 8, 128, base.kv_lens, block_size=128, workload=3400, q_tokens=4)
    kv_bytes = sum(c.kv_lens) * c.num_key_value_heads * 128 * 2 * 2
    q, tb = c.q.to(dev), c.block_table.to(dev)
    pools = [(c.k_pool.to(dev), c.v_pool.to(dev)) for _ in range(ROTATE)]
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, q.shape[2], 1), dtype=torch.float32, device=dev)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
    kw = dict(block_table=tb, block_size=c.block_size, actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads,
              num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD", sparse_mode=3,
              softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)
    fns = [lambda kp=kp, vp=vp: fia.fia_decode(q, kp, vp, **kw) for kp, vp in pools]
    step_ms, _ = timer.back_to_back(fns, steps, warmup)
    del pools
    cpu = pool.run(oracle_tasks_decode(c, mode=3), 1e9, "GB/s", "all 128 (batch, kv head) units") if pool else None
    return section("paged GQA decode, 4 query tokens causal, B=16 32/8 heads D=128 U[1,4096]",
                   kv_bytes / (step_ms * 1e-3) / 1e9, "GB/s", step_ms,
                   roofline("hbm", kv_bytes / (step_ms * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s",
                            traffic.get("decode_gqa_kernel_q4")), cpu)


def measure_mla(torch, dev, timer, steps, warmup, pk, traffic, pool):
    """MLA decode: B=32, 128 heads, latent 512 + rope 64, kv length 8192 (the
    302 MB cache exceeds L2: back to back without copies)."""
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

    step_ms, _ = timer.back_to_back([call], steps, warmup)
    cpu = pool.run(oracle_tasks_mla_decode(c)[:2 * pool.n], 1e9, "GB/s",
                   f"{min(32, 2 * pool.n)} of 32 batches") if pool else None
    gbs = cache_bytes / (step_ms * 1e-3) / 1e9
    return section("MLA decode B=32 128 heads latent 512 + rope 64 L=8192", gbs, "GB/s", step_ms,
                   roofline("hbm", gbs, pk["hbm_gbs"], "GB/s", traffic.get("mla_kernel")), cpu,
                   tflops=round(32 * 8192 * 128 * (2 * 576 + 2 * 512) / (step_ms * 1e-3) / 1e12, 1))


def _prefill_section(name, flops, call, timer, steps, warmup, pk, traffic_key, traffic, cpu, peak=None, extra=None):
    call_ms, kern_ms = timer.cold(call, steps, warmup)
    km = statistics.mean(kern_ms)
    tf = flops / (km * 1e-3) / 1e12
    roof = roofline("tensor", tf, peak or pk["bf16_tflops"], "TFLOP/s", traffic.get(traffic_key))
    if extra:
        roof.update(extra)
    return section(name, tf, "TFLOP/s", km, roof, cpu, call_ms=round(statistics.mean(call_ms), 5))


def measure_prefill_tnd(torch, dev, timer, steps, warmup, pk, traffic, pool):
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

    cpu = None
    if pool:
        units = sample_units(len(c.actual_seq_qlen), c.num_heads, 2 * pool.n, 1)
        cpu = pool.run(oracle_tasks_tnd(c, units, mode=3, flops_of=lambda L: L * (L + 1) // 2 * 4 * 128), 1e12,
                       "TFLOP/s", f"{len(units)} of 256 (sequence, head) units")
    return _prefill_section("varlen TND causal prefill, 8 seqs U[256,4096], 32/8 heads, D=128, LSE", flops, call,
                            timer, steps, warmup, pk, "prefill_pair_kernel", traffic, cpu)


def measure_prefill_band(torch, dev, timer, steps, warmup, pk, traffic, pool):
    """The varlen TND workload with a sliding window (sparse_mode 4,
    pre_tokens 1024, next_tokens 0): each row sees its 1025 latest keys."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_tnd_varlen()
    pre = 1024
    lens = [b - a for a, b in zip([0] + c.actual_seq_qlen[:-1], c.actual_seq_qlen)]

    def pairs_of(L):
        return sum(min(i + 1, pre + 1) for i in range(L))

    flops = sum(pairs_of(L) for L in lens) * c.num_heads * 4 * c.q.shape[-1]
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="TND", sparse_mode=4, pre_tokens=pre, next_tokens=0,
                        actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                        softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    cpu = None
    if pool:
        units = sample_units(len(lens), c.num_heads, 2 * pool.n, 2)
        cpu = pool.run(oracle_tasks_tnd(c, units, mode=4, pre=pre, nxt=0, flops_of=lambda L: pairs_of(L) * 4 * 128),
                       1e12, "TFLOP/s", f"{len(units)} of 256 (sequence, head) units")
    return _prefill_section("varlen TND band prefill (1024 keys back), 8 seqs U[256,4096], 32/8 heads", flops, call,
                            timer, steps, warmup, pk, "prefill_pair_kernel_band", traffic, cpu)


def measure_prefill_mask(torch, dev, timer, steps, warmup, pk, traffic, pool):
    """The varlen TND workload with an explicit mask (sparse_mode 1): a uint8
    lower-triangular (4096, 4096) mask, i.e. causal attention given as a mask;
    flops count the allowed pairs only."""
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_tnd_varlen()
    flops = prefill_tnd_flops(c)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    mask_h = fia_inputs.atten_mask((4096, 4096), "causal")
    mask = mask_h.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], c.num_heads, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="TND", sparse_mode=1, atten_mask=mask,
                        actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                        softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    cpu = None
    if pool:
        units = sample_units(len(c.actual_seq_qlen), c.num_heads, 2 * pool.n, 3)
        cpu = pool.run(oracle_tasks_tnd(c, units, mode=1, mask=mask_h.numpy(),
                                        flops_of=lambda L: L * (L + 1) // 2 * 4 * 128),
                       1e12, "TFLOP/s", f"{len(units)} of 256 (sequence, head) units")
    return _prefill_section("varlen TND prefill, explicit uint8 causal mask (sparse_mode 1)", flops, call, timer,
                            steps, warmup, pk, "prefill_pair_kernel_mask", traffic, cpu)


def measure_chunked_prefill(torch, dev, timer, steps, warmup, pk, traffic, pool):
    """Chunked prefill against a paged cache: 8 sequences, a 2048-token chunk
    after a cached context U[0, 14336], 256-token blocks, right-down causal."""
    import numpy as np
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

    cpu = None
    if pool:
        # one (batch, head) unit: its chunk against its paged keys, as a one-batch call
        qn, kpn, vpn, tn = _np32(c.q), _np32(c.k_pool), _np32(c.v_pool), c.block_table.numpy()
        g = c.num_heads // c.num_key_value_heads
        tasks = []
        for (b, h) in sample_units(len(c.kv_lens), c.num_heads, 2 * pool.n, 4):
            L, ql = c.kv_lens[b], c.q_lens[b]
            nb = (L + c.block_size - 1) // c.block_size
            k_sub, t_sub = _sub_pool(kpn[:, h // g:h // g + 1], tn[b], nb)
            v_sub, _ = _sub_pool(vpn[:, h // g:h // g + 1], tn[b], nb)
            kw = dict(q=qn[b:b + 1, h:h + 1, :ql], k=k_sub, v=v_sub, block_table=t_sub, block_size=c.block_size,
                      actual_seq_kvlen=[L], num_heads=1, num_key_value_heads=1, input_layout="BNSD",
                      scale_value=c.scale, sparse_mode=3, actual_seq_qlen=[ql])
            tasks.append(("fia_prefill_paged", kw, sum(L - ql + i + 1 for i in range(ql)) * 4 * D))
        cpu = pool.run(tasks, 1e12, "TFLOP/s", f"{len(tasks)} of 256 (batch, head) units")
    return _prefill_section("chunked prefill, paged cache: 8 x 2048-token chunks after U[0,14336] cached", flops,
                            call, timer, steps, warmup, pk, "prefill_pair_kernel_chunked", traffic, cpu)


def measure_mla_prefill(torch, dev, timer, steps, warmup, pk, traffic, pool):
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

    cpu = None
    if pool:
        cpu = pool.run(oracle_tasks_tnd(c, sample_units(len(lens), c.num_heads, 2 * pool.n, 5), mode=3,
                                        flops_of=lambda L: L * (L + 1) // 2 * 2 * (192 + 128)),
                       1e12, "TFLOP/s", f"{2 * pool.n} of 256 (sequence, head) units")
    return _prefill_section("MLA prefill TND, 8 seqs U[256,4096], 32 heads, D 192/128, causal", flops, call, timer,
                            steps, warmup, pk, "prefill_pair_kernel_mla", traffic, cpu)


def oracle_tasks_bsa(c, units, qblocks, fp8=None):
    """One task per (batch, head, run of query blocks): those query rows
    against the head's keys, with the matching rows of blockSparseMask."""
    import numpy as np
    q, k, v = _np32(c.q), _np32(c.k), _np32(c.v)
    m = c.mask.numpy()
    X, Y = c.block_shape
    g = c.num_heads // c.num_key_value_heads
    tasks = []
    for (b, h, qb0) in units:
        r0, r1 = qb0 * X, min((qb0 + qblocks) * X, q.shape[2])
        kw = dict(q=q[b:b + 1, h:h + 1, r0:r1], k=k[b:b + 1, h // g:h // g + 1], v=v[b:b + 1, h // g:h // g + 1],
                  block_sparse_mask=m[b:b + 1, h:h + 1, qb0:qb0 + qblocks], block_shape=c.block_shape, num_heads=1,
                  num_key_value_heads=1, scale_value=c.scale, input_layout="BNSD")
        if fp8 is not None:
            qs, ks, vs = (x.numpy() for x in fp8)
            kw.update(q_dequant_scale=qs[b:b + 1, h:h + 1, qb0:qb0 + qblocks],
                      k_dequant_scale=ks[b:b + 1, h // g:h // g + 1], v_dequant_scale=vs[b:b + 1, h // g:h // g + 1])
        rows = np.array([min(X, q.shape[2] - i * X) for i in range(qb0, qb0 + qblocks)])
        cols = np.array([min(Y, k.shape[2] - j * Y) for j in range(m.shape[3])])
        pairs = float(((m[b, h, qb0:qb0 + qblocks] != 0) * np.outer(rows, cols)).sum())
        tasks.append(("bsa_forward", kw, pairs * 4 * q.shape[-1]))
    return tasks


def measure_bsa(torch, dev, timer, steps, warmup, pk, traffic, pool):
    import numpy as np
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

    cpu = None
    if pool:
        rng = np.random.default_rng(6)
        units = [(int(rng.integers(2)), int(rng.integers(32)), 4 * int(rng.integers(32))) for _ in range(2 * pool.n)]
        cpu = pool.run(oracle_tasks_bsa(c, units, 4), 1e12, "TFLOP/s",
                       f"{len(units)} runs of 4 query blocks of one (batch, head)")
    return _prefill_section("block-sparse prefill B=2 32/8 heads S=16384 D=128, 128x128 blocks, diag + 25%", flops,
                            call, timer, max(3, steps // 4), max(3, warmup), pk, "bsa_kernel", traffic, cpu)


def measure_bsa_fp8(torch, dev, timer, steps, warmup, pk, traffic, pool):
    """FP8 block-sparse prefill: the bf16 workload's shapes in e4m3 with
    per-block dequant scales, 128 x 256 blocks (the quantisation blocks).
    Q K^T runs at the fp8 tensor rate (2x bf16, the recipe's nominal ratio),
    P V in bf16, so the peak is the harmonic blend of the two halves of the
    work: 2 / (1 / (2 P) + 1 / P) = 4/3 P -- a derived figure, not a measured
    fp8 peak."""
    import numpy as np
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

    cpu = None
    if pool:
        rng = np.random.default_rng(7)
        units = [(int(rng.integers(2)), int(rng.integers(32)), 4 * int(rng.integers(32))) for _ in range(2 * pool.n)]
        cpu = pool.run(oracle_tasks_bsa(c, units, 4, fp8=(f.q_scale, f.k_scale, f.v_scale)), 1e12, "TFLOP/s",
                       f"{len(units)} runs of 4 query blocks of one (batch, head)")
    peak = round(pk["bf16_tflops"] * 4 / 3, 1)
    return _prefill_section("FP8 e4m3 block-sparse prefill (per-block scales), 128x256 blocks, bf16 out", flops, call,
                            timer, max(3, steps // 4), max(3, warmup), pk, "bsa_fp8_kernel", traffic, cpu,
                            peak=peak, extra={"peak_source": "measured bf16 x 4/3, derived (nominal fp8 = 2x bf16)"})


def measure_fp8_dense(torch, dev, timer, steps, warmup, pk, traffic, pool):
    """Dense FP8 prefill (the FP8 block-sparse call without a mask: every
    key), B=2 32/8 heads S=4096 D=128, per-block scales; the same blended
    peak as the block-sparse FP8 section."""
    import numpy as np
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    f = fia_inputs.workload_fp8_dense()
    c = f.base
    flops = bsa_flops(c)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    qs, ks, vs = f.q_scale.to(dev), f.k_scale.to(dev), f.v_scale.to(dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[0], c.num_heads, q.shape[2], 1), dtype=torch.float32, device=dev)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.bsa_forward(q, k, v, None, c.block_shape, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                        scale_value=c.scale, input_layout="BNSD", softmax_lse_flag=True, out=out, softmax_lse=lse,
                        workspace=ws, q_dequant_scale=qs, k_dequant_scale=ks, v_dequant_scale=vs)

    cpu = None
    if pool:
        rng = np.random.default_rng(8)
        units = [(int(rng.integers(2)), int(rng.integers(32)), 4 * int(rng.integers(8))) for _ in range(pool.n)]
        cpu = pool.run(oracle_tasks_bsa(c, units, 4, fp8=(f.q_scale, f.k_scale, f.v_scale)), 1e12, "TFLOP/s",
                       f"{len(units)} runs of 4 query blocks of one (batch, head)")
    peak = round(pk["bf16_tflops"] * 4 / 3, 1)
    return _prefill_section("dense FP8 e4m3 prefill (per-block scales, no mask), B=2 32/8 heads S=4096, bf16 out",
                            flops, call, timer, max(3, steps // 4), max(3, warmup), pk, "bsa_fp8_kernel_dense",
                            traffic, cpu, peak=peak,
                            extra={"peak_source": "measured bf16 x 4/3, derived (nominal fp8 = 2x bf16)"})


def measure_small_prefill(torch, dev, timer, steps, warmup, pk, traffic, pool):
    import attention_fia_prefill_gb300 as fia
    import fia_inputs
    c = fia_inputs.workload_prefill_bnsd_f16_small()
    flops = 2 * (128 * 129 // 2) * 4 * 64
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((1, 2, 128, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)

    def call():
        fia.fia_prefill(q, k, v, num_heads=2, scale_value=c.scale, input_layout="BNSD", sparse_mode=2,
                        softmax_lse_flag=True, out=out, softmax_lse=lse, workspace=ws)

    call_ms, kern_ms = timer.cold(call, steps, warmup)
    km = statistics.mean(kern_ms)
    cpu = None
    if pool:
        kw = dict(q=_np32(c.q), k=_np32(c.k), v=_np32(c.v), num_heads=2, scale_value=c.scale, input_layout="BNSD",
                  sparse_mode=2)
        cpu = pool.run([("fia_prefill", kw, flops)] * pool.n, 1e12, "TFLOP/s", "the whole workload, once per core")
    return section("prefill BNSD fp16 B=1 N=2 S=128 D=64 causal (latency)", flops / (km * 1e-3) / 1e12, "TFLOP/s", km,
                   roofline("tensor", flops / (km * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s"), cpu,
                   call_us=round(statistics.mean(call_ms) * 1e3, 2))


# ------------------------------------------------------------------ CPU oracle baseline
# The fp64 oracle as it stands, run on the host cores by a pool of spawned
# worker processes (one per core, single-threaded BLAS each), over a bounded
# sample of each workload cut into independent units -- a (batch, kv head)
# for decode, a (sequence, head) for prefill, a few query blocks of one head
# for block-sparse.  Each unit's inputs are sliced here (fp32 numpy, exact for
# fp16/bf16 values) and passed to the oracle's public functions unchanged.

def _oracle_warm(_):
    from oracle import fia_oracle  # noqa: F401
    time.sleep(0.2)
    return os.getpid()


def _oracle_task(task):
    fn, kwargs, work = task
    from oracle import fia_oracle
    getattr(fia_oracle, fn)(**kwargs)
    return work


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """Worker processes for the oracle, started with spawn (safe after CUDA
    initialisation) and warmed before any timing."""

    def __init__(self, workers=None):
        import concurrent.futures as cf
        import multiprocessing as mp
        self.n = workers or host_cores()
        for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        self.ex = cf.ProcessPoolExecutor(self.n, mp_context=mp.get_context("spawn"))
        pids = set(self.ex.map(_oracle_warm, range(2 * self.n)))
        self.n = len(pids) if pids else self.n

    def run(self, tasks, scale, unit, sample):
        """Work per second of wall time over the tasks (work in the metric's
        base unit, divided by scale)."""
        t0 = time.perf_counter()
        done = sum(self.ex.map(_oracle_task, tasks))
        wall = time.perf_counter() - t0
        return {"value": round(done / wall / scale, 6), "unit": unit, "cores": self.n, "kind": "oracle",
                "sample": sample, "wall_s": round(wall, 2)}

    def close(self):
        self.ex.shutdown(wait=True, cancel_futures=True)


def _np32(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def _sub_pool(pool, table_row, nb):
    """The blocks of one sequence as a pool of their own, with the table that
    maps them in order (the gather the oracle does is unchanged)."""
    import numpy as np
    blocks = table_row[:nb].astype(np.int64)
    return pool[blocks], np.arange(nb, dtype=np.int32)[None, :]


def oracle_tasks_decode(c, q_tokens=1, mode=0, max_units=None):
    """One task per (batch, kv head): its query heads against its paged keys."""
    import numpy as np
    q = _np32(c.q)
    kp, vp, tab = _np32(c.k_pool), _np32(c.v_pool), c.block_table.numpy()
    N1, N2, D = c.num_heads, c.num_key_value_heads, q.shape[-1]
    g = N1 // N2
    tasks = []
    for b, L in enumerate(c.kv_lens):
        nb = (L + c.block_size - 1) // c.block_size
        if nb == 0:
            continue
        for kvh in range(N2):
            k_sub, t_sub = _sub_pool(kp[:, kvh:kvh + 1], tab[b], nb)
            v_sub, _ = _sub_pool(vp[:, kvh:kvh + 1], tab[b], nb)
            kw = dict(q=q[b:b + 1, kvh * g:(kvh + 1) * g], k=k_sub, v=v_sub, num_heads=g, num_key_value_heads=1,
                      scale_value=c.scale, input_layout="BNSD", actual_seq_kvlen=[L], block_table=t_sub,
                      block_size=c.block_size, sparse_mode=mode)
            tasks.append(("fia_decode", kw, L * D * 2 * 2))
    return tasks[:max_units] if max_units else tasks


def oracle_tasks_mla_decode(c):
    """One task per batch: 128 heads against the latent + rope cache."""
    q, qr = _np32(c.q), _np32(c.q_rope)
    lat, rope, tab = _np32(c.latent), _np32(c.rope), c.block_table.numpy()
    tasks = []
    for b, L in enumerate(c.kv_lens):
        nb = (L + c.block_size - 1) // c.block_size
        l_sub, t_sub = _sub_pool(lat, tab[b], nb)
        r_sub, _ = _sub_pool(rope, tab[b], nb)
        kw = dict(q=q[b:b + 1], k=l_sub, v=l_sub, query_rope=qr[b:b + 1], key_rope=r_sub, num_heads=c.num_heads,
                  num_key_value_heads=1, scale_value=c.scale, input_layout="BSND", actual_seq_kvlen=[L],
                  block_table=t_sub, block_size=c.block_size)
        tasks.append(("fia_decode", kw, L * (512 + 64) * 2))
    return tasks


def oracle_tasks_tnd(c, units, mode=3, pre=2147483647, nxt=2147483647, mask=None, flops_of=None):
    """One task per (sequence, head) of a TND workload: that sequence alone
    as a one-batch TND call."""
    q, k, v = _np32(c.q), _np32(c.k), _np32(c.v)
    ends = c.actual_seq_qlen
    starts = [0] + ends[:-1]
    g = c.num_heads // c.num_key_value_heads
    tasks = []
    for (b, h) in units:
        s0, L = starts[b], ends[b] - starts[b]
        kw = dict(q=q[s0:s0 + L, h:h + 1], k=k[s0:s0 + L, h // g:h // g + 1], v=v[s0:s0 + L, h // g:h // g + 1],
                  num_heads=1, scale_value=c.scale, input_layout="TND", sparse_mode=mode,
                  actual_seq_qlen=[L], actual_seq_kvlen=[L], pre_tokens=pre, next_tokens=nxt)
        if mask is not None:
            kw["atten_mask"] = mask[:L, :L]
        tasks.append(("fia_prefill", kw, flops_of(L)))
    return tasks


def sample_units(n_seq, n_heads, count, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    pairs = [(b, h) for b in range(n_seq) for h in range(n_heads)]
    idx = rng.permutation(len(pairs))[:count]
    return [pairs[i] for i in sorted(idx)]


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
    torch.cuda.synchronize()
    clocks = sampler.stop()
    sections = {}
    pool = None
    if rank == 0 and not args.no_cpu_baseline:
        pool = OraclePool()
    if not args.headline_only:
        # least important first: the driver keeps the tail of the line
        for name, fn in (("prefill_small", measure_small_prefill), ("fp8_dense", measure_fp8_dense),
                         ("bsa_fp8", measure_bsa_fp8),
                         ("mla_prefill", measure_mla_prefill), ("prefill_band", measure_prefill_band),
                         ("prefill_mask", measure_prefill_mask), ("chunked_prefill", measure_chunked_prefill),
                         ("decode_q4", measure_decode_tokens), ("bsa", measure_bsa), ("mla_decode", measure_mla),
                         ("prefill_tnd", measure_prefill_tnd)):
            try:
                sections[name] = fn(torch, dev, timer, args.steps, args.warmup, pk, traffic, pool)
            except Exception as e:  # a section failure is reported, not hidden
                sections[name] = {"error": repr(e)[:200]}
            torch.cuda.empty_cache()
    cpu = None
    if pool is not None:
        cpu = pool.run(oracle_tasks_decode(case), 1e9, "GB/s",
                       "the whole paged GQA decode workload, one task per (batch, kv head)")
        pool.close()
    dec["step_ms"], dec["e2e_ms"] = max_over_ranks([dec["step_ms"], dec["e2e_ms"]], device=dev)
    if rank != 0:
        return
    value = ws_ * dec["kv_bytes"] / (dec["step_ms"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dec["step_ms"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "paged GQA decode bf16: B=16, Q_N=32, KV_N=8, Q_S=1, D=128, "
                               "actual_seq_kvlen U[1,4096], block_size=128, random block_table",
                   "kv_bytes_per_step": dec["kv_bytes"],
                   "l2": f"inputs larger than L2: calls back to back over {ROTATE} copies of the KV pools",
                   "parallelism": f"replicas x{ws_}"},
        "e2e": {"value": round(ws_ * dec["kv_bytes"] / (dec["e2e_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": dec["h2d"], "d2h_bytes_per_step": dec["d2h"]},
        "gpu_launches": args.steps,
        "roofline": dict(dec["roofline"], peak_source=pk_src),
        "host_us_per_call": round(dec["host_us"], 2),
        "cold_us": {"call": round(dec["cold_call_us"], 2), "kernel": round(dec["cold_kernel_us"], 2)},
        "clocks": clocks,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    line["sections"] = sections
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The oracle (fp64, host cores) on the headline workload: every step runs
    a bounded sample of it -- a slice of the (batch, kv head) units -- on the
    worker pool."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    import fia_inputs
    c = fia_inputs.workload_paged_gqa_decode()
    pool = OraclePool()
    tasks = oracle_tasks_decode(c)
    per = max(pool.n, len(tasks) // 8)   # units per step
    times, done = [], 0
    for step in range(args.warmup + args.steps):
        i0 = (step * per) % len(tasks)
        chunk = (tasks + tasks)[i0:i0 + per]
        t0 = time.perf_counter()
        work = sum(pool.ex.map(_oracle_task, chunk))
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            done += work
    pool.close()
    total = sum(times)
    value = done / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "paged GQA decode bf16: B=16, Q_N=32, KV_N=8, Q_S=1, D=128, "
                                   "actual_seq_kvlen U[1,4096], block_size=128, random block_table"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": pool.n, "kind": "oracle",
                             "sample": f"{per} of {len(tasks)} (batch, kv head) units per step, cycling"},
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
    elif name in ("bsa_fp8", "fp8_dense"):
        f = fia_inputs.workload_bsa_fp8() if name == "bsa_fp8" else fia_inputs.workload_fp8_dense()
        c = f.base
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        m = c.mask.to(dev) if name == "bsa_fp8" else None
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
    elif name == "decode_q4":
        base = fia_inputs.workload_paged_gqa_decode()
        c = fia_inputs.paged_decode_case(16, 32, 8, 128, base.kv_lens, block_size=128, workload=3400, q_tokens=4)
        q, kp, vp, tb = c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev), c.block_table.to(dev)

        def call():
            fia.fia_decode(q, kp, vp, block_table=tb, block_size=c.block_size, actual_seq_kvlen=c.kv_lens,
                           num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                           input_layout="BNSD", sparse_mode=3, softmax_lse_flag=True)
    elif name == "chunked":
        c = fia_inputs.workload_chunked_prefill()
        q, kp, vp, tab = c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev), c.block_table.to(dev)

        def call():
            fia.fia_prefill_paged(q, kp, vp, tab, block_size=c.block_size, actual_seq_kvlen=c.kv_lens,
                                  actual_seq_qlen=c.actual_seq_qlen, num_heads=c.num_heads,
                                  num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                  input_layout="BNSD", sparse_mode=3, softmax_lse_flag=True)
    elif name in ("prefill_band", "prefill_mask"):
        c = fia_inputs.workload_tnd_varlen()
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        mask = fia_inputs.atten_mask((4096, 4096), "causal").to(dev) if name == "prefill_mask" else None
        kw = (dict(sparse_mode=4, pre_tokens=1024, next_tokens=0) if name == "prefill_band"
              else dict(sparse_mode=1, atten_mask=mask))

        def call():
            fia.fia_prefill(q, k, v, num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                            scale_value=c.scale, input_layout="TND", actual_seq_qlen=c.actual_seq_qlen,
                            actual_seq_kvlen=c.actual_seq_kvlen, softmax_lse_flag=True, **kw)
    else:
        raise SystemExit(f"unknown profile target {name}")
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    print(f"profile target {name}: {args.warmup + args.steps} calls done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", default=None, help="only run plain calls of one workload (decode, decode_q4, prefill_tnd, prefill_band, prefill_mask, chunked, bsa, bsa_fp8, fp8_dense, mla, mla_prefill)")
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
