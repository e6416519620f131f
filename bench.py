#!/usr/bin/env python
"""Benchmark of the quantized-KV MLA attention path on GB300.

Headline workload (``kv8_ragged``): long-context ragged decode, KV8.  32
sequences whose lengths are uniform in [1024, 131072] (splitmix64 seed 4,
2,256,568 cached rows in all), 128 heads sharing one 576-dim latent cache
(fp8 e4m3 codes + two f32 scales per row, 584 B), one bf16 query token per
sequence and head.  One step = one call of kv_attn_decode_append: the step's
32 new rows (the last row of each sequence's range) are encoded to KV8 and
stored, then attention runs over every row, the new ones included (split-T
partials + merge).  On the tensor-core path both happen in one launch, plus
the merge.  The cache (1.32 GB) is ten times the L2, so no flush is needed
between steps.

The same JSON line carries, under ``workloads``, the other timed workloads:

* ``tq4_ragged``   the same ragged decode step on a TQ4 cache (296 B/row; the
                   encoder launch, then the decode);
* ``kv8_prefill`` / ``tq4_prefill``  chunked causal prefill: 2048 new rows
                   encoded and appended to a 124 x 1024 = 126,976-row cache,
                   then 2048 tokens x 128 heads attend rows [0, P + j];
* ``kv8_8x4096`` / ``tq4_8x4096``  decode of 8 sequences x 4096 rows (KV8
                   19 MB, TQ4 9.7 MB, both fit in L2: a 256 MB buffer is
                   written between timed steps);
* ``pq4_8x4096`` / ``pq4t_8x4096``  the same short decode step on a PolarQuant
                   4-bit cache (296 B/row), on the fp32 consumer (the default
                   path for PolarQuant) and on the tensor-core consumer;
* ``k2v4_4x32768`` the K2/V4 GQA decode: 4 sequences x 32768 cells, 2 kv
                   heads x 256 dims, 16 query heads, sinks 8 + window 256 in
                   the fp16 overlay, K gain 1.10 (60.4 MB, fits in L2: flushed
                   between steps); its roofline is HBM (36 flop per byte).

Inputs are synthetic and seeded (quantized_kv_cache_kv8_gb300.synth): latent
rows N(0,1) x per-channel log-normal gains, N(0,1) queries rounded to bf16.
The ragged pool is built from one encoded master block of 131072 rows:
sequence b holds master rows (o_b + t) mod 131072, o_b = 40961 b mod 131072.

Metric: cache GB/s = rows read per step x row bytes / step time; rows/s and
the fraction of the measured HBM copy bandwidth beside it.  ``roofline`` is
the dominant kernel against the bf16 tensor roof (278,528 flop per row at 128
heads is above the GB300 ridge), timed by CUDA events the library records on
the launch stream (kvq_timing_enable).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--path auto|simt|tensor] [--workloads a,b,...]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, D, DV = 128, 576, 512
ROW_BYTES = {1: 576 + 2 * 4, 2: 288 + 2 * 4, 14: 288 + 2 * 4}   # KV8, TQ4, PolarQuant 4-bit
FORMAT_NAMES = {1: "KV8", 2: "TQ4", 14: "PolarQuant-4"}
FLOPS_PER_ROW = H * (D + DV) * 2
SM_SCALE = 1.0 / math.sqrt(192.0)
METRIC = "quantized-KV MLA decode attn: cache GB/s & % of HBM roofline; rows/s"

# ragged long-context decode
RAGGED_SEED, RAGGED_B, RAGGED_LO, RAGGED_HI, MASTER = 4, 32, 1024, 131072, 131072
# chunked causal prefill
PREFILL_PAST, PREFILL_NEW = 124 * 1024, 2048
# short decode (fits in L2)
SHORT_B, SHORT_T, SHORT_SEED = 8, 4096, 2
# K2/V4 GQA decode
K2_B, K2_H, K2_T, K2_D, K2_HQ, K2_SINK, K2_WINDOW, K2_SLACK, K2_GAIN, K2_SEED = 4, 2, 32768, 256, 16, 8, 256, 16, 1.10, 5

WORKLOAD_NAMES = {
    "kv8_ragged": "ragged decode, KV8: 32 seqs, lengths U[1024,131072] (seed 4), 128 heads, 576-dim latent "
                  "(512+64), bf16 query, the step's 32 new rows appended",
    "tq4_ragged": "ragged decode, TQ4: 32 seqs, lengths U[1024,131072] (seed 4), 128 heads, 576-dim latent "
                  "(512+64), bf16 query, the step's 32 new rows appended",
    "kv8_prefill": "chunked causal prefill, KV8: 2048 new rows encoded onto 126976 cached rows, "
                   "2048 tokens x 128 heads, bf16 query",
    "tq4_prefill": "chunked causal prefill, TQ4: 2048 new rows encoded onto 126976 cached rows, "
                   "2048 tokens x 128 heads, bf16 query",
    "kv8_8x4096": "decode, KV8: 8 seqs x 4096 rows, 128 heads, bf16 query, the step's 8 new rows appended",
    "tq4_8x4096": "decode, TQ4: 8 seqs x 4096 rows, 128 heads, bf16 query, the step's 8 new rows appended",
    "pq4_8x4096": "decode, PolarQuant 4-bit: 8 seqs x 4096 rows, 128 heads, bf16 query, the step's 8 new rows "
                  "appended (fp32 consumer, the default path)",
    "pq4t_8x4096": "decode, PolarQuant 4-bit: 8 seqs x 4096 rows, 128 heads, bf16 query, the step's 8 new rows "
                   "appended (tensor-core consumer, KVQ_PATH_TENSOR)",
    "k2v4_4x32768": "GQA decode, K2/V4: 4 seqs x 32768 cells, 2 kv heads x 256, 16 query heads, f32 query, "
                    "sinks 8 + window 256 fp16, K gain 1.10",
}
DEFAULT_WORKLOADS = ["kv8_ragged", "tq4_ragged", "kv8_prefill", "tq4_prefill", "kv8_8x4096", "tq4_8x4096",
                     "pq4_8x4096", "pq4t_8x4096", "k2v4_4x32768"]

# profile summaries holding the ncu DRAM traffic of a dominant kernel, keyed by workload
PROFILE_FOR = {"kv8_ragged": "decode_tc_kv8_ragged_b32_h128.md", "tq4_ragged": "decode_tc_tq4_ragged_b32_h128.md",
               "kv8_prefill": "prefill_tc_kv8_p126976_n2048_h128.md",
               "tq4_prefill": "prefill_tc_tq4_p126976_n2048_h128.md",
               "k2v4_4x32768": "decode_tc_k2v4_b4_t32768.md",
               "kv8_8x4096": "decode_tc_kv8_b8_t4096_h128.md", "tq4_8x4096": "decode_tc_tq4_b8_t4096_h128.md"}
# the sources whose hash a traffic figure is tied to (the kernel changed => no figure)
KERNEL_SOURCES = {1: ["attn_tc_kv8.cu", "tc_common.cuh", "attn_common.cuh", "kvq_internal.cuh"],
                  2: ["attn_tc_tq4.cu", "tc_common.cuh", "attn_common.cuh", "kvq_internal.cuh"],
                  "k2v4": ["k2v4.cu", "tc_common.cuh", "attn_common.cuh", "kvq_internal.cuh"]}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


def kernel_source_hash(fmt: int) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[fmt]:
        with open(os.path.join(ROOT, "quantized_kv_cache_kv8_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, fmt: int):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when there is none or the kernel source has changed since
    (the summary records the source hash it was taken on)."""
    name = PROFILE_FOR.get(workload)
    if not name:
        return None, "no capture for this workload"
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None, "no capture committed"
    with open(path) as f:
        text = f.read()
    m = re.search(r"traffic_bytes_per_launch=(\d+)\s+source_sha256=([0-9a-f]+)", text)
    if not m:
        return None, "capture has no traffic line"
    if m.group(2) != kernel_source_hash(fmt):
        return None, "kernel changed since the capture"
    return int(m.group(1)), f"ncu dram__bytes_read.sum + dram__bytes_write.sum, profiles/{name}"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[tuple[float, list[str]]] = []
        self.windows: list[tuple[float, float]] = []
        self._t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, begin: bool):
        if begin:
            self._t0 = time.time()
        else:
            self.windows.append((self._t0, time.time()))

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [f for t, f in self.lines if any(a <= t <= b for a, b in self.windows)]
        window = "timed"
        if len(inside) < 3:
            inside = [f for _, f in self.lines]
            window = "warmup+timed"
        sm = [float(f[1]) for f in inside if f[1].replace(".", "").isdigit()]
        mx = [float(f[2]) for f in inside if f[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for f in inside for i in range(4) if len(f) > 5 + i and f[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window}


def ragged_layout():
    from quantized_kv_cache_kv8_gb300 import synth
    lens = synth.ragged_lengths(RAGGED_SEED, RAGGED_B, RAGGED_LO, RAGGED_HI)
    cu = synth.cu_seqlens(lens)
    offs = (np.arange(RAGGED_B, dtype=np.int64) * 40961) % MASTER
    return lens, cu, offs


def max_over_ranks(vals, dist, device):
    """Each timing's maximum over the ranks: the slowest replica bounds the job."""
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.barrier()
    return t.tolist()


def job_rate_gbs(rows_per_rank, world, ms, row_bytes=ROW_BYTES[1]):
    """Whole-job cache throughput: every replica's rows over the slowest step time."""
    return rows_per_rank * world * row_bytes / (ms * 1e-3) / 1e9


class Ctx:
    """Device state shared by the workloads of one run."""

    def __init__(self, torch, kvq, args):
        self.torch, self.kvq, self.args = torch, kvq, args
        self.dev = torch.device("cuda")
        self.stream = torch.cuda.current_stream()
        self.path = {"auto": kvq.PATH_AUTO, "simt": kvq.PATH_SIMT, "tensor": kvq.PATH_TENSOR}[args.path]
        self._master_x = None
        self._prefill_q = None

    def prefill_q_bits(self):
        if self._prefill_q is None:
            from quantized_kv_cache_kv8_gb300 import synth
            self._prefill_q = synth.bf16_bits(synth.queries(42, (PREFILL_NEW, H, D)))
        return self._prefill_q

    def master_x(self):
        if self._master_x is None:
            from quantized_kv_cache_kv8_gb300 import synth
            self._master_x = synth.mla_rows(RAGGED_SEED, MASTER)
        return self._master_x

    def encode(self, fmt, x_dev, layout):
        torch, kvq = self.torch, self.kvq
        n = x_dev.shape[0]
        codes = torch.empty((n, kvq.row_bytes(fmt, layout)), dtype=torch.uint8, device=self.dev)
        scales = torch.empty((n, 2), dtype=torch.float32, device=self.dev)
        if fmt == 1:
            kvq.kv8_encode(x_dev, codes, scales, layout)
        elif fmt == 2:
            kvq.tq4_encode(x_dev, codes, scales, layout)
        else:
            kvq.pq_encode(fmt, x_dev, codes, scales, layout)
        return codes, scales


def timed_loop(torch, step, K, stream, flush=None, sampler=None):
    """Mean ms of K steps, each bracketed by CUDA events on the launch stream."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    for i in range(K):
        a, b = ev[i]
        a.record(stream)
        step()
        b.record(stream)
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    return sum(a.elapsed_time(b) for a, b in ev) / K


def kernel_timing(kvq, torch, step, K, flush=None):
    """The partial kernel and the merge alone: the library's launch events
    before each call's partial kernel and before and after its merge.  A loop of
    its own: the record between the two kernels ends the merge's programmatic
    overlap, so these calls are not the ones the step timing measures."""
    kvq.timing_enable(K)
    for _ in range(K):
        step()
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize()
    part_sum, merge_sum, n = kvq.timing_read()
    kvq.timing_enable(0)
    if n != K:
        raise RuntimeError(f"launch timing recorded {n} of {K} calls")
    return part_sum / K, merge_sum / K


def setup_decode(ctx, fmt, workload):
    """A decode workload: the resident pool, the step's inputs in one pinned
    staging buffer (bf16 queries, then the f32 new rows) and its device copy."""
    torch, kvq = ctx.torch, ctx.kvq
    from quantized_kv_cache_kv8_gb300 import synth
    layout = kvq.mla_layout(seed=RAGGED_SEED)
    if workload.endswith("ragged"):
        lens, cu, offs = ragged_layout()
        mc, ms = ctx.encode(fmt, torch.from_numpy(ctx.master_x()).to(ctx.dev), layout)
        idx = np.concatenate([(o + np.arange(T, dtype=np.int64)) % MASTER for o, T in zip(offs, lens)])
        idx_t = torch.from_numpy(idx).to(ctx.dev)
        codes, scales = mc[idx_t].contiguous(), ms[idx_t].contiguous()
        del mc, ms, idx_t
        q_seed, x_seed, B = RAGGED_SEED + 1, RAGGED_SEED + 100, RAGGED_B
    else:
        B = SHORT_B
        cu = synth.cu_seqlens([SHORT_T] * B)
        codes, scales = ctx.encode(fmt, torch.from_numpy(synth.mla_rows(SHORT_SEED, B * SHORT_T)).to(ctx.dev), layout)
        q_seed, x_seed = SHORT_SEED + 1, SHORT_SEED + 100
    total = int(cu[-1])
    q_bits = synth.bf16_bits(synth.queries(q_seed, (B, H, D)))
    new_rows = synth.mla_rows(x_seed, B)
    q_bytes, x_bytes = B * H * D * 2, B * D * 4
    stage_host = torch.empty(q_bytes + x_bytes, dtype=torch.uint8).pin_memory()
    stage_host[:q_bytes].view(torch.int16).copy_(torch.from_numpy(q_bits.view(np.int16).reshape(-1)))
    stage_host[q_bytes:].view(torch.float32).copy_(torch.from_numpy(new_rows.reshape(-1)))
    stage = stage_host.to(ctx.dev)
    q = stage[:q_bytes].view(torch.bfloat16).view(B, H, D)
    x_new = stage[q_bytes:].view(torch.float32).view(B, D)
    out = torch.empty((B, H, DV), dtype=torch.float32, device=ctx.dev)
    out_host = torch.empty((B, H, DV), dtype=torch.float32).pin_memory()
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, B, H, total, layout, ctx.path), dtype=torch.uint8,
                     device=ctx.dev)
    d = dict(layout=layout, codes=codes, scales=scales, cu=torch.from_numpy(cu).to(ctx.dev),
             dst=torch.from_numpy(cu[1:] - 1).to(ctx.dev), stage_host=stage_host, stage=stage, q=q, x_new=x_new,
             out=out, out_host=out_host, ws=ws, total=total, B=B, q_bytes=q_bytes)

    def step():
        kvq.kv_attn_decode_append(fmt, d["x_new"], d["dst"], d["q"], d["codes"], d["scales"], d["cu"], d["out"],
                                  d["ws"], total, layout=layout, path=ctx.path)
    d["step"] = step
    return d


def used_path(ctx, fmt):
    kvq = ctx.kvq
    if fmt not in (1, 2):
        # PolarQuant: the fp32 consumer unless the tensor path is asked for (4 bits)
        return "tensor" if (fmt == 14 and ctx.path == kvq.PATH_TENSOR) else "simt"
    return "tensor" if (ctx.path == kvq.PATH_TENSOR or (ctx.path == kvq.PATH_AUTO and H % 64 == 0)) else "simt"


def roofline(ctx, peaks, src, fmt, workload, rows, kernel_ms, sustained=False, kernel_name=""):
    path = used_path(ctx, fmt)
    flops = rows * FLOPS_PER_ROW
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    if path == "simt":
        peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        return {"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 2), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": None,
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 x max SM clock (MEASURED_PEAKS sm_max_mhz)",
                "kernel": kernel_name or "attn_partial_kernel (fp32 split-T partials)"}
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = peaks.get(key, peaks["bf16_tflops"])
    traffic, tsrc = profiled_traffic(workload, fmt)
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": tsrc,
            "algorithmic_bytes": int(rows * ROW_BYTES[fmt]),
            "peak_source": f"{key} ({src} of measured); f16 operands run at the bf16 dense rate",
            "kernel": kernel_name}


def pipelined_e2e(ctx, fmt, d, K, sampler=None):
    """End to end through the public call, two steps deep: step i's
    host-to-device copy of its inputs (pinned staging buffer) and its
    device-to-host copy of its result run on two copy streams beside the
    kernels, with the device inputs and outputs double-buffered, so that the
    copies of one step overlap the kernels of its neighbours.  Every step still
    moves its own inputs in and its own result out inside the timed region,
    which events on the launch stream bracket around all K steps (the first
    input copy waits for the opening event, the closing one for the last
    result copy).  Mean ms per step."""
    torch, kvq = ctx.torch, ctx.kvq
    stream = ctx.stream
    s_in, s_out = torch.cuda.Stream(device=ctx.dev), torch.cuda.Stream(device=ctx.dev)
    qb, B = d["q_bytes"], d["B"]
    stage = [d["stage"], torch.empty_like(d["stage"])]
    outs = [d["out"], torch.empty_like(d["out"])]
    out_host = [d["out_host"], torch.empty_like(d["out_host"]).pin_memory()]
    qs = [st[:qb].view(torch.bfloat16).view(d["q"].shape) for st in stage]
    xs = [st[qb:].view(torch.float32).view(B, -1) for st in stage]
    ev = lambda: torch.cuda.Event()
    in_ready, k_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    start.record(stream)
    for i in range(K):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(start if i < 2 else k_done[b])   # stage[b] last read by step i - 2
            stage[b].copy_(d["stage_host"], non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(d2h_done[b])                   # outs[b] last read by step i - 2's copy
        kvq.kv_attn_decode_append(fmt, xs[b], d["dst"], qs[b], d["codes"], d["scales"], d["cu"], outs[b], d["ws"],
                                  d["total"], layout=d["layout"], path=ctx.path, stream=stream)
        k_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(k_done[b])
            out_host[b].copy_(outs[b], non_blocking=True)
            d2h_done[b].record(s_out)
    stream.wait_event(d2h_done[0])
    stream.wait_event(d2h_done[1])
    end.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    return start.elapsed_time(end) / K


def run_decode(ctx, fmt, workload, K, W, peaks, src, sampler, world, dist, e2e=False):
    torch, kvq = ctx.torch, ctx.kvq
    d = setup_decode(ctx, fmt, workload)
    flush = None
    if workload.endswith("8x4096"):
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=ctx.dev)
    for _ in range(max(W, 3)):
        d["step"]()
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize()
    if kvq.read_device_error(d["ws"]) != 0:
        raise RuntimeError(f"{workload}: device error word set during warm-up")
    if dist:
        dist.barrier()
    kvq.read_exact_rescales(d["ws"])   # clears the counter
    step_ms = timed_loop(torch, d["step"], K, ctx.stream, flush, sampler)
    exact_per_step = kvq.read_exact_rescales(d["ws"]) / K
    part_ms, merge_ms = kernel_timing(kvq, torch, d["step"], K, flush)
    e2e_ms = e2e_serial_ms = None
    if e2e:
        def e2e_step():
            d["stage"].copy_(d["stage_host"], non_blocking=True)
            d["step"]()
            d["out_host"].copy_(d["out"], non_blocking=True)
        e2e_serial_ms = timed_loop(torch, e2e_step, K, ctx.stream, flush, sampler)
        e2e_ms = pipelined_e2e(ctx, fmt, d, K, sampler)
    err = kvq.read_device_error(d["ws"])
    if err != 0:
        raise RuntimeError(f"{workload}: device error word {err} after the timed region")
    vals = max_over_ranks([step_ms, part_ms, merge_ms, e2e_ms or 0.0, e2e_serial_ms or 0.0], dist, ctx.dev)
    step_ms, part_ms, merge_ms, e2e_ms_m, e2e_serial_m = vals
    rows, B = d["total"], d["B"]
    path = used_path(ctx, fmt)
    kname = {1: "attn_tc_kv8_kernel<APPEND> (tcgen05 split-T partials with the row append)",
             2: "attn_tc_tq4_kernel (tcgen05 split-T partials, query rotated in the prologue)",
             14: "attn_tc_tq4_kernel<PQ> (tcgen05 split-T partials, PolarQuant trees rebuilt into f16 operands)"
             if path == "tensor" else
             "attn_partial_kernel<PolarQuant> (fp32 split-T partials, rows rebuilt per tile)"}[fmt]
    res = {
        "workload": WORKLOAD_NAMES[workload], "format": FORMAT_NAMES[fmt], "path": path,
        "rows": rows, "row_bytes": ROW_BYTES[fmt], "ms_per_step": round(step_ms, 5),
        "value": round(job_rate_gbs(rows, world, step_ms, ROW_BYTES[fmt]), 3), "unit": "GB/s",
        "rows_per_s": round(rows * world / (step_ms * 1e-3), 1),
        "hbm_roof_frac": round(job_rate_gbs(rows, 1, step_ms, ROW_BYTES[fmt]) / peaks["hbm_gbs"], 5),
        "timing": {"partial_ms": round(part_ms, 5), "merge_ms": round(merge_ms, 5),
                   "partial_share": round(part_ms / (part_ms + merge_ms), 4), "launches": K,
                   "how": "CUDA events recorded by the library on the launch stream around each call's "
                          "partial kernel and merge (kvq_timing_enable), a loop of K calls of its own"},
        "roofline": roofline(ctx, peaks, src, fmt, workload, rows, part_ms, kernel_name=kname),
        # tensor KV8: the fused partial kernel + merge; otherwise encoder, partials, merge
        "gpu_launches_per_step": 2 if (path == "tensor" and fmt == 1) else 3,
        "exact_rescale_tiles_per_step": exact_per_step,
        "l2": "256 MB buffer written between timed steps (outside the events)" if flush is not None
        else "inputs larger than L2 (no flush)",
    }
    if e2e:
        res["e2e"] = {"value": round(job_rate_gbs(rows, world, e2e_serial_m, ROW_BYTES[fmt]), 3), "unit": "GB/s",
                      "ms_per_step": round(e2e_serial_m, 5),
                      "h2d_bytes_per_step": int(B * D * 4 + B * H * D * 2),
                      "d2h_bytes_per_step": int(B * H * DV * 4),
                      "how": "kv_attn_decode_append with host buffers: copy in from pinned memory, call, copy "
                             "out, one after another on the launch stream, each step bracketed by its own events",
                      "pipelined": {"value": round(job_rate_gbs(rows, world, e2e_ms_m, ROW_BYTES[fmt]), 3),
                                    "ms_per_step": round(e2e_ms_m, 5),
                                    "how": "the same steps two deep: each step's input and result copies on "
                                           "two copy streams beside the neighbouring steps' kernels (double-"
                                           "buffered device inputs and outputs); events around all K steps"}}
    del d
    torch.cuda.empty_cache()
    return res


def k2v4_bytes():
    """Bytes a K2/V4 decode reads: bulk cells' K codes and V blocks, every K
    scale group, and the overlay cells' fp16 K and V."""
    ov = K2_SINK + K2_WINDOW
    bulk = K2_T - ov
    per = bulk * (K2_D // 4 + (K2_D // 32) * 18) + ov * 4 * K2_D + (K2_T // 32) * K2_D * 2
    return K2_B * K2_H * per


def run_k2v4(ctx, workload, K, W, peaks, sampler, world, dist):
    torch, kvq = ctx.torch, ctx.kvq
    from quantized_kv_cache_kv8_gb300 import synth
    layout = kvq.k2v4_layout(K2_H, K2_D, K2_GAIN, K2_SINK, K2_WINDOW, K2_SLACK)
    k, v = synth.gqa_kv(K2_SEED, K2_B, K2_H, K2_T, K2_D)
    slots = K2_SINK + K2_WINDOW + K2_SLACK
    dev = ctx.dev
    kc = torch.zeros((K2_B, K2_H, K2_T, K2_D // 4), dtype=torch.uint8, device=dev)
    ks = torch.zeros((K2_B, K2_H, K2_T // 32, K2_D), dtype=torch.int16, device=dev)
    vb = torch.zeros((K2_B, K2_H, K2_T, K2_D // 32, 18), dtype=torch.uint8, device=dev)
    kw = torch.zeros((K2_B, K2_H, slots, K2_D), dtype=torch.int16, device=dev)
    vw = torch.zeros((K2_B, K2_H, slots, K2_D), dtype=torch.int16, device=dev)
    kvq.k2v4_encode(layout, torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), kc, ks, vb, kw, vw)
    del k, v
    q = torch.from_numpy(synth.queries(K2_SEED + 1, (K2_B, K2_HQ, K2_D))).to(dev)
    out = torch.empty((K2_B, K2_HQ, K2_D), dtype=torch.float32, device=dev)
    pth = ctx.path if ctx.path != kvq.PATH_AUTO else kvq.PATH_AUTO
    ws = torch.zeros(kvq.kv_attn_decode_k2v4_workspace_size(layout, K2_B, K2_HQ, K2_T, pth), dtype=torch.uint8,
                     device=dev)
    sm = 1.0 / math.sqrt(K2_D)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        kvq.kv_attn_decode_k2v4(layout, q, K2_T, kc, ks, vb, kw, vw, out, ws, sm, path=pth)
    for _ in range(max(W, 3)):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    if kvq.read_device_error(ws) != 0:
        raise RuntimeError(f"{workload}: device error word set during warm-up")
    if dist:
        dist.barrier()
    step_ms = timed_loop(torch, step, K, ctx.stream, flush, sampler)
    part_ms, merge_ms = kernel_timing(kvq, torch, step, K, flush)
    if kvq.read_device_error(ws) != 0:
        raise RuntimeError(f"{workload}: device error word set")
    step_ms, part_ms, merge_ms = max_over_ranks([step_ms, part_ms, merge_ms], dist, ctx.dev)
    nbytes = k2v4_bytes()
    tensor = ctx.path != kvq.PATH_SIMT
    traffic, tsrc = profiled_traffic(workload, "k2v4") if tensor else (None, "no capture for the fp32 kernel")
    achieved = nbytes / (part_ms * 1e-3) / 1e9
    res = {
        "workload": WORKLOAD_NAMES[workload], "format": "K2/V4", "path": "tensor" if tensor else "simt",
        "ms_per_step": round(step_ms, 5), "value": round(nbytes * world / (step_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
        "bytes_per_step": nbytes,
        "timing": {"partial_ms": round(part_ms, 5), "merge_ms": round(merge_ms, 5),
                   "how": "CUDA events recorded by the library around the partial kernel and the merge"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "traffic_source": tsrc, "algorithmic_bytes": nbytes,
                     "peak_source": "hbm_gbs (measured)",
                     "kernel": "k2v4_tc_kernel<256> (tcgen05, tiles dequantized to f16 in shared memory)"
                     if tensor else "k2v4_partial_kernel (fp32)"},
        "gpu_launches_per_step": 2,
        "l2": "256 MB buffer written between timed steps (outside the events)",
    }
    del kc, ks, vb, kw, vw, q, out, ws, flush
    torch.cuda.empty_cache()
    return res


def prefill_flops(n_past, n_new):
    return FLOPS_PER_ROW * sum(n_past + j + 1 for j in range(n_new))


def run_prefill(ctx, fmt, workload, K, W, peaks, src, sampler, world, dist):
    torch, kvq = ctx.torch, ctx.kvq
    from quantized_kv_cache_kv8_gb300 import synth
    layout = kvq.mla_layout(seed=RAGGED_SEED)
    P, N = PREFILL_PAST, PREFILL_NEW
    xm = ctx.master_x()
    codes_past, scales_past = ctx.encode(fmt, torch.from_numpy(xm[:P]).to(ctx.dev), layout)
    codes = torch.zeros((P + N, codes_past.shape[1]), dtype=torch.uint8, device=ctx.dev)
    scales = torch.zeros((P + N, 2), dtype=torch.float32, device=ctx.dev)
    codes[:P], scales[:P] = codes_past, scales_past
    del codes_past, scales_past
    x_new = torch.from_numpy(xm[P:P + N].copy()).to(ctx.dev)
    q_bits = ctx.prefill_q_bits()
    q = torch.from_numpy(q_bits.view(np.int16)).to(ctx.dev).view(torch.bfloat16)
    out = torch.empty((N, H, DV), dtype=torch.float32, device=ctx.dev)
    ws = torch.zeros(kvq.kv_attn_prefill_workspace_size(fmt, H, P, N, layout, ctx.path), dtype=torch.uint8,
                     device=ctx.dev)

    def step():
        kvq.kv_attn_prefill(fmt, x_new, q, codes, scales, P, out, ws, SM_SCALE, layout, ctx.path)
    for _ in range(max(W, 3)):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    kvq.read_exact_rescales(ws)   # clears the counter
    step_ms = timed_loop(torch, step, K, ctx.stream, None, sampler)
    exact_per_step = kvq.read_exact_rescales(ws) / K
    part_ms, merge_ms = kernel_timing(kvq, torch, step, K)
    if kvq.read_device_error(ws) != 0:
        raise RuntimeError(f"{workload}: device error word set")
    step_ms, part_ms, merge_ms = max_over_ranks([step_ms, part_ms, merge_ms], dist, ctx.dev)
    flops = prefill_flops(P, N)
    path = used_path(ctx, fmt)
    kname = ("attn_tc_kv8_kernel (prefill: one work item per token)" if fmt == 1
             else "attn_tc_tq4_kernel (prefill: one work item per token)")
    # rows read: every token's causal range once per head group
    rows_attended = sum(P + j + 1 for j in range(N))
    roof = roofline(ctx, peaks, src, fmt, workload, rows_attended, part_ms, sustained=True, kernel_name=kname)
    roof.pop("algorithmic_bytes", None)
    res = {
        "workload": WORKLOAD_NAMES[workload], "format": "KV8" if fmt == 1 else "TQ4", "path": path,
        "ms_per_step": round(step_ms, 4),
        "value": round(flops * world / (step_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
        "tokens_per_s": round(N * world / (step_ms * 1e-3), 1),
        "algorithmic_flops": flops,
        "timing": {"partial_ms": round(part_ms, 4), "merge_ms": round(merge_ms, 4),
                   "how": "CUDA events recorded by the library around the partial kernel and the merge"},
        "roofline": roof,
        "gpu_launches_per_step": 3,
        "exact_rescale_tiles_per_step": exact_per_step,
        "l2": "inputs larger than L2 (no flush)",
    }
    del codes, scales, q, out, ws, x_new
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world):
    import torch
    from quantized_kv_cache_kv8_gb300 import kvq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    ctx = Ctx(torch, kvq, args)
    peaks, src = load_peaks()
    workloads = [w for w in args.workloads.split(",") if w]
    for w in workloads:
        if w not in WORKLOAD_NAMES:
            raise SystemExit(f"unknown workload {w}")
    head = workloads[0]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    K, W = args.steps, max(args.warmup, 3)
    Kp = max(1, min(K, args.prefill_steps))
    results = {}
    for w in workloads:
        fmt = 1 if w.startswith("kv8") else (14 if w.startswith("pq4") else 2)
        saved = ctx.path
        if w.startswith("pq4t"):
            ctx.path = ctx.kvq.PATH_TENSOR
        if w.startswith("k2v4"):
            results[w] = run_k2v4(ctx, w, K, W, peaks, sampler, world, dist)
        elif w.endswith("prefill"):
            results[w] = run_prefill(ctx, fmt, w, Kp, W, peaks, src, sampler, world, dist)
        else:
            results[w] = run_decode(ctx, fmt, w, K, W, peaks, src, sampler, world, dist, e2e=(w == head))
        ctx.path = saved
    sampler.stop()
    if rank != 0:
        return None
    main = results[head]
    clocks = sampler.summary()
    line = {
        "metric": METRIC, "value": main["value"], "unit": main["unit"], "n_gpus": world,
        "steps": K if not head.endswith("prefill") else Kp, "warmup": W,
        "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if main["path"] == "tensor" else "f32",
        "precision": "e4m3 codes dequantized to f16 tensor-core operands, f32 accumulation and softmax"
        if main["path"] == "tensor" else "codes dequantized to f32, f32 accumulation and softmax",
        "data": "synthetic (seeded N(0,1) x log-normal channel gains; bf16 queries)",
        "config": {"workload": main["workload"], "heads": H, "row_bytes": main.get("row_bytes"),
                   "rows": main.get("rows"), "path": main["path"], "l2": main["l2"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "rows_per_s": main.get("rows_per_s"),
        "hbm_roof_frac": main.get("hbm_roof_frac"), "hbm_peak_gbs": peaks["hbm_gbs"], "peak_source": src,
        "gpu_launches": main["gpu_launches_per_step"] * (K if not head.endswith("prefill") else Kp),
        "roofline": main["roofline"],
        "timing": main["timing"],
        "exact_rescale_tiles_per_step": main.get("exact_rescale_tiles_per_step"),
        "clocks": clocks,
        "workloads": {w: r for w, r in results.items() if w != head},
    }
    if "e2e" in main:
        line["e2e"] = main["e2e"]
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    return line


# ---------------------------------------------------------------------------
# The oracle on the host cores (a reported baseline, not the target)
# ---------------------------------------------------------------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """The oracle's decode of the ragged KV8 workload on (sequence, 4-head block)
    units: reconstruct the sequence's rows from their codes, then f64 attention
    for 4 heads.  The cache is encoded once by the oracle beforehand (the
    decode's input is the quantized cache)."""

    HEADS = 4

    def __init__(self):
        from oracle import oracle as orc
        from quantized_kv_cache_kv8_gb300 import synth
        self.orc = orc
        orc.lib()
        self.lens, self.cu, self.offs = ragged_layout()
        x = synth.mla_rows(RAGGED_SEED, MASTER)
        self.mc, self.ms = orc.kv8_encode(x)
        bits = synth.bf16_bits(synth.queries(RAGGED_SEED + 1, (RAGGED_B, H, D)))
        self.q = synth.bf16_to_f32(bits)
        # units in a fixed order: sequences in turn, each with its next head block
        self.units = [(b, hb) for hb in range(H // self.HEADS) for b in range(RAGGED_B)]

    def run(self, k: int) -> int:
        """Runs unit k (mod the unit count); returns rows x heads processed."""
        b, hb = self.units[k % len(self.units)]
        rows = (self.offs[b] + np.arange(self.lens[b], dtype=np.int64)) % MASTER
        xh = self.orc.kv8_decode(np.ascontiguousarray(self.mc[rows]), np.ascontiguousarray(self.ms[rows]))
        heads = slice(hb * self.HEADS, (hb + 1) * self.HEADS)
        self.orc.attn_dense(xh, np.ascontiguousarray(self.q[b, heads]), SM_SCALE, DV)
        return int(self.lens[b]) * self.HEADS


def _rate_gbs(row_heads: int, seconds: float) -> float:
    # a row read once serves all 128 heads: rows x heads / 128 rows' worth of cache bytes
    return row_heads / H * ROW_BYTES[1] / seconds / 1e9


def cpu_baseline(seconds: float = 10.0):
    """The oracle as it stands on the host: one thread, then one thread per host
    core over distinct (sequence, head block) units (the C oracle releases the
    GIL), each for about `seconds`."""
    from concurrent.futures import ThreadPoolExecutor
    s = OracleSample()
    t0 = time.perf_counter()
    done = work = 0
    while done == 0 or time.perf_counter() - t0 < seconds:
        work += s.run(done)
        done += 1
    single = _rate_gbs(work, time.perf_counter() - t0)
    single_units = done

    cores = min(host_cores(), 32)
    counter = iter(range(10 ** 9))
    lock = threading.Lock()
    deadline = time.perf_counter() + seconds

    def worker(_):
        w = n = 0
        while time.perf_counter() < deadline or n == 0:
            with lock:
                k = next(counter)
            w += s.run(single_units + k)
            n += 1
        return w, n
    t1 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        parts = list(ex.map(worker, range(cores)))
    dt = time.perf_counter() - t1
    all_work = sum(w for w, _ in parts)
    all_units = sum(n for _, n in parts)
    return {"value": round(_rate_gbs(all_work, dt), 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "host_cores": host_cores(),
            "sample": f"{all_units} units of (one sequence of the ragged batch, 4 of 128 heads): reconstruct "
                      f"+ f64 attention, one thread per host core for {dt:.1f} s; rate scaled to all heads "
                      f"(a row is read once for the 128 heads)",
            "single_core": {"value": round(single, 6), "unit": "GB/s", "cores": 1,
                            "sample": f"{single_units} units in turn on one thread"}}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step one (sequence, 4-head) unit of
    the ragged KV8 decode on one host thread, rate scaled to all heads."""
    if rank != 0:
        return None
    K = max(args.steps, 1)
    W = max(args.warmup, 0)
    s = OracleSample()
    times, work = [], []
    for i in range(W + K):
        t0 = time.perf_counter()
        wk = s.run(i)
        dt = time.perf_counter() - t0
        if i >= W:
            times.append(dt)
            work.append(wk)
        if sum(times) > 120:
            break
    K = len(times)
    gbs = _rate_gbs(sum(work), sum(times))
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": W, "ms_per_step": round(sum(times) / K * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "precision": "the oracle: f32 codecs, f64 attention", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES["kv8_ragged"] + " (each step: one sequence x 4 of 128 heads)",
                       "heads": H, "row_bytes": ROW_BYTES[1]},
            "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{K} steps of one (sequence, 4-head) unit each; rate scaled to all heads"},
            "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--prefill-steps", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["auto", "simt", "tensor"], default="auto")
    ap.add_argument("--workloads", default=",".join(DEFAULT_WORKLOADS),
                    help="comma-separated; the first is the headline")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
