#!/usr/bin/env python
"""Benchmark of the quantized-KV MLA decode step on GB300.

Workload: KV8 decode, 8 sequences x 4096 cached rows, 128 heads sharing one
576-dim latent cache (fp8 e4m3 + two f32 scales per row, 584 B), one bf16
query token per sequence and head.  Inputs are synthetic and seeded
(quantized_kv_cache_kv8_gb300.synth): latent rows N(0,1) x per-channel
log-normal gains.

One step = the whole hot path for one decode token of every sequence, one
call of kv_attn_decode_append:
  1. the 8 new rows (one per sequence, the last row of its range of the
     resident pool) are encoded to KV8 and stored,
  2. attention over all 8 x 4096 rows, the new ones included (split-T
     partials + merge).
On the tensor-core path both run in one launch (plus the merge); on the fp32
path (--path simt) the encoder is its own launch.
The cache (19 MB) fits in L2, so a 256 MB buffer is written between timed
steps (outside the timed events) to flush it.

Metric: cache GB/s = rows read per step x 584 B / step time; rows/s and the
fraction of the measured HBM copy bandwidth are reported beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--path auto|simt|tensor]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, T, H, D, DV = 8, 4096, 128, 576, 512
ROW_BYTES = 576 + 2 * 4
FLOPS_PER_ROW = H * (D + DV) * 2
SEED = 2
METRIC = "quantized-KV MLA decode attn: cache GB/s & % of HBM roofline; rows/s"
WORKLOAD = "KV8 decode: 8 seqs x 4096 rows, 128 heads, 576-dim latent (512+64), bf16 query"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[tuple[float, list[str]]] = []
        self.t0 = self.t1 = None

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
            self.t0 = time.time()
        else:
            self.t1 = time.time()

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
        inside = [f for t, f in self.lines if self.t0 and self.t1 and self.t0 <= t <= self.t1]
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


def make_inputs(torch, kvq):
    from quantized_kv_cache_kv8_gb300 import synth
    rows = synth.mla_rows(SEED, B * T)
    cu = synth.cu_seqlens([T] * B)
    dev = torch.device("cuda")
    codes = torch.empty((B * T, D), dtype=torch.uint8, device=dev)
    scales = torch.empty((B * T, 2), dtype=torch.float32, device=dev)
    kvq.kv8_encode(torch.from_numpy(rows).to(dev), codes, scales)
    new_rows = synth.mla_rows(SEED + 100, B)
    q = synth.queries(SEED + 1, (B, H, D))
    q_bits = synth.bf16_bits(q)
    # the step's host inputs share one pinned staging buffer (bf16 queries, then
    # the f32 new rows), so that they cross to the device in one copy
    q_bytes, x_bytes = B * H * D * 2, B * D * 4
    stage_host = torch.empty(q_bytes + x_bytes, dtype=torch.uint8).pin_memory()
    stage_host[:q_bytes].view(torch.int16).copy_(torch.from_numpy(q_bits.view(np.int16).reshape(-1)))
    stage_host[q_bytes:].view(torch.float32).copy_(torch.from_numpy(new_rows.reshape(-1)))
    return dict(codes=codes, scales=scales, cu=torch.from_numpy(cu).to(dev), cu_np=cu,
                dst=torch.from_numpy(cu[1:] - 1).to(dev), stage_host=stage_host)


def stage_views(stage):
    """The bf16 queries [B][H][576] and the f32 new rows [B][576] inside a staging buffer."""
    import torch
    q_bytes = B * H * D * 2
    q = stage[:q_bytes].view(torch.bfloat16).view(B, H, D)
    x_new = stage[q_bytes:].view(torch.float32).view(B, D)
    return q, x_new


def max_over_ranks(vals, dist, device):
    """Each timing's maximum over the ranks: the slowest replica bounds the job."""
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.barrier()
    return t.tolist()


def job_rate_gbs(rows_per_rank, world, ms):
    """Whole-job cache throughput: every replica's rows over the slowest step time."""
    return rows_per_rank * world * ROW_BYTES / (ms * 1e-3) / 1e9


def run_ours(args, rank, world):
    import torch
    from quantized_kv_cache_kv8_gb300 import kvq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    path = {"auto": kvq.PATH_AUTO, "simt": kvq.PATH_SIMT, "tensor": kvq.PATH_TENSOR}[args.path]
    inp = make_inputs(torch, kvq)
    stream = torch.cuda.current_stream()
    dev = torch.device("cuda")
    stage = inp["stage_host"].to(dev)
    q, x_new = stage_views(stage)
    out = torch.empty((B, H, DV), dtype=torch.float32, device=dev)
    out_host = torch.empty((B, H, DV), dtype=torch.float32).pin_memory()
    ws = torch.zeros(kvq.kv_attn_workspace_size(kvq.KVQ_KV8, B, H, B * T, path=path), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step(xn, qq):
        kvq.kv_attn_decode_append(kvq.KVQ_KV8, xn, inp["dst"], qq, inp["codes"], inp["scales"], inp["cu"], out, ws,
                                  B * T, path=path)

    for _ in range(max(args.warmup, 3)):
        step(x_new, q)
        flush.zero_()
    torch.cuda.synchronize()
    if kvq.read_device_error(ws) != 0:
        raise RuntimeError("device error word set during warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark(True)
    for i in range(K):
        e0, e2 = ev[i]
        e0.record(stream)
        step(x_new, q)
        e2.record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    sampler.mark(False)
    step_ms = sum(e0.elapsed_time(e2) for e0, e2 in ev) / K

    # the dominant kernel alone, for the roofline: the library's launch events
    # before each call's partial kernel and before and after its merge.  A loop
    # of its own: the record between the two kernels ends the merge's
    # programmatic overlap, so these steps are not the ones timed above.
    kvq.timing_enable(K)
    for i in range(K):
        step(x_new, q)
        flush.zero_()
    torch.cuda.synchronize()
    part_sum, merge_sum, n_timed = kvq.timing_read()
    kvq.timing_enable(0)
    if n_timed != K:
        raise RuntimeError(f"launch timing recorded {n_timed} of {K} calls")
    partial_ms, merge_ms = part_sum / K, merge_sum / K

    # end to end through the public API: pinned host inputs in, result out, every step
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        a, b = e2e_ev[i]
        a.record(stream)
        stage.copy_(inp["stage_host"], non_blocking=True)
        step(x_new, q)
        out_host.copy_(out, non_blocking=True)
        b.record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    sampler.stop()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / K
    err = kvq.read_device_error(ws)
    if err != 0:
        raise RuntimeError(f"device error word {err} after the timed region")

    step_ms, e2e_ms, partial_ms, merge_ms = max_over_ranks([step_ms, e2e_ms, partial_ms, merge_ms], dist, dev)
    if rank != 0:
        return None

    rows = B * T * world
    peaks, src = load_peaks()
    gbs = job_rate_gbs(B * T, world, step_ms)
    e2e_gbs = job_rate_gbs(B * T, world, e2e_ms)
    clocks = sampler.summary()
    # the decode's tensor-core path is bound by the bf16 tensor pipe; the SIMT
    # path by the fp32 FMA pipe (152 SMs x 128 lanes x 2 flop x max SM clock)
    used_path = "tensor" if (path == kvq.PATH_TENSOR or (path == kvq.PATH_AUTO and H % 64 == 0)) else "simt"
    flops = B * T * FLOPS_PER_ROW
    # per launch of the partial kernel: every row of the step, all 128 heads
    achieved_tf = flops / (partial_ms * 1e-3) / 1e12
    timing = {"partial_ms": round(partial_ms, 5), "merge_ms": round(merge_ms, 5),
              "partial_share": round(partial_ms / (partial_ms + merge_ms), 4), "launches": K,
              "how": "CUDA events recorded by the library on the launch stream around each call's "
                     "partial kernel and merge (kvq_timing_enable), a loop of K steps of its own"}
    if used_path == "simt":
        peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": round(achieved_tf, 3), "peak": round(peak, 2), "unit": "TFLOP/s",
                "frac": round(achieved_tf / peak, 4), "traffic": None,
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 x max SM clock (MEASURED_PEAKS sm_max_mhz)",
                "kernel": "attn_partial_kernel (fp32 split-T partials), timed alone", "timing": timing}
    else:
        peak = peaks["bf16_tflops"]
        # DRAM bytes of one launch of the partial kernel of this step, from the full
        # ncu capture summarised in profiles/decode_tc_kv8_b8_t4096_h128.md
        # (dram__bytes_read.sum + dram__bytes_write.sum)
        roof = {"bound": "tensor", "achieved": round(achieved_tf, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved_tf / peak, 4), "traffic": 20428032 + 0,
                "peak_source": f"bf16_tflops ({src}); f16 operands run at the bf16 dense rate",
                "kernel": "attn_tc_kv8_kernel<APPEND> (tcgen05 split-T partials with the row append), timed alone",
                "timing": timing}
    line = {
        "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16" if used_path == "tensor" else "f32",
        "precision": "e4m3 codes dequantized to f16 tensor-core operands, f32 accumulation and softmax"
        if used_path == "tensor" else "e4m3 codes dequantized to f32, f32 accumulation and softmax",
        "data": "synthetic (seeded N(0,1) x log-normal channel gains; bf16 queries)",
        "config": {"workload": WORKLOAD, "batch": B, "seq_len": T, "heads": H, "row_bytes": ROW_BYTES,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "256 MB buffer written between timed steps (outside the events)", "path": used_path},
        "rows_per_s": round(rows / (step_ms * 1e-3), 1),
        "hbm_roof_frac": round(gbs / peaks["hbm_gbs"], 5),
        "hbm_peak_gbs": peaks["hbm_gbs"], "peak_source": src,
        "e2e": {"value": round(e2e_gbs, 3), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(B * D * 4 + B * H * D * 2), "d2h_bytes_per_step": int(B * H * DV * 4)},
        # tensor path: the fused partial kernel + the merge; fp32 path: encoder, partials, merge
        "gpu_launches": (2 if used_path == "tensor" else 3) * K,
        "roofline": roof,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    return line


def cpu_baseline(seconds: float = 10.0, sample_seqs: int | None = None, heads: int = H):
    """The oracle as it stands, single-threaded on the host, on a bounded sample
    of the same workload: sequences of 4096 rows x `heads` of the 128 heads, in
    turn and again from the first, until the time budget is spent (at least one;
    with `sample_seqs`, at most that many).  The rate is scaled to the metric's
    unit: rows read once for all 128 heads."""
    from oracle import oracle as orc
    from quantized_kv_cache_kv8_gb300 import synth
    orc.lib()
    rows = synth.mla_rows(SEED, B * T)
    q = synth.bf16_to_f32(synth.bf16_bits(synth.queries(SEED + 1, (B, H, D))))
    cu = synth.cu_seqlens([T] * B)
    t0 = time.perf_counter()
    done = 0
    while True:
        b = done % B
        codes, scales = orc.kv8_encode(rows[cu[b]:cu[b + 1]])
        xh = orc.kv8_decode(codes, scales)
        orc.attn_dense(xh, q[b, :heads], 1.0 / math.sqrt(192.0), DV)
        done += 1
        if time.perf_counter() - t0 > seconds or (sample_seqs is not None and done >= sample_seqs):
            break
    dt = time.perf_counter() - t0
    gbs = done * T * ROW_BYTES * (heads / H) / dt / 1e9
    return {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} sequence{'s' if done > 1 else ''} ({done / B:.2g} passes over the {B}) x {T} rows x "
                      f"{heads} of {H} heads "
                      f"(encode + f64 attention), {dt:.1f} s; rate scaled to all {H} heads"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    K = max(args.steps, 1)
    W = max(args.warmup, 0)
    times = []
    for i in range(W + K):
        t0 = time.perf_counter()
        cpu_baseline(seconds=0.0, sample_seqs=1, heads=8)
        dt = time.perf_counter() - t0
        if i >= W:
            times.append(dt)
        if sum(times) > 120:
            K = len(times)
            break
    step_s = sum(times) / len(times)
    gbs = T * ROW_BYTES * (8 / H) / step_s / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": W, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "precision": "the oracle: f32 codecs, f64 attention", "data": "synthetic",
            "config": {"workload": WORKLOAD + " (each step: one sequence of the batch, 8 of 128 heads)", "batch": B,
                       "seq_len": T, "heads": H},
            "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "per step: 1 of 8 sequences x 4096 rows x 8 of 128 heads; rate scaled "
                                       "to all heads"},
            "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["auto", "simt", "tensor"], default="auto")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
