"""Benchmark of the grouped-query attention hot path on B300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gqa,reference}]

A step is one gqa_decode call (split-KV partial attention, the in-kernel
log-sum-exp merge, over the bf16 [B, Hkv, Lmax, D] cache) on the Llama-3-8B
shaped workload B=16, Hq=32, Hkv=8, D=128, L=4096, inputs resident in HBM.
The headline value is K/V bytes read per second (the visible cache rows, once
per KV head) -- decode is bound by reading the KV cache.  The causal prefill
(B=4, L=2048, Hq=32, Hkv=8, D=128) is timed in the same run and reported in
TFLOP/s under "prefill"; the other decode workloads under "decode_workloads".

L2 (126 MB) is flushed before every timed launch: a 256 MiB buffer is written,
then a second 256 MiB buffer is read, so that the flush's own dirty lines are
written back before the launch instead of during it.  Each launch is bracketed
by its own CUDA events on the launching stream, and ms_per_step is the mean of
those event intervals.

Under torchrun (N > 1) every rank runs its own batch of the same shape
(independent sequences: no data-path collective; weak scaling); the value is
the bytes of all ranks divided by the slowest rank's time.

Also timed in the same run (reported as extra keys): FP8 (E4M3) cache decode,
paged-cache decode (bf16 and FP8 pages), the rotary embedding + cache append of the new token, a
chunked prefill after a cached prefix, and the MHA -> GQA mean-pool conversion
of a K projection.

--impl reference times the fp64 CPU oracle on the same workload, metric and
unit (a bounded sample of (b, h) rows, extrapolated to the full step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GQA decode K/V-read GB/s (% HBM peak); causal prefill TFLOP/s; 1xB300"
HEADLINE = "llama3_8b"

# DRAM bytes (read + write) per launch from one ncu capture of a workload,
# keyed by the SHA-256 of the kernel source they were taken on; reported as
# null as soon as the source differs.
NCU_TRAFFIC = {
    ("decode.cu", "llama3_8b"): {
        "sha256": "b918ae2d7261ee9169222504ac93d8554e5ad00d19b0d10ec0f80aed94a9eb77",
        "bytes_per_launch": 268635904.0 + 2781184.0,
        "capture": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum, one launch of "
                   "python bench.py --only llama3_8b --steps 3 --warmup 3"},
    ("decode_tc.cu", "mqa"): {
        "sha256": "2fe2a8f7fbb80615831d71f094ab0487200f592a3f237431e344a05edbf23241",
        "bytes_per_launch": 44320256.0 + 33280.0,
        "capture": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum, one launch of "
                   "python bench.py --only mqa --steps 3 --warmup 3"},
    ("prefill.cu", "prefill"): {
        "sha256": "49ae9b16a18d68d9188749b389271f3474d5de3d207fe4995edf217030fd0403",
        "bytes_per_launch": 100837376.0 + 14577920.0,
        "capture": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum, one launch of "
                   "python bench.py --only prefill --steps 3 --warmup 3"},
}


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_for(kernel_file, workload):
    rec = NCU_TRAFFIC.get((os.path.basename(kernel_file), workload))
    if not rec or not rec["bytes_per_launch"] or rec["sha256"] != _sha(kernel_file):
        return None
    return rec["bytes_per_launch"]


def _csrc(name):
    return os.path.join(ROOT, "grouped_query_attention_09_b300", "csrc", name)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ timing
class L2Flush:
    """Evicts L2 (126 MB on B300): writes a 256 MiB buffer, then reads another
    256 MiB buffer so the written lines are cleaned out before the next launch."""

    def __init__(self, dev, nbytes=256 * 2**20):
        import torch
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def timed_launches(fn, steps, warmup, flush, stream):
    """Runs fn() warmup times, then `steps` times with an L2 flush before each
    launch; returns the per-launch event durations in ms."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def bench_decode(g, W, name, dev, steps, warmup, flush, seed_offset=0):
    import torch
    w = W.WORKLOADS[name]
    if seed_offset:
        w = W.DecodeWorkload(w.name, w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.len_lo, w.len_hi, w.seed + seed_offset)
    q, k, v, sl = W.make_decode_inputs(w)
    qd, kd, vd, sld = q.to(dev), k.to(dev), v.to(dev), sl.to(dev)
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    ts = timed_launches(lambda: g.gqa_decode(qd, kd, vd, sld, out=out, scale=w.scale, stream=stream),
                        steps, warmup, flush, stream)
    flags = g.gqa_get_device_status()
    if flags:
        raise RuntimeError(f"decode {name}: device status {flags:#x}")
    nbytes = W.decode_kv_bytes(sl, w.Hkv, w.D)
    return {"w": w, "inputs": (q, k, v, sl), "ms": ts, "bytes": nbytes,
            "flops": W.decode_flops(sl, w.Hq, w.D)}


def bench_decode_fp8(g, W, name, dev, steps, warmup, flush):
    """gqa_decode_fp8 on workload `name` with its cache quantised to E4M3."""
    import torch
    w = W.WORKLOADS[name]
    q, k8, v8, ks, vs, sl = W.make_decode_fp8_inputs(w)
    qd, kd, vd, ksd, vsd, sld = (t.to(dev) for t in (q, k8, v8, ks, vs, sl))
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    ts = timed_launches(lambda: g.gqa_decode_fp8(qd, kd, vd, ksd, vsd, sld, out=out, scale=w.scale, stream=stream),
                        steps, warmup, flush, stream)
    flags = g.gqa_get_device_status()
    if flags:
        raise RuntimeError(f"decode fp8 {name}: device status {flags:#x}")
    return {"w": w, "ms": ts, "bytes": W.decode_kv_bytes_fp8(sl, w.Hkv, w.D)}


def bench_decode_paged(g, W, name, page_size, dev, steps, warmup, flush):
    """gqa_decode_paged on workload `name` with its cache cut into pages of
    page_size rows, handed out in a seeded random order."""
    import torch
    w = W.WORKLOADS[name]
    q, k, v, sl = W.make_decode_inputs(w)
    kp, vp, bt = W.page_cache(k, v, page_size, seed=w.seed + 50)
    del k, v
    qd, kd, vd, btd, sld = (t.to(dev) for t in (q, kp, vp, bt, sl))
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    ts = timed_launches(lambda: g.gqa_decode_paged(qd, kd, vd, btd, sld, out=out, scale=w.scale, stream=stream),
                        steps, warmup, flush, stream)
    flags = g.gqa_get_device_status()
    if flags:
        raise RuntimeError(f"decode paged {name}: device status {flags:#x}")
    return {"w": w, "ms": ts, "bytes": W.decode_kv_bytes(sl, w.Hkv, w.D)}


def bench_decode_fp8_paged(g, W, name, page_size, dev, steps, warmup, flush):
    """gqa_decode_fp8_paged on workload `name`: its E4M3 cache cut into pages
    of page_size rows, handed out in a seeded random order."""
    import torch
    w = W.WORKLOADS[name]
    q, k8, v8, ks, vs, sl = W.make_decode_fp8_inputs(w)
    kp, vp, bt = W.page_cache(k8, v8, page_size, seed=w.seed + 60)
    del k8, v8
    qd, kd, vd, ksd, vsd, btd, sld = (t.to(dev) for t in (q, kp, vp, ks, vs, bt, sl))
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    ts = timed_launches(lambda: g.gqa_decode_fp8_paged(qd, kd, vd, ksd, vsd, btd, sld, out=out, scale=w.scale,
                                                       stream=stream),
                        steps, warmup, flush, stream)
    flags = g.gqa_get_device_status()
    if flags:
        raise RuntimeError(f"decode fp8 paged {name}: device status {flags:#x}")
    return {"w": w, "ms": ts, "bytes": W.decode_kv_bytes_fp8(sl, w.Hkv, w.D)}


def bench_rope_append(g, W, name, dev, steps, warmup, flush):
    """gqa_rope_append for the new token of every sequence of decode workload
    `name` (cache at its workload lengths); seqlens is reset before each launch
    (outside the timed region) so every call appends at the same positions."""
    import torch
    w = W.WORKLOADS[name]
    q, k, v, sl = W.make_decode_inputs(w)
    gen = torch.Generator().manual_seed(w.seed + 100)
    kn = torch.randn(w.B, w.Hkv, w.D, generator=gen).to(torch.bfloat16)
    vn = torch.randn(w.B, w.Hkv, w.D, generator=gen).to(torch.bfloat16)
    sl = (sl - 1).clamp(min=0)  # the new token becomes the last visible key
    qd, kd, vd, knd, vnd, sl0 = (t.to(dev) for t in (q, k, v, kn, vn, sl))
    sld = sl0.clone()
    qo = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)

    def prep():
        flush()
        sld.copy_(sl0)

    ts = timed_launches(lambda: g.gqa_rope_append(qd, knd, vnd, kd, vd, sld, q_out=qo, stream=stream),
                        steps, warmup, prep, stream)
    flags = g.gqa_get_device_status()
    if flags:
        raise RuntimeError(f"rope_append {name}: device status {flags:#x}")
    moved = 2 * (2 * w.B * w.Hq * w.D + 4 * w.B * w.Hkv * w.D) + 8 * w.B
    return {"w": w, "ms": ts, "bytes": moved}


def bench_meanpool(g, W, dev, steps, warmup, flush, H=32, Hkv=8, D=128, d_model=4096):
    """gqa_meanpool_kv_heads on a Llama-3-8B-shaped K projection: 32 heads of
    [128, 4096] bf16 -> 8 groups (synthetic weights, N(0, 0.02^2))."""
    import torch
    gen = torch.Generator().manual_seed(77)
    w = (torch.randn(H, D, d_model, generator=gen) * 0.02).to(torch.bfloat16).to(dev)
    out = torch.empty(Hkv, D, d_model, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    ts = timed_launches(lambda: g.gqa_meanpool_kv_heads(w, Hkv, out=out, stream=stream), steps, warmup, flush, stream)
    return {"ms": ts, "bytes": (H + Hkv) * D * d_model * 2, "shape": (H, Hkv, D, d_model)}


def bench_prefill(g, W, dev, steps, warmup, flush, D=128):
    """The causal prefill workload (B=4, L=2048, Hq=32, Hkv=8); D = 64 runs the
    same shape at half the head size."""
    import torch
    w = W.WORKLOADS["prefill"]
    if D != w.D:
        w = W.PrefillWorkload(f"prefill_d{D}", w.B, w.L, w.Hq, w.Hkv, D, w.causal, w.seed)
    q, k, v = W.make_prefill_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    try:
        g.gqa_prefill(qd, kd, vd, out=out, causal=w.causal, stream=stream)
    except g.GQAError as e:
        if e.status == g.GQA_ERR_UNSUPPORTED:
            return None
        raise
    ts = timed_launches(lambda: g.gqa_prefill(qd, kd, vd, out=out, causal=w.causal, stream=stream),
                        steps, warmup, flush, stream)
    return {"w": w, "ms": ts, "flops": W.prefill_flops(w.B, w.Hq, w.L, w.D, w.causal)}


def bench_prefill_chunk(g, W, dev, steps, warmup, flush, Lq=512, Lk=2048):
    """gqa_prefill_chunk: a chunk of Lq tokens after Lk - Lq cached ones at the
    prefill workload's head shape (B=4, Hq=32, Hkv=8, D=128), causal."""
    import torch
    w = W.WORKLOADS["prefill"]
    gen = torch.Generator().manual_seed(w.seed + 7)
    q = torch.randn(w.B, w.Hq, Lq, w.D, generator=gen).to(torch.bfloat16).to(dev)
    k = torch.randn(w.B, w.Hkv, Lk, w.D, generator=gen).to(torch.bfloat16).to(dev)
    v = torch.randn(w.B, w.Hkv, Lk, w.D, generator=gen).to(torch.bfloat16).to(dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    ts = timed_launches(lambda: g.gqa_prefill_chunk(q, k, v, out=out, causal=True, stream=stream),
                        steps, warmup, flush, stream)
    return {"ms": ts, "flops": W.prefill_chunk_flops(w.B, w.Hq, Lq, Lk, w.D, True), "Lq": Lq, "Lk": Lk}


def e2e_decode(g, W, name, steps, warmup):
    """Same metric through gqa_decode_host: pinned host inputs copied in and the
    output copied back inside the timed region, every step."""
    import torch
    w = W.WORKLOADS[name]
    q, k, v, sl = W.make_decode_inputs(w)
    q, k, v, sl = q.pin_memory(), k.pin_memory(), v.pin_memory(), sl.pin_memory()
    out = torch.empty_like(q).pin_memory()
    for _ in range(warmup):
        g.gqa_decode_host(q, k, v, sl, out=out, scale=w.scale)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        g.gqa_decode_host(q, k, v, sl, out=out, scale=w.scale)
    dt = (time.perf_counter() - t0) / steps
    nbytes = W.decode_kv_bytes(sl, w.Hkv, w.D)
    h2d = q.numel() * 2 + k.numel() * 2 + v.numel() * 2 + sl.numel() * 4
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": out.numel() * 2, "ms_per_step": dt * 1e3}


# ------------------------------------------------------------------ CPU oracle
def oracle_decode_rate(W, name, budget_s=12.0, max_rows=None, cycle=False):
    """fp64 oracle on the host cores: time a sample of (b, h) rows, extrapolate
    to the whole step and return (GB/s of the step's K/V bytes, sample text, threads).
    cycle: when one step takes less than budget_s, go round the step's rows
    again until the budget is spent (the rate then averages several steps)."""
    import numpy as np
    import oracle
    w = W.WORKLOADS[name]
    q, k, v, sl = W.make_decode_inputs(w)
    qb, kb, vb, sln = W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), sl.numpy()
    rows_all = np.array([(b, h) for b in range(w.B) for h in range(w.Hq)], dtype=np.int32)
    n = 8
    elapsed, done = 0.0, 0
    while elapsed < budget_s and (cycle or done < len(rows_all)):
        at = done % len(rows_all)
        take = rows_all[at:at + n] if max_rows is None else rows_all[at:at + min(n, max_rows - done)]
        if len(take) == 0:
            break
        t0 = time.perf_counter()
        oracle.decode(qb, kb, vb, sln, w.scale, rows=take)
        elapsed += time.perf_counter() - t0
        done += len(take)
        n = min(n * 2, 256)
        if max_rows is not None and done >= max_rows:
            break
    rows_per_s = done / elapsed
    step_s = len(rows_all) / rows_per_s
    nbytes = W.decode_kv_bytes(sl, w.Hkv, w.D)
    if done > len(rows_all):
        sample = f"{done} (b, h) rows = {done / len(rows_all):.1f} steps of {len(rows_all)} rows in {elapsed:.1f} s"
    else:
        sample = f"{done} of {len(rows_all)} (b, h) rows of one step in {elapsed:.1f} s, extrapolated to the step"
    return nbytes / step_s / 1e9, step_s, sample, oracle.num_threads()


# ------------------------------------------------------------------ main
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("GQA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def max_over_ranks(x, world, dev=None):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev if dev is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_step, world, steps, total_ms):
    """Whole-job throughput in GB/s: every rank runs `steps` steps of its own
    batch (weak scaling), the job takes the slowest rank's total time."""
    return bytes_per_step * world * steps / (total_ms / 1e3) / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from grouped_query_attention_09_b300 import workloads as W
    steps = []
    for _ in range(args.warmup):
        oracle_decode_rate(W, HEADLINE, budget_s=1.0, max_rows=16)
    sample = threads = None
    for _ in range(args.steps):
        gbs, step_s, sample, threads = oracle_decode_rate(W, HEADLINE, budget_s=args.ref_budget)
        steps.append(step_s)
    step_s = statistics.mean(steps)
    w = W.WORKLOADS[HEADLINE]
    nbytes = W.decode_kv_bytes(W.make_decode_inputs(W.DecodeWorkload("x", w.B, w.Hq, w.Hkv, w.D, 1, 1, 1, 0))[3]
                               * w.len_lo, w.Hkv, w.D)
    value = nbytes / step_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "llama3_8b decode: B=16, Hq=32, Hkv=8, D=128, L=4096, bf16 inputs widened to fp64",
                       "reference": "fp64 CPU oracle (oracle/gqa_oracle.c), no installable reference exists"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def run_only(g, W, args, dev, flush, peaks):
    """One workload, for profiling and sweeps: prints the per-launch mean time and rate."""
    if args.only in ("prefill", "prefill_d64"):
        r = bench_prefill(g, W, dev, args.steps, args.warmup, flush, D=64 if args.only == "prefill_d64" else 128)
        if r is None:
            print(json.dumps({"only": args.only, "status": "not built"}))
            return 0
        ms = statistics.mean(r["ms"])
        tf = r["flops"] / (ms / 1e3) / 1e12
        print(json.dumps({"only": args.only, "us": ms * 1e3, "TFLOP/s": tf, "frac": tf / peaks["bf16_tflops"]}))
        return 0
    if args.only == "prefill_chunk":
        r = bench_prefill_chunk(g, W, dev, args.steps, args.warmup, flush)
        ms = statistics.mean(r["ms"])
        tf = r["flops"] / (ms / 1e3) / 1e12
        print(json.dumps({"only": args.only, "us": ms * 1e3, "TFLOP/s": tf, "frac": tf / peaks["bf16_tflops"]}))
        return 0
    if args.only.endswith("_fp8_paged"):
        name = args.only[:-10]
        r = bench_decode_fp8_paged(g, W, name, 128 if name == "mqa" else 256, dev, args.steps, args.warmup, flush)
        ms = statistics.mean(r["ms"])
        gbs = r["bytes"] / (ms / 1e3) / 1e9
        print(json.dumps({"only": args.only, "us": ms * 1e3, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"]}))
        return 0
    if args.only.endswith("_paged"):
        name = args.only[:-6]
        r = bench_decode_paged(g, W, name, 128 if name == "mqa" else 256, dev, args.steps, args.warmup, flush)
        ms = statistics.mean(r["ms"])
        gbs = r["bytes"] / (ms / 1e3) / 1e9
        print(json.dumps({"only": args.only, "us": ms * 1e3, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"]}))
        return 0
    if args.only == "rope_append":
        r = bench_rope_append(g, W, "llama3_8b", dev, args.steps, args.warmup, flush)
        ms = statistics.mean(r["ms"])
        print(json.dumps({"only": "rope_append", "us": ms * 1e3, "GB/s": r["bytes"] / (ms / 1e3) / 1e9}))
        return 0
    if args.only == "kv_meanpool":
        r = bench_meanpool(g, W, dev, args.steps, args.warmup, flush)
        ms = statistics.mean(r["ms"])
        gbs = r["bytes"] / (ms / 1e3) / 1e9
        print(json.dumps({"only": "kv_meanpool", "us": ms * 1e3, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"]}))
        return 0
    if args.only.endswith("_fp8"):
        r = bench_decode_fp8(g, W, args.only[:-4], dev, args.steps, args.warmup, flush)
    else:
        r = bench_decode(g, W, args.only, dev, args.steps, args.warmup, flush)
    ms = statistics.mean(r["ms"])
    gbs = r["bytes"] / (ms / 1e3) / 1e9
    print(json.dumps({"only": args.only, "us": ms * 1e3, "us_min": min(r["ms"]) * 1e3, "GB/s": gbs,
                      "frac": gbs / peaks["hbm_gbs"]}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gqa", choices=["gqa", "reference"])
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="headline only (for profiling runs)")
    ap.add_argument("--only", default=None,
                    help="time one workload and print its line: a decode workload name (tiny, llama3_8b, "
                         "llama2_70b, mqa), optionally with _fp8, _paged or _fp8_paged; prefill; prefill_d64; prefill_chunk; rope_append; "
                         "kv_meanpool")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank, world, local = dist_setup()
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
        barrier(world)
        return rc

    import torch
    import grouped_query_attention_09_b300 as g
    from grouped_query_attention_09_b300 import workloads as W

    g.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    flush = L2Flush(dev)
    if args.only:
        return run_only(g, W, args, dev, flush, peaks)

    barrier(world)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        res = bench_decode(g, W, HEADLINE, dev, args.steps, args.warmup, flush, seed_offset=rank)
        torch.cuda.synchronize()
    barrier(world)
    mean_ms = statistics.mean(res["ms"])
    total_ms = max_over_ranks(sum(res["ms"]), world, dev)
    value = job_value(res["bytes"], world, args.steps, total_ms)
    achieved = res["bytes"] / (mean_ms / 1e3) / 1e9

    extras = {}
    if not args.no_extras:
        small_steps = max(50, min(args.steps, 400))
        dw = {}
        for name in ("tiny", "llama2_70b", "mqa"):
            r = bench_decode(g, W, name, dev, small_steps, args.warmup, flush)
            ms = statistics.mean(r["ms"])
            gbs = r["bytes"] / (ms / 1e3) / 1e9
            dw[name] = {"us": ms * 1e3, "kv_bytes": r["bytes"], "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                        "TFLOP/s": r["flops"] / (ms / 1e3) / 1e12}
            if name == "mqa":
                dw[name]["kernel"] = "decode_tc_kernel<false>"
                dw[name]["traffic"] = traffic_for(_csrc("decode_tc.cu"), "mqa")
        dw[HEADLINE] = {"us": mean_ms * 1e3, "kv_bytes": res["bytes"], "GB/s": achieved,
                        "frac_hbm": achieved / peaks["hbm_gbs"], "TFLOP/s": res["flops"] / (mean_ms / 1e3) / 1e12}
        extras["decode_workloads"] = dw
        d8 = {}
        for name in ("llama3_8b", "llama2_70b", "mqa"):
            r = bench_decode_fp8(g, W, name, dev, small_steps, args.warmup, flush)
            ms = statistics.mean(r["ms"])
            gbs = r["bytes"] / (ms / 1e3) / 1e9
            d8[name] = {"us": ms * 1e3, "kv_bytes_fp8": r["bytes"], "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                        "speedup_vs_bf16": dw[name]["us"] / (ms * 1e3)}
        extras["decode_fp8_kv"] = d8
        dp = {}
        for name, ps in (("llama3_8b", 256), ("mqa", 128)):
            r = bench_decode_paged(g, W, name, ps, dev, small_steps, args.warmup, flush)
            ms = statistics.mean(r["ms"])
            gbs = r["bytes"] / (ms / 1e3) / 1e9
            dp[name] = {"page_size": ps, "us": ms * 1e3, "kv_bytes": r["bytes"], "GB/s": gbs,
                        "frac_hbm": gbs / peaks["hbm_gbs"]}
        extras["decode_paged"] = dp
        d8p = {}
        for name, ps in (("llama3_8b", 256), ("mqa", 128)):
            r = bench_decode_fp8_paged(g, W, name, ps, dev, small_steps, args.warmup, flush)
            ms = statistics.mean(r["ms"])
            gbs = r["bytes"] / (ms / 1e3) / 1e9
            d8p[name] = {"page_size": ps, "us": ms * 1e3, "kv_bytes_fp8": r["bytes"], "GB/s": gbs,
                         "frac_hbm": gbs / peaks["hbm_gbs"]}
        extras["decode_fp8_paged"] = d8p
        ra = bench_rope_append(g, W, "llama3_8b", dev, small_steps, args.warmup, flush)
        rms = statistics.mean(ra["ms"])
        extras["rope_append"] = {"workload": "new token of llama3_8b: B=16, Hq=32, Hkv=8, D=128, appended at 4095",
                                 "us": rms * 1e3, "bytes_moved": ra["bytes"],
                                 "GB/s": ra["bytes"] / (rms / 1e3) / 1e9,
                                 "frac_hbm": ra["bytes"] / (rms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        mp = bench_meanpool(g, W, dev, small_steps, args.warmup, flush)
        mms = statistics.mean(mp["ms"])
        extras["kv_meanpool"] = {
            "workload": "MHA -> GQA conversion of a Llama-3-8B K projection: [32, 128, 4096] bf16 -> 8 groups",
            "us": mms * 1e3, "bytes_moved": mp["bytes"], "GB/s": mp["bytes"] / (mms / 1e3) / 1e9,
            "frac_hbm": mp["bytes"] / (mms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        pr = bench_prefill(g, W, dev, small_steps, args.warmup, flush)
        if pr is not None:
            pms = statistics.mean(pr["ms"])
            tf = pr["flops"] / (pms / 1e3) / 1e12
            extras["prefill"] = {
                "workload": "causal prefill: B=4, L=2048, Hq=32, Hkv=8, D=128", "us": pms * 1e3,
                "flops": pr["flops"], "TFLOP/s": tf,
                "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": tf / peaks["bf16_tflops"],
                             "frac_sustained": tf / peaks["bf16_tflops_sustained"]
                             if peaks.get("bf16_tflops_sustained") else None,
                             "traffic": traffic_for(_csrc("prefill.cu"), "prefill")}}
        else:
            extras["prefill"] = {"status": "not built"}
        p64 = bench_prefill(g, W, dev, small_steps, args.warmup, flush, D=64)
        if p64 is not None:
            pms = statistics.mean(p64["ms"])
            tf = p64["flops"] / (pms / 1e3) / 1e12
            extras["prefill_d64"] = {"workload": "causal prefill: B=4, L=2048, Hq=32, Hkv=8, D=64", "us": pms * 1e3,
                                     "flops": p64["flops"], "TFLOP/s": tf, "frac_tensor": tf / peaks["bf16_tflops"]}
        pc = bench_prefill_chunk(g, W, dev, small_steps, args.warmup, flush)
        cms = statistics.mean(pc["ms"])
        ctf = pc["flops"] / (cms / 1e3) / 1e12
        extras["prefill_chunk"] = {"workload": f"causal chunk of {pc['Lq']} tokens after {pc['Lk'] - pc['Lq']} cached: "
                                               "B=4, Hq=32, Hkv=8, D=128", "us": cms * 1e3, "flops": pc["flops"],
                                   "TFLOP/s": ctf, "frac_tensor": ctf / peaks["bf16_tflops"]}
        if rank == 0:
            extras["e2e"] = e2e_decode(g, W, HEADLINE, steps=max(5, min(args.steps, 20)), warmup=2)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, step_s, sample, threads = oracle_decode_rate(W, HEADLINE, budget_s=12.0, cycle=True)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "llama3_8b decode: B=16, Hq=32, Hkv=8, D=128, L=4096 (bf16 KV cache "
                                   "[16, 8, 4096, 128] + q [16, 32, 128], N(0,1) seed 2)",
                       "l2": "flushed before every timed launch (256 MiB write, then 256 MiB read of another buffer)",
                       "parallelism": f"replica per GPU x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                         "kernel": "decode_kernel<128,1>",
                         "traffic": traffic_for(_csrc("decode.cu"), HEADLINE)},
            "cpu_baseline": cpu,
            "e2e": extras.pop("e2e", None),
            "gpu_launches": args.steps,
            "clocks": clocks.summary(),
        }
        line.update(extras)
        print(json.dumps(line), flush=True)
    barrier(world)
    return 0


if __name__ == "__main__":
    sys.exit(main())
