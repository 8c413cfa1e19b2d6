#!/usr/bin/env python
"""Benchmark: quantized exact attention throughput on the headline workload.

One step = the whole path on one batch: sattn_prepare (K smoothing, INT8 Q/K,
FP8 V) then sattn_forward (INT8 QK^T, online softmax, FP8 P, two-level PV,
BF16 output), on B=4, Hq=32 / Hkv=8 (GQA), Nq=Nkv=8192, D=128, causal, with
synthetic seeded inputs.  The metric is TOPS = 4*B*Hq*Nq*Nkv*D / t.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs its own
replica of the workload (weak scaling, no collective on the data path); the
time is the maximum over ranks.  --impl reference times the CPU oracle on the
host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "quantized attention TOPS (4*B*H*Nq*Nkv*D / t)"
UNIT = "TOPS"
DTYPE = "int8-qk+e4m3-pv"     # INT8 codes (FP16 carrier) for QK^T, FP8 E4M3 for PV, FP32 state


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- peaks

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def mixed_peak(bf16_tflops: float) -> dict:
    """Roofline of the forward kernel: half of the algorithmic operations are
    QK^T on the FP16 carrier (FP16 rate = BF16 rate), half are PV in FP8 (twice
    the BF16 rate, by the nominal 4.5 / 2.25 PFLOP/s ratio)."""
    r16, r8 = bf16_tflops, 2.0 * bf16_tflops
    return {"mixed": 2.0 / (1.0 / r16 + 1.0 / r8), "fp8": r8, "fp16": r16}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the run."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        if not rows:
            return None
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if len(inside) < 3:
            inside = [r for r in rows if r[0] <= t1 + 0.05]
            window = "whole run (timed region shorter than the sampling period)"
        reasons = sorted({self.REASONS[i] for r in inside for i, v in enumerate(r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample(w: synth.Workload, rows_per_step: int | None, heads: int, seed_inputs=None):
    """Time the oracle (prepare + forward) on a bounded sample of the workload.

    The sample is the query heads 0 .. heads-1 of batch 0 (one GQA group per
    KV head they read); prepare runs on exactly those heads, forward on all
    their rows, or on `rows_per_step` rows spread evenly over head 0.
    Returns (seconds, literal_ops, description, threads).
    """
    import oracle
    g = w.Hq // w.Hkv
    kv_needed = (heads + g - 1) // g
    if seed_inputs is None:
        q, k, v = synth.make_inputs(w, kv_heads=(0, kv_needed))
        seed_inputs = (q[:1, :heads].copy(), k[:1].copy(), v[:1].copy())
    q, k, v = seed_inputs
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    prep = oracle.prepare(q, k, v)
    if rows_per_step is None:
        rows = np.arange(heads * w.Nq, dtype=np.int64)
    else:
        rows = np.linspace(0, w.Nq - 1, rows_per_step).astype(np.int64)
    oracle.forward(prep, w.Nq, w.Nkv, w.causal, rows=rows, nthreads=threads)
    secs = time.perf_counter() - t0
    ops = 4.0 * rows.size * w.Nkv * w.D
    desc = (f"batch 0, query heads 0..{heads - 1} of {w.B}x{w.Hq}: prepare of those heads and "
            f"their KV head(s), forward of {rows.size} query rows "
            f"({'all rows' if rows_per_step is None else 'evenly spaced over head 0'}); "
            f"literal ops of those rows over all {w.Nkv} keys")
    return secs, ops, desc, threads, seed_inputs


def cpu_baseline(w: synth.Workload, budget_s: float = 15.0) -> dict:
    """Oracle throughput on the host cores: whole query heads, grown until the
    sample takes about `budget_s` seconds."""
    import oracle
    oracle.build()
    heads = 1
    secs, ops, desc, threads, _ = oracle_sample(w, None, heads)
    while secs < budget_s / 2 and heads * 2 <= min(8, w.Hq):
        heads *= 2
        secs, ops, desc, threads, _ = oracle_sample(w, None, heads)
    return {"value": ops / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc, "seconds": round(secs, 3)}


# ----------------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import torch
    import quantized_exact_attention_smoothing_gb300 as sattn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    sattn.load_library()
    w = synth.workload(args.workload)
    if args.batch:
        w = synth.workload(args.workload, B=args.batch)
    log(f"[rank {rank}] generating {w.name} inputs ...")
    q, k, v = synth.make_inputs(w)
    pin = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    hq, hk, hv = pin(q), pin(k), pin(v)
    dq, dk, dv = hq.to(dev), hk.to(dev), hv.to(dev)
    del q, k, v
    shape = sattn.make_shape(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.causal)
    sizes = sattn.query_sizes(shape)
    buf = sattn.prepare_buffers(shape, dev)
    fws = torch.empty(sizes["forward_workspace"], dtype=torch.uint8, device=dev)
    out = torch.empty((w.B, w.Hq, w.Nq, 128), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        prep = sattn.prepare(dq, dk, dv, w.causal, buffers=buf, stream=stream)
        sattn.forward(prep, out=out, workspace=fws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sattn.check_status(fws) != 0:
        raise RuntimeError("device status reports a timeout during warm-up")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_host0 = time.time()
    start.record(stream)
    for e in evs:
        e[0].record(stream)
        prep = sattn.prepare(dq, dk, dv, w.causal, buffers=buf, stream=stream)
        e[1].record(stream)
        sattn.forward(prep, out=out, workspace=fws, stream=stream)
        e[2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(world)
    clk = clocks.stop(t_host0, t_host1)
    if sattn.check_status(fws) != 0:
        raise RuntimeError("device status reports a timeout in the timed region")
    ms_total = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_prep = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    ms_fwd = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    per_step = [e[0].elapsed_time(e[2]) for e in evs]
    step_median = statistics.median(per_step)
    step_cv = statistics.pstdev(per_step) / statistics.fmean(per_step) if K > 1 else 0.0
    ms_step = ms_total / K
    value = world * w.literal_ops / (ms_step * 1e-3) / 1e12

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        arena = torch.empty(sizes["arena"], dtype=torch.uint8, device=dev)
        oh = torch.empty((w.B, w.Hq, w.Nq, 128), dtype=torch.bfloat16, pin_memory=True)
        for _ in range(2):
            sattn.attention_host(hq, hk, hv, w.causal, out=oh, arena=arena, stream=stream)
        torch.cuda.synchronize()
        ke = max(3, K // 10)
        barrier(world)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(ke):
            sattn.attention_host(hq, hk, hv, w.causal, out=oh, arena=arena, stream=stream)
        e2.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms_e2e = max_over_ranks(s2.elapsed_time(e2), world, dev) / ke
        e2e = {"value": world * w.literal_ops / (ms_e2e * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": ms_e2e, "steps": ke,
               "h2d_bytes_per_step": hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2,
               "d2h_bytes_per_step": oh.numel() * 2,
               "path": "sattn_attention_host (pinned host buffers, copies + both passes)"}

    peaks = load_peaks()
    mp = mixed_peak(peaks["bf16_tflops"])
    # DRAM bytes of one attn_fwd_kernel launch from the ncu capture summarised in
    # profiles/attn_fwd_c5_b3_full.md (c5 at batch 3: 495.3 MB read + 159.7 MB
    # written), scaled by the units processed; other workloads were not captured.
    traffic = 655.01e6 * w.B / 3.0 if w.name == "c5" else None
    achieved = w.algorithmic_ops / (ms_fwd * 1e-3) / 1e12
    prep_bytes = (hq.numel() + hk.numel() + hv.numel()) * 2 + \
        (buf["q_codes"].numel() + buf["k_codes"].numel() + w.B * w.Hkv * 128 * w.Nkv) + \
        4 * (buf["q_scales"].numel() + buf["k_scales"].numel() + buf["k_mean"].numel() + buf["v_scales"].numel())
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": f"{w.name}: B{w.B} Hq{w.Hq}/Hkv{w.Hkv} (GQA) Nq=Nkv={w.Nq} D128 "
                               f"{'causal' if w.causal else 'non-causal'}",
                   "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv, "D": 128,
                   "causal": w.causal, "step": "sattn_prepare + sattn_forward",
                   "l2": f"inputs larger than L2 ({prep_bytes / 1e6:.0f} MB streamed per step)",
                   "parallelism": f"replica x{world}"},
        "algorithmic_tops": round(world * w.algorithmic_ops / (ms_step * 1e-3) / 1e12, 3),
        "ms_prepare": round(ms_prep, 5), "ms_forward": round(ms_fwd, 5),
        "ms_per_step_median": round(step_median, 5), "step_cv": round(step_cv, 4),
        "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel (the only kernel of sattn_forward)",
                     "achieved": round(achieved, 2), "peak": round(mp["mixed"], 2), "unit": "TFLOP/s",
                     "frac": round(achieved / mp["mixed"], 4),
                     "traffic": round(traffic) if traffic else None,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, c5 batch 3, "
                                       "scaled by batch" if traffic else None,
                     "peak_basis": f"mixed FP16/FP8 roofline from {peaks['source']} bf16 "
                                   f"{peaks['bf16_tflops']} TFLOP/s (burst) x nominal ratios",
                     "frac_of_fp8_dense": round(achieved / mp["fp8"], 4)},
        "prepare_roofline": {"bound": "hbm", "achieved": round(prep_bytes / (ms_prep * 1e-3) / 1e9, 1),
                             "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(prep_bytes / (ms_prep * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                             "algorithmic_bytes": prep_bytes},
        # per step: 5 prepare kernels + the attention kernel (+ one status memset)
        "gpu_launches": 6 * K,
        "clocks": clk,
    }
    if e2e is not None:
        result["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        log("[rank 0] timing the CPU oracle sample ...")
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    """The CPU oracle on the host cores, on the same workload, metric and unit.
    Each step is a bounded sample: prepare of query head 0 of batch 0 and its
    KV head, forward of rows evenly spaced over that head."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = synth.workload(args.workload)
    rows = args.reference_rows
    _, _, _, _, inputs = oracle_sample(w, rows, 1)
    for _ in range(args.warmup):
        oracle_sample(w, rows, 1, inputs)
    t0 = time.perf_counter()
    ops = 0.0
    for _ in range(args.steps):
        _, o, desc, threads, _ = oracle_sample(w, rows, 1, inputs)
        ops += o
    secs = time.perf_counter() - t0
    value = ops / secs / 1e12
    ms = secs / args.steps * 1e3
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": f"{w.name}: B{w.B} Hq{w.Hq}/Hkv{w.Hkv} (GQA) Nq=Nkv={w.Nq} D128 "
                               f"{'causal' if w.causal else 'non-causal'}",
                   "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv, "D": 128,
                   "causal": w.causal, "step": f"oracle prepare + forward on a {rows}-row sample"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c5", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-rows", type=int, default=256)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (smaller profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
