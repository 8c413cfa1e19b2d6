#!/usr/bin/env python
"""Benchmark: quantized exact attention throughput on the five synthetic workloads.

One step = the whole path on one batch: sattn_prepare (K smoothing, INT8 Q/K,
FP8 V) then sattn_forward (K carrier, INT8 QK^T, online softmax, FP8 P,
two-level PV, BF16 output), with synthetic seeded inputs.  The metric is
TOPS = 4*B*Hq*Nq*Nkv*D / t.  The headline line is the B=4, Hq=32 / Hkv=8
(GQA), Nq=Nkv=8192, D=128, causal workload (c5); the other four workloads
(c1-c4) are measured the same way and reported under "workloads".

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


# The FP8 / FP16 throughput ratio of tcgen05.mma, measured in each run with
# sattn_measure_mma_rate on the forward's own shapes (kind::f16 N = 256 as
# QK^T, kind::f8f6f4 N = 144 as PV); this value (the ratio measured when the
# hook was added: 16366 / 8183 FLOP per SM-clock) stands in if that fails.
FP8_OVER_FP16 = 2.0


def tcgen05_rates(sattn) -> dict:
    try:
        f16 = sattn.measure_mma_rate("f16", 256)
        f8 = sattn.measure_mma_rate("f8", 144)
    except Exception as e:  # reported, not fatal: the recorded ratio is used
        return {"error": str(e), "fp8_over_fp16": FP8_OVER_FP16, "source": "recorded"}
    return {"f16_n256_flop_per_clk_sm": round(f16["flop_per_clk_sm"], 1), "f16_n256_tflops": round(f16["tflops"], 1),
            "f8_n144_flop_per_clk_sm": round(f8["flop_per_clk_sm"], 1), "f8_n144_tflops": round(f8["tflops"], 1),
            "fp8_over_fp16": round(f8["flop_per_clk_sm"] / f16["flop_per_clk_sm"], 4), "source": "measured"}


def mixed_peak(bf16_tflops: float, fp8_over_fp16: float = FP8_OVER_FP16) -> dict:
    """Roofline of the forward kernel: half of the algorithmic operations are
    QK^T on the FP16 carrier (FP16 rate = the measured BF16 GEMM rate), half
    are PV in FP8 at the measured FP8 / FP16 ratio of tcgen05.mma."""
    r16, r8 = bf16_tflops, fp8_over_fp16 * bf16_tflops
    return {"mixed": 2.0 / (1.0 / r16 + 1.0 / r8), "fp8": r8, "fp16": r16}


# DRAM bytes of attn_fwd_kernel from ncu (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by the SHA-256 of the kernel source it was
# captured on; a capture of another source is not used (traffic null).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_dram_bytes.json")
KERNEL_SOURCE = os.path.join(ROOT, "quantized_exact_attention_smoothing_gb300", "csrc", "attn_fwd.cu")


def kernel_source_sha() -> str:
    import hashlib
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def measured_traffic(w) -> dict | None:
    """Per-launch DRAM bytes of the attention kernel for workload w, scaled from
    its capture by the number of (batch, head) units, if the capture was taken
    on the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        data = json.load(f)
    if data.get("source_sha256") != kernel_source_sha():
        return None
    cap = data.get("captures", {}).get(w.name)
    if not cap:
        return None
    units_full = w.B * w.Hq
    scale = units_full / float(cap["units"])
    return {"bytes": (cap["read"] + cap["write"]) * scale, "captured": cap["case"],
            "scaled_by": round(scale, 4)}


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
    """Oracle throughput on the host cores: whole query heads, grown (or the
    whole problem repeated, when it has one head) until the sample takes
    about `budget_s` seconds."""
    import oracle
    oracle.build()
    heads = 1
    secs, ops, desc, threads, inputs = oracle_sample(w, None, heads)
    while secs < budget_s / 2 and heads * 2 <= min(8, w.Hq):
        heads *= 2
        secs, ops, desc, threads, inputs = oracle_sample(w, None, heads)
    reps = 1
    if secs < budget_s / 8:   # a tiny problem: repeat it
        reps = max(1, int(budget_s / 4 / max(secs, 1e-4)))
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle_sample(w, None, heads, inputs)
        secs = (time.perf_counter() - t0) / reps
        desc += f"; mean of {reps} repetitions"
    return {"value": ops / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc, "seconds": round(secs * reps, 3)}


# ----------------------------------------------------------------------------- our arm

# The page's own latency for the single-head case (Q128 x KV192 x D128): the
# p50 of its VEA-B kernel, measured on an SM121 device.  Other hardware and
# another kernel boundary: quoted as context, never as the target.
PAGE_CONTEXT = {"c1": {"page_p50_ms": 0.014426, "what": "VEA-B p50, Q128 x KV192 x D128, SM121 device "
                                                        "(the page's own measurement; context only)"}}
L2_FLUSH_BYTES = 512 << 20   # written between steps of workloads whose inputs fit in L2


def describe(w) -> str:
    return (f"{w.name}: B{w.B} Hq{w.Hq}/Hkv{w.Hkv}{' (GQA)' if w.Hq != w.Hkv else ''} Nq={w.Nq} "
            f"Nkv={w.Nkv} D128 {'causal' if w.causal else 'non-causal'}")


class Runner:
    """Device buffers and one timed step (prepare + forward) of a workload."""

    def __init__(self, sattn, torch, w, dev, stream):
        self.sattn, self.torch, self.w, self.dev, self.stream = sattn, torch, w, dev, stream
        q, k, v = synth.make_inputs(w)
        pin = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
        self.hq, self.hk, self.hv = pin(q), pin(k), pin(v)
        self.dq, self.dk, self.dv = self.hq.to(dev), self.hk.to(dev), self.hv.to(dev)
        del q, k, v
        self.shape = sattn.make_shape(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.causal)
        self.sizes = sattn.query_sizes(self.shape)
        self.buf = sattn.prepare_buffers(self.shape, dev)
        self.fws = torch.empty(self.sizes["forward_workspace"], dtype=torch.uint8, device=dev)
        self.out = torch.empty((w.B, w.Hq, w.Nq, 128), dtype=torch.bfloat16, device=dev)
        self.input_bytes = (self.hq.numel() + self.hk.numel() + self.hv.numel()) * 2

    def step(self, ev=None):
        """prepare + forward; ev = 5 events (step start, forward start, attention
        kernel start and end, step end) or None."""
        sattn, st = self.sattn, self.stream
        if ev is not None:
            ev[0].record(st)
        prep = sattn.prepare(self.dq, self.dk, self.dv, self.w.causal, buffers=self.buf, stream=st)
        if ev is not None:
            ev[1].record(st)
            sattn.profile_events(ev[2], ev[3])
        sattn.forward(prep, out=self.out, workspace=self.fws, stream=st)
        if ev is not None:
            sattn.profile_events()
            ev[4].record(st)

    def prep_bytes(self) -> int:
        b, w = self.buf, self.w
        return self.input_bytes + (b["q_codes"].numel() + b["k_codes"].numel() + w.B * w.Hkv * 128 * w.Nkv) + \
            4 * (b["q_scales"].numel() + b["k_scales"].numel() + b["k_mean"].numel() + b["v_scales"].numel())

    def check(self, where: str):
        if self.sattn.check_status(self.fws) != 0:
            raise RuntimeError(f"device status reports a timeout {where}")


def summarise(w, evs, peaks) -> dict:
    """Per-step means of the five events of each step, and the rooflines."""
    K = len(evs)
    ms_prep = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    ms_fwd = sum(e[1].elapsed_time(e[4]) for e in evs) / K
    ms_attn = sum(e[2].elapsed_time(e[3]) for e in evs) / K
    per_step = [e[0].elapsed_time(e[4]) for e in evs]
    ratio = peaks.get("fp8_over_fp16", FP8_OVER_FP16)
    mp = mixed_peak(peaks["bf16_tflops"], ratio)
    achieved = w.algorithmic_ops / (ms_attn * 1e-3) / 1e12
    tr = measured_traffic(w)
    return {
        "ms_prepare": round(ms_prep, 5), "ms_forward": round(ms_fwd, 5), "ms_attention_kernel": round(ms_attn, 5),
        "ms_step_mean": round(statistics.fmean(per_step), 5), "ms_step_median": round(statistics.median(per_step), 5),
        "step_cv": round(statistics.pstdev(per_step) / statistics.fmean(per_step), 4) if K > 1 else 0.0,
        "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel",
                     "achieved": round(achieved, 2), "peak": round(mp["mixed"], 2), "unit": "TFLOP/s",
                     "frac": round(achieved / mp["mixed"], 4),
                     "traffic": round(tr["bytes"]) if tr else None,
                     "traffic_source": (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of {tr['captured']}, "
                                        f"scaled x{tr['scaled_by']} by (batch, head) units") if tr else
                                       "no capture of the current kernel source",
                     "achieved_basis": "algorithmic ops (4 * D per unmasked query-key pair) / mean duration of "
                                       "the attention kernel (CUDA events recorded by sattn_profile_events)",
                     "peak_basis": f"{peaks['source']} bf16 {peaks['bf16_tflops']} TFLOP/s (burst) for the FP16 "
                                   f"half, x{ratio:.2f} (tcgen05 FP8/FP16, {peaks.get('ratio_source', 'recorded')}) "
                                   f"for the FP8 half",
                     "frac_of_fp8_dense": round(achieved / mp["fp8"], 4)},
    }


def measure_workload(r: Runner, steps: int, warmup: int, peaks: dict, flush: bool) -> dict:
    """Steps timed one by one with CUDA events; with `flush` an L2-sized
    buffer is written between steps (outside the events)."""
    torch, st = r.torch, r.stream
    scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=r.dev) if flush else None
    for _ in range(warmup):
        r.step()
    torch.cuda.synchronize()
    r.check("during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for e in evs:
        if scratch is not None:
            scratch.zero_()
        r.step(e)
    torch.cuda.synchronize()
    r.check("in the timed steps")
    res = summarise(r.w, evs, peaks)
    ms = res["ms_step_mean"]
    res.update({"config": describe(r.w), "value": round(r.w.literal_ops / (ms * 1e-3) / 1e12, 4), "unit": UNIT,
                "algorithmic_tops": round(r.w.algorithmic_ops / (ms * 1e-3) / 1e12, 4), "steps": steps,
                "l2": "L2 flushed between steps (512 MB written)" if flush else
                      f"inputs larger than L2 ({r.prep_bytes() / 1e6:.0f} MB streamed per step)"})
    res["prepare_roofline"] = prepare_roofline(r, res["ms_prepare"], peaks)
    if r.w.name in PAGE_CONTEXT:
        res["context"] = dict(PAGE_CONTEXT[r.w.name], ours_ms_forward=res["ms_forward"],
                              ours_ms_attention_kernel=res["ms_attention_kernel"])
    return res


def measure_small(sattn, torch, r: Runner, steps: int, warmup: int, flush: bool) -> dict:
    """The same step through sattn_attention_small (preparation and attention
    in one launch), timed like measure_workload."""
    st = r.stream
    buf = sattn.prepare_buffers(r.shape, r.dev)
    ws = torch.empty(r.sizes["forward_workspace"], dtype=torch.uint8, device=r.dev)
    out = torch.empty_like(r.out)
    call = lambda: sattn.attention_small(r.dq, r.dk, r.dv, r.w.causal, buffers=buf, out=out, workspace=ws, stream=st)
    scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=r.dev) if flush else None
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in evs:
        if scratch is not None:
            scratch.zero_()
        e[0].record(st)
        call()
        e[1].record(st)
    torch.cuda.synchronize()
    if sattn.check_status(ws) != 0:
        raise RuntimeError("device status reports a timeout in the small-path steps")
    same = bool(torch.equal(out.view(torch.int16), r.out.view(torch.int16)))
    ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in evs)
    return {"ms_step_mean": round(ms, 5), "value": round(r.w.literal_ops / (ms * 1e-3) / 1e12, 4),
            "launches_per_step": 1, "output_equals_two_calls": same,
            "path": "sattn_attention_small (preparation inside the attention kernel)"}


def prepare_roofline(r: Runner, ms_prep: float, peaks: dict) -> dict:
    pb = r.prep_bytes()
    gbs = pb / (ms_prep * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": pb}


def run_ours(args, world, rank, local):
    import torch
    import quantized_exact_attention_smoothing_gb300 as sattn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    sattn.load_library()
    peaks = load_peaks()
    rates = tcgen05_rates(sattn)
    peaks["fp8_over_fp16"] = rates["fp8_over_fp16"]
    peaks["ratio_source"] = rates["source"]
    if args.mma_rates:
        if rank == 0:
            print(json.dumps({"tcgen05": rates, "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count}),
                  flush=True)
        return
    stream = torch.cuda.current_stream()
    w = synth.workload(args.workload)
    if args.batch:
        w = synth.workload(args.workload, B=args.batch)
    if args.heads:
        w = synth.workload(w.name, B=w.B, Hq=args.heads, Hkv=min(w.Hkv, args.heads))
    log(f"[rank {rank}] generating {w.name} inputs ...")
    r = Runner(sattn, torch, w, dev, stream)

    for _ in range(args.warmup):
        r.step()
    torch.cuda.synchronize()
    r.check("during warm-up")

    # the headline: exactly K steps between two events, barrier and synchronize on both sides
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_host0 = time.time()
    start.record(stream)
    for e in evs:
        r.step(e)
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(world)
    clk = clocks.stop(t_host0, t_host1)
    r.check("in the timed region")
    ms_total = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_step = ms_total / K
    value = world * w.literal_ops / (ms_step * 1e-3) / 1e12
    summ = summarise(w, evs, peaks)

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        arena = torch.empty(r.sizes["arena"], dtype=torch.uint8, device=dev)
        oh = torch.empty((w.B, w.Hq, w.Nq, 128), dtype=torch.bfloat16, pin_memory=True)
        for _ in range(2):
            sattn.attention_host(r.hq, r.hk, r.hv, w.causal, out=oh, arena=arena, stream=stream)
        torch.cuda.synchronize()
        ke = max(3, K // 10)
        barrier(world)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(ke):
            sattn.attention_host(r.hq, r.hk, r.hv, w.causal, out=oh, arena=arena, stream=stream)
        e2.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms_e2e = max_over_ranks(s2.elapsed_time(e2), world, dev) / ke
        e2e = {"value": world * w.literal_ops / (ms_e2e * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": ms_e2e, "steps": ke, "h2d_bytes_per_step": r.input_bytes,
               "d2h_bytes_per_step": oh.numel() * 2,
               "path": "sattn_attention_host (pinned host buffers, copies + both passes)"}
        del arena, oh

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": describe(w), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv,
                   "D": 128, "causal": w.causal, "step": "sattn_prepare + sattn_forward",
                   "l2": f"inputs larger than L2 ({r.prep_bytes() / 1e6:.0f} MB streamed per step)",
                   "parallelism": f"replica x{world}"},
        "algorithmic_tops": round(world * w.algorithmic_ops / (ms_step * 1e-3) / 1e12, 3),
        "ms_prepare": summ["ms_prepare"], "ms_forward": summ["ms_forward"],
        "ms_attention_kernel": summ["ms_attention_kernel"],
        "ms_per_step_median": summ["ms_step_median"], "step_cv": summ["step_cv"],
        "roofline": summ["roofline"],
        "prepare_roofline": prepare_roofline(r, summ["ms_prepare"], peaks),
        # per step: five prepare kernels, the K carrier conversion and the attention kernel
        "gpu_launches": 7 * K,
        "clocks": clk,
        "tcgen05": rates,
    }
    if e2e is not None:
        result["e2e"] = e2e
    del r
    torch.cuda.empty_cache()

    # the other four workloads (rank 0 of a single-GPU run only: they are not scaled)
    if world == 1 and not args.headline_only:
        others = {}
        for name in ("c1", "c2", "c3", "c4"):
            if name == w.name:
                continue
            wo = synth.workload(name)
            log(f"[rank {rank}] measuring {name} ...")
            ro = Runner(sattn, torch, wo, dev, stream)
            flush = ro.prep_bytes() < 4 * 129e6
            steps = 50 if wo.literal_ops < 1e13 else 20
            res = measure_workload(ro, steps, args.warmup, peaks, flush)
            if sattn.small_shape_ok(wo.B, wo.Hq, wo.Hkv, wo.Nq, wo.Nkv):
                res["small_path"] = measure_small(sattn, torch, ro, steps, args.warmup, flush)
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = cpu_baseline(wo, budget_s=6.0)
            others[name] = res
            del ro
            torch.cuda.empty_cache()
        result["workloads"] = others
        result["gpu_launches_workloads"] = 7 * sum((args.warmup + o["steps"]) for o in others.values())
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
        "config": {"workload": describe(w),
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
    ap.add_argument("--heads", type=int, default=None,
                    help="override the workload's query heads (smaller profiling captures)")
    ap.add_argument("--mma-rates", action="store_true",
                    help="print the measured tcgen05.mma rates and exit")
    ap.add_argument("--headline-only", action="store_true",
                    help="measure the headline workload only (no c1-c4 lines)")
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
