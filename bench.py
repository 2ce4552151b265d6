#!/usr/bin/env python
"""Benchmark of the weight-quantized SwiGLU MLP on GB300.

Headline (one JSON line on stdout): microseconds per MLP call of the dense
27B-class NVFP4 decode MLP (hidden K=5120, intermediate I=17408, M=1 token),
i.e. the gate/up GEMV with fused SwiGLU followed by the down GEMV, on
synthetic seeded weights. One "step" = one MLP call. Inputs are resident in
HBM; the weights rotate over several independent device copies whose total
exceeds twice the L2 size, so every call streams its weights from HBM.

Also reported: the HBM roofline fraction of the dominant kernel (the
single-launch decode MLP, timed with CUDA events on its stream), the
end-to-end time through the host-buffer entry point, the CPU oracle timed on
this host, and secondary workloads (tiny NVFP4, FP8 W8A16 decode,
routed-expert AWQ, NVFP4 and FP8 prefill on the tensor-core GEMM).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]
"""
from __future__ import annotations

import argparse
import hashlib
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

from weight_quantized_swiglu_gb300 import inputs as gen  # noqa: E402

METRIC = "MLP us/call (dense NVFP4 decode, M=1)"
UNIT = "us/call"
K_HID, I_INT = gen.DENSE_K, gen.DENSE_I


def nvfp4_bytes(K, I):
    """Algorithmic bytes of one NVFP4 MLP call: packed codes + E4M3 scales of
    gate, up, down + the three fp32 globals (activations excluded)."""
    return 3 * (I * K // 2 + I * K // 16) + 12


def nvfp4_gateup_bytes(K, I):
    return 2 * (I * K // 2 + I * K // 16)


def fp8_bytes(K, I):
    return 3 * I * K + 4 * (I + I + K)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_src_sha(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    if d.get("src_sha") != kernel_src_sha(d["src_files"]):
        return None
    return d.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(device_index)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


def parse_clock_samples(text):
    """Median SM clock, max SM clock and the throttle reasons seen in the
    `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits`
    lines; None when no line carries a clock."""
    sm, smax, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax = float(parts[2])
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
            "samples": len(sm)}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ----------------------------------------------------------------------------
def dist_setup(n_gpus):
    """Rank layout from the torchrun environment; one process per GPU over
    NCCL (gloo when there is no GPU: the host logic alone, as in the tests)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    """The largest v over the ranks (timings: the job is as slow as its
    slowest replica)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# measurements
# ----------------------------------------------------------------------------
def n_rotating_copies(bytes_per_copy):
    import torch
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    return max(2, math.ceil(2 * l2 / bytes_per_copy) + 1), l2


def capture(calls, stream):
    """CUDA graph of the given zero-argument launch closures (run once first)."""
    import torch
    with torch.cuda.stream(stream):
        for f in calls:
            f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for f in calls:
            f()
    return g


def time_graph(g, reps, stream):
    """Replay `g` reps times on `stream`, timed by CUDA events on that stream."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def time_graph_samples(g, stream, min_samples=7, min_seconds=1.0):
    """Replays of `g` on `stream`, each timed by its own pair of CUDA events
    on that stream, back to back: at least `min_samples` of them and at least
    `min_seconds` of device time (so the clock sampler sees the timed region).
    Returns the per-replay times in ms."""
    import torch
    times, total = [], 0.0
    while len(times) < min_samples or total < min_seconds * 1e3:
        n = max(min_samples, 64)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(n):
                g.replay()
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
        batch = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
        times += batch
        total += sum(batch)
    return times


def bench_headline(args, world, rank, local, pk):
    import torch
    import weight_quantized_swiglu_gb300 as q
    case = gen.workload_case("dense_nvfp4_decode", 0)
    R, l2 = n_rotating_copies(nvfp4_bytes(K_HID, I_INT))
    mlps = [q.QuantMLP.from_case(case) for _ in range(R)]
    x = torch.from_numpy(case.x.view(np.int16)).cuda()
    out = torch.empty((1, K_HID), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    # one graph of exactly K = --steps calls (the weights rotate over the R
    # copies), replayed back to back; every replay is one timed sample
    K = max(1, args.steps)
    g = capture([(lambda m=mlps[i % R]: m.forward(x, out, stream=s)) for i in range(K)], s)
    with torch.cuda.stream(s):
        for _ in range(max(1, math.ceil(args.warmup / K))):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    time.sleep(0.25)
    barrier(world)
    torch.cuda.synchronize()
    samples = time_graph_samples(g, s)
    barrier(world)
    clocks = sampler.stop()
    med_ms = max_over_ranks(world, statistics.median(samples))
    us_per_call = med_ms * 1e3 / K
    mlps[0].check()
    del g

    # per-projection kernels (stage launches) for diagnostics
    per_graph = R * max(1, 24 // R)
    g0 = capture([(lambda m=mlps[i % R]: m.forward_stage(0, x, None, 1, stream=s)) for i in range(per_graph)], s)
    g1 = capture([(lambda m=mlps[i % R]: m.forward_stage(1, None, out, 1, stream=s)) for i in range(per_graph)], s)
    gu_us = statistics.median(time_graph_samples(g0, s, min_seconds=0.2)) * 1e3 / per_graph
    dn_us = statistics.median(time_graph_samples(g1, s, min_seconds=0.2)) * 1e3 / per_graph
    del g0, g1

    # end-to-end through the host-buffer entry point (pinned buffers; the
    # copies and the completion wait are inside the timed region)
    xh = torch.from_numpy(case.x.view(np.int16)).pin_memory()
    oh = torch.empty((1, K_HID), dtype=torch.int16).pin_memory()
    for i in range(3):
        mlps[i % R].forward_host(xh, oh, stream=s)
    n_e2e = max(200, min(K, 2000))
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        mlps[i % R].forward_host(xh, oh, stream=s)
    e2e_s = max_over_ranks(world, time.perf_counter() - t0)
    for m in mlps:
        m.close()

    call_bytes = nvfp4_bytes(K_HID, I_INT)
    achieved = call_bytes / (us_per_call * 1e-6) / 1e9
    res = {
        "us_per_call": us_per_call,
        "steps": K,
        "samples": len(samples),
        "sample_spread_us": [min(samples) * 1e3 / K, max(samples) * 1e3 / K],
        "ms_per_step": med_ms / K,
        "gu_us": gu_us,
        "down_us": dn_us,
        "hbm_gbs_call": achieved,
        "roofline": {"bound": "hbm", "kernel": "gemv_split_kernel<NVFP4, M=1> (whole MLP, I partitioned over CTAs, "
                                               "in-kernel reduction; time = the whole call)",
                     "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"],
                     "algorithmic_bytes_per_launch": call_bytes,
                     "traffic": ncu_traffic("gemv_split_nvfp4_m1")},
        "e2e": {"value": e2e_s * 1e6 / n_e2e, "unit": UNIT, "h2d_bytes_per_step": K_HID * 2,
                "d2h_bytes_per_step": K_HID * 2, "steps": n_e2e},
        "clocks": clocks,
        "rotating_copies": R,
        "l2_bytes": l2,
        # one kernel per call at M=1 (NVFP4: in-kernel reduction), K calls per
        # timed replay
        "gpu_launches": K * len(samples),
    }
    return res, case


def oracle_time(fn, budget_s=2.0):
    """Wall time of one call of an oracle function on this host's cores:
    repeated until `budget_s` has passed (at least once). Returns (seconds
    per call, calls)."""
    if budget_s > 0:
        fn()  # tables, page-in (skipped for the long, single-call timings)
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el / n, n


def oracle_baseline(fn, unit_scale, unit, what, budget_s=2.0, extrapolate=None):
    """cpu_baseline object of one workload: the oracle as it stands, timed on
    the host cores. extrapolate = (factor, how) scales a timed sample to the
    whole workload and says so."""
    import oracle
    oracle.build()
    sec, n = oracle_time(fn, budget_s)
    value = sec * unit_scale
    sample = f"{n} oracle call(s) of {what}, {sec:.3f} s each"
    kind = "oracle"
    if extrapolate:
        value *= extrapolate[0]
        sample += f"; extrapolated to the whole workload: {extrapolate[1]}"
        kind = "oracle (extrapolated)"
    return {"value": value, "unit": unit, "cores": oracle.num_threads(), "kind": kind, "sample": sample}


def bench_dense_secondary(name, variant, fmt_bytes):
    """us/call of another dense workload (rotating copies, CUDA-graph replay,
    median of >= 7 timed replays), with the oracle timed beside it."""
    import torch
    import weight_quantized_swiglu_gb300 as q
    case = gen.workload_case(name, variant)
    R, _ = n_rotating_copies(fmt_bytes)
    mlps = [q.QuantMLP.from_case(case) for _ in range(R)]
    x = torch.from_numpy(case.x.view(np.int16)).cuda()
    out = torch.empty((case.M, case.K), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    per_graph = R * max(1, 24 // R)
    g = capture([(lambda m=mlps[i % R]: m.forward(x, out, stream=s)) for i in range(per_graph)], s)
    time_graph(g, 1, s)
    samples = time_graph_samples(g, s, min_seconds=0.3)
    us = statistics.median(samples) * 1e3 / per_graph
    del g
    for m in mlps:
        m.close()
    import oracle
    cpu = oracle_baseline(lambda: oracle.dense_forward(case), 1e6, UNIT,
                          f"the full MLP (K={case.K}, I={case.I}, M={case.M}, fp64)")
    return {"M": case.M, "us_per_call": us, "samples": len(samples), "gbs": fmt_bytes / (us * 1e-6) / 1e9,
            "tokens_per_s": case.M / (us * 1e-6), "cpu_baseline": cpu}


def bench_moe(meta_bytes=4):
    """Routed-expert M=1: CUDA-graph replay of 48 calls, 7 samples, median
    (hot = the same 10 experts; rotating = 480 experts cycled)."""
    import torch
    import weight_quantized_swiglu_gb300 as q
    c = gen.gen_moe_case(gen.seed_for(4, 0))
    moe = q.MoeAWQ.from_case(c, meta_bytes)
    x = torch.from_numpy(c.x_fp16.view(np.int16)).cuda()
    rw = torch.from_numpy(c.router_w).cuda()
    hot_ids = torch.from_numpy(c.ids).cuda()
    # one 16-entry (64-byte) row per call keeps every row 16-byte aligned
    rot = np.full((48, 16), -1, np.int32)
    for k in range(48):
        rot[k, :10] = gen.rotating_ids(k)
    rot_ids = torch.from_numpy(rot).cuda()
    out = torch.empty(c.K, dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    res = {}
    for mode in ("hot", "rotating"):
        with torch.cuda.stream(s):
            for k in range(3):
                moe.forward(x, q.DT_FP16, hot_ids if mode == "hot" else rot_ids[k, :10], rw, out, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for k in range(48):
                moe.forward(x, q.DT_FP16, hot_ids if mode == "hot" else rot_ids[k, :10], rw, out, stream=s)
        g.replay()
        torch.cuda.synchronize()
        samples = []
        for _ in range(7):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            samples.append(e0.elapsed_time(e1))
        ms48 = statistics.median(samples)
        uniq = len({int(i) for i in (c.ids if mode == "hot" else gen.rotating_ids(0)) if 0 <= i < c.E})
        per_exp = 2 * c.I * c.K // 2 + 2 * c.I * (c.K // 32) * meta_bytes + c.K * c.I // 2 + c.K * (c.I // 32) * meta_bytes
        res[mode] = {"ms_per_48_calls": ms48, "us_per_call": ms48 * 1e3 / 48,
                     "gbs": uniq * per_exp / (ms48 * 1e-3 / 48) / 1e9}
    moe.close()
    import oracle
    res["cpu_baseline"] = oracle_baseline(lambda: oracle.moe_m1_forward(c, meta_bytes, "fp16"), 1e6, "us/call",
                                          f"the routed-expert step (E={c.E}, top-{c.topk}, {meta_bytes}-byte "
                                          f"metadata, the hot id set)")
    return res


def bench_moe_tokens(Ms=(16, 512), meta_bytes=4):
    """Routed experts for M tokens (grouped by expert on the device), E=512
    K=2560 I=160 top-10: CUDA-graph replay of 20 calls, 7 samples, median.
    Bytes = the unique valid experts' codes + metadata (each read once when
    the grouping shares them)."""
    import torch
    import weight_quantized_swiglu_gb300 as q
    tok = gen.gen_moe_tokens(gen.seed_for(6, 0), max(Ms))
    c = tok.case
    moe = q.MoeAWQ.from_case(c, meta_bytes)
    moe.reserve(max(Ms))
    per_exp = 2 * c.I * c.K // 2 + 2 * c.I * (c.K // 32) * meta_bytes + c.K * c.I // 2 + c.K * (c.I // 32) * meta_bytes
    s = torch.cuda.Stream()
    res = {}
    for M in Ms:
        x = torch.from_numpy(tok.x16[:M].view(np.int16).copy()).cuda()
        ids = torch.from_numpy(tok.ids[:M].copy()).cuda()
        rw = torch.from_numpy(tok.rw[:M].copy()).cuda()
        out = torch.empty((M, c.K), dtype=torch.int16, device="cuda")
        with torch.cuda.stream(s):
            for _ in range(3):
                moe.forward_tokens(x, q.DT_FP16, ids, rw, out, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(20):
                moe.forward_tokens(x, q.DT_FP16, ids, rw, out, stream=s)
        g.replay()
        torch.cuda.synchronize()
        samples = []
        for _ in range(7):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            samples.append(e0.elapsed_time(e1))
        us = statistics.median(samples) * 1e3 / 20
        uniq = len({int(i) for i in tok.ids[:M].ravel() if 0 <= i < c.E})
        import oracle
        from dataclasses import replace
        nt = min(M, 32)  # tokens are independent: a sample of them, scaled by M / nt

        def run_tokens(nt=nt):
            for t in range(nt):
                oracle.moe_m1_forward(replace(c, x_fp16=tok.x16[t]), meta_bytes, "fp16", ids=tok.ids[t],
                                      rw=tok.rw[t])
        cpu = oracle_baseline(run_tokens, 1e6, "us/call", f"{nt} tokens' routed-expert steps",
                              extrapolate=None if nt == M else (M / nt, f"x {M}/{nt} tokens"))
        res[f"M{M}"] = {"us_per_call": us, "tokens_per_s": M / (us * 1e-6), "unique_experts": uniq,
                        "gbs_unique_bytes": uniq * per_exp / (us * 1e-6) / 1e9, "cpu_baseline": cpu}
        del g
    moe.check()
    moe.close()
    return res


DQ_MIN_M = 768  # the automatic path decodes the weights once per call from here on


def bench_prefill(M, reps, pk, fmt="nvfp4", path=None, cpu=True):
    import torch
    import weight_quantized_swiglu_gb300 as q
    case = gen.gen_dense_case(fmt, K_HID, I_INT, M, gen.seed_for(3 if fmt == "nvfp4" else 5, 0 if M == 512 else 1))
    mlp = q.QuantMLP.from_case(case)
    x = torch.from_numpy(case.x.view(np.int16)).cuda()
    out = torch.empty((M, K_HID), dtype=torch.int16, device="cuda")
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    path = q.PATH_AUTO if path is None else path
    name = {q.PATH_GEMM: "gemm (decoder warps)", q.PATH_GEMM_PAIR: "gemm_pair (decoder warps, CTA pairs)",
            q.PATH_GEMM_DQ: "gemm_dq (weights decoded once per call)"}.get(path)
    if name is None:
        name = "auto: " + ("gemm_dq (weights decoded once per call)" if M >= DQ_MIN_M else "gemm (decoder warps)")
    for _ in range(3):
        mlp.forward(x, out, path=path)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mlp.forward(x, out, path=path)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    mlp.check()
    mlp.close()
    ms = statistics.median(times)
    flops = 2.0 * M * 3 * I_INT * K_HID
    tf = flops / (ms * 1e-3) / 1e12
    import oracle
    if not cpu:
        cpu = None
    elif M <= 512:
        cpu = oracle_baseline(lambda: oracle.dense_forward(case), 1e3, "ms/call",
                              f"the full MLP (K={K_HID}, I={I_INT}, M={M}, fp64)", budget_s=0.0)
    else:
        rows = np.arange(0, M, M // 64, dtype=np.int32)[:64]
        cpu = oracle_baseline(lambda: oracle.dense_forward(case, rows=rows), 1e3, "ms/call",
                              f"64 token rows of the M={M} MLP (fp64; every call decodes all weights once)",
                              budget_s=0.0, extrapolate=(M / 64, f"x {M}/64 rows (an upper bound: the weight "
                                                                 f"decode is counted once per 64 rows)"))
    # each call is timed alone (L2 flushed between calls): the burst peak applies
    return {"M": M, "path": name, "ms_per_call": ms, "tflops": tf, "frac_bf16_peak": tf / pk["bf16_tflops"],
            "peak_tflops": pk["bf16_tflops"], "peak_kind": "bf16 burst (cuBLAS, isolated calls), " + pk["source"],
            "tokens_per_s": M / (ms * 1e-3), "l2": "512 MB buffer written between calls", "cpu_baseline": cpu}


def cpu_baseline(case, budget_s=10.0):
    import oracle
    oracle.build()
    oracle.dense_forward(case)  # warm (tables, page-in)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.dense_forward(case)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": el * 1e6 / n, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} full oracle MLP calls (K=5120, I=17408, M=1, fp64) in {el:.1f} s"}


# ----------------------------------------------------------------------------
# the reference arm: the CPU oracle as it stands
# ----------------------------------------------------------------------------
def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    case = gen.workload_case("dense_nvfp4_decode", 0)
    t0 = time.perf_counter()
    oracle.dense_forward(case)
    t_full = time.perf_counter() - t0
    budget = 150.0
    frac = min(1.0, budget / max(1e-9, (args.steps + args.warmup) * t_full))
    sub = None
    if frac < 1.0:
        # each step computes a row block of gate, up and down (a fixed fraction
        # of the weights) with the oracle's projection routine; the time is
        # scaled by the fraction of weights processed
        ni = max(16, int(I_INT * frac) // 16 * 16)
        nk = max(16, int(K_HID * frac) // 16 * 16)
        cut = lambda p, n: gen.Proj(p.fmt, n, p.K, p.w[:n], p.scale[:n], p.global_scale)
        sub = (cut(case.gate, ni), cut(case.up, ni), cut(case.down, nk))
        xact = gen.gen_x_only(7, 1, I_INT)
        wfrac = (2 * ni * K_HID + nk * I_INT) / (2 * I_INT * K_HID + K_HID * I_INT)

    def step():
        if sub is None:
            oracle.dense_forward(case)
        else:
            oracle.project(sub[0], case.x)
            oracle.project(sub[1], case.x)
            oracle.project(sub[2], xact)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    per_step_us = el * 1e6 / args.steps
    value = per_step_us if sub is None else per_step_us / wfrac
    sample = ("full oracle MLP call per step" if sub is None else
              f"per step: rows 0:{sub[0].N} of gate/up and 0:{sub[2].N} of down ({wfrac:.4f} of the weights); "
              f"us/call scaled by 1/{wfrac:.4f}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded NVFP4 weights, x ~ N(0,1) bf16)",
            "config": {"workload": "dense_nvfp4_decode K=5120 I=17408 M=1", "K": K_HID, "I": I_INT, "M": 1,
                       "fmt": "nvfp4"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# eager launches of one operation, for ncu (no JSON output)
# ----------------------------------------------------------------------------
def run_profile(args):
    import torch
    import weight_quantized_swiglu_gb300 as q
    from weight_quantized_swiglu_gb300 import build
    build.build()
    n = args.warmup + args.steps
    if args.profile in ("fused", "fusedM4", "stage0", "stage1", "fp8_fused", "fp8_fusedM16"):
        name = "dense_fp8_decode" if args.profile.startswith("fp8_fused") else "dense_nvfp4_decode"
        case = gen.workload_case(name, 1 if args.profile in ("fusedM4", "fp8_fusedM16") else 0)
        mlp = q.QuantMLP.from_case(case)
        x = torch.from_numpy(case.x.view(np.int16)).cuda()
        out = torch.empty((case.M, case.K), dtype=torch.int16, device="cuda")
        for _ in range(n):
            if args.profile in ("fused", "fusedM4", "fp8_fused", "fp8_fusedM16"):
                mlp.forward(x, out)
            elif args.profile == "stage0":
                mlp.forward_stage(0, x, None, 1)
            else:
                mlp.forward_stage(0, x, None, 1)
                mlp.forward_stage(1, None, out, 1)
        torch.cuda.synchronize()
        mlp.check()
    elif args.profile == "moe":
        c = gen.gen_moe_case(gen.seed_for(4, 0))
        moe = q.MoeAWQ.from_case(c, 4)
        x = torch.from_numpy(c.x_fp16.view(np.int16)).cuda()
        ids = torch.from_numpy(c.ids).cuda()
        rw = torch.from_numpy(c.router_w).cuda()
        out = torch.empty(c.K, dtype=torch.int16, device="cuda")
        for _ in range(n):
            moe.forward(x, q.DT_FP16, ids, rw, out)
        torch.cuda.synchronize()
        moe.check()
    elif args.profile.startswith("moetokens"):
        M = int(args.profile[len("moetokens"):] or 16)
        tok = gen.gen_moe_tokens(gen.seed_for(6, 0), M)
        moe = q.MoeAWQ.from_case(tok.case, 4)
        moe.reserve(M)
        x = torch.from_numpy(tok.x16.view(np.int16).copy()).cuda()
        ids = torch.from_numpy(tok.ids.copy()).cuda()
        rw = torch.from_numpy(tok.rw.copy()).cuda()
        out = torch.empty((M, tok.case.K), dtype=torch.int16, device="cuda")
        for _ in range(n):
            moe.forward_tokens(x, q.DT_FP16, ids, rw, out)
        torch.cuda.synchronize()
        moe.check()
    elif any(args.profile.startswith(p) for p in ("prefill", "fp8prefill", "pairprefill", "fp8pairprefill",
                                                  "dqprefill", "fp8dqprefill")):
        fp8 = args.profile.startswith("fp8")
        pair = "pair" in args.profile
        path = q.PATH_GEMM_PAIR if pair else q.PATH_GEMM_DQ if "dq" in args.profile else q.PATH_GEMM
        M = int(args.profile.split("prefill", 1)[1] or 512)
        case = gen.gen_dense_case("fp8" if fp8 else "nvfp4", K_HID, I_INT, M, gen.seed_for(5 if fp8 else 3, 0))
        mlp = q.QuantMLP.from_case(case)
        x = torch.from_numpy(case.x.view(np.int16)).cuda()
        out = torch.empty((M, K_HID), dtype=torch.int16, device="cuda")
        for _ in range(n):
            mlp.forward(x, out, path=path)
        torch.cuda.synchronize()
        mlp.check()
    print(f"profile {args.profile}: {n} calls ok", flush=True)


# ----------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--extras", default="all",
                    help="comma list of extra workloads to time (decode,fp8,tiny,moe,prefill) or 'all'")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--profile", default=None,
                    help="eager launches of one operation for ncu: fused|fusedM4|stage0|stage1|fp8_fused|fp8_fusedM16|moe|"
                         "moetokensM|prefillM|fp8prefillM|pairprefillM|fp8pairprefillM|dqprefillM|fp8dqprefillM "
                         "(prefill: the decoder-warp GEMM; dq: weights decoded once per call)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.profile:
        run_profile(args)
        return

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path in this library)")
    world, rank, local = dist_setup(args.gpus)
    from weight_quantized_swiglu_gb300 import build
    if rank == 0:
        build.build()
    barrier(world)
    pk = peaks()
    head, case = bench_headline(args, world, rank, local, pk)

    extras = {}
    if not args.no_extras and rank == 0:
        import weight_quantized_swiglu_gb300 as q
        want = set(args.extras.split(",")) if args.extras != "all" else {"decode", "fp8", "tiny", "moe", "prefill"}
        if "decode" in want:
            extras["dense_nvfp4_decode_M4"] = bench_dense_secondary("dense_nvfp4_decode", 1,
                                                                    nvfp4_bytes(K_HID, I_INT))
        if "fp8" in want:
            extras["dense_fp8_decode_M1"] = bench_dense_secondary("dense_fp8_decode", 0, fp8_bytes(K_HID, I_INT))
            extras["dense_fp8_decode_M16"] = bench_dense_secondary("dense_fp8_decode", 1, fp8_bytes(K_HID, I_INT))
        if "tiny" in want:
            extras["tiny_nvfp4_M1"] = bench_dense_secondary("tiny_nvfp4", 0, nvfp4_bytes(gen.TINY_K, gen.TINY_I))
        if "moe" in want:
            extras["moe_awq_m1_4B"] = bench_moe(4)
            extras["moe_awq_m1_3B"] = bench_moe(3)
            extras["moe_awq_tokens_4B"] = bench_moe_tokens()
        if "prefill" in want:
            for fmt in ("nvfp4", "fp8"):
                try:
                    extras[f"{fmt}_mid_M64"] = bench_prefill(64, 5, pk, fmt)
                    extras[f"{fmt}_prefill_M512"] = bench_prefill(512, 5, pk, fmt)
                    extras[f"{fmt}_prefill_M8192"] = bench_prefill(8192, 3, pk, fmt)
                    # the explicit paths the automatic one (above) does not take at
                    # this size: the decoder-warp GEMM, single CTAs and CTA pairs
                    for key, path in (("decwarps", q.PATH_GEMM), ("pair", q.PATH_GEMM_PAIR)):
                        line = bench_prefill(8192, 3, pk, fmt, path=path, cpu=False)
                        # same workload and inputs as the automatic line: its oracle timing applies
                        line["cpu_baseline"] = extras[f"{fmt}_prefill_M8192"]["cpu_baseline"]
                        extras[f"{fmt}_prefill_{key}_M8192"] = line
                except q.QmlpError as e:
                    extras[f"{fmt}_prefill"] = {"unavailable": str(e)}
        torch.cuda.synchronize()

    cpu = cpu_baseline(case, args.cpu_budget) if rank == 0 else None
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": head["us_per_call"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": head["steps"],
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 weights, fp16 x fp16 -> fp32 MMA, bf16 act/out",
        "data": "synthetic (seeded NVFP4 weights, x ~ N(0,1) bf16)",
        "config": {"workload": "dense_nvfp4_decode K=5120 I=17408 M=1", "K": K_HID, "I": I_INT, "M": 1,
                   "fmt": "nvfp4", "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": f"{head['rotating_copies']} rotating weight copies "
                         f"({head['rotating_copies'] * nvfp4_bytes(K_HID, I_INT) / 1e6:.0f} MB > 2x L2 "
                         f"{head['l2_bytes'] / 1e6:.0f} MB)"},
        "hbm_gbs": head["hbm_gbs_call"],
        "kernel_us": {"gate_up_stage_alone": head["gu_us"], "down_stage_alone": head["down_us"]},
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "cpu_baseline": cpu,
        "extras": extras,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
