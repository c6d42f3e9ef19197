#!/usr/bin/env python3
"""Benchmark of the MXFP4 GEMM hot path on GB300.

One step = one complete mxfp4_gemm call (A quantized inside the call, MMA, split-K
reduction, bf16 epilogue) on the M=8, N=2112, K=7168 weight-streaming workload; B is
quantized and prepacked once, outside the timed region (the pages prepare B in their
harness too). Inputs are resident in HBM and rotate over enough copies that every step
streams its weights from DRAM rather than L2.

Prints ONE JSON line. `value` is microseconds per call (lower is better); TFLOPS, GB/s and
the roofline fraction ride along, with the same measurement for every workload in
`per_shape`. `--impl reference` times the CPU oracle instead (the method has no runnable
reference implementation here): `--warmup` untimed and `--steps` timed whole calls on a sample
of the output columns sized to about two minutes, time scaled to all of N.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_mxfp4_bf16_gb300 import workloads  # noqa: E402

METRIC = "µs/call and TFLOPS (2MNK/t) per shape; % of HBM or FP4 tensor roofline"
# DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) of one GEMM launch from one ncu
# capture (profiles/), valid only for the device code and the launch plan it was taken with (both
# checked at run time; reported as null otherwise).
# Per workload: (GEMM launch bytes, standalone token-block quantizer launch bytes or None, source
# hash, plan signature); from the per-configuration ncu capture in profiles/.
MEASURED_TRAFFIC = {
    "M16_N3072_K1536": (2594816, None, "1b5a93632b1fd20e",
                        "path=3,splits=3,m_tile=16,ctas=72,stages=2,issuers=2,reduction=4,recv_dedicated=1"),
    "M8_N2112_K7168": (8439808, None, "1b5a93632b1fd20e",
                       "path=3,splits=6,m_tile=16,ctas=102,stages=5,issuers=3,reduction=4,recv_dedicated=1"),
    "M32_N4096_K512": (1185536, None, "1b5a93632b1fd20e",
                       "path=3,splits=1,m_tile=16,ctas=64,stages=2,issuers=2,reduction=0,recv_dedicated=0"),
    "M64_N7168_K2048": (7940864, 270848, "8b89230104543f78",
                        "path=2,splits=1,m_tile=64,ctas=56,stages=8,issuers=3,reduction=0,recv_dedicated=0"),
    "M256_N4096_K7168": (16641024, 3679744, "8b89230104543f78",
                         "path=2,splits=2,m_tile=128,ctas=128,stages=6,issuers=2,reduction=3,recv_dedicated=0"),
    "M4_N2880_K512": (843520, None, "1b5a93632b1fd20e",
                      "path=3,splits=1,m_tile=16,ctas=23,stages=2,issuers=2,reduction=0,recv_dedicated=0"),
    "M32_N2880_K512": (872192, None, "1b5a93632b1fd20e",
                       "path=3,splits=1,m_tile=16,ctas=46,stages=2,issuers=2,reduction=0,recv_dedicated=0"),
    "M16_N2112_K7168": (8554240, None, "1b5a93632b1fd20e",
                        "path=3,splits=6,m_tile=16,ctas=102,stages=5,issuers=3,reduction=4,recv_dedicated=1"),
    "M256_N3072_K1536": (2796800, 795136, "8b89230104543f78",
                         "path=2,splits=1,m_tile=64,ctas=96,stages=6,issuers=3,reduction=0,recv_dedicated=0"),
}
NOMINAL_HBM_GBS = 8000.0             # the ~8 TB/s the method's throughput target is stated against
STEADY_STEPS = 1000                  # calls in a steady-state region
HEADLINE = "M8_N2112_K7168"
SUBMIT_COVER_CYCLES = 200_000        # ~0.1 ms of device time ahead of each timed region
FALLBACK_HBM_GBS = 6800.0
L2_BYTES_DEFAULT = 126 * 1024 * 1024


# Per plan path, the translation units of the kernels one call launches and everything they
# include: a capture stays valid while these are unchanged (the two-kernel path also launches the
# token-block quantizer of mxfp4_quant.cu).
KERNEL_SOURCES = {
    1: ("mxfp4_gemm.cu", "mma_desc.cuh", "ptx.cuh", "quant_device.cuh", "internal.h"),
    2: ("mxfp4_gemm.cu", "mxfp4_quant.cu", "mma_desc.cuh", "ptx.cuh", "quant_device.cuh", "internal.h"),
    3: ("mxfp4_gemm_resident.cu", "mma_desc.cuh", "ptx.cuh", "quant_device.cuh", "internal.h"),
}


def product_code_lines(text: str) -> list[str]:
    """The lines of a CUDA source that the product build compiles: comments, blank lines and the
    timing build's `#ifdef MXFP4_TRACE` branches (up to their `#else` or `#endif`) left out."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out, skip, depth = [], False, 0
    for ln in (ln.split("//", 1)[0].rstrip() for ln in text.splitlines()):
        d = ln.strip()
        if not skip:
            if d == "#ifdef MXFP4_TRACE":
                skip, depth = True, 0
            elif ln:
                out.append(ln)
            continue
        if d.startswith("#if"):
            depth += 1
        elif d == "#endif" and depth > 0:
            depth -= 1
        elif depth == 0 and d in ("#else", "#endif"):
            skip = False
    return out


def kernel_source_hash(path: int) -> str:
    """Hash of the device code a call on plan path `path` launches (the kernels' source files and
    the headers they include, as the product build compiles them), so that editing a comment or
    the timing build's stamps keeps the measured traffic."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[path]:
        h.update(name.encode())
        with open(os.path.join(ROOT, "block_scaled_mxfp4_bf16_gb300", "csrc", name)) as fh:
            h.update("\n".join(product_code_lines(fh.read())).encode())
    return h.hexdigest()[:16]


def plan_signature(plan: dict) -> str:
    keys = ("path", "splits", "m_tile", "ctas", "stages", "issuers", "reduction", "recv_dedicated")
    return ",".join(f"{k}={plan[k]}" for k in keys)


def measured_traffic(name: str, plan: dict):
    """(GEMM bytes, quantizer bytes or None) of one launch, or None when the kernels' source or
    the plan differ from the ones captured."""
    entry = MEASURED_TRAFFIC.get(name)
    if entry is None or entry[2] != kernel_source_hash(plan["path"]) or entry[3] != plan_signature(plan):
        return None
    return entry[0], entry[1]


def max_over_ranks(value: float) -> float:
    """Largest value over all ranks (the slowest rank's time decides the job's time)."""
    if not torch.distributed.is_initialized():
        return value
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background while the GPU is under load."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) >= 9 for i in range(4) if r[5 + i].strip() == "Active"})
        busy = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def _events():
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def bench_workload(mx, w, steps: int, warmup: int, l2_bytes: int, soak_s: float = 0.0, e2e: bool = False,
                   warm: bool = False, timings: int = 7, a_ready: bool = False):
    """Time exactly `steps` back-to-back mxfp4_gemm calls of workload w (`timings` times; the
    median counts).

    The calls are captured in CUDA graphs (programmatic-launch edges kept) and replayed, so
    the number is device time per call with host launch cost out of the way; each call uses
    its own copy of A, packed B and C, rotating over enough copies (> 3x L2) that the
    weights stream from HBM -- or, with warm=True, one copy that stays in L2. a_ready: every
    call declares MXFP4_GEMM_A_READY (true here: the copies of A are written once, before the
    timed calls), so it reads its A while the call before it still runs. Returns a dict."""
    dev = torch.device("cuda")
    a_cpu, b_cpu = workloads.make_inputs(w, seed=0)
    b = b_cpu.to(dev)
    bq, bs = mx.mxfp4_quantize(b)
    packed0 = mx.mxfp4_prepack_b(bq, bs)
    del b, bq, bs
    a0 = a_cpu.to(dev)
    per_copy = packed0.numel() + a0.numel() * 2 + w.M * w.N * 2
    copies = 1 if warm else max(2, min(512, -(-3 * l2_bytes // per_copy)))
    packs = [packed0] + [packed0.clone() for _ in range(copies - 1)]
    As = [a0] + [a0.clone() for _ in range(copies - 1)]
    Cs = [torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    plan = mx.mxfp4_gemm_plan(w.M, w.N, w.K, a_ready=a_ready)
    ws = torch.empty(max(1, mx.mxfp4_gemm_workspace_size(w.M, w.N, w.K)), dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()

    def step(i, stream):
        j = i % copies
        mx.mxfp4_gemm(As[j], packs[j], w.N, c=Cs[j], workspace=ws, stream=stream, a_ready=a_ready)

    with torch.cuda.stream(side):
        for i in range(max(warmup, copies)):
            step(i, side)
    torch.cuda.synchronize()

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(n):
                step(i, side)
        return g

    chunk = min(steps, 1024)
    g_main = capture(chunk)
    tail = steps % chunk
    g_tail = capture(tail) if tail else None
    reps = steps // chunk
    for _ in range(2):
        g_main.replay()
    torch.cuda.synchronize()
    if soak_s > 0:
        t_end = time.time() + soak_s
        while time.time() < t_end:
            g_main.replay()
            torch.cuda.synchronize()
    e0, e1 = _events()
    # The timed region -- exactly `steps` calls, a barrier and a synchronize on both sides -- is
    # measured `timings` times; the median is reported, with every timing beside it.
    elapsed = []
    for _ in range(timings):
        if torch.distributed.is_initialized():
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            # a short spin ahead of the start event keeps the stream busy while the host submits
            # the graph, so the region holds the K calls and not the host's submission latency
            torch.cuda._sleep(SUBMIT_COVER_CYCLES)
            e0.record(side)
            for _ in range(reps):
                g_main.replay()
            if g_tail is not None:
                g_tail.replay()
            e1.record(side)
        e1.synchronize()
        torch.cuda.synchronize()
        elapsed.append(e0.elapsed_time(e1))
    ms = statistics.median(elapsed)
    status = mx.mxfp4_device_status()
    res = {"us_per_call": 1000.0 * ms / steps, "elapsed_ms": ms, "copies": copies, "plan": plan,
           "kernels_per_call": 2 if plan["path"] == 2 else 1, "status": status,
           "timings_us_per_call": [round(1000.0 * t / steps, 3) for t in elapsed]}
    # the same calls launched one by one from the host (no graph, each copy's call prepared
    # once), for comparison
    n_direct = min(steps, 2000)
    dev_calls = [mx.prepare_gemm(As[j], packs[j], w.N, Cs[j], workspace=ws, stream=side, a_ready=a_ready)
                 for j in range(copies)]
    with torch.cuda.stream(side):
        e0.record(side)
        for i in range(n_direct):
            dev_calls[i % copies]()
        e1.record(side)
    e1.synchronize()
    res["direct_us_per_call"] = 1000.0 * e0.elapsed_time(e1) / n_direct
    if e2e:
        # end to end through the C-ABI host-buffer call (mxfp4_gemm_host): pinned host A ->
        # device, GEMM, C -> pinned host, all enqueued by the library. A serving loop keeps its
        # buffers, so each rotating copy's call is prepared once (mxfp4_call_create_host: checks,
        # plan and host-pointer queries outside the timed region), and each step is one run.
        # A is written by the host only (a serving loop's input), which the call is told
        # (MXFP4_CALL_A_HOST_WRITTEN): A crosses the link while the previous call still runs.
        a_host = a_cpu.pin_memory()
        c_host = torch.empty(w.M, w.N, dtype=torch.bfloat16).pin_memory()
        n_e2e = max(20, min(steps, 2000))
        host_calls = [mx.prepare_gemm_host(a_host, packs[j], w.N, c_host, As[j], Cs[j], workspace=ws, stream=side,
                                           a_host_written=True)
                      for j in range(copies)]

        def step_host(j):
            host_calls[j]()

        with torch.cuda.stream(side):
            for i in range(3):
                step_host(0)
            side.synchronize()
            e0.record(side)
            for i in range(n_e2e):
                step_host(i % copies)
            e1.record(side)
        e1.synchronize()
        res["e2e_us_per_call"] = 1000.0 * e0.elapsed_time(e1) / n_e2e
        res["h2d_bytes"] = w.M * w.K * 2
        res["d2h_bytes"] = w.M * w.N * 2
    del packs, As, Cs, ws, g_main, g_tail, dev_calls
    host_calls = None
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def bench_quantizer(mx, rows: int, K: int, steps: int, warmup: int, l2_bytes: int) -> dict:
    """The standalone quantizer on a large activation: `steps` mxfp4_quantize calls of a bf16
    [rows, K] matrix in a CUDA graph, rotating over enough copies (> 3x L2) that every call reads
    from HBM. Algorithmic bytes: the bf16 read, the e2m1 and e8m0 writes."""
    dev = torch.device("cuda")
    x0 = workloads.random_bf16(rows, K, seed=11).to(dev)
    per_copy = rows * K * 2 + rows * K // 2 + rows * K // 32
    copies = max(2, -(-3 * l2_bytes // per_copy))
    xs = [x0] + [x0.clone() for _ in range(copies - 1)]
    qs = [torch.empty(rows, K // 2, dtype=torch.uint8, device=dev) for _ in range(copies)]
    ss = [torch.empty(rows, K // 32, dtype=torch.uint8, device=dev) for _ in range(copies)]
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        for i in range(max(warmup, copies)):
            mx.mxfp4_quantize(xs[i % copies], qs[i % copies], ss[i % copies], stream=side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(steps):
            mx.mxfp4_quantize(xs[i % copies], qs[i % copies], ss[i % copies], stream=side)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = _events()
    with torch.cuda.stream(side):
        torch.cuda._sleep(SUBMIT_COVER_CYCLES)
        e0.record(side)
        g.replay()
        e1.record(side)
    e1.synchronize()
    us = 1000.0 * e0.elapsed_time(e1) / steps
    status = mx.mxfp4_device_status()
    del xs, qs, ss, g
    torch.cuda.empty_cache()
    return {"rows": rows, "K": K, "us_per_call": round(us, 3), "algorithmic_bytes": per_copy,
            "gbs": round(per_copy / (us * 1e-6) / 1e9, 1), "status": status}


def bench_two_kernel_parts(mx, w, plan: dict, steps: int, warmup: int, l2_bytes: int) -> dict:
    """The two kernels of a two-kernel plan timed apart, through the public token-block entry
    points: `steps` back-to-back mxfp4_quantize_tokens calls of A [M, K], then `steps`
    mxfp4_gemm_tokens calls on the blocks, each chain in a CUDA graph over enough rotating copies
    (> 3x L2) that every call reads from HBM. The quantizer's algorithmic bytes: A's bf16 read,
    the codes' and scales' writes."""
    dev = torch.device("cuda")
    a_cpu, b_cpu = workloads.make_inputs(w, seed=0)
    bq, bs = mx.mxfp4_quantize(b_cpu.to(dev))
    packed0 = mx.mxfp4_prepack_b(bq, bs)
    a0 = a_cpu.to(dev)
    mt, splits = plan["m_tile"], plan["splits"]
    tok_bytes = mx.mxfp4_token_blocks_size(w.M, w.K, mt)
    per_copy = packed0.numel() + a0.numel() * 2 + tok_bytes + w.M * w.N * 2
    copies = max(2, min(512, -(-3 * l2_bytes // per_copy)))
    As = [a0] + [a0.clone() for _ in range(copies - 1)]
    packs = [packed0] + [packed0.clone() for _ in range(copies - 1)]
    toks = [mx.mxfp4_quantize_tokens(As[j], mt) for j in range(copies)]
    Cs = [torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    side = torch.cuda.Stream()

    def quant(i):
        j = i % copies
        mx.mxfp4_quantize_tokens(As[j], mt, out=toks[j].data, stream=side)

    def gemm(i):
        j = i % copies
        mx.mxfp4_gemm_tokens(toks[j], packs[j], w.N, c=Cs[j], splits=splits, stream=side)

    out = {}
    for name, fn in (("token_quantizer", quant), ("gemm_tokens", gemm)):
        with torch.cuda.stream(side):
            for i in range(max(warmup, copies)):
                fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(steps):
                fn(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = _events()
        with torch.cuda.stream(side):
            torch.cuda._sleep(SUBMIT_COVER_CYCLES)
            e0.record(side)
            g.replay()
            e1.record(side)
        e1.synchronize()
        out[name] = 1000.0 * e0.elapsed_time(e1) / steps
        del g
    out["quant_algorithmic_bytes"] = w.M * w.K * 2 + w.M * w.K // 2 + w.M * ((w.K + 31) // 32)
    out["status"] = mx.mxfp4_device_status()
    del As, packs, toks, Cs
    torch.cuda.empty_cache()
    return out


def fp4_peak_tflops():
    """Dense FP4 peak: the measured bf16 burst figure times the nominal fp4 / bf16 ratio (13.5 / 2.25
    PFLOP/s), else the nominal 13.5 PFLOP/s. Returns (TFLOP/s, kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]) * 13.5 / 2.25, "measured bf16 x nominal fp4/bf16 ratio"
    except (OSError, KeyError, ValueError):
        return 13500.0, "nominal"


def cpu_oracle_step_time(w, budget_s: float = 12.0, threads: int = 0):
    """The oracle as it stands on the host cores: quantize A, dequantize, fp64 GEMM, bf16 cast.
    Bounded sample: whole calls of workload w, repeated until budget_s has passed (min 1).
    threads > 0 runs it on that many threads (then restores the default)."""
    import oracle
    if threads > 0:
        default = oracle.num_threads()
        oracle.set_num_threads(threads)
        try:
            return cpu_oracle_step_time(w, budget_s)
        finally:
            oracle.set_num_threads(default)
    a_cpu, b_cpu = workloads.make_inputs(w, seed=0)
    bq, bs = oracle.quantize(workloads.bf16_bits(b_cpu))     # B pre-quantized: not timed
    a_bits = workloads.bf16_bits(a_cpu)
    # a sample of rows keeps one step of the big workloads inside the budget
    rows = w.M if w.M * w.N * w.K <= 4e9 else max(1, int(4e9 // (w.N * w.K)))
    a_bits = np.ascontiguousarray(a_bits[:rows])
    n, t0 = 0, time.time()
    while True:
        aq, as_ = oracle.quantize(a_bits)
        c = oracle.mxfp4_gemm_ref(aq, as_, bq, bs)
        oracle.to_bf16(c)
        n += 1
        if time.time() - t0 >= budget_s:
            break
    dt = (time.time() - t0) / n
    scale = w.M / rows
    return {"us_per_call": 1e6 * dt * scale, "cores": oracle.num_threads(),
            "sample": f"{n} oracle call(s) on {rows} of {w.M} rows of {w.name}, time scaled by {scale:g}"}


def reference_arm(w, steps: int, warmup: int, budget_s: float = 120.0) -> dict:
    """--impl reference: the oracle as it stands on the host cores, `warmup` untimed steps then
    `steps` timed ones. A step is the whole call (quantize A, dequantize, fp64 GEMM, bf16 cast) on
    the first `cols` weight rows, i.e. output columns; its cost grows in proportion to them, so
    the time is scaled by N / cols. cols is all of N unless that would take the run past budget_s
    (sized from an untimed probe on a few columns)."""
    import oracle
    a_cpu, b_cpu = workloads.make_inputs(w, seed=0)
    bq, bs = oracle.quantize(workloads.bf16_bits(b_cpu))     # B pre-quantized: not timed
    a_bits = workloads.bf16_bits(a_cpu)

    def call(cols):
        aq, as_ = oracle.quantize(a_bits)
        oracle.to_bf16(oracle.mxfp4_gemm_ref(aq, as_, bq[:cols], bs[:cols]))

    probe = min(w.N, 128)
    t0 = time.perf_counter()
    call(probe)
    per_col = (time.perf_counter() - t0) / probe
    cols = max(1, min(w.N, int(budget_s / (max(1, steps + warmup) * per_col))))
    for _ in range(warmup):
        call(cols)
    t0 = time.perf_counter()
    for _ in range(steps):
        call(cols)
    dt = (time.perf_counter() - t0) / max(1, steps)
    return {"us_per_call": 1e6 * dt * w.N / cols, "cores": oracle.num_threads(),
            "sample": f"{steps} timed steps after {warmup} untimed, each the whole call on {cols} of {w.N} "
                      f"output columns of {w.name}, time scaled by {w.N / cols:g}"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-shapes", action="store_true", help="skip the per-shape sweep")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = workloads.by_name(args.workload)

    if args.impl == "reference":
        if rank != 0:
            return
        r = reference_arm(w, args.steps, args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": r["us_per_call"], "unit": "us/call",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": r["us_per_call"] / 1000.0, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K},
                "cpu_baseline": {"value": r["us_per_call"], "unit": "us/call", "cores": r["cores"],
                                 "kind": "oracle", "sample": r["sample"]},
                "e2e": {"value": r["us_per_call"], "unit": "us/call", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    import block_scaled_mxfp4_bf16_gb300 as mx
    mx.load_library()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size or L2_BYTES_DEFAULT
    peak, peak_kind = measured_peaks()

    sampler = ClockSampler(local)
    sampler.start()
    main_res = bench_workload(mx, w, args.steps, args.warmup, l2, soak_s=1.0, e2e=True)
    clocks = sampler.stop()

    # whole-job figure: every rank runs its own copy of the workload (independent problems, no
    # collective on the data path); the job's time is the slowest rank's
    t_us = 1000.0 * max_over_ranks(main_res["elapsed_ms"]) / (args.steps * world)

    per_shape = {}
    if not args.no_shapes:
        fp4_peak, _ = fp4_peak_tflops()
        for ws_ in workloads.WORKLOADS + workloads.EXTRA_WORKLOADS:
            # the same --steps region as the headline (so the two agree for the same workload; a
            # short region carries the first call, which no earlier call overlaps), a long
            # region for the steady state, and a long region with one copy resident in L2
            r = bench_workload(mx, ws_, args.steps, args.warmup, l2)
            rs = bench_workload(mx, ws_, STEADY_STEPS, args.warmup, l2)
            rw = bench_workload(mx, ws_, STEADY_STEPS, args.warmup, l2, warm=True)
            # the steady state again with A declared ready before each call (MXFP4_GEMM_A_READY:
            # the A load and quantization overlap the call before); not the headline, whose
            # calls stand for a chain in which each A may come from the work just before
            ra = bench_workload(mx, ws_, STEADY_STEPS, args.warmup, l2, a_ready=True)
            gbs = ws_.algorithmic_bytes / (r["us_per_call"] * 1e-6) / 1e9
            gbs_s = ws_.algorithmic_bytes / (rs["us_per_call"] * 1e-6) / 1e9
            tf = ws_.flops / (r["us_per_call"] * 1e-6) / 1e12
            tf_warm = ws_.flops / (rw["us_per_call"] * 1e-6) / 1e12
            traffic = measured_traffic(ws_.name, r["plan"])
            per_shape[ws_.name] = {"us_per_call": round(r["us_per_call"], 3),
                                   "steady_us_per_call": round(rs["us_per_call"], 3),
                                   "steady_hbm_frac": round(gbs_s / peak, 4),
                                   "direct_us_per_call": round(rs["direct_us_per_call"], 3),
                                   "tflops": round(tf, 2),
                                   "algorithmic_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4),
                                   "hbm_frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                                   "fp4_frac": round(tf / fp4_peak, 4),
                                   "warm_l2_us_per_call": round(rw["us_per_call"], 3),
                                   "a_ready_steady_us_per_call": round(ra["us_per_call"], 3),
                                   "a_ready_plan": {k: ra["plan"][k] for k in ("path", "splits", "ctas", "a_early")},
                                   "warm_l2_fp4_frac": round(tf_warm / fp4_peak, 4),
                                   "gemm_dram_bytes": traffic[0] if traffic else None,
                                   "quantizer_dram_bytes": traffic[1] if traffic else None,
                                   "path": r["plan"]["path"], "splits": r["plan"]["splits"],
                                   "ctas": r["plan"]["ctas"],
                                   "status": max(r["status"], rs["status"], rw["status"], ra["status"])}
            if r["plan"]["path"] == 2:
                # the two kernels of the call apart (each chain alone, back to back)
                parts = bench_two_kernel_parts(mx, ws_, r["plan"], STEADY_STEPS, args.warmup, l2)
                q_gbs = parts["quant_algorithmic_bytes"] / (parts["token_quantizer"] * 1e-6) / 1e9
                per_shape[ws_.name].update({
                    "token_quantizer_us_per_call": round(parts["token_quantizer"], 3),
                    "token_quantizer_algorithmic_gbs": round(q_gbs, 1),
                    "token_quantizer_hbm_frac": round(q_gbs / peak, 4),
                    "gemm_tokens_us_per_call": round(parts["gemm_tokens"], 3),
                    "gemm_tokens_fp4_frac": round(ws_.flops / (parts["gemm_tokens"] * 1e-6) / 1e12 / fp4_peak, 4)})
                per_shape[ws_.name]["status"] = max(per_shape[ws_.name]["status"], parts["status"])

    quantizer = None
    if not args.no_shapes:
        quantizer = bench_quantizer(mx, 4096, 7168, 50, args.warmup, l2)
        quantizer["hbm_frac"] = round(quantizer["gbs"] / peak, 4)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu:
        c = cpu_oracle_step_time(w)
        c1 = cpu_oracle_step_time(w, budget_s=6.0, threads=1)
        cpu = {"value": c["us_per_call"], "unit": "us/call", "cores": c["cores"], "kind": "oracle",
               "sample": c["sample"],
               "single_core": {"value": c1["us_per_call"], "unit": "us/call", "cores": c1["cores"],
                               "sample": c1["sample"]}}
    gbs = w.algorithmic_bytes / (main_res["us_per_call"] * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(t_us, 4), "unit": "us/call", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_us / 1000.0, 7), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1xe2m1->f32->bf16", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                   "l2": f"inputs rotate over {main_res['copies']} copies (> 3x L2) so weights stream from HBM",
                   "path": main_res["plan"]["path"], "splits": main_res["plan"]["splits"],
                   "ctas": main_res["plan"]["ctas"]},
        "tflops": round(w.flops / (t_us * 1e-6) / 1e12, 3),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4),
                     "traffic": (measured_traffic(w.name, main_res["plan"]) or (None,))[0],
                     "peak_kind": peak_kind, "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                     "algorithmic_bytes_per_launch": w.algorithmic_bytes},
        "e2e": {"value": round(main_res["e2e_us_per_call"], 3), "unit": "us/call",
                "h2d_bytes_per_step": main_res["h2d_bytes"], "d2h_bytes_per_step": main_res["d2h_bytes"]},
        "gpu_launches": args.steps * main_res["kernels_per_call"],
        "timing": f"CUDA-graph replay of back-to-back calls, the {args.steps}-call region timed "
                  f"{len(main_res['timings_us_per_call'])} times, median reported; direct host launches: "
                  f"{main_res['direct_us_per_call']:.3f} us/call",
        "timings_us_per_call": main_res["timings_us_per_call"],
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_shape": per_shape,
        "quantizer": quantizer,
        "device_status": main_res["status"],
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
