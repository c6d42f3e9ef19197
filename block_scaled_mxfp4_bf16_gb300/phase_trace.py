"""Phase timeline of the GEMM kernels in steady state, from the library's timing build.

    python -m block_scaled_mxfp4_bf16_gb300.phase_trace --workload M8_N2112_K7168 [--path 3]

Builds the library with -DMXFP4_TRACE into its own file (the product library is left alone),
replays a CUDA graph of back-to-back calls of the workload (inputs rotating over more than 3x
L2, as the benchmark does), and reads the trace rows back: every CTA records its grid id, block
index and SM, the global timer and the SM clock when it starts and when it stores C, and the SM
clock at each phase. Phases are reported per call as the median over the call's CTAs of the time
since that CTA's dependency wait returned (SM clock deltas, converted with each call's measured
clock rate), plus the gap from the previous call's last C store to this call's median wait.
Prints one JSON line per workload.

With --steps (streaming-kernel plans), also the weight and token ring step by step: when each
256-K step's stage was seen full by its MMA thread, when the copy thread saw the stage it
refills for a step released (the MMAs of the step `stages` earlier complete), and the refill's
latency from that release to the step's stage being full again.
"""
from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np
import torch

from . import build as _build
from . import workloads

# trace slots of the weight-resident kernel and of the two-kernel / fused kernel
PHASES = {
    3: {2: "wait", 3: "first_block_quantized", 4: "quantized", 5: "mma_go", 6: "mma_issued", 7: "acc_ready",
        1: "tmem_loaded", 8: "posted", 9: "received"},
    2: {1: "weights_requested", 2: "wait", 3: "mma_start", 4: "first_step", 5: "last_step", 6: "acc_ready",
        7: "reduction_start", 8: "posted", 9: "received"},
}
PHASES[1] = PHASES[2]


def _library():
    path = _build.build_variant("trace", ["-DMXFP4_TRACE"])
    L = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    for name in ("mxfp4_trace_read", "mxfp4_trace_read_resident", "mxfp4_ring_read"):
        getattr(L, name).argtypes = [vp, ctypes.c_size_t]
        getattr(L, name).restype = ctypes.c_int
    L.mxfp4_quantize.argtypes = [vp, i64, i64, i64, vp, vp, vp]
    L.mxfp4_prepack_b.argtypes = [vp, vp, i64, i64, vp, vp]
    L.mxfp4_prepack_b_size.argtypes = [i64, i64]
    L.mxfp4_prepack_b_size.restype = ctypes.c_size_t
    return L


class _Opts(ctypes.Structure):   # mxfp4_gemm_options (flags 0: the flagless plans)
    _fields_ = [("path", ctypes.c_int), ("splits", ctypes.c_int), ("m_tile", ctypes.c_int),
                ("flags", ctypes.c_int), ("reserved", ctypes.c_int * 4)]


def trace(w: workloads.Workload, path: int = 0, splits: int = 0, m_tile: int = 0, calls: int = 60,
          steps: bool = False) -> dict:
    import block_scaled_mxfp4_bf16_gb300 as mx
    L = _library()
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    L.mxfp4_gemm_ex.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, ctypes.c_size_t, ctypes.POINTER(_Opts), vp]
    plan = mx.mxfp4_gemm_plan(w.M, w.N, w.K, path, splits, m_tile)
    dev = torch.device("cuda")
    a_cpu, b_cpu = workloads.make_inputs(w, seed=0)
    bq, bs = mx.mxfp4_quantize(b_cpu.to(dev))
    packed0 = mx.mxfp4_prepack_b(bq, bs)
    a0 = a_cpu.to(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(2, min(512, -(-3 * l2 // (packed0.numel() + a0.numel() * 2 + w.M * w.N * 2))))
    packs = [packed0] + [packed0.clone() for _ in range(copies - 1)]
    As = [a0] + [a0.clone() for _ in range(copies - 1)]
    Cs = [torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    ws = torch.zeros(max(1, mx.mxfp4_gemm_workspace_size(w.M, w.N, w.K, path, splits, m_tile)), dtype=torch.uint8,
                     device=dev)
    opts = _Opts(path, splits, m_tile)
    side = torch.cuda.Stream()

    def step(i):
        j = i % copies
        st = L.mxfp4_gemm_ex(As[j].data_ptr(), w.M, w.K, w.K, packs[j].data_ptr(), w.N, Cs[j].data_ptr(), w.N,
                             ws.data_ptr(), ws.numel(), ctypes.byref(opts), side.cuda_stream)
        assert st == 0, st

    with torch.cuda.stream(side):
        for i in range(copies):
            step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(calls):
            step(i)
    g.replay()
    torch.cuda.synchronize()
    buf = np.zeros((4096, 16), dtype=np.uint64)
    read = L.mxfp4_trace_read_resident if plan["path"] == 3 else L.mxfp4_trace_read
    assert read(buf.ctypes.data, buf.nbytes) == 0
    t = np.concatenate([buf.astype(np.int64), np.arange(4096, dtype=np.int64)[:, None]], axis=1)   # [16]: row
    t = t[(t[:, 0] > 0) & (t[:, 13] > 0)]
    grids: dict = {}
    for row in t:
        grids.setdefault(int(row[14]), []).append(row)
    order = sorted(grids, key=lambda gid: min(r[0] for r in grids[gid]))
    steady = [gid for gid in order if len(grids[gid]) == plan["ctas"]][-12:-2]
    names = PHASES[plan["path"]]
    agg: dict = {name: [] for name in names.values()}
    agg.update(cta_start=[], cta_end=[], gap_from_previous_call=[], sm_ghz=[])
    prev_end = None
    for gid in steady:
        rows = np.array(grids[gid])
        ghz = float(np.median((rows[:, 11] - rows[:, 10]) / np.maximum(1, rows[:, 13] - rows[:, 0])))
        for slot, name in names.items():
            ok = rows[:, slot] >= rows[:, 10]        # stamped by this launch (not left from another)
            if ok.any():
                agg[name].append(float(np.median((rows[ok, slot] - rows[ok, 2]) / ghz)))
        agg["cta_start"].append(float(np.median((rows[:, 10] - rows[:, 2]) / ghz)))
        agg["cta_end"].append(float(np.median((rows[:, 11] - rows[:, 2]) / ghz)))
        agg["sm_ghz"].append(ghz)
        wait_ns = rows[:, 0] + (rows[:, 2] - rows[:, 10]) / ghz
        if prev_end is not None:
            agg["gap_from_previous_call"].append(float(np.median(wait_ns)) - prev_end)
        prev_end = float(np.max(rows[:, 13]))
    out = {"workload": w.name, "plan": plan, "calls": len(steady),
           "ns_after_dependency_wait": {k: round(float(np.median(v)), 0 if k != "sm_ghz" else 3)
                                        for k, v in agg.items() if v}}
    if steps and plan["path"] != 3:
        out["ring"] = _ring(L, grids, steady, plan, w)
    return out


def _ring(L, grids: dict, steady: list, plan: dict, w: workloads.Workload) -> dict:
    ring = np.zeros((4096, 64), dtype=np.uint64)
    assert L.mxfp4_ring_read(ring.ctypes.data, ring.nbytes) == 0
    return ring_summary(ring.astype(np.int64), grids, steady, plan, w.K)


def ring_summary(r: np.ndarray, grids: dict, steady: list, plan: dict, K: int) -> dict:
    """Per-step medians (ns after each CTA's dependency wait) of the ring stamps `r` [row][64] of
    the steady calls' CTAs, whose trace rows (`grids[gid]`, 17 columns: the 16 trace slots and
    the row index) give the clock base and rate."""
    na = min(32, -(-(-(-K // 256)) // plan["splits"]))   # steps of the longest slice (stamped up to 32)
    stages = plan["stages"]
    ready: dict = {j: [] for j in range(na)}
    released: dict = {j: [] for j in range(stages, na)}
    latency: dict = {j: [] for j in range(stages, na)}
    for gid in steady:
        rows = np.array(grids[gid])
        ghz = float(np.median((rows[:, 11] - rows[:, 10]) / np.maximum(1, rows[:, 13] - rows[:, 0])))
        for row in rows:
            tr = r[int(row[16])]
            for j in range(na):
                if tr[j] >= row[10]:   # stamped by this launch
                    ready[j].append((tr[j] - row[2]) / ghz)
            for j in range(stages, na):
                if tr[32 + j] >= row[10] and tr[j] >= row[10]:
                    released[j].append((tr[32 + j] - row[2]) / ghz)
                    latency[j].append((tr[j] - tr[32 + j]) / ghz)

    def med(d):
        return [round(float(np.median(v))) for _, v in sorted(d.items()) if v]
    return {"step_ready": med(ready), "refill_released_from_step": stages, "refill_released": med(released),
            "refill_latency": med(latency)}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", action="append", required=True)
    ap.add_argument("--path", type=int, default=0)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--m-tile", type=int, default=0)
    ap.add_argument("--steps", action="store_true", help="also the ring, step by step (streaming plans)")
    ap.add_argument("--calls", type=int, default=60)
    args = ap.parse_args()
    torch.cuda.set_device(0)
    for name in args.workload:
        print(json.dumps(trace(workloads.by_name(name), args.path, args.splits, args.m_tile, args.calls,
                               args.steps)), flush=True)


if __name__ == "__main__":
    main()
