"""Host logic of the multi-process benchmark path, on CPU with gloo and two ranks: the job time
is the slowest rank's, and each rank's workload is independent (no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(float(10 + 5 * rank))
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_two_ranks_gloo():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5


def test_traffic_is_dropped_when_kernel_sources_or_plan_change(monkeypatch):
    import bench
    name = next(iter(bench.MEASURED_TRAFFIC))
    plan = {"path": 1, "splits": 6, "m_tile": 16, "ctas": 102, "stages": 5, "issuers": 2, "reduction": 2,
            "recv_dedicated": 1}
    sig = bench.plan_signature(plan)
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, name, (123, 45, bench.kernel_source_hash(1), sig))
    assert bench.measured_traffic(name, plan) == (123, 45)
    assert bench.measured_traffic(name, dict(plan, splits=5)) is None          # another launch plan
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, name, (123, 45, "0000000000000000", sig))
    assert bench.measured_traffic(name, plan) is None                          # other device code


def test_source_hash_sees_only_the_product_build():
    # comments, blank lines and the timing build's stamps leave the hash alone; code in the
    # product build (including an #else branch of the timing guard) changes it
    import bench
    base = "int a;\n#ifdef MXFP4_TRACE\nstamp();\n#if 1\nmore();\n#endif\n#else\nnop();\n#endif\nint b;\n"
    same = base.replace("stamp();", "stamp(); other_stamp();  // note") + "\n/* c */\n"
    assert bench.product_code_lines(base) == bench.product_code_lines(same) == ["int a;", "nop();", "#endif", "int b;"]
    assert bench.product_code_lines(base.replace("nop();", "op();")) != bench.product_code_lines(base)
    assert bench.product_code_lines(base.replace("int b;", "int c;")) != bench.product_code_lines(base)


def test_recorded_traffic_matches_the_current_sources_and_plans():
    # every recorded capture belongs to the device code in the tree and to the plan the planner
    # makes for that workload on a GB300 (152 SMs; the cluster limits of the planner tests)
    import bench
    import block_scaled_mxfp4_bf16_gb300 as mx
    from block_scaled_mxfp4_bf16_gb300 import workloads
    from test_planner import CLUSTER_CAPS, SM_COUNT
    for name, (gemm, quant, h, sig) in bench.MEASURED_TRAFFIC.items():
        w = workloads.by_name(name)
        plan = mx.mxfp4_gemm_plan_model(w.M, w.N, w.K, SM_COUNT, CLUSTER_CAPS)
        assert h == bench.kernel_source_hash(plan["path"]), name
        assert bench.plan_signature(plan) == sig, name
        assert 0.95 * w.algorithmic_bytes - 2 * w.M * w.N <= gemm + (quant or 0) <= 1.3 * w.algorithmic_bytes, name


def test_reference_arm_counts_steps_and_bounds_its_sample(monkeypatch):
    # the reference arm runs `warmup` untimed and `steps` timed oracle calls on a column sample
    # sized to its time budget, and scales the time by N / columns
    import bench
    import oracle
    from block_scaled_mxfp4_bf16_gb300 import workloads
    w = workloads.Workload("tiny", 4, 256, 128)
    calls = []
    real = oracle.mxfp4_gemm_ref
    monkeypatch.setattr(oracle, "mxfp4_gemm_ref", lambda aq, as_, bq, bs: calls.append(bq.shape[0]) or
                        real(aq, as_, bq, bs))
    r = bench.reference_arm(w, steps=4, warmup=2)
    assert calls == [128] + [256] * 6            # probe, then whole-N steps within the budget
    assert r["us_per_call"] > 0 and "4 timed steps after 2 untimed" in r["sample"]
    calls.clear()
    r = bench.reference_arm(w, steps=4, warmup=2, budget_s=1e-9)
    assert calls == [128] + [1] * 6              # a budget too small for anything: one column
    assert "on 1 of 256 output columns" in r["sample"] and "scaled by 256" in r["sample"]


def _run_bench(args, env_extra):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **env_extra)
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], env=env, cwd=root,
                         capture_output=True, text=True, timeout=600, check=True).stdout
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def test_reference_arm_json_line():
    lines = _run_bench(["--impl", "reference", "--workload", "M4_N2880_K512", "--steps", "2", "--warmup", "3"],
                       {"RANK": "0", "WORLD_SIZE": "1"})
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["unit"] == "us/call" and line["higher_is_better"] is False and line["value"] > 0
    assert line["config"]["workload"] == "M4_N2880_K512"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1 and "2 timed steps after 3 untimed" in line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "us/call", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    assert _run_bench(["--impl", "reference", "--workload", "M4_N2880_K512", "--steps", "2"],
                      {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
