"""Host logic of the timing build's step-by-step ring report (no GPU): synthetic trace rows with
known clock rate, dependency-wait stamp and per-step stamps give back the per-step medians."""
import numpy as np

from block_scaled_mxfp4_bf16_gb300 import phase_trace


def _row(idx, start, wait, ghz):
    row = np.zeros(17, dtype=np.int64)
    row[0], row[13] = 1_000, 11_000                      # global timer at start / at C store (ns)
    row[10], row[11] = start, start + int(10_000 * ghz)  # SM clock at the same two points
    row[2] = wait                                        # SM clock when the dependency wait returned
    row[16] = idx
    return row


def test_ring_summary_medians_and_latency():
    ghz, stages, K = 2.0, 2, 1024                        # 4 steps, stages refilled from step 2 on
    plan = {"splits": 1, "stages": stages}
    r = np.zeros((4096, 64), dtype=np.int64)
    rows = []
    for idx, base in ((5, 100_000), (9, 200_000)):
        wait = base + 1_000
        rows.append(_row(idx, base, wait, ghz))
        for j in range(4):
            r[idx, j] = wait + int((300 + 200 * j) * ghz)          # stage full: 300, 500, 700, 900 ns
        for j in range(stages, 4):
            r[idx, 32 + j] = wait + int((150 + 200 * j) * ghz)     # released: 550, 750 ns
    r[7, :] = 123                                                  # a row of another call: ignored
    out = phase_trace.ring_summary(r, {1: rows}, [1], plan, K)
    assert out["step_ready"] == [300, 500, 700, 900]
    assert out["refill_released_from_step"] == 2 and out["refill_released"] == [550, 750]
    assert out["refill_latency"] == [150, 150]


def test_ring_summary_skips_stamps_older_than_the_launch():
    plan = {"splits": 2, "stages": 1}
    r = np.zeros((4096, 64), dtype=np.int64)
    row = _row(3, 50_000, 51_000, 1.0)
    r[3, 0] = 40_000                                   # left from an earlier launch on this row
    r[3, 1] = 51_400
    r[3, 33] = 51_100
    out = phase_trace.ring_summary(r, {7: [row]}, [7], plan, 1024)   # 2 steps per slice
    assert out["step_ready"] == [400]                  # step 0's stale stamp is not counted
    assert out["refill_released"] == [100] and out["refill_latency"] == [300]
