"""GPU quantizer parity: e2m1 bytes and e8m0 scales from mxfp4_quantize (CUDA, through the C
ABI) must equal the CPU oracle's bit for bit."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads
from mxfp4_testlib import assert_bytes_equal, quantize_both, to_np_u8

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.json")


@pytest.mark.parametrize("w", workloads.WORKLOADS, ids=lambda w: w.name)
def test_quantize_workload_a_and_b_bit_exact(w):
    a, b = workloads.make_inputs(w, seed=0)
    for name, x in (("A", a), ("B", b)):
        q, s, rq, rs = quantize_both(x)
        assert_bytes_equal(s, rs, f"{w.name} {name} scales")
        assert_bytes_equal(q, rq, f"{w.name} {name} e2m1")


def test_quantize_hand_blocks():
    with open(GOLD) as f:
        blocks = json.load(f)["blocks"]
    rows = []
    for blk in blocks:
        fill = int(blk.get("fill", "0000"), 16)
        rows.append([int(h, 16) for h in blk["x"]] + [fill] * (32 - len(blk["x"])))
    x = torch.from_numpy(np.array(rows, np.uint16).view(np.int16)).view(torch.bfloat16)
    q, s, _, _ = quantize_both(x)
    for i, blk in enumerate(blocks):
        assert int(s[i, 0]) == blk["scale_byte"], blk["name"]
        assert bytes(q[i]).hex() == blk["packed_hex"], blk["name"]


def test_quantize_every_bf16_value_under_many_scales():
    # every finite bf16 pattern appears as an element of a block whose amax fixes the scale:
    # 32640 magnitudes x 2 signs, placed after a block-max element that sweeps the range
    pats = np.arange(0, 0x7F80, dtype=np.uint16)
    vals = np.concatenate([pats, pats | 0x8000])
    rng = np.random.default_rng(5)
    vals = vals[rng.permutation(vals.size)]
    nblk = (vals.size + 30) // 31
    nblk += nblk & 1
    x = np.zeros((nblk, 32), np.uint16)
    flat = np.zeros(nblk * 31, np.uint16)
    flat[:vals.size] = vals
    x[:, 1:] = flat.reshape(nblk, 31)
    # block max element: random exponents over the whole range (some blocks get their amax
    # from the swept values instead)
    x[:, 0] = rng.integers(0, 0x7F80, nblk).astype(np.uint16)
    t = torch.from_numpy(x.reshape(-1, 64).view(np.int16)).view(torch.bfloat16)
    q, s, rq, rs = quantize_both(t)
    assert_bytes_equal(s, rs, "scales")
    assert_bytes_equal(q, rq, "e2m1")


def test_quantize_strided_rows_and_small_shapes():
    x = workloads.random_bf16(7, 96 + 40, seed=3, scale=5.0)
    xs = x[:, :96]                              # row stride 136 elements
    import block_scaled_mxfp4_bf16_gb300 as mx
    q, s = mx.mxfp4_quantize(x.cuda()[:, :96])
    rq, rs = oracle.quantize(workloads.bf16_bits(xs.contiguous()))
    torch.cuda.synchronize()
    assert_bytes_equal(to_np_u8(q), rq, "e2m1")
    assert_bytes_equal(to_np_u8(s), rs, "scales")
    for rows, K in [(1, 32), (1, 64), (3, 160), (129, 32)]:
        xx = workloads.random_bf16(rows, K, seed=rows * K)
        q, s, rq, rs = quantize_both(xx)
        assert_bytes_equal(q, rq, f"e2m1 {rows}x{K}")
        assert_bytes_equal(s, rs, f"scales {rows}x{K}")


def test_quantize_rejects_bad_arguments():
    import block_scaled_mxfp4_bf16_gb300 as mx
    L = mx.load_library()
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(4, 32, dtype=torch.uint8, device="cuda")
    s = torch.empty(4, 2, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert L.mxfp4_quantize(x.data_ptr(), 4, 48, 64, q.data_ptr(), s.data_ptr(), st) == 2    # K % 32
    assert L.mxfp4_quantize(x.data_ptr(), 4, 64, 60, q.data_ptr(), s.data_ptr(), st) == 2    # ld < K
    assert L.mxfp4_quantize(x.data_ptr() + 2, 4, 64, 64, q.data_ptr(), s.data_ptr(), st) == 3  # misaligned
    assert L.mxfp4_quantize(None, 4, 64, 64, q.data_ptr(), s.data_ptr(), st) == 1
    assert L.mxfp4_quantize(x.data_ptr(), 0, 64, 64, q.data_ptr(), s.data_ptr(), st) == 0    # empty no-op
