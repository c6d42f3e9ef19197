"""GPU quantizer parity: e2m1 bytes and e8m0 scales from mxfp4_quantize (CUDA, through the C
ABI) must equal the CPU oracle's bit for bit."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads
from mxfp4_testlib import assert_bytes_equal, expected_token_blocks, quantize_both, to_np_u8

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


@pytest.mark.parametrize("rows,K", [(1, 8), (3, 40), (5, 72), (64, 200), (129, 7176), (4096, 7176)])
def test_quantize_k_tail_bit_exact(rows, K):
    # K % 32 != 0: the last block is cut by K and its missing elements count as zeros; the row
    # padding past K holds huge values, which would change the last block's scale if read
    import block_scaled_mxfp4_bf16_gb300 as mx
    x = workloads.random_bf16(rows, K, seed=rows + 3 * K, scale=2.0)
    store = torch.full((rows, K + 40), 1.0e30, dtype=torch.bfloat16)
    store[:, :K] = x
    q, s = mx.mxfp4_quantize(store.cuda()[:, :K])
    rq, rs = oracle.quantize(workloads.bf16_bits(x))
    torch.cuda.synchronize()
    nblk = (K + 31) // 32
    assert tuple(q.shape) == (rows, nblk * 16) and tuple(s.shape) == (rows, nblk)
    assert_bytes_equal(to_np_u8(q), rq, f"e2m1 {rows}x{K}")
    assert_bytes_equal(to_np_u8(s), rs, f"scales {rows}x{K}")


def test_quantize_tail_rows_hand_worked():
    # the hand-derived rows of tests/golden/tail_blocks.json, on the GPU
    import block_scaled_mxfp4_bf16_gb300 as mx
    from test_oracle_pins import _load_tail_rows, tail_row_input
    for row in _load_tail_rows():
        x = torch.from_numpy(tail_row_input(row).view(np.int16)).view(torch.bfloat16)
        q, s = mx.mxfp4_quantize(x.cuda())
        torch.cuda.synchronize()
        assert [int(v) for v in to_np_u8(s)[0]] == row["scale_bytes"], row["name"]
        assert bytes(to_np_u8(q)[0]).hex() == row["packed_hex"], row["name"]


def test_quantize_rejects_bad_arguments():
    import block_scaled_mxfp4_bf16_gb300 as mx
    L = mx.load_library()
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(4, 32, dtype=torch.uint8, device="cuda")
    s = torch.empty(4, 2, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert L.mxfp4_quantize(x.data_ptr(), 4, 44, 64, q.data_ptr(), s.data_ptr(), st) == 2    # K % 8
    assert L.mxfp4_quantize(x.data_ptr(), 4, 64, 60, q.data_ptr(), s.data_ptr(), st) == 2    # ld < K
    assert L.mxfp4_quantize(x.data_ptr() + 2, 4, 64, 64, q.data_ptr(), s.data_ptr(), st) == 3  # misaligned
    assert L.mxfp4_quantize(None, 4, 64, 64, q.data_ptr(), s.data_ptr(), st) == 1
    assert L.mxfp4_quantize(x.data_ptr(), 0, 64, 64, q.data_ptr(), s.data_ptr(), st) == 0    # empty no-op


@pytest.mark.parametrize("M,K,m_tile", [(40, 768, 0), (300, 512, 0), (33, 320, 0), (100, 1024, 64), (200, 7168, 0),
                                         (40, 776, 0), (33, 344, 0), (7, 8, 0), (200, 7176, 0)])
def test_two_kernel_token_blocks_bit_exact(M, K, m_tile):
    # the standalone quantizer's output in the GEMM's token-block layout, read back from the
    # workspace, byte for byte against the oracle's quantization of A (the (200, K) cases have
    # enough blocks for the one-lane-per-block kernel, the others use four lanes per block; the
    # K % 32 != 0 cases cut the last block, and A's row padding holds huge values that would
    # change that block's scale if anything past K were read)
    import block_scaled_mxfp4_bf16_gb300 as mx
    N = 256
    a = workloads.random_bf16(M, K, seed=M * 7 + K)
    a_store = torch.full((M, K + 24), 1.0e30, dtype=torch.bfloat16)
    a_store[:, :K] = a
    plan = mx.mxfp4_gemm_plan(M, N, K, 2, 1, m_tile)
    assert plan["path"] == 2
    need = mx.mxfp4_gemm_workspace_size(M, N, K, 2, 1, m_tile)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=5).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    mx.mxfp4_gemm(a_store.cuda()[:, :K], packed, N, workspace=ws, path=2, splits=1, m_tile=m_tile)
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    rq, rs = oracle.quantize(workloads.bf16_bits(a))
    want, defined = expected_token_blocks(rq, rs, M, K, plan["m_tile"])
    got = to_np_u8(ws)
    assert got.size == want.size, (got.size, want.size)
    bad = np.flatnonzero((got != want) & defined)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[0]}: got {got[bad[0]]:#04x} want {want[bad[0]]:#04x}"
