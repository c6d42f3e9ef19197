"""The token-block entry points: mxfp4_quantize_tokens writes the oracle's codes and scales in the
layout the GEMM reads (byte for byte, every m_tile, K tails, padded rows), and mxfp4_gemm_tokens
on those blocks gives the two-kernel GEMM's bits and the oracle's product within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads
from mxfp4_testlib import check_tolerance, expected_token_blocks, bf16_to_f64, to_np_u8

pytestmark = pytest.mark.gpu


def _mx():
    import block_scaled_mxfp4_bf16_gb300 as mx
    return mx


@pytest.mark.parametrize("M,K,m_tile", [(64, 2048, 0), (256, 7168, 0), (300, 520, 0), (40, 776, 32), (7, 8, 0),
                                         (100, 1024, 64), (200, 512, 256), (33, 344, 16), (129, 264, 128)])
def test_quantize_tokens_bytes_match_oracle(M, K, m_tile):
    # A's row padding holds 1e30 (reading past K would change a scale); the buffer starts as
    # 0xA5 and has a guard band after the layout that must stay untouched
    mx = _mx()
    a = workloads.random_bf16(M, K, seed=M * 5 + K)
    a_store = torch.full((M, K + 40), 1.0e30, dtype=torch.bfloat16, device="cuda")
    a_store[:, :K] = a.cuda()
    mt = mx.mxfp4_token_tile(M, K, m_tile)
    size = mx.mxfp4_token_blocks_size(M, K, m_tile)
    buf = torch.full((size + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    tokens = mx.mxfp4_quantize_tokens(a_store[:, :K], m_tile, out=buf[:size])
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    assert tokens.m_tile == mt and (tokens.M, tokens.K) == (M, K)
    rq, rs = oracle.quantize(workloads.bf16_bits(a))
    want, defined = expected_token_blocks(rq, rs, M, K, mt)
    got = to_np_u8(buf)
    assert want.size == size
    bad = np.flatnonzero((got[:size] != want) & defined)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[0]}: got {got[bad[0]]:#04x} want {want[bad[0]]:#04x}"
    assert np.all(got[size:] == 0xA5), "wrote past the token blocks"


@pytest.mark.parametrize("w", [workloads.by_name("M64_N7168_K2048"), workloads.by_name("M256_N4096_K7168")],
                         ids=lambda w: w.name)
def test_gemm_tokens_equals_two_kernel_gemm_on_workloads(w):
    # the public two-step form on the benchmark's two-kernel workloads: the GEMM's own bits, and
    # a sample of outputs against the oracle
    mx = _mx()
    a, b = workloads.make_inputs(w, seed=0)
    bq, bs = mx.mxfp4_quantize(b.cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    plan = mx.mxfp4_gemm_plan(w.M, w.N, w.K)
    assert plan["path"] == 2
    a_dev = a.cuda()
    want = mx.mxfp4_gemm(a_dev, packed, w.N)
    tokens = mx.mxfp4_quantize_tokens(a_dev, plan["m_tile"])
    c = mx.mxfp4_gemm_tokens(tokens, packed, w.N, splits=plan["splits"])
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    assert torch.equal(c.view(torch.int16), want.view(torch.int16))
    aq, as_ = oracle.quantize(workloads.bf16_bits(a))
    rq, rs = oracle.quantize(workloads.bf16_bits(b))
    rng = np.random.default_rng(3)
    rows = rng.choice(w.M, min(w.M, 24), replace=False)
    cols = np.concatenate([rng.choice(w.N, 60, replace=False), [0, w.N - 1]])
    im, inn = np.repeat(rows, cols.size), np.tile(cols, rows.size)
    ref = oracle.gemm_entries(aq, as_, rq, rs, im, inn)
    check_tolerance(bf16_to_f64(c.cpu())[im, inn], ref, w.name)


@pytest.mark.parametrize("M,N,K,m_tile,splits", [(40, 200, 776, 32, 1), (300, 384, 1024, 128, 2), (5, 130, 72, 16, 1),
                                                  (129, 256, 2048, 0, 0), (600, 200, 512, 256, 1)])
def test_gemm_tokens_vs_oracle_and_reuse(M, N, K, m_tile, splits):
    # one quantization of A feeds two GEMMs with different weights; both match the oracle over
    # every output and the path-2 call of mxfp4_gemm bit for bit
    mx = _mx()
    a = workloads.random_bf16(M, K, seed=M + K)
    a_dev = a.cuda()
    tokens = mx.mxfp4_quantize_tokens(a_dev, m_tile)
    aq, as_ = oracle.quantize(workloads.bf16_bits(a))
    for seed in (1, 2):
        b = workloads.random_bf16(N, K, seed=seed * 100 + N)
        bq, bs = mx.mxfp4_quantize(b.cuda())
        packed = mx.mxfp4_prepack_b(bq, bs)
        c_store = torch.full((M + 1, N + 5), 777.0, dtype=torch.bfloat16, device="cuda")
        c = mx.mxfp4_gemm_tokens(tokens, packed, N, c=c_store[:M, :N], splits=splits)
        want = mx.mxfp4_gemm(a_dev, packed, N, path=2, splits=splits, m_tile=tokens.m_tile)
        torch.cuda.synchronize()
        assert mx.mxfp4_device_status() == 0
        assert torch.equal(c.view(torch.int16), want.view(torch.int16)), seed
        outside = torch.ones_like(c_store, dtype=torch.bool)
        outside[:M, :N] = False
        assert bool((c_store[outside] == 777.0).all()), "GEMM wrote outside C"
        rq, rs = oracle.quantize(workloads.bf16_bits(b))
        check_tolerance(bf16_to_f64(c.cpu()), oracle.mxfp4_gemm_ref(aq, as_, rq, rs), f"{M}x{N}x{K} seed {seed}")


def test_token_entry_points_refuse_bad_arguments():
    mx = _mx()
    L = mx.load_library()
    st = torch.cuda.current_stream().cuda_stream
    M, K, N = 40, 512, 256
    a = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    size = mx.mxfp4_token_blocks_size(M, K, 32)
    blk = torch.full((size + 512,), 0x5A, dtype=torch.uint8, device="cuda")
    base = blk.data_ptr() + (-blk.data_ptr()) % 256
    bq, bs = mx.mxfp4_quantize(torch.zeros(N, K, dtype=torch.bfloat16, device="cuda"))
    packed = mx.mxfp4_prepack_b(bq, bs)
    c = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    q = L.mxfp4_quantize_tokens
    g = L.mxfp4_gemm_tokens
    assert q(a.data_ptr(), M, K, K, 32, base, size - 1, st) == 7          # blocks too small
    assert q(a.data_ptr(), M, K, K, 32, base + 16, size, st) == 3         # blocks not 256-byte aligned
    assert q(a.data_ptr(), M, K, K, 24, base, size, st) == 1              # m_tile not a multiple of 16
    assert q(a.data_ptr(), M, K, K, 272, base, size, st) == 1             # m_tile above 256
    assert q(a.data_ptr(), M, 100, K, 32, base, size, st) == 2            # K not a multiple of 8
    assert q(a.data_ptr(), M, K, K - 8, 32, base, size, st) == 2          # lda < K
    assert q(a.data_ptr() + 2, M, K, K, 32, base, size, st) == 3          # A misaligned
    assert q(None, M, K, K, 32, base, size, st) == 1
    assert q(a.data_ptr(), 0, K, K, 32, base, size, st) == 0              # no tokens: no-op
    assert g(base, size - 1, M, K, 32, packed.data_ptr(), N, c.data_ptr(), N, 0, st) == 7
    assert g(base + 16, size, M, K, 32, packed.data_ptr(), N, c.data_ptr(), N, 0, st) == 3
    assert g(base, size, M, K, 24, packed.data_ptr(), N, c.data_ptr(), N, 0, st) == 1
    assert g(base, size, M, K, 32, packed.data_ptr(), N, c.data_ptr(), N, -1, st) == 1
    assert g(base, size, M, K, 32, packed.data_ptr(), N, c.data_ptr(), N - 1, 0, st) == 2   # ldc < N
    assert g(base, size, 0, K, 32, packed.data_ptr(), N, c.data_ptr(), N, 0, st) == 0       # no-op
    torch.cuda.synchronize()
    assert bool((blk == 0x5A).all()) and bool((c == 3.0).all())
    assert mx.mxfp4_device_status() == 0
