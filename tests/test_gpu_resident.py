"""The weight-resident kernel (plan path 3: each CTA holds its whole K slice of weights, quantizes
A from registers and reduces the K slices by weight-row owners) against the fp64 oracle, through
the C ABI: C within the tolerance, B's bytes bit-exact, nothing written outside C, A's row
padding past K never read (it holds 1e30)."""
import numpy as np
import pytest
import torch

from block_scaled_mxfp4_bf16_gb300 import workloads
from mxfp4_testlib import assert_bytes_equal, check_tolerance, oracle_c, run_gemm

import oracle

pytestmark = pytest.mark.gpu


def _mx():
    import block_scaled_mxfp4_bf16_gb300 as mx
    return mx


# M, N, K, splits, m_tile: K tails inside a block and past the last 256, N tails, one and two
# token tiles, a ragged second token tile, every owner split from 1 to 8
CASES = [
    (1, 128, 256, 0, 0),
    (1, 1, 8, 0, 0),
    (3, 129, 40, 1, 0),
    (5, 200, 520, 2, 0),
    (8, 2112, 7168, 0, 0),
    (8, 2112, 7176, 6, 0),
    (16, 384, 1536, 3, 0),
    (16, 640, 2072, 5, 16),
    (17, 300, 1032, 4, 0),
    (32, 4096, 512, 0, 0),
    (32, 200, 2048, 8, 32),
    (33, 200, 512, 2, 0),
    (13, 257, 1800, 7, 16),
    (24, 130, 768, 3, 32),
    (2, 512, 4096, 8, 0),
    # 16-token tiles of 3 to 8 steps a slice: a quantizing warp joins as the third MMA issuer
    (7, 128, 768, 1, 16),
    (3, 140, 1024, 1, 16),
    (10, 384, 1288, 1, 16),
    (6, 300, 1792, 1, 16),
    (4, 256, 2048, 1, 16),
    (9, 200, 3840, 2, 16),
    # more than two 1x32 blocks of A per quantizing thread (the kernel variant that loads three at
    # a time): three, four, six; a ragged token tile; a K tail
    (16, 300, 7168, 4, 16),
    (24, 260, 7168, 4, 32),
    (32, 200, 7168, 4, 32),
    (20, 129, 2040, 1, 32),
]


@pytest.mark.parametrize("M,N,K,splits,m_tile", CASES)
def test_resident_vs_oracle(M, N, K, splits, m_tile):
    mx = _mx()
    plan = mx.mxfp4_gemm_plan(M, N, K, path=3, splits=splits, m_tile=m_tile)
    assert plan["path"] == 3
    if splits:
        assert plan["splits"] == min(splits, -(-K // 256))
    a = workloads.random_bf16(M, K, seed=M * 31 + K)
    b = workloads.random_bf16(N, K, seed=N * 17 + K, scale=0.5)
    c, bq, bs = run_gemm(a, b, path=3, splits=splits, m_tile=m_tile, lda_pad=8, ldc_pad=3)
    rq, rs = oracle.quantize(workloads.bf16_bits(b))
    assert_bytes_equal(bq, rq, "B e2m1")
    assert_bytes_equal(bs, rs, "B scales")
    check_tolerance(c, oracle_c(a, bq, bs), f"{M}x{N}x{K} resident splits {splits} m_tile {m_tile}")


@pytest.mark.parametrize("name", ["M8_N2112_K7168", "M16_N3072_K1536", "M32_N4096_K512", "M16_N2112_K7168",
                                  "M4_N2880_K512", "M32_N2880_K512"])
def test_resident_workloads_full_oracle(name):
    """The benchmark's small-M workloads (the outlier recipe of 32x4096x512 included) in the
    automatic weight-resident plan, every output against the oracle."""
    w = workloads.by_name(name)
    a, b = workloads.make_inputs(w, seed=0)
    c, bq, bs = run_gemm(a, b, path=3)
    check_tolerance(c, oracle_c(a, bq, bs), name)


def test_resident_run_to_run_identical():
    mx = _mx()
    w = workloads.by_name("M8_N2112_K7168")
    a, b = workloads.make_inputs(w, seed=0)
    bq, bs = mx.mxfp4_quantize(b.cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a = a.cuda()
    outs = [mx.mxfp4_gemm(a, packed, w.N, path=3).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    for c in outs[1:]:
        assert torch.equal(c.view(torch.int16), outs[0].view(torch.int16))


def test_resident_single_product_lands_in_place():
    """One nonzero A element and one nonzero B element: C is exactly their product at (m, n)."""
    mx = _mx()
    M, N, K = 9, 300, 1800
    for (m, n, k) in [(0, 0, 0), (8, 299, 1799), (3, 130, 1024), (5, 64, 257)]:
        a = torch.zeros(M, K, dtype=torch.bfloat16)
        b = torch.zeros(N, K, dtype=torch.bfloat16)
        a[m, k] = 1.5
        b[n, k] = -4.0
        c, _, _ = run_gemm(a, b, path=3, splits=5)
        want = np.zeros((M, N))
        want[m, n] = -6.0
        assert np.array_equal(c, want), (m, n, k)


def test_resident_plan_is_refused_where_the_slice_cannot_fit():
    mx = _mx()
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_gemm_plan(1, 128, 65536, path=3, splits=2)        # 128 steps per slice
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_gemm_plan(32, 128, 7168, path=3, splits=1)        # 28 steps per slice
