"""The fused GEMM quantizer maps a work item to its (1x32 block, token row) by a multiply-high with
the reciprocal 0xFFFFFFFF / m + 1 of the tile's row count m, instead of a division. That is exact
only for item indices below 2^16 and m <= 256. Checked here on the CPU: the identity for every
m and index in that range, and that no fused plan the planner makes (forced or automatic) deals an
index past it (its items are rows x blocks of the CTA's K slice, plus one pass of the CTA's
threads)."""
import numpy as np
import pytest

SM_COUNT = 152
CTA_THREADS = 352


def test_reciprocal_quotient_is_exact_below_2_16():
    idx = np.arange(1 << 16, dtype=np.uint64)
    for m in range(2, 257):
        magic = np.uint64(0xFFFFFFFF // m + 1)
        q = (idx * magic) >> np.uint64(32)
        assert np.array_equal(q, idx // np.uint64(m)), m


def test_reciprocal_quotient_fails_where_the_error_term_predicts():
    # magic * m = 2^32 + e with e < m, so the quotient is exact while idx * e < 2^32; for m = 255
    # (e = 254) the first failure is at the largest remainder past 2^32 / 254, far above 2^16: the
    # bound used is conservative, and the identity is not unconditional
    m = 255
    magic = 0xFFFFFFFF // m + 1
    e = magic * m - (1 << 32)
    assert e == 254
    idx = np.arange(1, (1 << 25) // m, dtype=np.uint64) * np.uint64(m) + np.uint64(m - 1)   # remainder m - 1
    bad = idx[((idx * np.uint64(magic)) >> np.uint64(32)) != idx // np.uint64(m)]
    first = int(bad[0])
    # with remainder m - 1 the quotient is wrong exactly when idx * e >= 2^32
    assert first * e >= 1 << 32 > (first - m) * e
    assert first > 1 << 24
    assert all(((i * magic) >> 32) == i // m for i in range(first - 4 * m, first))


@pytest.fixture(scope="module")
def mx():
    import block_scaled_mxfp4_bf16_gb300 as m
    m.load_library()
    return m


def test_fused_plans_keep_item_indices_below_2_16(mx):
    checked = 0
    for M in (1, 2, 7, 16, 31, 64, 100, 128, 200, 256, 1000):
        for N in (128, 2112, 7168):
            for K in (8, 40, 256, 1288, 2048, 7168, 16384, 65536):
                for splits in (0, 1, 2, 4, 8, 16):
                    for m_tile in (0, 16, 64, 128, 256):
                        for path in (0, 1):
                            try:
                                p = mx.mxfp4_gemm_plan_model(M, N, K, SM_COUNT, None, path=path, splits=splits,
                                                             m_tile=m_tile)
                            except mx.Mxfp4Error:
                                continue    # a forced fused slice too large for shared memory is refused
                            if p["path"] != 1:
                                continue
                            atoms_max = -(-(-(-K // 256)) // p["splits"])
                            rows = min(M, p["m_tile"])
                            assert rows <= 256
                            assert rows * 8 * atoms_max + CTA_THREADS < 1 << 16, (M, N, K, splits, m_tile, p)
                            checked += 1
    assert checked > 500
