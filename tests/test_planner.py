"""CPU tests of the host planner through mxfp4_gemm_plan_model (no GPU, no CUDA call): the
plans it picks for the five workloads on a GB300-like device, the invariants the GEMM kernel
relies on, the split-K form of every case the GPU tests run, and the cluster-residency limit."""
import pytest

from mxfp4_testlib import REDUCTION_CASES

# GB300: 152 SMs; clusters of s CTAs resident at once, s = 1..16 (cudaOccupancyMaxActiveClusters
# on the GEMM kernel, the same for 90 KB, 130 KB and 210 KB of shared memory per CTA)
SM_COUNT = 152
CLUSTER_CAPS = [152, 76, 46, 36, 28, 23, 15, 15, 15, 13, 8, 8, 7, 7, 7, 7]


@pytest.fixture(scope="module")
def mx():
    import block_scaled_mxfp4_bf16_gb300 as m
    m.load_library()
    return m


def plan(mx, M, N, K, **kw):
    return mx.mxfp4_gemm_plan_model(M, N, K, SM_COUNT, CLUSTER_CAPS, **kw)


@pytest.mark.parametrize("M,N,K,path,splits,m_tile", [
    (16, 3072, 1536, 3, 3, 16),      # weight-resident, two 256-K steps per slice, 72 CTAs
    (8, 2112, 7168, 3, 6, 16),       # weight-resident, 6-slice clusters, 102 CTAs
    (32, 4096, 512, 3, 1, 16),       # weight-resident in two 16-token tiles, unsplit, 64 CTAs
    (64, 7168, 2048, 2, 1, 64),      # longer K keeps one token tile
    (256, 4096, 7168, 2, 2, 128),    # 128-token tiles, 2 slices (bulk split-K)
    (16, 2112, 7168, 3, 6, 16),      # weight-resident: two 1x32 blocks of A per thread
    (4, 2880, 512, 3, 1, 16),
    (32, 2880, 512, 3, 1, 16),
    (24, 2112, 7168, 2, 5, 32),      # too many A blocks per thread for the resident kernel
    (1, 128, 65536, 1, 8, 16),       # slices too long for the resident kernel: fused path
    (256, 3072, 1536, 2, 1, 64),     # 129..512 tokens: 64-token tiles while one wave, unsplit, no refill
    (512, 2048, 2048, 2, 1, 64),
    (160, 7168, 2048, 2, 1, 128),    # 64-token tiles would be 168 CTAs: more than one wave
])
def test_workload_plans(mx, M, N, K, path, splits, m_tile):
    p = plan(mx, M, N, K)
    assert (p["path"], p["splits"], p["m_tile"]) == (path, splits, m_tile), p
    m_tiles = -(-M // p["m_tile"])
    assert p["ctas"] == m_tiles * -(-N // 128) * p["splits"]


def test_invariants_over_a_grid(mx):
    checked = 0
    for M in (1, 5, 8, 16, 17, 33, 64, 100, 128, 200, 256, 300, 512, 1000, 4096):
        for N in (128, 2112, 7168):
            for K in (8, 40, 64, 256, 1280, 1288, 4096, 7168, 16384, 65536):   # with K tails
                for path in (0, 1, 2, 3):
                    for splits in (0, 1, 2, 3, 5, 8, 16):
                        try:
                            p = plan(mx, M, N, K, path=path, splits=splits)
                        except Exception:
                            continue
                        checked += 1
                        steps = -(-(-(-K // 256)) // p["splits"])     # 256-K steps of the longest slice
                        assert 1 <= p["issuers"] <= (3 if p["path"] in (2, 3) else 2) and 1 <= p["stages"] <= 8, p
                        if p["path"] == 3:    # the whole slice resident, two A blocks per thread at most
                            assert p["stages"] == steps and p["m_tile"] in (16, 32), p
                            # a third issuing warp only for 16-token tiles of three or more steps
                            assert p["issuers"] == (3 if p["m_tile"] == 16 and steps >= 3 else 2), p
                            assert p["issuers"] * p["m_tile"] + 16 * steps <= p["tmem_cols"], p
                            # explicit plans may take the kernel variant with up to six blocks
                            # of A per quantizing thread
                            assert min(M, p["m_tile"]) * steps * 8 <= 320 * 6, (M, N, K, p)
                            assert p["smem_bytes"] <= 227 * 1024, p
                        if p["issuers"] == 3 and p["path"] == 2:   # the lent epilogue warp: only without refills
                            assert p["stages"] == steps and p["m_tile"] <= 128, p
                        # scale factors by tensor-memory stores on the two-kernel path, where the
                        # tensor pipe is the limit: two issuers sharing each step, or a refilled ring
                        wide = p["m_tile"] > 128 and p["issuers"] == 2
                        assert p["scale_stores"] == int(p["path"] == 2 and (wide or steps > p["stages"])), p
                        if p["m_tile"] > 128:   # two issuers, each with part of every step's tokens
                            assert p["issuers"] == 2, p
                            assert p["m_tile"] + 32 * p["stages"] <= p["tmem_cols"], p
                        elif steps > p["stages"]:   # refilled stages: one MMA thread per stage
                            assert p["stages"] % p["issuers"] == 0, (M, N, K, path, splits, p)
                        t = p["tmem_cols"]
                        assert 32 <= t <= 512 and t & (t - 1) == 0, p
                        assert p["smem_bytes"] <= 227 * 1024, p
                        assert p["m_tile"] % 16 == 0 and 16 <= p["m_tile"] <= 256
                        assert p["splits"] <= min(16, -(-K // 256))
                        if splits:
                            assert p["splits"] == min(splits, -(-K // 256), 16)
                        if path:
                            assert p["path"] == path
                        if p["splits"] == 1:
                            assert p["reduction"] == 0
    assert checked > 1500


@pytest.mark.parametrize("M,N,K,path,splits,form", REDUCTION_CASES)
def test_split_k_forms(mx, M, N, K, path, splits, form):
    p = plan(mx, M, N, K, path=path, splits=splits)
    assert (p["reduction"], p["recv_dedicated"]) == form, p


def test_cluster_residency_limits_the_split(mx):
    # the headline shape has 17 output tiles: 6-CTA clusters need 17 resident at once
    caps = list(CLUSTER_CAPS)
    assert mx.mxfp4_gemm_plan_model(8, 2112, 7168, SM_COUNT, caps)["splits"] == 6
    caps[5] = 16                     # only 16 clusters of 6 fit: fall back to 5 slices
    assert mx.mxfp4_gemm_plan_model(8, 2112, 7168, SM_COUNT, caps)["splits"] == 5
    # without a limit the automatic plan still stays within portable cluster sizes (<= 8)
    assert mx.mxfp4_gemm_plan_model(1, 128, 65536, SM_COUNT, None)["splits"] <= 8


def test_automatic_small_m_plans_keep_their_limits_and_one_wave(mx):
    # up to 32 tokens the automatic plan is the weight-resident kernel wherever its slices fit
    # (at most two 1x32 blocks of A per quantizing thread, eight 256-K steps per slice); where
    # they do not, the fused plan only while its quantization is at most one block per thread
    # (352 threads); the CTAs fit one wave either way
    resident = fused = two_kernel = 0
    for M in (1, 4, 8, 13, 16, 17, 24, 32, 33, 64):
        for N in (128, 2112, 2880, 4096, 7168):
            for K in (64, 512, 1536, 2048, 7168, 16384):
                p = plan(mx, M, N, K)
                atoms_max = -(-(-(-K // 256)) // p["splits"])
                if p["path"] == 3:
                    resident += 1
                    assert M <= 32 and p["m_tile"] in (16, 32), (M, N, K, p)
                    assert min(M, p["m_tile"]) * 8 * atoms_max <= 640 and atoms_max <= 8, (M, N, K, p)
                    assert p["splits"] == 1 or atoms_max >= 2, (M, N, K, p)
                    assert p["ctas"] <= SM_COUNT, (M, N, K, p)
                elif p["path"] == 1:
                    fused += 1
                    assert M <= 32 and p["m_tile"] == 16, (M, N, K, p)
                    assert min(M, 16) * 8 * atoms_max <= 352, (M, N, K, p)
                    assert p["ctas"] <= SM_COUNT, (M, N, K, p)
                else:
                    two_kernel += 1
    assert resident and two_kernel


def test_errors(mx):
    import block_scaled_mxfp4_bf16_gb300 as m
    with pytest.raises(m.Mxfp4Error):
        plan(mx, 8, 2112, 7204)          # K not a multiple of 8
    with pytest.raises(m.Mxfp4Error):
        plan(mx, 0, 2112, 7168)
    with pytest.raises(m.Mxfp4Error):
        mx.mxfp4_gemm_plan_model(8, 2112, 7168, 0, CLUSTER_CAPS)
    with pytest.raises(m.Mxfp4Error):
        plan(mx, 8, 2112, 7168, m_tile=24)   # token tile must be a multiple of 16


@pytest.mark.parametrize("M,N,K,plain,ready,early", [
    (8, 2112, 7168, (3, 6, 102), (3, 4, 68), 1),    # six 112 KB slices leave no room: four on 68 SMs
    (4, 2112, 7168, (3, 6, 102), (3, 4, 68), 1),
    (16, 2112, 7168, (3, 6, 102), (3, 4, 68), 1),   # three blocks of A per quantizing thread
    (32, 2112, 7168, (2, 5, 85), (3, 4, 68), 1),    # six: no flagless resident plan fits
    (24, 2112, 7168, (2, 5, 85), (3, 4, 68), 1),
    (8, 4096, 5120, (3, 4, 128), (3, 4, 128), 0),   # two slices would take ten steps each: it waits
    (16, 3072, 1536, (3, 3, 72), (3, 3, 72), 1),    # room to read A early: the same plan
    (32, 4096, 512, (3, 1, 64), (3, 1, 64), 1),
    (8, 2112, 5120, (3, 6, 102), (3, 6, 102), 1),
])
def test_plans_with_a_declared_ready(mx, M, N, K, plain, ready, early):
    # MXFP4_GEMM_A_READY: A is read before the dependency wait where two CTAs of 112 KB do not
    # share an SM; where they would (or no flagless resident plan fits), the most slices whose
    # CTAs fill at most half the SMs, one per SM, if the slices fit; otherwise the flagless plan,
    # waiting as before
    p = plan(mx, M, N, K)
    r = plan(mx, M, N, K, a_ready=True)
    assert (p["path"], p["splits"], p["ctas"], p["a_early"]) == plain + (0,)
    assert (r["path"], r["splits"], r["ctas"], r["a_early"]) == ready + (early,)
    if ready != plain:
        assert 2 * r["ctas"] <= SM_COUNT and 2 * (r["smem_bytes"] + 1024) > 233472
        # the same slices can be forced without the flag (the kernel then waits before reading A)
        f = plan(mx, M, N, K, path=3, splits=r["splits"], m_tile=r["m_tile"])
        assert (f["splits"], f["ctas"], f["a_early"]) == (r["splits"], r["ctas"], 0)


def test_a_early_only_where_it_is_read(mx):
    # the flag changes nothing on the streaming paths, and an explicit resident plan keeps its
    # slices: it reads early only where the shared memory leaves room
    for M, N, K in ((64, 7168, 2048), (256, 4096, 7168), (300, 384, 1536)):
        assert plan(mx, M, N, K, a_ready=True) == plan(mx, M, N, K)
    six = plan(mx, 8, 2112, 7168, path=3, splits=6, a_ready=True)
    four = plan(mx, 8, 2112, 7168, path=3, splits=4, a_ready=True)
    assert (six["splits"], six["a_early"]) == (6, 0)
    assert (four["splits"], four["a_early"]) == (4, 1)
    assert plan(mx, 8, 2112, 7168, path=3, splits=4)["a_early"] == 0
