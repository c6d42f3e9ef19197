"""GPU GEMM parity: C from mxfp4_gemm (tcgen05 kind::mxf4, through the C ABI) against the
fp64 oracle, within |C - C_ref| <= 8e-3 |C_ref| + 1e-3 rms(C_ref)."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads
from mxfp4_testlib import (REDUCTION_CASES, assert_bytes_equal, bf16_to_f64, check_tolerance, oracle_c,
                           run_gemm, to_np_u8)

pytestmark = pytest.mark.gpu


def _mx():
    import block_scaled_mxfp4_bf16_gb300 as mx
    return mx


def test_single_product_lands_in_place():
    # one nonzero per operand: exposes any error in operand, scale-factor or output layout
    M, N, K = 5, 200, 512
    for (m, n, k) in [(0, 0, 0), (3, 131, 300), (4, 199, 511), (1, 64, 33)]:
        a = torch.zeros(M, K, dtype=torch.bfloat16)
        b = torch.zeros(N, K, dtype=torch.bfloat16)
        a[m, k] = 3.0
        b[n, k] = -0.75
        for path in (1, 2):
            c, _, _ = run_gemm(a, b, path=path)
            want = np.zeros((M, N))
            want[m, n] = -2.25
            assert np.array_equal(c, want), (m, n, k, path, np.argwhere(c != want)[:5])


SMALL = [
    # M, N, K -- tails in every dimension, K not a multiple of 256, M past one 256-token tile
    (1, 128, 64), (5, 200, 192), (16, 384, 512), (8, 2112, 1024), (17, 130, 320),
    (32, 256, 1536), (33, 640, 256), (64, 512, 768), (100, 300, 512), (256, 256, 256), (300, 136, 128),
    # K % 32 != 0: the last 1x32 block is cut by K (zeros past K), also inside a split's last step
    (3, 200, 40), (16, 136, 8), (8, 256, 72), (33, 300, 200), (100, 128, 456), (8, 2112, 7176),
]


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_gemm_small_shapes_vs_oracle(M, N, K, path):
    a = workloads.random_bf16(M, K, seed=M * 1000 + K)
    b = workloads.random_bf16(N, K, seed=N * 1000 + K + 1, scale=0.5)
    for splits in (0, 1, 3):
        c, bq, bs = run_gemm(a, b, path=path, splits=splits, lda_pad=8, ldc_pad=3)
        rq, rs = oracle.quantize(workloads.bf16_bits(b))
        assert_bytes_equal(bq, rq, "B e2m1")
        assert_bytes_equal(bs, rs, "B scales")
        check_tolerance(c, oracle_c(a, bq, bs), f"{M}x{N}x{K} path {path} splits {splits}")


@pytest.mark.parametrize("w", workloads.WORKLOADS, ids=lambda w: w.name)
def test_gemm_workloads_sampled_vs_oracle(w):
    # full-size workloads in the automatic plan the benchmark times; the oracle computes a
    # sample of outputs one by one (every row, 384 random columns)
    a, b = workloads.make_inputs(w, seed=0)
    c, bq, bs = run_gemm(a, b)
    rq, rs = oracle.quantize(workloads.bf16_bits(b))
    assert_bytes_equal(bs, rs, "B scales")
    assert_bytes_equal(bq, rq, "B e2m1")
    aq, as_ = oracle.quantize(workloads.bf16_bits(a))
    rng = np.random.default_rng(1)
    cols = np.concatenate([rng.choice(w.N, 380, replace=False), [0, w.N - 1, 127, 128]])
    im = np.repeat(np.arange(w.M), cols.size)
    inn = np.tile(cols, w.M)
    ref = oracle.gemm_entries(aq, as_, bq, bs, im, inn)
    check_tolerance(c[im, inn], ref, w.name)


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 7168), (8, 2112, 32768), (1, 128, 65536), (520, 7168, 1032)])
def test_gemm_large_shapes_sampled_vs_oracle(M, N, K):
    # sizes past the benchmark's: 256-token tiles over many token tiles, long K slices that refill
    # every pipeline stage several times, one weight tile with the widest automatic split, a K
    # cut inside a block at 520 tokens; automatic plans, sampled outputs against the oracle
    a = workloads.random_bf16(M, K, seed=M + 3 * K)
    b = workloads.random_bf16(N, K, seed=N + 5 * K, scale=0.5)
    c, bq, bs = run_gemm(a, b)
    rq, rs = oracle.quantize(workloads.bf16_bits(b))
    assert_bytes_equal(bs, rs, "B scales")
    assert_bytes_equal(bq, rq, "B e2m1")
    aq, as_ = oracle.quantize(workloads.bf16_bits(a))
    rng = np.random.default_rng(M + N + K)
    rows = np.unique(np.concatenate([rng.choice(M, min(M, 96), replace=False), [0, M - 1]]))
    cols = np.unique(np.concatenate([rng.choice(N, min(N, 96), replace=False), [0, N - 1]]))
    im = np.repeat(rows, cols.size)
    inn = np.tile(cols, rows.size)
    ref = oracle.gemm_entries(aq, as_, bq, bs, im, inn)
    check_tolerance(c[im, inn], ref, f"{M}x{N}x{K}")


@pytest.mark.parametrize("w", workloads.EXTRA_WORKLOADS, ids=lambda w: w.name)
def test_gemm_leaderboard_shapes_full_oracle(w):
    a, b = workloads.make_inputs(w, seed=2)
    c, bq, bs = run_gemm(a, b)
    check_tolerance(c, oracle_c(a, bq, bs), w.name)


def test_gemm_outlier_workload_full_oracle_both_paths():
    w = workloads.by_name("M32_N4096_K512")
    a, b = workloads.make_inputs(w, seed=0)
    for path in (1, 2):
        c, bq, bs = run_gemm(a, b, path=path)
        check_tolerance(c, oracle_c(a, bq, bs), f"{w.name} path {path}")


@pytest.mark.parametrize("name,path,splits", [("M8_N2112_K7168", 0, 0), ("M256_N4096_K7168", 2, 2)])
def test_gemm_run_to_run_identical(name, path, splits):
    # split-K sums in a fixed order: short runs (posted stores) and long runs (bulk copies)
    mx = _mx()
    w = workloads.by_name(name)
    a, b = workloads.make_inputs(w, seed=4)
    a, b = a.cuda(), b.cuda()
    bq, bs = mx.mxfp4_quantize(b)
    packed = mx.mxfp4_prepack_b(bq, bs)
    c1 = mx.mxfp4_gemm(a, packed, w.N, path=path, splits=splits).clone()
    c2 = mx.mxfp4_gemm(a, packed, w.N, path=path, splits=splits).clone()
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert mx.mxfp4_gemm_plan(w.M, w.N, w.K, path, splits)["splits"] > 1


def test_gemm_empty_and_errors():
    mx = _mx()
    L = mx.load_library()
    st = torch.cuda.current_stream().cuda_stream
    a = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    bq = torch.zeros(64, 64, dtype=torch.uint8, device="cuda")
    bs = torch.zeros(64, 4, dtype=torch.uint8, device="cuda")
    packed = mx.mxfp4_prepack_b(bq, bs)
    c = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    # M == 0 and N == 0 are no-ops
    assert L.mxfp4_gemm(a.data_ptr(), 0, 128, 128, packed.data_ptr(), 64, c.data_ptr(), 64, None, 0, st) == 0
    assert L.mxfp4_gemm(a.data_ptr(), 4, 128, 128, packed.data_ptr(), 0, c.data_ptr(), 64, None, 0, st) == 0
    # K not a multiple of 8, lda < K, misaligned A, missing workspace
    assert L.mxfp4_gemm(a.data_ptr(), 4, 100, 128, packed.data_ptr(), 64, c.data_ptr(), 64, None, 0, st) == 2
    assert L.mxfp4_gemm(a.data_ptr(), 4, 128, 64, packed.data_ptr(), 64, c.data_ptr(), 64, None, 0, st) == 2
    assert L.mxfp4_gemm(a.data_ptr() + 2, 4, 128, 128, packed.data_ptr(), 64, c.data_ptr(), 64, None, 0, st) == 3
    need = mx.mxfp4_gemm_workspace_size(4, 64, 128)
    if need:
        assert L.mxfp4_gemm(a.data_ptr(), 4, 128, 128, packed.data_ptr(), 64, c.data_ptr(), 64, None, 0, st) == 7
    assert L.mxfp4_prepack_b_size(64, 100) == 0
    # the binding refuses packed weights smaller than the shape needs, before any launch
    with pytest.raises(ValueError):
        mx.mxfp4_gemm(a, packed[:1024], 64)
    with pytest.raises(ValueError):
        mx.mxfp4_gemm(a, packed, 64 + 128)        # N past the packed tiles


def test_concurrent_streams_use_their_own_default_workspace():
    # two-kernel GEMMs (the workspace holds the quantized A between the two kernels) on two streams
    # at once through the binding's default workspaces: each stream must get its own, or the
    # calls would overwrite each other's token blocks
    mx = _mx()
    M, N, K = 64, 512, 2048
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=31).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a = [workloads.random_bf16(M, K, seed=32 + i).cuda() for i in range(2)]
    want = [mx.mxfp4_gemm(x, packed, N).clone() for x in a]
    assert mx.mxfp4_gemm_plan(M, N, K)["path"] == 2
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    outs = [[], []]
    for rep in range(20):
        for i, s in enumerate(streams):
            with torch.cuda.stream(s):
                outs[i].append(mx.mxfp4_gemm(a[i], packed, N, stream=s))
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    for i in range(2):
        for c in outs[i]:
            assert torch.equal(c.view(torch.int16), want[i].view(torch.int16))


def test_gemm_host_empty_and_errors():
    # the host-buffer call checks everything before it copies anything: empty shapes are no-ops,
    # bad strides, misaligned device buffers and missing host buffers are refused, and none of
    # them touches the host or device buffers
    mx = _mx()
    L = mx.load_library()
    st = torch.cuda.current_stream().cuda_stream
    M, N, K = 4, 128, 64
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=1).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a_host = workloads.random_bf16(M, K, seed=2).pin_memory()
    c_host = torch.full((M, N), 5.0, dtype=torch.bfloat16).pin_memory()
    a_dev = torch.full((M, K), 7.0, dtype=torch.bfloat16, device="cuda")
    c_dev = torch.full((M, N), 9.0, dtype=torch.bfloat16, device="cuda")

    def call(a=a_host.data_ptr(), m=M, k=K, lda=K, n=N, c=c_host.data_ptr(), ldc=N, ad=a_dev.data_ptr(),
             cd=c_dev.data_ptr()):
        return L.mxfp4_gemm_host(a, m, k, lda, packed.data_ptr(), n, c, ldc, ad, cd, None, 0, st)

    assert call(m=0) == 0 and call(n=0) == 0          # no-ops
    assert call(lda=K - 8) == 2                         # host row stride shorter than K
    assert call(ldc=N - 1) == 2                         # host C stride shorter than N
    assert call(k=K + 4) == 2                           # K not a multiple of 8
    assert call(ad=a_dev.data_ptr() + 2) == 3           # misaligned device A
    assert call(a=None) == 1 and call(c=None) == 1      # missing host buffers
    torch.cuda.synchronize()
    assert torch.all(c_host == 5.0) and torch.all(a_dev == 7.0) and torch.all(c_dev == 9.0)
    assert mx.mxfp4_device_status() == 0


def test_timeout_is_reported_not_hung():
    mx = _mx()
    assert mx.mxfp4_device_status() == 0
    mx.mxfp4_selftest_timeout(2000)          # waits 2 ms on a barrier nobody signals
    assert mx.mxfp4_device_status() == 6     # MXFP4_ERR_TIMEOUT, context still usable
    assert mx.mxfp4_device_status() == 0     # cleared by the read
    x = torch.ones(2, 64, dtype=torch.bfloat16, device="cuda")
    q, s = mx.mxfp4_quantize(x)
    torch.cuda.synchronize()
    assert int(s[0, 0].item()) == 125


@pytest.mark.parametrize("M,N,K,m_tile", [(256, 384, 1024, 128), (100, 256, 768, 64), (64, 512, 512, 16)])
def test_gemm_token_tile_override_vs_oracle(M, N, K, m_tile):
    # several token tiles per weight tile (m_tiles > 1), with and without split-K, both paths
    mx = _mx()
    a = workloads.random_bf16(M, K, seed=M + m_tile)
    b = workloads.random_bf16(N, K, seed=N + m_tile)
    bq, bs = mx.mxfp4_quantize(b.cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    ref = oracle_c(a, to_np_u8(bq), to_np_u8(bs))
    for path in (1, 2):
        for splits in (1, 2):
            try:
                mx.mxfp4_gemm_plan(M, N, K, path, splits, m_tile)
            except mx.Mxfp4Error as e:
                # a forced fused path whose staged A slice exceeds shared memory is refused
                assert path == 1 and e.status == 2
                continue
            c = mx.mxfp4_gemm(a.cuda(), packed, N, path=path, splits=splits, m_tile=m_tile)
            torch.cuda.synchronize()
            assert mx.mxfp4_gemm_plan(M, N, K, path, splits, m_tile)["m_tile"] == m_tile
            check_tolerance(bf16_to_f64(c.cpu()), ref, f"{M}x{N}x{K} m_tile {m_tile} path {path} splits {splits}")


@pytest.mark.parametrize("M,N,K,path,splits,form", REDUCTION_CASES)
def test_every_split_k_form_vs_oracle(M, N, K, path, splits, form):
    mx = _mx()
    plan = mx.mxfp4_gemm_plan(M, N, K, path, splits)
    assert (plan["reduction"], plan["recv_dedicated"]) == form, plan
    assert plan["path"] == path and plan["splits"] == splits
    a = workloads.random_bf16(M, K, seed=M * 31 + K)
    b = workloads.random_bf16(N, K, seed=N * 37 + K, scale=0.5)
    c, bq, bs = run_gemm(a, b, path=path, splits=splits, ldc_pad=5)
    check_tolerance(c, oracle_c(a, bq, bs), f"{M}x{N}x{K} path {path} splits {splits} form {form}")


def test_plan_invariants_over_a_shape_grid():
    # Planner invariants the kernel relies on, over tiny to large shapes and every option:
    # a refilled stage has a single MMA issuer (stages % issuers == 0), tensor memory fits one
    # power-of-two allocation, shared memory fits the opt-in limit.
    mx = _mx()
    checked = 0
    for M in (1, 8, 16, 33, 64, 100, 200, 256, 1000):
        for K in (256, 1280, 4096, 7168, 16384):
            for path in (0, 1, 2):
                for splits in (0, 1, 2, 3, 5):
                    try:
                        pl = mx.mxfp4_gemm_plan(M, 2112, K, path, splits)
                    except Exception:
                        continue
                    checked += 1
                    steps = -(-(-(-K // 256)) // pl["splits"])      # 256-K steps of the longest slice
                    assert 1 <= pl["issuers"] <= (3 if pl["path"] in (2, 3) else 2), pl
                    halves = pl["m_tile"] > 128 and pl["issuers"] == 2   # both issuers take every stage
                    if steps > pl["stages"] and not halves:
                        assert pl["stages"] % pl["issuers"] == 0, (M, K, path, splits, pl)
                    t = pl["tmem_cols"]
                    assert 32 <= t <= 512 and t & (t - 1) == 0, pl
                    assert pl["smem_bytes"] <= 227 * 1024, pl
    assert checked > 200


def test_gemm_host_buffers_match_device_call():
    # mxfp4_gemm_host: strided host A in, strided host C out, bit-identical to the device call,
    # for every way A and C can travel -- A from mapped page-locked memory by the staging kernel
    # (16-byte rows) or by a copy (pageable memory, or a row stride that is not a multiple of 8),
    # C written by the GEMM into mapped page-locked memory or copied back; an undersized
    # workspace is refused before anything is copied.
    mx = _mx()
    for M, N, K in ((8, 2112, 7168), (40, 300, 512), (5, 200, 72)):
        a = workloads.random_bf16(M, K, seed=M + 7)
        b = workloads.random_bf16(N, K, seed=N + 7)
        bq, bs = mx.mxfp4_quantize(b.cuda())
        packed = mx.mxfp4_prepack_b(bq, bs)
        want = mx.mxfp4_gemm(a.cuda(), packed, N)
        for a_kind, pad in (("pinned", 64), ("pageable", 64), ("pinned", 3)):
            a_store = torch.full((M, K + pad), 1.0e30, dtype=torch.bfloat16)
            if a_kind == "pinned":
                a_store = a_store.pin_memory()
            a_store[:, :K] = a
            for c_pinned in (True, False):   # mapped page-locked C (written by the GEMM) or a copy
                c_store = torch.full((M, N + 3), 5.0, dtype=torch.bfloat16)
                if c_pinned:
                    c_store = c_store.pin_memory()
                a_dev = torch.full((M, K), 7.0, dtype=torch.bfloat16, device="cuda")
                c_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
                mx.mxfp4_gemm_host(a_store[:, :K], packed, N, c_store[:, :N], a_dev, c_dev)
                torch.cuda.synchronize()
                assert mx.mxfp4_device_status() == 0
                what = (M, N, K, a_kind, pad, c_pinned)
                assert torch.equal(a_dev.cpu().view(torch.int16), a.view(torch.int16)), what
                assert torch.equal(c_store[:, :N].view(torch.int16), want.cpu().view(torch.int16)), what
                assert torch.all(c_store[:, N:] == 5.0)
    # chained host-buffer calls: the first call's C (stored by its GEMM into mapped page-locked
    # memory) is the second call's A, so the second call must see the first one's stores
    M, N = 8, 512
    a1 = workloads.random_bf16(M, 512, seed=21).pin_memory()
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, 512, seed=22).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    c1 = torch.full((M, N), 3.0, dtype=torch.bfloat16).pin_memory()
    c2 = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    a_dev = [torch.empty(M, 512, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    c_dev = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for _ in range(3):
        c1.fill_(3.0)
        mx.mxfp4_gemm_host(a1, packed, N, c1, a_dev[0], c_dev[0])
        mx.mxfp4_gemm_host(c1, packed, N, c2, a_dev[1], c_dev[1])
        torch.cuda.synchronize()
        want1 = mx.mxfp4_gemm(a1.cuda(), packed, N)
        want2 = mx.mxfp4_gemm(want1, packed, N)
        assert torch.equal(c1.view(torch.int16), want1.cpu().view(torch.int16))
        assert torch.equal(c2.view(torch.int16), want2.cpu().view(torch.int16))
    # M = 300 needs a workspace (two-kernel path): a one-byte one is refused, C untouched
    M, N, K = 300, 256, 256
    need = mx.mxfp4_gemm_workspace_size(M, N, K)
    assert need > 0
    a_host = workloads.random_bf16(M, K, seed=3).pin_memory()
    c_host = torch.full((M, N), 5.0, dtype=torch.bfloat16).pin_memory()
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=4).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a_dev = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    c_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    tiny = torch.empty(1, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_gemm_host(a_host, packed, N, c_host, a_dev, c_dev, workspace=tiny)
    torch.cuda.synchronize()
    assert torch.all(c_host == 5.0)


def test_prepared_calls_match_plain_calls():
    # prepared calls on fixed buffers, replayed with new contents in those buffers, give the
    # plain calls' bits every time; the host-buffer form returns C through pinned memory
    mx = _mx()
    M, N, K = 8, 2112, 7168
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=31).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    a_host = torch.empty(M, K, dtype=torch.bfloat16).pin_memory()
    c_host = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    a_dev = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    c_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    call = mx.prepare_gemm(a, packed, N, c)
    host_call = mx.prepare_gemm_host(a_host, packed, N, c_host, a_dev, c_dev)
    for seed in (1, 2, 3):
        x = workloads.random_bf16(M, K, seed=seed)
        a.copy_(x)
        a_host.copy_(x)
        call()
        host_call()
        torch.cuda.synchronize()
        want = mx.mxfp4_gemm(x.cuda(), packed, N)
        assert torch.equal(c.view(torch.int16), want.view(torch.int16)), seed
        assert torch.equal(c_host.view(torch.int16), want.cpu().view(torch.int16)), seed
    assert mx.mxfp4_device_status() == 0


@pytest.mark.parametrize("M,N,K,path,splits,m_tile", [
    (16, 3072, 1536, 0, 0, 0),       # weight-resident, split K
    (5, 300, 520, 1, 2, 0),          # fused, K tail
    (64, 7168, 2048, 0, 0, 0),       # two-kernel (workspace)
    (300, 384, 1536, 2, 1, 192),     # two issuers sharing every step, scale factors stored by warps
])
def test_prepared_calls_every_plan(M, N, K, path, splits, m_tile):
    # the library's prepared calls (created once, run many times) against the plain calls on the
    # same buffers, for each kind of plan; host buffers both page-locked (A staged by a kernel, C
    # stored straight into them; A read before or after the work ahead of it) and pageable
    # (copied both ways)
    mx = _mx()
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=M + 3).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    call = mx.prepare_gemm(a, packed, N, c, path=path, splits=splits, m_tile=m_tile)
    a_dev = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    c_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    hosts = []
    for pinned, early in ((True, False), (True, True), (False, False)):
        a_host = torch.empty(M, K, dtype=torch.bfloat16)
        c_host = torch.empty(M, N, dtype=torch.bfloat16)
        if pinned:
            a_host, c_host = a_host.pin_memory(), c_host.pin_memory()
        # early: A declared host-written only, staged without waiting for the work before it
        hosts.append((a_host, c_host, mx.prepare_gemm_host(a_host, packed, N, c_host, a_dev, c_dev,
                                                           a_host_written=early)))
    for seed in (5, 6):
        x = workloads.random_bf16(M, K, seed=seed)
        want = mx.mxfp4_gemm(x.cuda(), packed, N, path=path, splits=splits, m_tile=m_tile)
        a.copy_(x)
        call()
        torch.cuda.synchronize()
        assert torch.equal(c.view(torch.int16), want.view(torch.int16)), seed
        auto = mx.mxfp4_gemm(x.cuda(), packed, N)   # host calls run the automatic plan
        for a_host, c_host, host_call in hosts:
            a_host.copy_(x)
            c_host.zero_()
            host_call()
            torch.cuda.synchronize()
            assert torch.equal(c_host.view(torch.int16), auto.cpu().view(torch.int16)), (seed, a_host.is_pinned())
    assert mx.mxfp4_device_status() == 0


@pytest.mark.parametrize("M,N,K,path,splits,m_tile", [
    (8, 2112, 7168, 0, 0, 0),        # weight-resident, six K slices (four with the flag)
    (16, 2112, 7168, 0, 0, 0),       # four slices with the flag: three blocks of A per thread
    (32, 2112, 7168, 0, 0, 0),       # two-kernel without the flag, weight-resident with it
    (16, 3072, 1536, 0, 0, 0),       # weight-resident, three K slices
    (5, 300, 520, 1, 2, 0),          # fused, K tail
    (64, 7168, 2048, 0, 0, 0),       # two-kernel, four-lane quantizer
    (300, 384, 1536, 2, 1, 192),     # two-kernel, one-lane quantizer, wide token tile
])
def test_a_ready_gives_the_same_bits(M, N, K, path, splits, m_tile):
    # MXFP4_GEMM_A_READY used as its contract allows: A rewritten by an ordinary copy, read by a
    # call without the flag, then by calls with it (their predecessor began after the copy had
    # finished). Each seed rewrites A, so a flagged call that read A too early would see the
    # previous seed's values. Every call gives the bits of a flagless call on the plan the flag
    # selects (the same plan, except where the automatic weight-resident plan changes with it).
    mx = _mx()
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=M + 11).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    kw = dict(path=path, splits=splits, m_tile=m_tile)
    rp = mx.mxfp4_gemm_plan(M, N, K, a_ready=True, **kw)
    kw_plan = dict(path=rp["path"], splits=rp["splits"], m_tile=rp["m_tile"])
    if (M, N, K) == (8, 2112, 7168):   # the flagless six slices leave no room: side by side
        assert rp["path"] == 3 and rp["a_early"] == 1 and 2 * rp["ctas"] <= 152, rp
    prepared = mx.prepare_gemm(a, packed, N, outs[3], a_ready=True, **kw)
    xs = [workloads.random_bf16(M, K, seed=s).cuda() for s in (21, 22, 23)]
    wants = [mx.mxfp4_gemm(x, packed, N, **kw_plan) for x in xs]
    torch.cuda.synchronize()
    for rep in range(2):
        for x, want in zip(xs, wants):
            a.copy_(x)
            mx.mxfp4_gemm(a, packed, N, c=outs[0], **kw_plan)
            mx.mxfp4_gemm(a, packed, N, c=outs[1], a_ready=True, **kw)
            mx.mxfp4_gemm(a, packed, N, c=outs[2], a_ready=True, **kw)
            prepared()
            torch.cuda.synchronize()
            for i, c in enumerate(outs):
                assert torch.equal(c.view(torch.int16), want.view(torch.int16)), (rep, i)
    assert mx.mxfp4_device_status() == 0

def test_prepared_host_calls_chain_through_host_memory():
    # C of one prepared host call is A of the next (K == N): the second call's staging must read
    # the first call's C only once it is complete
    mx = _mx()
    M, N = 8, 1024
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, N, seed=41, scale=0.05).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    bufs = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    a_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    c_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    first = mx.prepare_gemm_host(bufs[0], packed, N, bufs[1], a_dev, c_dev)
    second = mx.prepare_gemm_host(bufs[1], packed, N, bufs[2], a_dev, c_dev)
    x = workloads.random_bf16(M, N, seed=42)
    bufs[0].copy_(x)
    for _ in range(3):
        first()
        second()
    torch.cuda.synchronize()
    once = mx.mxfp4_gemm(x.cuda(), packed, N)
    twice = mx.mxfp4_gemm(once, packed, N)
    assert torch.equal(bufs[2].view(torch.int16), twice.cpu().view(torch.int16))
    assert mx.mxfp4_device_status() == 0


def test_prepared_call_of_an_empty_product():
    # M = 0: the call is created and each run enqueues nothing
    mx = _mx()
    N, K = 256, 512
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=9).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
    call = mx.prepare_gemm(a, packed, N, c)
    call()
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0


@pytest.mark.parametrize("M,N,K,path,splits,m_tile,stores", [
    (200, 384, 4096, 2, 1, 128, 1),   # 16 steps over 6 stages: refilled, scale factors stored by warps
    (100, 300, 5128, 2, 2, 64, 1),    # split-K, K tail, ragged weight tile, 11 steps over 8 stages
    (40, 256, 12288, 2, 3, 48, 1),    # three slices of 16 steps, 48-token tiles
    (40, 256, 2304, 2, 3, 48, 0),     # three steps per slice, a stage each: the MMA threads copy them
    (64, 256, 2048, 2, 1, 64, 0),     # the same unsplit, three issuers
])
def test_gemm_scale_factor_stores_vs_oracle(M, N, K, path, splits, m_tile, stores):
    # On the two-kernel path with a refilling ring, epilogue warps 4..7 write each stage's weight
    # and token scale factors into tensor memory (one lane quarter each) instead of the MMA
    # threads copying them; both forms against the oracle
    mx = _mx()
    plan = mx.mxfp4_gemm_plan(M, N, K, path, splits, m_tile)
    assert plan["scale_stores"] == stores and plan["m_tile"] == m_tile, plan
    a = workloads.random_bf16(M, K, seed=M + K + 7)
    b = workloads.random_bf16(N, K, seed=N + K + 7, scale=0.5)
    bq, bs = mx.mxfp4_quantize(b.cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    c = mx.mxfp4_gemm(a.cuda(), packed, N, path=path, splits=splits, m_tile=m_tile)
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    ref = oracle_c(a, to_np_u8(bq), to_np_u8(bs))
    check_tolerance(bf16_to_f64(c.cpu()), ref, f"{M}x{N}x{K} splits {splits} m_tile {m_tile} stores {stores}")


@pytest.mark.parametrize("M,N,K,path,splits,m_tile", [
    (600, 200, 512, 2, 1, 0), (600, 200, 1024, 2, 2, 0), (300, 384, 768, 2, 1, 256),
    (600, 200, 2048, 2, 1, 0),       # 8 steps over 4 stages: both issuers release every refilled stage
    (700, 300, 3072, 2, 1, 0),       # 12 steps, three tiles, the last one ragged (188 tokens)
    (300, 384, 1536, 2, 1, 192),     # 6 steps over 5 stages; the second issuer's MMAs take 64 tokens
    (200, 256, 1024, 2, 2, 160),     # split-K over a 160-token tile: 32-token MMAs for the second issuer
    (300, 256, 256, 1, 1, 256),      # the fused path with a 256-token tile
])
def test_gemm_wide_token_tiles_vs_oracle(M, N, K, path, splits, m_tile):
    # Tiles of more than 128 tokens (M > 512 by default, or forced): two 128-row scale chunks per
    # token block, and two MMA issuers, the first taking tokens 0..127 of every step, the second
    # the rest, into one accumulator; ragged last tiles
    mx = _mx()
    plan = mx.mxfp4_gemm_plan(M, N, K, path, splits, m_tile)
    assert plan["m_tile"] == (m_tile or 256) and plan["issuers"] == 2, plan
    assert plan["scale_stores"] == (1 if path == 2 else 0), plan
    assert plan["tmem_cols"] >= plan["m_tile"] + 32 * plan["stages"], plan
    a = workloads.random_bf16(M, K, seed=M + K + 256)
    b = workloads.random_bf16(N, K, seed=N + K + 256, scale=0.5)
    bq, bs = mx.mxfp4_quantize(b.cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    c = mx.mxfp4_gemm(a.cuda(), packed, N, path=path, splits=splits, m_tile=m_tile)
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status() == 0
    ref = oracle_c(a, to_np_u8(bq), to_np_u8(bs))
    check_tolerance(bf16_to_f64(c.cpu()), ref, f"{M}x{N}x{K} path {path} splits {splits} m_tile {plan['m_tile']}")


@pytest.mark.parametrize("M,K,path,splits", [(8, 512, 1, 1), (16, 1536, 1, 3), (5, 1280, 1, 2), (13, 2048, 1, 4),
                                              (40, 768, 2, 1), (8, 1024, 2, 2), (8, 520, 1, 1), (13, 2056, 1, 4),
                                              (40, 776, 2, 1), (3, 72, 1, 1)])
def test_quantized_a_read_back_through_one_hot_b(M, K, path, splits):
    # With B one-hot (B[n, n] = 1, all else 0: exactly representable, so its quantization is the
    # identity), C[m, n] is dequant(quantized A)[m, n] exactly: C shows the codes and scales the
    # call's own A quantization produced -- inside the GEMM on the fused path -- and must equal the
    # oracle's bit for bit, not just within the GEMM tolerance.
    N = K
    a = workloads.random_bf16(M, K, seed=M * 13 + K)
    b = torch.zeros(N, K, dtype=torch.bfloat16)
    idx = torch.arange(N)
    b[idx, idx] = 1.0
    c, bq, bs = run_gemm(a, b, path=path, splits=splits)
    aq, as_ = oracle.quantize(workloads.bf16_bits(a))
    want = oracle.bf16_to_f64(oracle.to_bf16(oracle.mxfp4_gemm_ref(aq, as_, bq, bs)))
    assert np.array_equal(want, oracle.dequantize(aq, as_)[:, :K]), "one-hot B must read A back"
    bad = np.argwhere(c != want)
    assert bad.size == 0, f"{len(bad)} entries differ, first at {tuple(bad[0])}: got {c[tuple(bad[0])]!r} want {want[tuple(bad[0])]!r}"


@pytest.mark.parametrize("M,N,K", [(8, 2112, 7168), (5, 300, 520), (64, 1024, 2048), (300, 384, 1536)])
def test_unpacked_gemm_matches_prepacked(M, N, K):
    # B as the quantizer writes it, prepacked inside the call: the prepacked call's bits, and
    # back-to-back calls with different weights on one workspace each see their own weights
    mx = _mx()
    a = workloads.random_bf16(M, K, seed=M + 17).cuda()
    outs = []
    for seed in (1, 2):
        bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=N + seed).cuda())
        want = mx.mxfp4_gemm(a, mx.mxfp4_prepack_b(bq, bs), N)
        outs.append((bq, bs, want))
    ws = None
    for bq, bs, want in outs + outs:        # alternate the weights on the same stream and workspace
        c = mx.mxfp4_gemm_unpacked(a, bq, bs, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(c.view(torch.int16), want.view(torch.int16))
    assert mx.mxfp4_device_status() == 0
    L = mx.load_library()
    need = L.mxfp4_gemm_unpacked_workspace_size(M, N, K)
    assert need >= mx.mxfp4_prepack_b_size(N, K) + mx.mxfp4_gemm_workspace_size(M, N, K)
    raw = torch.empty(need + 1024, dtype=torch.uint8, device="cuda")
    small = raw[(-raw.data_ptr()) % 1024:][:mx.mxfp4_prepack_b_size(N, K) - 1]
    with pytest.raises(ValueError):   # the binding refuses a workspace below the size query
        mx.mxfp4_gemm_unpacked(a, outs[0][0], outs[0][1], workspace=small)
