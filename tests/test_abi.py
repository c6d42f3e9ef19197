"""CPU-only checks of the boundary: the library builds for sm_103a, loads without a GPU and
exports every function include/mxfp4_gb300.h declares; pure host helpers answer correctly."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp4_gb300.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from block_scaled_mxfp4_bf16_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_three_calls():
    names = _declared_functions()
    for required in ("mxfp4_quantize", "mxfp4_prepack_b", "mxfp4_gemm"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.mxfp4_status_string.restype = ctypes.c_char_p
    assert lib.mxfp4_status_string(0) == b"MXFP4_OK"
    assert lib.mxfp4_status_string(6) == b"MXFP4_ERR_TIMEOUT"
    assert lib.mxfp4_version() >= 100


def test_prepack_size_is_pure_host_arithmetic(lib):
    lib.mxfp4_prepack_b_size.restype = ctypes.c_size_t
    lib.mxfp4_prepack_b_size.argtypes = [ctypes.c_int64, ctypes.c_int64]
    # one 17408-byte block (16 KB of swizzled e2m1 rows + 1 KB of scales) per 128-row tile
    # and 256-element K step
    assert lib.mxfp4_prepack_b_size(2112, 7168) == 17 * 28 * 17408
    assert lib.mxfp4_prepack_b_size(100, 64) == 1 * 1 * 17408
    assert lib.mxfp4_prepack_b_size(100, 96) == 1 * 1 * 17408   # K tails are zero padding
    assert lib.mxfp4_prepack_b_size(100, 8) == 1 * 1 * 17408
    assert lib.mxfp4_prepack_b_size(100, 100) == 0    # K must be a multiple of 8
    assert lib.mxfp4_prepack_b_size(0, 64) == 0
    # the GEMM's size limits: N below 2^31, K at most 2^30
    assert lib.mxfp4_prepack_b_size(128, 1 << 30) == (1 << 30) // 256 * 17408
    assert lib.mxfp4_prepack_b_size(128, (1 << 30) + 8) == 0
    assert lib.mxfp4_prepack_b_size((1 << 31) - 1, 256) == (1 << 24) * 17408
    assert lib.mxfp4_prepack_b_size(1 << 31, 256) == 0


def test_no_cpu_fallback_when_cuda_missing(lib):
    # without a GPU every compute entry point must refuse, not compute on the host
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib.mxfp4_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    buf = ctypes.create_string_buffer(256)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert lib.mxfp4_quantize(p, 1, 32, 32, p, p, None) != 0
    # the host-buffer GEMM refuses too (no device to plan for), before touching any buffer
    big = ctypes.create_string_buffer(8192)
    q = ctypes.addressof(big) + (-ctypes.addressof(big)) % 1024
    lib.mxfp4_gemm_host.restype = ctypes.c_int
    lib.mxfp4_gemm_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.c_void_p]
    before = big.raw
    assert lib.mxfp4_gemm_host(q, 1, 64, 64, q, 16, q + 2048, 16, q + 4096, q + 6144, None, 0, None) != 0
    assert big.raw == before


def test_plan_info_layout_and_null_check(lib):
    # the binding's struct mirrors mxfp4_plan_info: ten ints and six reserved (64 bytes)
    import block_scaled_mxfp4_bf16_gb300 as mx
    assert ctypes.sizeof(mx._PlanInfo) == 64
    lib.mxfp4_gemm_plan_info.restype = ctypes.c_int
    lib.mxfp4_gemm_plan_info.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p]
    assert lib.mxfp4_gemm_plan_info(8, 2112, 7168, None, None) == 1      # MXFP4_ERR_ARG, no device needed



def test_prepared_call_null_checks(lib):
    # a prepared call's entry points refuse a missing handle or output slot before touching a
    # device, and destroying no handle is a no-op
    vp = ctypes.c_void_p
    lib.mxfp4_call_run.argtypes = [vp, vp]
    lib.mxfp4_call_run.restype = ctypes.c_int
    lib.mxfp4_call_destroy.argtypes = [vp]
    lib.mxfp4_call_destroy.restype = None
    i64, sz = ctypes.c_int64, ctypes.c_size_t
    lib.mxfp4_call_create.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, sz, vp, vp]
    lib.mxfp4_call_create.restype = ctypes.c_int
    lib.mxfp4_call_create_host.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, vp, vp, sz, ctypes.c_uint, vp]
    lib.mxfp4_call_create_host.restype = ctypes.c_int
    assert lib.mxfp4_call_run(None, None) == 1          # MXFP4_ERR_ARG
    lib.mxfp4_call_destroy(None)
    assert lib.mxfp4_call_create(None, 8, 512, 512, None, 256, None, 256, None, 0, None, None) == 1
    assert lib.mxfp4_call_create_host(None, 8, 512, 512, None, 256, None, 256, None, None, None, 0, 0, None) == 1
    out = vp(1234)
    # a null A is refused by the argument checks and leaves no handle behind
    assert lib.mxfp4_call_create(None, 8, 512, 512, None, 256, None, 256, None, 0, None, ctypes.byref(out)) == 1
    assert out.value is None


def test_gemm_options_flags_are_checked_first(lib):
    # mxfp4_gemm_options is {path, splits, m_tile, flags, reserved[4]}; a flag bit other than
    # MXFP4_GEMM_A_READY is an argument error found before any device query, while the known
    # bit passes the argument checks (and the call then fails only for want of a device)
    import torch
    import block_scaled_mxfp4_bf16_gb300 as mx
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert ctypes.sizeof(mx._Options) == 32 and mx._Options.flags.offset == 12
    assert "#define MXFP4_GEMM_A_READY 1" in open(HEADER).read() and mx.GEMM_A_READY == 1
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.mxfp4_gemm_ex.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, ctypes.c_size_t, vp, vp]
    lib.mxfp4_gemm_ex.restype = ctypes.c_int
    big = ctypes.create_string_buffer(8192)
    q = ctypes.addressof(big) + (-ctypes.addressof(big)) % 1024
    before = big.raw
    for flags, refused in ((2, True), (1 << 30, True), (3, True), (1, False), (0, False)):
        opts = mx._Options(0, 0, 0, flags)
        st = lib.mxfp4_gemm_ex(q, 1, 64, 64, q, 16, q + 2048, 16, q + 4096, 4096, ctypes.byref(opts), None)
        assert (st == 1) == refused, (flags, st)
        assert st != 0
    assert big.raw == before
