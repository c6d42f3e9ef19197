"""mxfp4_gemm_noalloc: the GEMM for callers that cannot allocate device memory (an engine
plugin whose host owns the memory plan, a serving loop that must never call cudaMalloc or
cudaFree because they can synchronize the device). Its scratch is a fixed array inside the
library instead of a caller workspace.

Checked through the C ABI against the regular mxfp4_gemm, within the same tolerance the
parity tests use, on two calls in a row. The array keeps the previous call's contents and
nothing in it is cleared between calls, so the second call of each shape shows that a call
reads only bytes it has written itself; a larger call followed by a smaller one with a
different tile shape shows the same when the stale bytes differ from the new ones. This file
is collected last on purpose; it passes alone in a fresh process as well as after the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_TOL, RMS_TOL = 8e-3, 1e-3
NOALLOC_BYTES = 32 * 1024 * 1024


def _lib():
    import block_scaled_mxfp4_bf16_gb300 as mx
    L = mx.load_library()
    L.mxfp4_gemm_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                     ctypes.c_void_p]
    L.mxfp4_gemm_noalloc.restype = ctypes.c_int
    return mx, L


def _as_f64(c: torch.Tensor) -> np.ndarray:
    return oracle.bf16_to_f64(workloads.bf16_bits(c.cpu()))


@pytest.mark.parametrize("M,N,K", [(8, 2112, 7168), (16, 384, 1536), (64, 1024, 2048), (5, 200, 320)])
def test_noalloc_matches_gemm_twice(M, N, K):
    mx, L = _lib()
    a = workloads.random_bf16(M, K, seed=M + K).cuda()
    b = workloads.random_bf16(N, K, seed=N + K).cuda()
    bq, bs = mx.mxfp4_quantize(b)
    packed = mx.mxfp4_prepack_b(bq, bs)
    want = _as_f64(mx.mxfp4_gemm(a, packed, N))
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        c = torch.full((M, N), 777.0, dtype=torch.bfloat16, device="cuda")
        st = L.mxfp4_gemm_noalloc(a.data_ptr(), M, K, K, packed.data_ptr(), N, c.data_ptr(), N, stream)
        assert st == 0, L.mxfp4_status_string(st)
        torch.cuda.synchronize()
        assert mx.mxfp4_device_status() == 0
        ok, worst = oracle.tolerance_ok(_as_f64(c), want, REL_TOL, RMS_TOL)
        assert ok, f"call {call}: worst ratio {worst:.3g}"


def test_noalloc_python_binding_matches_c_call():
    mx, L = _lib()
    M, N, K = 40, 300, 520                  # two-kernel path (scratch in use), K cut inside a block
    a = workloads.random_bf16(M, K, seed=9).cuda()
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=10).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    c_py = mx.mxfp4_gemm_noalloc(a, packed, N)
    c_c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = L.mxfp4_gemm_noalloc(a.data_ptr(), M, K, K, packed.data_ptr(), N, c_c.data_ptr(), N,
                              torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(c_py.view(torch.int16), c_c.view(torch.int16))
    # same automatic plan, deterministic kernels: bit-identical to the workspace call
    assert torch.equal(c_py.view(torch.int16), mx.mxfp4_gemm(a, packed, N).view(torch.int16))


def test_noalloc_rejects_scratch_beyond_its_limit():
    mx, L = _lib()
    # the two-kernel path keeps the quantized A (M*K/2 bytes) in the scratch: 8192 x 8192
    # needs 32 MiB for it alone, more than the array holds even without split-K
    M, N, K = 8192, 128, 8192
    assert M * K // 2 >= NOALLOC_BYTES
    a = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    packed = mx.mxfp4_prepack_b(torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda"),
                                torch.zeros(N, K // 32, dtype=torch.uint8, device="cuda"))
    c = torch.full((M, N), 777.0, dtype=torch.bfloat16, device="cuda")
    st = L.mxfp4_gemm_noalloc(a.data_ptr(), M, K, K, packed.data_ptr(), N, c.data_ptr(), N,
                              torch.cuda.current_stream().cuda_stream)
    assert st == 7, L.mxfp4_status_string(st)          # MXFP4_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert bool((c == 777.0).all())


def test_noalloc_stale_larger_call_does_not_leak():
    """A large two-kernel call with large-magnitude A leaves its quantized A in the array; a
    smaller two-kernel call with another token tile and K-step count then reuses the same
    bytes. The second result must be bit-identical to mxfp4_gemm with its own workspace."""
    mx, L = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    big = (256, 512, 4096)
    small = (40, 300, 520)
    plans = [mx.mxfp4_gemm_plan(*s) for s in (big, small)]
    assert all(p["path"] == 2 for p in plans)                     # both use the scratch
    assert plans[0]["m_tile"] != plans[1]["m_tile"]
    assert mx.mxfp4_gemm_workspace_size(*big) > mx.mxfp4_gemm_workspace_size(*small)
    outs = []
    for (M, N, K), scale in ((big, 1e3), (small, 1.0)):
        a = workloads.random_bf16(M, K, seed=M + 3, scale=scale).cuda()
        bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=N + 4).cuda())
        packed = mx.mxfp4_prepack_b(bq, bs)
        c = torch.full((M, N), 777.0, dtype=torch.bfloat16, device="cuda")
        st = L.mxfp4_gemm_noalloc(a.data_ptr(), M, K, K, packed.data_ptr(), N, c.data_ptr(), N, stream)
        assert st == 0, L.mxfp4_status_string(st)
        torch.cuda.synchronize()
        assert mx.mxfp4_device_status() == 0
        outs.append((c, mx.mxfp4_gemm(a, packed, N)))
    c_small, want_small = outs[1]
    torch.cuda.synchronize()
    assert torch.equal(c_small.view(torch.int16), want_small.view(torch.int16))
