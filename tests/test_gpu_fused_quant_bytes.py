"""The A quantization that the GEMM performs inside its own kernel (the weight-resident path and
the fused path), byte for byte against the oracle: codes, scale bytes and the sign of zero codes
(0x8 for -0.0 and for negative values that round to zero), which a product read back through C
cannot show. A test build of the library (-DMXFP4_TEST_HOOKS, its own .so; the product library
has no such hook) makes the CTAs of weight tile 0 copy the token blocks they quantized to a
buffer; the rest of the call runs as in the product build."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads
from mxfp4_testlib import to_np_u8

pytestmark = pytest.mark.gpu


class _Opts(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("splits", ctypes.c_int), ("m_tile", ctypes.c_int),
                ("reserved", ctypes.c_int * 5)]


@pytest.fixture(scope="module")
def hooks():
    from block_scaled_mxfp4_bf16_gb300 import build
    L = ctypes.CDLL(build.build_variant("hooks", ["-DMXFP4_TEST_HOOKS"]))
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    L.mxfp4_test_token_dump.argtypes = [vp]
    L.mxfp4_test_token_dump.restype = None
    L.mxfp4_gemm_ex.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, ctypes.c_size_t, ctypes.POINTER(_Opts), vp]
    L.mxfp4_gemm_ex.restype = ctypes.c_int
    L.mxfp4_device_status.argtypes = [vp]
    L.mxfp4_device_status.restype = ctypes.c_int
    return L


def _expected(rq: np.ndarray, rs: np.ndarray, M: int, K: int, m_tile: int):
    """The oracle's bytes in the token-block layout the MMAs read: per (token tile, 256-K step)
    the tile's rows (row r at r*128, its eight 16-byte chunks at (c ^ r%8)*16), then two 512-byte
    scale chunks (row r at (r%32)*16 + block%4 for these tiles of at most 32 rows). Only the rows
    of real tokens are defined (the kernels leave the padding rows of a tile alone); K past the
    end is zero."""
    a_block = m_tile * 128 + 1024
    m_tiles, k_atoms, nblk = -(-M // m_tile), -(-K // 256), (K + 31) // 32
    out = np.zeros((m_tiles, k_atoms, a_block), dtype=np.uint8)
    defined = np.zeros_like(out, dtype=bool)
    for mt in range(m_tiles):
        for r in range(min(m_tile, M - mt * m_tile)):
            row = mt * m_tile + r
            for j in range(k_atoms):
                for c in range(8):
                    kb = j * 8 + c
                    off = r * 128 + (c ^ (r % 8)) * 16
                    sf = m_tile * 128 + (c >> 2) * 512 + (r % 32) * 16 + (c & 3)
                    defined[mt, j, off:off + 16] = True
                    defined[mt, j, sf] = True
                    if kb < nblk:
                        out[mt, j, off:off + 16] = rq[row, kb * 16:kb * 16 + 16]
                        out[mt, j, sf] = rs[row, kb]
    return out.reshape(-1), defined.reshape(-1)


def _signed_zero_a(M: int, K: int, seed: int) -> torch.Tensor:
    """Seeded normal A with blocks that exercise the sign of zero: a block of -0.0 only, a block
    mixing +0.0, -0.0 and negative values far below the block's scale, and a block of tiny
    negative values only."""
    a = workloads.random_bf16(M, K, seed=seed).float()
    nb = (K + 31) // 32
    a[0, 0:32] = -0.0
    if M > 1 and nb > 1:
        blk = a[1, 32:64]
        blk[0::4] = 0.0
        blk[1::4] = -0.0
        blk[2::4] = -1e-6
    if M > 2:
        a[M - 1, 0:min(32, K)] = -1e-30
    return a.to(torch.bfloat16)


@pytest.mark.parametrize("M,N,K,path,splits,m_tile", [
    (8, 2112, 7168, 3, 0, 0),        # the benchmark's weight-streaming shape, automatic plan
    (16, 384, 1536, 3, 3, 16),
    (8, 256, 2048, 3, 1, 16),        # eight steps: three MMA-issuing warps, one of them a quantizer
    (32, 256, 512, 3, 1, 16),        # two 16-token tiles
    (24, 300, 2072, 3, 4, 32),       # a 32-token tile with 24 tokens; K cuts the last step
    (5, 200, 520, 3, 2, 16),         # K cuts a 1x32 block
    (1, 128, 8, 3, 1, 16),
    (8, 256, 1536, 1, 3, 16),        # the fused path of the other kernel
    (3, 200, 520, 1, 2, 16),
])
def test_in_kernel_quantization_bytes_match_oracle(hooks, M, N, K, path, splits, m_tile):
    import block_scaled_mxfp4_bf16_gb300 as mx
    a = _signed_zero_a(M, K, seed=M * 13 + K)
    plan = mx.mxfp4_gemm_plan(M, N, K, path, splits, m_tile)
    assert plan["path"] == path
    mt = plan["m_tile"]
    m_tiles, k_atoms = -(-M // mt), -(-K // 256)
    dump = torch.full((m_tiles * k_atoms * (mt * 128 + 1024),), 0xA5, dtype=torch.uint8, device="cuda")
    bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=3).cuda())
    packed = mx.mxfp4_prepack_b(bq, bs)
    a_dev = a.cuda()
    c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    hooks.mxfp4_test_token_dump(dump.data_ptr())
    try:
        opts = _Opts(path, splits, m_tile)
        st = hooks.mxfp4_gemm_ex(a_dev.data_ptr(), M, K, K, packed.data_ptr(), N, c.data_ptr(), N, None, 0,
                                 ctypes.byref(opts), torch.cuda.current_stream().cuda_stream)
        assert st == 0, st
        torch.cuda.synchronize()
        assert hooks.mxfp4_device_status(torch.cuda.current_stream().cuda_stream) == 0
    finally:
        hooks.mxfp4_test_token_dump(None)
    rq, rs = oracle.quantize(workloads.bf16_bits(a))
    assert rq[0, 0] == 0x88 and rs[0, 0] == 0          # the -0.0 block, as the oracle reads it
    want, defined = _expected(rq, rs, M, K, mt)
    got = to_np_u8(dump)
    bad = np.flatnonzero((got != want) & defined)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[0]}: got {got[bad[0]]:#04x} want {want[bad[0]]:#04x}"
    # and the product of that call is the product's: the hook only copies
    want_c = mx.mxfp4_gemm(a_dev, packed, N, path=path, splits=splits, m_tile=m_tile)
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16), want_c.view(torch.int16))
