"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI binding and the
CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_scaled_mxfp4_bf16_gb300 import workloads

REL_TOL = 8e-3       # |C - C_ref| <= REL_TOL * |C_ref| + RMS_TOL * rms(C_ref)
RMS_TOL = 1e-3


def gpu_available() -> bool:
    return torch.cuda.is_available()


def to_np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_to_f64(workloads.bf16_bits(t))


def quantize_both(x_cpu: torch.Tensor):
    """(gpu_q, gpu_s, ref_q, ref_s) for a CPU bf16 matrix."""
    import block_scaled_mxfp4_bf16_gb300 as mx
    q, s = mx.mxfp4_quantize(x_cpu.cuda())
    rq, rs = oracle.quantize(workloads.bf16_bits(x_cpu))
    torch.cuda.synchronize()
    return to_np_u8(q), to_np_u8(s), rq, rs


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str) -> None:
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        r, c = bad[0]
        raise AssertionError(f"{what}: {len(bad)} mismatching bytes, first at {tuple(bad[0])}: "
                             f"got {got[r, c]:#04x} want {want[r, c]:#04x}")


def check_tolerance(c: np.ndarray, c_ref: np.ndarray, what: str) -> float:
    ok, worst = oracle.tolerance_ok(c, c_ref, REL_TOL, RMS_TOL)
    if not ok:
        err = np.abs(c - c_ref)
        i = np.unravel_index(np.argmax(err - REL_TOL * np.abs(c_ref)), c.shape)
        raise AssertionError(f"{what}: tolerance exceeded (worst ratio {worst:.3g}); at {i}: "
                             f"got {c[i]!r} want {c_ref[i]!r}")
    return worst


def run_gemm(a_cpu: torch.Tensor, b_cpu: torch.Tensor, path: int = 0, splits: int = 0, lda_pad: int = 0,
             ldc_pad: int = 0, canary: float = 777.0, m_tile: int = 0, also_a_ready: bool = False):
    """Quantize B and prepack it on the GPU, run mxfp4_gemm, check the B bytes against the
    oracle and that nothing outside C[:M,:N] was written. Returns (C as fp64 [M,N], Bq, Bs).
    also_a_ready: run the call again with A declared ready (its predecessor began after A was
    written) into a second canaried C, which must hold the bits of a flagless call on the plan
    the flag selects (the automatic plan may differ with it)."""
    import block_scaled_mxfp4_bf16_gb300 as mx
    M, K = a_cpu.shape
    N = b_cpu.shape[0]
    b = b_cpu.cuda()
    bq, bs = mx.mxfp4_quantize(b)
    packed = mx.mxfp4_prepack_b(bq, bs)
    # the row padding past K holds huge values: reading any of it would show in C
    a_store = torch.full((M, K + lda_pad), 1.0e30, dtype=torch.bfloat16, device="cuda")
    a_store[:, :K] = a_cpu.cuda()
    a = a_store[:, :K]
    c_store = torch.full((M + 1, N + ldc_pad), canary, dtype=torch.bfloat16, device="cuda")
    c = c_store[:M, :N]
    mx.mxfp4_gemm(a, packed, N, c=c, path=path, splits=splits, m_tile=m_tile)
    torch.cuda.synchronize()
    st = mx.mxfp4_device_status()
    assert st == 0, f"device status {st}"
    outside = torch.ones_like(c_store, dtype=torch.bool)
    outside[:M, :N] = False
    assert bool((c_store[outside] == canary).all()), "GEMM wrote outside C"
    if also_a_ready:
        rp = mx.mxfp4_gemm_plan(M, N, K, path, splits, m_tile, a_ready=True)
        c2_store = torch.full_like(c_store, canary)
        c3_store = torch.full_like(c_store, canary)
        c2, c3 = c2_store[:M, :N], c3_store[:M, :N]
        mx.mxfp4_gemm(a, packed, N, c=c3, path=rp["path"], splits=rp["splits"], m_tile=rp["m_tile"])
        mx.mxfp4_gemm(a, packed, N, c=c2, path=path, splits=splits, m_tile=m_tile, a_ready=True)
        torch.cuda.synchronize()
        assert mx.mxfp4_device_status() == 0
        assert bool((c2_store[outside] == canary).all()), "GEMM with A declared ready wrote outside C"
        assert torch.equal(c2.view(torch.int16), c3.view(torch.int16)), "A declared ready changed C"
    return bf16_to_f64(c.cpu()), to_np_u8(bq), to_np_u8(bs)


def oracle_c(a_cpu: torch.Tensor, bq: np.ndarray, bs: np.ndarray) -> np.ndarray:
    aq, as_ = oracle.quantize(workloads.bf16_bits(a_cpu))
    return oracle.mxfp4_gemm_ref(aq, as_, bq, bs)


# One case per split-K form the planner can pick (mxfp4_plan_info.reduction: 1 posted rows,
# 2 st.async short runs, 3 bulk copies), with and without a dedicated receive buffer, for
# both paths; the expected form is asserted so a planner change cannot silently drop one.
REDUCTION_CASES = [
    # M, N, K, path, splits, (reduction, recv_dedicated)
    (100, 200, 512, 1, 2, (1, 0)),
    (100, 200, 768, 2, 2, (1, 0)),
    (64, 200, 512, 2, 2, (1, 1)),
    (1, 200, 4096, 1, 12, (2, 0)),
    (5, 200, 4096, 2, 12, (2, 0)),
    (1, 200, 512, 1, 2, (2, 1)),
    (7, 200, 512, 2, 2, (2, 1)),
    (33, 200, 4096, 1, 2, (3, 0)),
    (33, 200, 2048, 2, 2, (3, 0)),
    (33, 200, 512, 1, 2, (3, 1)),
    (40, 200, 512, 2, 2, (3, 1)),
]


def expected_token_blocks(rq: np.ndarray, rs: np.ndarray, M: int, K: int, m_tile: int):
    """Token blocks (the two-kernel path's workspace, mxfp4_quantize_tokens' output) laid out
    from the oracle's bytes: per (token tile, 256-K step) a block of the tile's rows (row r at
    r*128, its eight 16-byte chunks at (c ^ r%8)*16), then per 128 rows two 512-byte scale
    chunks (row r at (r%32)*16 + ((r/32)%4)*4 + block%4).
    Rows past M and K past the end are zero. Returns (bytes, mask of the defined bytes): the
    scale slots of rows past the tile (a tile of < 128 rows) are not part of the layout."""
    nmc = (m_tile + 127) // 128
    a_block = m_tile * 128 + nmc * 1024
    m_tiles = -(-M // m_tile)
    k_atoms = -(-K // 256)
    out = np.zeros((m_tiles, k_atoms, a_block), dtype=np.uint8)
    defined = np.zeros((m_tiles, k_atoms, a_block), dtype=bool)
    nblk = (K + 31) // 32
    for mt in range(m_tiles):
        for r in range(m_tile):
            row = mt * m_tile + r
            for j in range(k_atoms):
                defined[mt, j, r * 128:(r + 1) * 128] = True
                for c in range(8):
                    sf = m_tile * 128 + ((r >> 7) * 2 + (c >> 2)) * 512 + (r % 32) * 16 + ((r >> 5) & 3) * 4 + (c & 3)
                    defined[mt, j, sf] = True
                    kb = j * 8 + c
                    if row >= M or kb >= nblk:
                        continue
                    off = r * 128 + ((c ^ (r % 8)) * 16)
                    out[mt, j, off:off + 16] = rq[row, kb * 16:kb * 16 + 16]
                    out[mt, j, sf] = rs[row, kb]
    return out.reshape(-1), defined.reshape(-1)
