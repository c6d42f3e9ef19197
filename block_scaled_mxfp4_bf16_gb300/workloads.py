"""Seeded synthetic workloads for the MXFP4 GEMM (shared by the tests and the benchmark).

This module only draws random inputs; it holds none of the quantizer's or the GEMM's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs from it.

Recipe (after the input generator quoted in amd-mxfp4-mm submission 608632, the
``_new_generate_input`` it removes: one seeded generator, A then B, bf16 normal; the public
leaderboard harness itself is not available, so these stand in for its inputs):
  * ``g = torch.Generator("cpu").manual_seed(seed)`` -- a CPU generator, so the host
    oracle and the GPU see identical bytes;
  * ``A = randn(M, K)`` then ``B = sigma_B * randn(N, K)`` in fp32, each cast to bf16;
  * outlier workload (M=32, N=4096, K=512): after B, ``perm = randperm(M*K/32)``; the
    first 5% of A's 1x32 blocks (floor) are multiplied by 1e3 and the next 5% are set to
    +0.0, in fp32 before the bf16 cast, to hit saturating and zero-scale blocks.
"""
from __future__ import annotations

import re
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    b_sigma: float = 1.0
    outlier_blocks: bool = False

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """A bf16 read + B e2m1 read + B e8m0 read + C bf16 write, each once."""
        return 2 * self.M * self.K + self.N * self.K // 2 + self.N * self.K // 32 + 2 * self.M * self.N


# The five shapes the method is measured on (weight-streaming decode to compute-bound).
WORKLOADS = [
    Workload("M16_N3072_K1536", 16, 3072, 1536),
    Workload("M8_N2112_K7168", 8, 2112, 7168),
    Workload("M32_N4096_K512", 32, 4096, 512, outlier_blocks=True),
    Workload("M64_N7168_K2048", 64, 7168, 2048, b_sigma=0.02),
    Workload("M256_N4096_K7168", 256, 4096, 7168),
]

# More shapes from the pages' leaderboard list (N tails, M=4) for parity coverage.
EXTRA_WORKLOADS = [
    Workload("M4_N2880_K512", 4, 2880, 512),
    Workload("M32_N2880_K512", 32, 2880, 512),
    Workload("M16_N2112_K7168", 16, 2112, 7168),
    Workload("M256_N3072_K1536", 256, 3072, 1536),
]


def by_name(name: str) -> Workload:
    """A listed workload by name, else any shape named ``M<m>_N<n>_K<k>`` (B with sigma 1, no
    outlier blocks), e.g. a large token count to time the compute-bound regime."""
    for w in WORKLOADS + EXTRA_WORKLOADS:
        if w.name == name:
            return w
    m = re.fullmatch(r"M(\d+)_N(\d+)_K(\d+)", name)
    if m is None or min(int(v) for v in m.groups()) < 1:
        raise KeyError(name)
    return Workload(name, int(m.group(1)), int(m.group(2)), int(m.group(3)))


def make_inputs(w: Workload, seed: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
    """(A bf16 [M,K], B bf16 [N,K]) on the CPU, drawn as described in the module docstring."""
    g = torch.Generator("cpu").manual_seed(seed)
    a = torch.randn(w.M, w.K, generator=g, dtype=torch.float32)
    b = torch.randn(w.N, w.K, generator=g, dtype=torch.float32) * w.b_sigma
    if w.outlier_blocks:
        nblk = w.M * w.K // 32
        n5 = nblk * 5 // 100
        perm = torch.randperm(nblk, generator=g)
        blocks = a.view(nblk, 32)
        blocks[perm[:n5]] *= 1e3
        blocks[perm[n5:2 * n5]] = 0.0
    return a.to(torch.bfloat16), b.to(torch.bfloat16)


def random_bf16(rows: int, cols: int, seed: int, scale: float = 1.0) -> torch.Tensor:
    """Plain seeded normal bf16 matrix (CPU) for small parity cases."""
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(rows, cols, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (a view of the same bytes, copied to host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
