"""Layout helpers shared by the host planner and the kernels (csrc/internal.h), checked on the CPU
against the layouts they are documented to produce:
- the 128-byte swizzle of a weight or token tile places every 16-byte chunk of every row exactly
  once inside its own row, and eight consecutive rows reading one chunk column hit eight distinct
  16-byte bank groups;
- the scale-factor offsets fill the tile's scale chunks exactly once, one byte per (row, block);
- the split-K receive stride and the staged-A pitch put consecutive rows in distinct bank groups;
- the receive buffer holds every source's run of rows.
A wrong helper would still pass on shapes the GPU tests happen to cover."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_scaled_mxfp4_bf16_gb300", "csrc")
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

HARNESS = r"""
#include <cstdio>
#include <vector>
#include "internal.h"
using namespace mxfp4;

int main() {
    long bad_swz = 0, bad_bank = 0, bad_sf = 0, bad_red = 0, bad_pitch = 0;
    // swizzle: a permutation of the 128 x 128-byte tile, each chunk inside its own row
    std::vector<int> seen(kTileN * 128 / 16, 0);
    for (uint32_t r = 0; r < 128; ++r)
        for (uint32_t c = 0; c < 8; ++c) {
            const uint32_t off = swz_chunk_offset(r, c);
            if (off % 16 != 0 || off / 128 != r) ++bad_swz;
            else ++seen[off / 16];
        }
    for (int v : seen) if (v != 1) ++bad_swz;
    // eight consecutive rows, one chunk column: eight distinct 16-byte groups of the 128-byte bank line
    for (uint32_t r0 = 0; r0 < 128; r0 += 8)
        for (uint32_t c = 0; c < 8; ++c) {
            int group[8] = {0};
            for (uint32_t r = r0; r < r0 + 8; ++r) ++group[(swz_chunk_offset(r, c) % 128) / 16];
            for (int g : group) if (g != 1) ++bad_bank;
        }
    // scale offsets: for nmc 128-row groups, each of the 2 * nmc 512-byte chunks filled exactly once
    for (uint32_t nmc = 1; nmc <= 2; ++nmc) {
        std::vector<int> sf(2 * nmc * kSfChunk, 0);
        for (uint32_t r = 0; r < 128 * nmc; ++r)
            for (uint32_t kb = 0; kb < 8; ++kb) {
                const uint32_t off = block_sf_offset(r, kb);
                if (off >= sf.size()) ++bad_sf;
                else ++sf[off];
            }
        for (int v : sf) if (v != 1) ++bad_sf;
    }
    // split-K receive rows: stride covers the run, is an odd number of 16-byte units, and eight
    // consecutive weight rows n land in distinct 16-byte bank groups
    for (int m_valid = 1; m_valid <= 256; ++m_valid)
        for (int splits = 2; splits <= kMaxSplits; ++splits) {
            const int rp = red_rows_per(m_valid, splits);
            if (rp % 4 != 0 || rp * splits < m_valid || (rp - 4) * splits >= m_valid + 3 * splits) ++bad_red;
            if (rp > kRedVecMaxRows) continue;
            const int st = red_stride(rp);
            if (st < rp || st % 4 != 0 || (st / 4) % 2 != 1) ++bad_red;
            int group[8] = {0};
            for (int n = 0; n < 8; ++n) ++group[(n * st * 4 % 128) / 16];
            for (int g : group) if (g != 1) ++bad_red;
            if (red_recv_floats(rp, splits) < static_cast<size_t>(splits) * 128 * rp) ++bad_red;
        }
    // staged bf16 A rows: pitch = atoms * 512 + 16 bytes, so consecutive rows sit one group apart
    for (int atoms = 1; atoms <= 64; ++atoms) {
        const uint32_t pitch = raw_pitch(atoms);
        if (pitch % 128 != 16 || pitch < static_cast<uint32_t>(atoms) * kAtomK * 2) ++bad_pitch;
    }
    std::printf("%ld %ld %ld %ld %ld\n", bad_swz, bad_bank, bad_sf, bad_red, bad_pitch);
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")),
                    reason="needs g++ and the CUDA headers")
def test_layout_helpers(tmp_path):
    src = tmp_path / "layout.cpp"
    src.write_text(HARNESS)
    exe = tmp_path / "layout"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, "-I", CUDA_INC, "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout.split()
    names = ("swizzle placement", "swizzle bank groups", "scale offsets", "split-K receive rows", "A row pitch")
    assert dict(zip(names, map(int, out))) == dict.fromkeys(names, 0)
