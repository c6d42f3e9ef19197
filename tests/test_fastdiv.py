"""The exact-division constants the token-block quantizers divide item indices by (make_fastdiv,
host code shared with the kernels): for every divisor 1..2^20 and a random sample up to 2^31,
the round-up multiplier and shifts give n / d exactly at the dividends where a wrong constant
shows first (around multiples of d and at the top of the 32-bit range). The device side is the
three-operation quotient of Granlund and Montgomery, "Division by invariant integers using
multiplication" (1994), restated below on the host."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_scaled_mxfp4_bf16_gb300", "csrc")
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

HARNESS = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "internal.h"

static uint32_t quotient(uint32_t n, const mxfp4::FastDiv& f) {
    const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(f.m) * n) >> 32);
    return (t + ((n - t) >> f.s1)) >> f.s2;
}

static long check(uint32_t d) {
    const mxfp4::FastDiv f = mxfp4::make_fastdiv(d);
    long bad = 0;
    auto one = [&](uint64_t n) {
        if (n > 0xFFFFFFFFull) return;
        if (quotient(static_cast<uint32_t>(n), f) != static_cast<uint32_t>(n / d)) ++bad;
    };
    const uint64_t top = 0xFFFFFFFFull;
    for (uint64_t n = 0; n < 4 * static_cast<uint64_t>(d) + 4 && n < 512; ++n) one(n);
    for (uint64_t k = 1; k < 64; ++k) { one(k * d - 1); one(k * d); one(k * d + 1); }
    const uint64_t kmax = top / d;
    for (uint64_t k = (kmax > 64 ? kmax - 64 : 1); k <= kmax + 1; ++k) { one(k * d - 1); one(k * d); one(k * d + 1); }
    for (uint64_t n = top - 512; n <= top; ++n) one(n);
    return bad;
}

int main() {
    long bad = 0, divisors = 0;
    for (uint32_t d = 1; d <= (1u << 20); ++d, ++divisors) bad += check(d);
    std::mt19937 g(7);
    std::uniform_int_distribution<uint32_t> big(1u << 20, (1u << 31) - 1);
    for (int i = 0; i < 20000; ++i, ++divisors) bad += check(big(g));
    for (uint32_t d : {(1u << 31) - 1, (1u << 30), (1u << 30) + 1, 3u << 29}) { bad += check(d); ++divisors; }
    std::printf("%ld %ld\n", divisors, bad);
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")),
                    reason="needs g++ and the CUDA headers")
def test_fastdiv_constants_divide_exactly(tmp_path):
    src = tmp_path / "fastdiv.cpp"
    src.write_text(HARNESS)
    exe = tmp_path / "fastdiv"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, "-I", CUDA_INC, "-o", str(exe), str(src)], check=True)
    divisors, bad = map(int, subprocess.run([str(exe)], check=True, capture_output=True, text=True,
                                            timeout=600).stdout.split())
    assert divisors == (1 << 20) + 20004
    assert bad == 0
