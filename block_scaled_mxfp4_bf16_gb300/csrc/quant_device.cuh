// Device-side MXFP4 block quantizer: 32 bf16 values -> 16 packed e2m1 bytes + 1 e8m0 byte.
//
// The arithmetic is the one submission 711914 of the amd-mxfp4-mm leaderboard spells out in
// `_mxfp4_quant_tile`:
//   amax   = max |x| over the block (fp32);
//   amax_r = bits(amax) + 0x200000, mantissa cleared  (power of two, rounding up from 1.75);
//   s      = clamp(floor(log2(amax_r)) - 2, -127, 127), stored as s + 127;
//   code   = e2m1(x * 2^-s): nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to even,
//            saturating at 6, sign in bit 3 even when the magnitude rounds to 0;
//   byte   = code(even element) | code(odd element) << 4.
// Here amax is a depth-4 tree of max.xorsign.abs.bf16x2 over the block's bf16 pairs (the
// magnitude of the larger |x|, exactly; inputs are finite by contract), floor(log2) is read off
// the exponent field, the scaling is one fp32 multiply per element (exact for a power of two)
// and the element rounding uses the sm_100+ conversion cvt.rn.satfinite.e2m1x2.f32. (Measured
// against a chain of integer maxima, and against f32x2 multiplies with prmt packing: the tree
// with scalar multiplies was the fastest inside the fused GEMM and the quantize kernels.)
#pragma once
#include <cstdint>

namespace mxfp4 {

// Unbiased scale exponent s from the fp32 bit pattern of the block's max |x|.
__device__ __forceinline__ int scale_exponent(uint32_t amax_bits) {
    const uint32_t r = (amax_bits + 0x200000u) & 0xFF800000u;
    if (r == 0u) return -127;              // log2(0) = -inf, clamped
    if (r >= 0x7F800000u) return 127;      // rounded up to +inf, clamped
    const int e = static_cast<int>(r >> 23) - 127 - 2;
    return e < -127 ? -127 : e;            // e <= 125 here
}

// 2^-s as an fp32 (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float inv_scale(int s) {
    const uint32_t bits = (s == 127) ? 0x00400000u : static_cast<uint32_t>(127 - s) << 23;
    return __uint_as_float(bits);
}

// Two scaled fp32 values -> one byte: `lo` in bits 0..3, `hi` in bits 4..7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
#ifndef MXFP4_SOFTWARE_ENCODE
    uint16_t r;
    // the first source operand lands in the upper nibble, the second in the lower
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r;
#else
    // Threshold count: the code is the number of grid midpoints below |v|, where a value
    // sitting exactly on a midpoint moves up only if that lands on an even code.
    auto enc = [](float v) -> uint32_t {
        const float a = fabsf(v);
        uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
        return c | ((__float_as_uint(v) >> 28) & 8u);
    };
    return enc(lo) | (enc(hi) << 4);
#endif
}

// max(|a|, |b|) per bf16 half (the sign bit of each half is junk: mask it off).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Codes of 8 elements (4 words) scaled by m: 4 bytes, element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t encode_words4(const uint32_t* w, float m) {
    uint32_t packed = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float even = __fmul_rn(__uint_as_float(w[i] << 16), m);
        const float odd = __fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), m);
        packed |= e2m1x2(even, odd) << (8 * i);
    }
    return packed;
}

// Quantize one 1x32 block held as 16 words of bf16 pairs (element 2i in the low half of
// word i). Writes 4 words of packed codes (element 2i in the low nibble of its byte) and
// returns the e8m0 byte.
__device__ __forceinline__ uint32_t quantize_block32(const uint32_t (&w)[16], uint32_t (&out)[4]) {
    uint32_t m8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = absmax_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) m8[i] = absmax_bf16x2(m8[2 * i], m8[2 * i + 1]);
    const uint32_t mx = absmax_bf16x2(absmax_bf16x2(m8[0], m8[1]), absmax_bf16x2(m8[2], m8[3]));
    const uint32_t amax_bits = max(mx & 0x7FFFu, (mx >> 16) & 0x7FFFu) << 16;
    const int s = scale_exponent(amax_bits);
    const float m = inv_scale(s);
#pragma unroll
    for (int j = 0; j < 4; ++j) out[j] = encode_words4(&w[4 * j], m);
    return static_cast<uint32_t>(s + 127);
}

// A quarter of a 1x32 block: 8 bf16 as 4 words, quantized with the block's scale multiplier m
// (inv_scale of the block's exponent); returns 4 bytes of packed codes (element 2i in the low
// nibble of byte i). Same arithmetic per element as quantize_block32.
__device__ __forceinline__ uint32_t quantize_quarter(const uint32_t (&w)[4], float m) {
    return encode_words4(w, m);
}

// Max |x| bit pattern (as a bf16 in the low half) over 4 words of bf16 pairs.
__device__ __forceinline__ uint32_t amax_quarter(const uint32_t (&w)[4]) {
    const uint32_t m = absmax_bf16x2(absmax_bf16x2(w[0], w[1]), absmax_bf16x2(w[2], w[3]));
    return max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
}

// Load 32 consecutive bf16 (64 bytes, 16-byte aligned) as 16 words.
__device__ __forceinline__ void load_block32(const uint16_t* src, uint32_t (&w)[16]) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(p + i);
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
}

// The block starting at src when only `avail` elements remain in the row (avail > 0, a
// multiple of 8): the 16-byte pieces at or past the row's end are not read and count as zeros.
__device__ __forceinline__ void load_block32_upto(const uint16_t* src, int64_t avail, uint32_t (&w)[16]) {
    if (avail >= 32) {
        load_block32(src, w);
        return;
    }
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = 8 * i < avail ? __ldg(p + i) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
}

}  // namespace mxfp4
