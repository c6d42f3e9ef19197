// Descriptors of the tcgen05 block-scaled MMA (kind::mxf4) as the GEMM kernels use it: 128-byte
// swizzled operand rows in shared memory, scale factors copied into tensor memory, fp32
// accumulators, bf16 output packing.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

// Operand rows of 128 bytes, 128-byte swizzle, 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) { return smem_desc(addr, 16, 1024, 2); }
// A 512-byte scale-factor chunk (32 rows of 16 bytes) for tcgen05.cp 32x128b.warpx4.
__device__ __forceinline__ uint64_t desc_sf(uint32_t addr) { return smem_desc(addr, 0, 128, 0); }

// Instruction descriptor, kind::mxf4: e2m1 x e2m1, both K-major, UE8M0 scales, M = 128.
__device__ __forceinline__ uint32_t idesc_mxf4(uint32_t n_mma) {
    return (1u << 7)                        // A format: e2m1
         | (1u << 10)                       // B format: e2m1
         | ((n_mma >> 3) << 17)             // N / 8
         | (1u << 23)                       // scale factor type UE8M0
         | ((uint32_t(kTileN) >> 4) << 24); // M / 16
}

// Two fp32 -> two bf16 (round to nearest even) in one word, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace mxfp4
