// Standalone MXFP4 quantizer and the B scale-factor prepack.
//
// quantize_kernel: one thread per (row, group of four 1x32 blocks) = 128 bf16 in, 64 bytes of
// packed e2m1 + 4 scale bytes out, all with 16-byte vector accesses. The scales go either to
// the natural [rows, K/32] layout (public mxfp4_quantize) or straight into the 512-byte
// tensor-core chunks the GEMM copies into tensor memory (two-kernel GEMM path), padding
// included, so the GEMM never reads an unwritten scale byte.
#include "internal.h"
#include "ptx.cuh"
#include "quant_device.cuh"

namespace mxfp4 {

template <bool kChunkLayout>
__global__ void __launch_bounds__(256)
quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ld,
                uint8_t* __restrict__ q, uint8_t* __restrict__ scales,
                int64_t rows_cover, int groups_cover) {
    pdl_launch_dependents();
    pdl_wait_prior_grid();   // x may come from the previous kernel; q/scales may still be read by it
    const int64_t nblk = K / 32;
    const int64_t items = rows_cover * groups_cover;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items; it += stride) {
        const int64_t r = it / groups_cover;
        const int g = static_cast<int>(it - r * groups_cover);
        uint32_t sc = 0u;
        if (r < rows) {
            const uint16_t* xrow = x + r * ld;
            uint8_t* qrow = q + r * (K / 2);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int64_t kb = 4 * static_cast<int64_t>(g) + b;
                if (kb < nblk) {
                    uint32_t w[16], out[4];
                    load_block32(xrow + kb * 32, w);
                    const uint32_t byte = quantize_block32(w, out);
                    *reinterpret_cast<uint4*>(qrow + kb * 16) = make_uint4(out[0], out[1], out[2], out[3]);
                    sc |= byte << (8 * b);
                    if (!kChunkLayout) scales[r * nblk + kb] = static_cast<uint8_t>(byte);
                }
            }
        }
        if (kChunkLayout)
            *reinterpret_cast<uint32_t*>(scales + sf_chunk_offset(static_cast<uint32_t>(r), 4u * g, groups_cover)) = sc;
    }
}

// Scale bytes of a pre-quantized B [N, K/32] -> tensor-core chunks, zero padded to whole
// 128-row tiles and to `groups` 4-block groups per row.
__global__ void __launch_bounds__(256)
prepack_sf_kernel(const uint8_t* __restrict__ bs, int64_t N, int64_t K, uint8_t* __restrict__ out, int groups) {
    const int64_t nblk = K / 32;
    const int64_t rows_cover = (N + 127) / 128 * 128;
    const int64_t items = rows_cover * groups;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items; it += stride) {
        const int64_t r = it / groups;
        const int g = static_cast<int>(it - r * groups);
        uint32_t v = 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int64_t kb = 4 * static_cast<int64_t>(g) + b;
            if (r < N && kb < nblk) v |= static_cast<uint32_t>(bs[r * nblk + kb]) << (8 * b);
        }
        *reinterpret_cast<uint32_t*>(out + sf_chunk_offset(static_cast<uint32_t>(r), 4u * g, groups)) = v;
    }
}

static int grid_for(int64_t items, int threads) {
    int64_t blocks = (items + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;   // grid-stride loops cover the rest
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* q,
                            uint8_t* scales, int64_t chunk_rows, int groups, cudaStream_t s) {
    const int threads = 256;
    if (chunk_rows > 0) {
        const int64_t rows_cover = chunk_rows;
        return launch_pdl(quantize_kernel<true>, dim3(grid_for(rows_cover * groups, threads)), dim3(threads), 0, s,
                          x, rows, K, ld, q, scales, rows_cover, groups);
    }
    const int gc = static_cast<int>((K / 32 + 3) / 4);
    return launch_pdl(quantize_kernel<false>, dim3(grid_for(rows * gc, threads)), dim3(threads), 0, s,
                      x, rows, K, ld, q, scales, rows, gc);
}

cudaError_t launch_prepack_sf(const uint8_t* bs, int64_t N, int64_t K, uint8_t* sf_out, int groups, cudaStream_t s) {
    const int threads = 256;
    const int64_t rows_cover = (N + 127) / 128 * 128;
    prepack_sf_kernel<<<grid_for(rows_cover * groups, threads), threads, 0, s>>>(bs, N, K, sf_out, groups);
    return cudaGetLastError();
}

}  // namespace mxfp4
