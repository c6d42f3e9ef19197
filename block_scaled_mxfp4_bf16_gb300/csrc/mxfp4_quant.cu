// Standalone MXFP4 quantizer (natural layout and the GEMM's token blocks) and the weight
// prepack. One thread per 1x32 block: 64 bytes of bf16 in (four 16-byte loads in flight),
// 16 bytes of packed e2m1 and one e8m0 byte out.
// K is a multiple of 8. A row has ceil(K/32) blocks; in the last one the elements past K count
// as zeros (submission 711914 `_standalone_quant_kernel` loads A under the mask offs_k < K with
// 0 as the fill value), so they give zero codes and do not change the block's scale. The
// 16-byte pieces past K are never read.
#include "internal.h"
#include "ptx.cuh"
#include "quant_device.cuh"

namespace mxfp4 {

// Natural layout: q [rows, nblk*16], scales [rows, nblk], nblk = ceil(K/32).
__global__ void __launch_bounds__(256)
quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ld,
                uint8_t* __restrict__ q, uint8_t* __restrict__ scales) {
    pdl_launch_dependents();
    const int64_t nblk = (K + 31) / 32;
    const int64_t items = rows * nblk;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (first < items) prefetch_l2(x + (first / nblk) * ld + (first % nblk) * 32);   // see prefetch_l2
    pdl_wait_prior_grid();   // x may come from the previous kernel; q/scales may still be read by it
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items; it += stride) {
        const int64_t r = it / nblk;
        const int64_t kb = it - r * nblk;
        uint32_t w[16], out[4];
        load_block32_upto(x + r * ld + kb * 32, K - kb * 32, w);
        const uint32_t byte = quantize_block32(w, out);
        *reinterpret_cast<uint4*>(q + r * (nblk * 16) + kb * 16) = make_uint4(out[0], out[1], out[2], out[3]);
        scales[it] = static_cast<uint8_t>(byte);
    }
}

// Item index -> (quotient by a launch-fixed divisor): FastDiv when every item index fits 32 bits
// (kNarrow), a 64-bit division otherwise.
template <bool kNarrow>
__device__ __forceinline__ int64_t div_items(int64_t n, int64_t d, const FastDiv& f) {
    if constexpr (kNarrow) return fast_div(static_cast<uint32_t>(n), f);
    else return n / d;
}

// Token blocks, one lane per 1x32 block (layout in internal.h): block (mt, j) at
// (mt * k_atoms + j) * a_block. Items run
// over every (row, block) of the padded [m_tiles*m_tile, k_atoms*256] matrix, so padding rows and
// the K tail are written as zeros. Four consecutive lanes own the four blocks of one scale word.
// fd_row divides by the items of a padded row (8 * k_atoms), fd_mtile by m_tile.
template <bool kNarrow>
__global__ void __launch_bounds__(256)
quantize_blocks_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ld,
                       uint8_t* __restrict__ blocks, int m_tile, int m_tiles, int k_atoms, uint32_t a_block,
                       FastDiv fd_row, FastDiv fd_mtile, int a_ready) {
    pdl_launch_dependents();
    const int64_t nblk = (K + 31) / 32;
    const int64_t row_items = 8 * static_cast<int64_t>(k_atoms);
    const int64_t items = static_cast<int64_t>(m_tiles) * m_tile * row_items;   // multiple of 8
    {   // warm L2 with this thread's first block while the previous grid finishes (see prefetch_l2)
        const int64_t it0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        const int64_t r = div_items<kNarrow>(it0, row_items, fd_row), kbp = it0 - r * row_items;
        if (it0 < items && r < rows && kbp < nblk) prefetch_l2(x + r * ld + kbp * 32);
    }
    // x may come from the previous grid, which may also still read `blocks`: wait before the
    // first load -- or, when the caller declared A ready, only before the first store
    if (!a_ready) pdl_wait_prior_grid();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int lane = threadIdx.x & 31;
    // the loop bound is uniform per warp (warps start at multiples of 32) so the shuffles below
    // always see all 32 lanes
    for (int64_t wbase = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); wbase < items;
         wbase += stride) {
        const int64_t it = wbase + lane;
        const bool in_range = it < items;
        const int64_t r = in_range ? div_items<kNarrow>(it, row_items, fd_row) : 0;
        const int64_t kbp = in_range ? it - r * row_items : 0;     // block index within the padded row
        const bool live = in_range && r < rows && kbp < nblk;
        uint32_t w[16], out[4] = {0u, 0u, 0u, 0u}, byte = 0u;
        if (live) {
            load_block32_upto(x + r * ld + kbp * 32, K - kbp * 32, w);
            byte = quantize_block32(w, out);
        }
        uint32_t word = byte << (8 * (lane & 3));
        word |= __shfl_xor_sync(0xffffffffu, word, 1);
        word |= __shfl_xor_sync(0xffffffffu, word, 2);
        if (a_ready) pdl_wait_prior_grid();
        if (in_range) {
            const int mt = static_cast<int>(div_items<kNarrow>(r, m_tile, fd_mtile));
            const uint32_t rr = static_cast<uint32_t>(r - static_cast<int64_t>(mt) * m_tile);
            const uint32_t c = static_cast<uint32_t>(kbp & 7);
            uint8_t* blk = blocks + (static_cast<size_t>(mt) * k_atoms + static_cast<size_t>(kbp >> 3)) * a_block;
            *reinterpret_cast<uint4*>(blk + swz_chunk_offset(rr, c)) = make_uint4(out[0], out[1], out[2], out[3]);
            if ((lane & 3) == 0)
                *reinterpret_cast<uint32_t*>(blk + static_cast<uint32_t>(m_tile) * 128u + block_sf_offset(rr, c)) = word;
        }
    }
}

// Token blocks (layout in internal.h): block (mt, j) at (mt * k_atoms + j) * a_block; items run
// over every (row, block) of the padded [m_tiles*m_tile, k_atoms*256] matrix, so padding rows and
// the K tail are written as zeros. Four lanes per 1x32 block: lane part p of a block loads
// elements 8p..8p+7 (16 bytes; a warp reads eight consecutive blocks, 512 contiguous bytes), the
// block's amax is combined over the four lanes, and each lane writes its 4 bytes of codes. The
// eight blocks of a warp are two scale words (four consecutive blocks of one row each),
// assembled by shuffles. Shorter per-thread chains than one lane per block: the kernel sits
// between two GEMMs on the critical path, so its latency is what counts (launched for at most
// kQuantFourLaneMaxBlocks items, so item indices fit 32 bits and divide by FastDiv).
__global__ void __launch_bounds__(256)
quantize_blocks4_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ld,
                        uint8_t* __restrict__ blocks, int m_tile, int m_tiles, int k_atoms, uint32_t a_block,
                        FastDiv fd_row, FastDiv fd_mtile, int a_ready) {
    pdl_launch_dependents();
    const int64_t nblk = (K + 31) / 32;
    const int64_t row_items = 8 * static_cast<int64_t>(k_atoms);
    const int64_t items = static_cast<int64_t>(m_tiles) * m_tile * row_items;   // multiple of 8
    const int lane = threadIdx.x & 31;
    const int part = lane & 3;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    {   // warm L2 with this lane's first 16 bytes while the previous grid finishes (see prefetch_l2)
        const int64_t it0 = warp_id * 8 + (lane >> 2);
        const int64_t r = fast_div(static_cast<uint32_t>(it0), fd_row), kbp = it0 - r * row_items;
        if (it0 < items && r < rows && kbp * 32 + part * 8 < K) prefetch_l2(x + r * ld + kbp * 32 + part * 8);
    }
    if (!a_ready) pdl_wait_prior_grid();   // as in quantize_blocks_kernel
    // the loop bound is uniform per warp, so the shuffles below always see all 32 lanes
    for (int64_t base = warp_id * 8; base < items; base += warps * 8) {
        const int64_t it = base + (lane >> 2);
        const int64_t r = fast_div(static_cast<uint32_t>(it), fd_row);
        const int64_t kbp = it - r * row_items;          // block index within the padded row
        const bool live = r < rows && kbp < nblk;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (live && kbp * 32 + part * 8 < K) {   // a piece past K in the last block stays zero
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + r * ld + kbp * 32 + part * 8));
            w[0] = v.x;
            w[1] = v.y;
            w[2] = v.z;
            w[3] = v.w;
        }
        uint32_t amax = amax_quarter(w);
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int s = scale_exponent(amax << 16);
        const uint32_t codes = live ? quantize_quarter(w, inv_scale(s)) : 0u;
        const uint32_t byte = live ? static_cast<uint32_t>(s + 127) : 0u;
        // scale word of four consecutive blocks: the part-0 lanes 0, 4, 8, 12 (and 16..28)
        uint32_t word = part == 0 ? byte << (8 * ((lane >> 2) & 3)) : 0u;
        word |= __shfl_xor_sync(0xffffffffu, word, 4);
        word |= __shfl_xor_sync(0xffffffffu, word, 8);
        const int mt = static_cast<int>(fast_div(static_cast<uint32_t>(r), fd_mtile));
        const uint32_t rr = static_cast<uint32_t>(r - static_cast<int64_t>(mt) * m_tile);
        const uint32_t c = static_cast<uint32_t>(kbp & 7);
        uint8_t* blk = blocks + (static_cast<size_t>(mt) * k_atoms + static_cast<size_t>(kbp >> 3)) * a_block;
        if (a_ready) pdl_wait_prior_grid();
        *reinterpret_cast<uint32_t*>(blk + swz_chunk_offset(rr, c) + part * 4) = codes;
        if ((lane & 15) == 0)
            *reinterpret_cast<uint32_t*>(blk + static_cast<uint32_t>(m_tile) * 128u + block_sf_offset(rr, c)) = word;
    }
}

// Weight prepack: one thread per (row, block) of the padded [n_tiles*128, k_atoms*256] matrix;
// copies 16 bytes of e2m1 into the swizzled rows and the scale byte into its chunk. Input rows
// are the natural layout: nblk = ceil(K/32) blocks of 16 code bytes and one scale byte each.
__global__ void __launch_bounds__(256)
prepack_kernel(const uint8_t* __restrict__ bq, const uint8_t* __restrict__ bs, int64_t N, int64_t K,
               uint8_t* __restrict__ out, int k_atoms) {
    const int64_t nblk = (K + 31) / 32;
    const int64_t row_items = 8 * static_cast<int64_t>(k_atoms);
    const int64_t rows_cover = (N + kTileN - 1) / kTileN * kTileN;
    const int64_t items = rows_cover * row_items;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items; it += stride) {
        const int64_t r = it / row_items;
        const int64_t kbp = it - r * row_items;
        const uint32_t rr = static_cast<uint32_t>(r % kTileN);
        const uint32_t c = static_cast<uint32_t>(kbp & 7);
        uint8_t* blk = out + (static_cast<size_t>(r / kTileN) * k_atoms + static_cast<size_t>(kbp >> 3)) * kWBlock;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        uint8_t sc = 0;
        if (r < N && kbp < nblk) {
            v = __ldg(reinterpret_cast<const uint4*>(bq + r * (nblk * 16) + kbp * 16));
            sc = bs[r * nblk + kbp];
        }
        *reinterpret_cast<uint4*>(blk + swz_chunk_offset(rr, c)) = v;
        blk[kBRowsBytes + block_sf_offset(rr, c)] = sc;
    }
}

// Host rows -> device rows for the host-buffer GEMM: one 16-byte piece per thread, read from
// page-locked host memory mapped into the device's address space (zero-copy). The store comes
// after the wait on the previous grid, which may still read the destination. So does the read,
// unless the caller has declared the source written by the host only (kEarly): otherwise that
// grid may be writing it (a chained call whose C, stored into mapped host memory, is this
// call's A), and the stream order a copy would give is kept. With kEarly the read crosses the
// link while the previous grid still runs. Unlike a copy-engine transfer, a kernel keeps the
// programmatic-dependent-launch chain from the previous GEMM through this copy to the next
// GEMM, so their launches still overlap.
template <bool kEarly>
__global__ void __launch_bounds__(256)
stage_rows_kernel(const uint4* __restrict__ src, int64_t src_row16, uint4* __restrict__ dst, int64_t row16,
                  int64_t pieces) {
    pdl_launch_dependents();
    if (!kEarly) pdl_wait_prior_grid();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t r = i / row16;
    const int64_t c = i - r * row16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (i < pieces) v = src[r * src_row16 + c];
    if (kEarly) pdl_wait_prior_grid();
    if (i < pieces) dst[r * row16 + c] = v;
}

constexpr int64_t kQuantFourLaneMaxBlocks = 16384;

static int grid_for(int64_t items, int threads) {
    int64_t blocks = (items + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;   // grid-stride loops cover the rest
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* q, uint8_t* scales,
                            cudaStream_t s) {
    const int threads = 256;
    return launch_pdl(quantize_kernel, dim3(grid_for(rows * ((K + 31) / 32), threads)), dim3(threads), 0, s, x, rows, K,
                      ld, q, scales);
}

cudaError_t launch_quantize_blocks(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* blocks,
                                   int m_tile, int m_tiles, int k_atoms, uint32_t a_block, bool a_ready,
                                   cudaStream_t s) {
    const int ready = a_ready ? 1 : 0;
    const int threads = 256;
    const int64_t items = static_cast<int64_t>(m_tiles) * m_tile * 8 * k_atoms;
    // few blocks: four lanes each (shorter chains, the launch is latency-bound); many blocks: one
    // lane each (less total work; measured faster for 256x7168 and slower for 64x2048)
    const FastDiv fd_row = make_fastdiv(8u * static_cast<uint32_t>(k_atoms));
    const FastDiv fd_mtile = make_fastdiv(static_cast<uint32_t>(m_tile));
    if (items <= kQuantFourLaneMaxBlocks)
        return launch_pdl(quantize_blocks4_kernel, dim3(grid_for(items * 4, threads)), dim3(threads), 0, s, x, rows,
                          K, ld, blocks, m_tile, m_tiles, k_atoms, a_block, fd_row, fd_mtile, ready);
    // One lane per block in 128-thread blocks: more, smaller blocks than 256-thread ones shorten
    // the launch's tail (256x4096x7168 11.85 -> 11.65 us per call, 512x4096x7168 14.23 -> 13.60;
    // the four-lane kernel above measured mixed with 128 threads and keeps 256).
    const int threads1 = 128;
    // item indices (and the grid-stride overshoot, below one more grid) within 32 bits: FastDiv
    const int64_t span = items + static_cast<int64_t>(grid_for(items, threads1)) * threads1;
    if (span <= static_cast<int64_t>(UINT32_MAX))
        return launch_pdl(quantize_blocks_kernel<true>, dim3(grid_for(items, threads1)), dim3(threads1), 0, s, x, rows,
                          K, ld, blocks, m_tile, m_tiles, k_atoms, a_block, fd_row, fd_mtile, ready);
    return launch_pdl(quantize_blocks_kernel<false>, dim3(grid_for(items, threads1)), dim3(threads1), 0, s, x, rows, K,
                      ld, blocks, m_tile, m_tiles, k_atoms, a_block, fd_row, fd_mtile, ready);
}

cudaError_t launch_stage_rows(const void* src, int64_t lda, void* dst, int64_t rows, int64_t K, bool early,
                              cudaStream_t s) {
    const int threads = 256;
    const int64_t row16 = K / 8, pieces = rows * row16;
    const int64_t blocks = (pieces + threads - 1) / threads;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const auto* in = static_cast<const uint4*>(src);
    auto* out = static_cast<uint4*>(dst);
    return early ? launch_pdl(stage_rows_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, in,
                              lda / 8, out, row16, pieces)
                 : launch_pdl(stage_rows_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, in,
                              lda / 8, out, row16, pieces);
}

cudaError_t launch_prepack(const uint8_t* bq, const uint8_t* bs, int64_t N, int64_t K, uint8_t* out, cudaStream_t s) {
    const int threads = 256;
    const int k_atoms = static_cast<int>((K + kAtomK - 1) / kAtomK);
    const int64_t rows_cover = (N + kTileN - 1) / kTileN * kTileN;
    prepack_kernel<<<grid_for(rows_cover * 8 * k_atoms, threads), threads, 0, s>>>(bq, bs, N, K, out, k_atoms);
    return cudaGetLastError();
}

}  // namespace mxfp4
