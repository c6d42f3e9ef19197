// Host/device shared definitions of the MXFP4 library (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxfp4 {

constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 8;               // warps 3..10: A quantization (fused path) and the epilogue
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kGemmThreads = 96 + kEpiThreads;   // warp 0 copies, warps 1-2 MMA
constexpr int kTileN = 128;                // weight rows per MMA (the MMA's M)
constexpr int kAtomK = 256;                // K elements per pipeline step (128-byte rows)
constexpr int kMaxMTile = 256;             // tokens per tile (the MMA's N)
constexpr int kMaxSplits = 16;             // K slices per tile = cluster size (> 8 needs the non-portable opt-in)
constexpr int kAutoMaxSplits = 8;          // the automatic plan stays within portable cluster sizes
constexpr int kAutoMaxSplitsTwoKernel = 5;  // two-kernel path: 6 slices measured slower than 5
constexpr uint32_t kBRowsBytes = kTileN * kAtomK / 2;    // 16 KB of e2m1 per weight tile per atom
constexpr uint32_t kSfChunk = 512;         // 128 rows x 4 scale bytes
constexpr size_t kSmemLimit = 227 * 1024;

// Operand blocks. Each (tile, 256-K atom) of an operand is stored in global memory as the exact
// shared-memory image the MMA reads, so one contiguous bulk copy fills a pipeline stage:
//   rows:   row r of the tile at byte r*128; its eight 16-byte chunks (chunk c = 32 e2m1 values =
//           one 1x32 block) at (c ^ (r % 8)) * 16 -- the 128-byte swizzle the MMA descriptor
//           names (the 1 KB-aligned base keeps the pattern aligned);
//   scales: after the rows, for every 128 rows two 512-byte chunks (4-block groups 2j and 2j+1 of
//           atom j); in a chunk, row r sits at (r%32)*16 + ((r/32)%4)*4 + (block%4), the layout
//           tcgen05.cp 32x128b.warpx4 spreads over tensor memory.
// Weight block (128 rows): 16384 + 1024 = 17408 bytes. Token block of m rows:
// m*128 + ceil(m/128)*1024 bytes.
constexpr uint32_t kWBlock = kBRowsBytes + 2 * kSfChunk;

// Split-K reduction: the tile's rows are dealt to the cluster's CTAs in runs of rows_per (a
// multiple of 4); an owner receives [source][weight row n][recv_stride] fp32, where the stride
// (in floats) pads the run so that consecutive rows n land 16 bytes apart modulo 32 banks.
__host__ __device__ inline int red_rows_per(int m_valid, int splits) {
    return ((m_valid + splits - 1) / splits + 3) / 4 * 4;
}
__host__ __device__ inline int red_stride(int rows_per) {
    const int units = rows_per / 4 + 1;          // 16-byte units, made odd
    return 4 * (units + ((units & 1) == 0 ? 1 : 0));
}
// Short runs go as 16-byte stores into [source][n][stride]; long runs as rows of the tile,
// [source][row][n], one contiguous 128-byte segment per warp store (remote stores coalesce
// per contiguous segment).
constexpr int kRedVecMaxRows = 16;
__host__ __device__ inline size_t red_recv_floats(int rows_per, int splits) {
    return rows_per <= kRedVecMaxRows ? static_cast<size_t>(splits) * 128 * red_stride(rows_per)
                                      : static_cast<size_t>(splits) * rows_per * 128;
}

// Fused path: bytes from one staged bf16 token row to the next. 16 bytes beyond the row's
// atoms_max * 256 values move consecutive rows four banks apart, so eight threads reading the
// same 1x32 block of eight consecutive rows hit distinct banks.
__host__ __device__ inline uint32_t raw_pitch(int atoms_max) {
    return static_cast<uint32_t>(atoms_max) * kAtomK * 2u + 16u;
}

__host__ __device__ inline uint32_t swz_chunk_offset(uint32_t r, uint32_t c) {
    return r * 128u + ((c ^ (r & 7u)) << 4);
}
__host__ __device__ inline uint32_t block_sf_offset(uint32_t r, uint32_t kb_in_atom) {
    return ((r >> 7) * 2u + (kb_in_atom >> 2)) * kSfChunk + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u +
           (kb_in_atom & 3u);
}

// Weight-resident kernel (path 3, small token counts): each CTA requests its whole K slice of
// weights (at most kResMaxAtoms 256-K steps) the moment it starts, loads its bf16 A blocks
// straight into registers once the previous grid is done, quantizes them into token blocks in
// shared memory, runs every MMA of the slice from one thread and reduces the K slices of a tile
// by weight-row owners through distributed shared memory.
constexpr int kResThreads = 384;           // 12 warps: warps 1-2 run tensor memory and the MMAs,
constexpr int kResQuantThreads = kResThreads - 64;   // the other 10 quantize A
constexpr int kResMaxAtoms = 8;
constexpr int kResMaxMTile = 32;
constexpr int kResMaxItemsPerThread = 2;   // 1x32 blocks of A per quantizing thread
// ... on plans that read A before the dependency wait, where the A phase overlaps the call ahead
// (a separate instantiation of the kernel, three blocks in flight per thread at a time)
constexpr int kResManyItemsPerThread = 6;
// Rows of the 128-row weight tile each cluster rank owns in the split-K reduction, and the
// fp32 words one owned row takes per source in the receive buffer (tokens rounded up to 4).
__host__ __device__ inline int res_rows_per_owner(int splits) { return (kTileN + splits - 1) / splits; }
__host__ __device__ inline int res_row_words(int m_valid) { return (m_valid + 3) / 4 * 4; }

// Tiling of one mxfp4_gemm call.
struct GemmPlan {
    int path;          // 1: A quantized by the GEMM's own warps; 2: standalone quantize first;
                       // 3: the weight-resident kernel (A quantized inside it)
    int splits;        // K slices per output tile (= thread-block cluster size)
    int m_tile;        // tokens per tile = MMA N (multiple of 16, <= 256)
    int nmc;           // 128-row scale chunks per token tile
    int m_tiles, n_tiles;
    int k_atoms;       // ceil(K / 256)
    int atoms_max;     // most atoms any split gets
    int raw_rows;      // fused path: token rows staged as bf16 (the real rows of a tile)
    int stages;
    int issuers;       // MMA-issuing threads (1 to 3); one accumulator each, or halves of one
    int sf_stores;     // two-kernel path: scale factors written into tensor memory by epilogue warps
    int a_early;       // weight-resident path: A read before the dependency wait (the caller
                       // declared it ready and the plan leaves the SM room for it)
    int many_items;    // weight-resident path: more than kResMaxItemsPerThread blocks of A per
                       // quantizing thread (only with a_early)
    int ctas;
    uint32_t a_block;  // bytes of one token block
    // shared-memory layout (bytes from a 1 KB-aligned base): weight stages at 0, token blocks
    // at off_a, the fused path's bf16 A slice at off_araw, the reduction's receive buffer at
    // off_recv (over the pipeline buffers unless recv_dedicated), barriers at off_bar
    uint32_t off_a, off_araw, off_recv, off_bar;
    int recv_dedicated;
    // split-K by bulk copies: each CTA stages its fp32 tile [row][n] at off_stage (inside the
    // pipeline buffers, clear of the receive buffer) and copies each owner's rows in one piece
    int red_bulk;
    uint32_t off_stage;
    size_t smem_bytes;
    uint32_t tmem_cols;
    size_t ws_total;   // workspace: the two-kernel path's token blocks [m_tiles][k_atoms][a_block]
};

struct GemmArgs {
    const uint16_t* a;     // bf16 A (fused path)
    int64_t lda;
    const uint8_t* ablk;   // token blocks (two-kernel path)
    const uint8_t* bblk;   // weight blocks (packed B)
    uint16_t* c;
    int64_t ldc;
    uint32_t* status;      // device error word
    int M, N, K;
    int m_tile, nmc, m_tiles, n_tiles, splits, k_atoms, stages, atoms_max, issuers;
    uint32_t a_block, off_a, off_araw, off_recv, off_bar;
    int recv_dedicated;
    int red_bulk;
    uint32_t off_stage;
    uint32_t tmem_cols;
    int fused;
    int sf_stores;         // scale factors into tensor memory by epilogue warps (two-kernel path)
    int a_ready;           // the fused path's A rows may be requested before the previous grid finishes
    int c_vec4;            // C rows allow 8-byte stores of 4 bf16 (ldc % 4 == 0, C 8-byte aligned)
    uint64_t wait_limit_ns;
#ifdef MXFP4_TEST_HOOKS
    uint8_t* token_dump;   // test build only: the fused CTAs of weight tile 0 copy their token blocks here
#endif
};

struct ResidentArgs {
    const uint16_t* a;     // bf16 A [M, lda]
    int64_t lda;
    const uint8_t* bblk;   // weight blocks (packed B)
    uint16_t* c;
    int64_t ldc;
    uint32_t* status;      // device error word
    int M, N, K;
    int m_tile, m_tiles, n_tiles, splits, k_atoms;
    int issuers;           // MMA-issuing warps: 2, or 3 (16-token tiles of at least three steps)
    int a_early;           // A loaded before the previous grid has finished (GemmPlan::a_early)
    uint32_t a_block;      // bytes of one token block
    uint32_t off_a, off_recv, off_bar;   // shared-memory offsets from the 1 KB-aligned base
    uint32_t tmem_cols;
    uint64_t wait_limit_ns;
#ifdef MXFP4_TEST_HOOKS
    uint8_t* token_dump;   // test build only: the CTAs of weight tile 0 copy their token blocks here
#endif
};

// Device properties the planner needs (cached per device).
struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;
    uint32_t* status;      // address of the device error word on this device
};

int device_info(DeviceInfo* out);   // MXFP4_OK or an error status
// cluster_caps: if not null, cluster_caps[s] (s = 1..kMaxSplits) is how many clusters of s CTAs
// can be resident at once, used instead of asking the current device (no CUDA call is made).
// a_ready: the caller declared A ready (MXFP4_GEMM_A_READY), which can change the weight-resident
// plan (GemmPlan::a_early).
int make_plan(int64_t M, int64_t N, int64_t K, int path_req, int splits_req, int mtile_req, int sm_count,
              GemmPlan* plan, const int* cluster_caps = nullptr, bool a_ready = false);
size_t packed_b_bytes(int64_t N, int64_t K);

// Exact unsigned 32-bit division by a divisor fixed at launch: the round-up multiplier with one
// correction step of Granlund and Montgomery, "Division by invariant integers using
// multiplication" (1994): q = (t + ((n - t) >> s1)) >> s2 with t = umulhi(m, n), for every
// n < 2^32 and 1 <= d < 2^31. A runtime integer division costs tens of dependent instructions
// on the quantizers' critical path; this costs four.
struct FastDiv {
    uint32_t m, s1, s2;
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;   // ceil(log2 d)
    while ((uint64_t(1) << l) < d) ++l;
    FastDiv f;
    f.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
    f.s1 = l < 1 ? l : 1;
    f.s2 = l > 1 ? l - 1 : 0;
    return f;
}
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
    const uint32_t t = __umulhi(f.m, n);
    return (t + ((n - t) >> f.s1)) >> f.s2;
}
#endif

// Kernel launchers (return cudaError_t).
// Natural layout: q [rows, nblk*16], scales [rows, nblk], nblk = ceil(K/32) (K % 8 == 0).
cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* q,
                            uint8_t* scales, cudaStream_t s);
// Token blocks for the GEMM, [m_tiles][k_atoms][a_block]; rows past `rows` and K past `K` zeroed.
// a_ready: x may be read before the previous grid finishes (the stores still wait for it).
cudaError_t launch_quantize_blocks(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* blocks,
                                   int m_tile, int m_tiles, int k_atoms, uint32_t a_block, bool a_ready,
                                   cudaStream_t s);
// bf16 rows [rows, K] at row stride lda (elements; 16-byte aligned rows, K % 8 == 0) from
// device-accessible host memory -> packed device rows [rows, K]; PDL-chained (see the kernel).
// early: read src before waiting for the previous grid (the caller declared it host-written only)
cudaError_t launch_stage_rows(const void* src, int64_t lda, void* dst, int64_t rows, int64_t K, bool early,
                              cudaStream_t s);
// Pre-quantized B (natural layout) -> weight blocks [n_tiles][k_atoms][kWBlock].
cudaError_t launch_prepack(const uint8_t* bq, const uint8_t* bs, int64_t N, int64_t K, uint8_t* out,
                           cudaStream_t s);
cudaError_t launch_gemm(const GemmPlan& plan, const GemmArgs& args, cudaStream_t s);
cudaError_t launch_gemm_resident(const GemmPlan& plan, const ResidentArgs& args, cudaStream_t s);
// Clusters of `cluster_size` weight-resident CTAs with this much shared memory resident at once.
int max_active_clusters_resident(int cluster_size, size_t smem_bytes);
cudaError_t launch_timeout_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s);
// Clusters of `cluster_size` GEMM CTAs with this much shared memory resident at once (0 if unknown).
int max_active_clusters(int cluster_size, size_t smem_bytes);

// Launch with programmatic stream serialization so a dependent kernel can start early.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace mxfp4
