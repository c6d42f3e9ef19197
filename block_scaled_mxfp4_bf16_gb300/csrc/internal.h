// Host/device shared definitions of the MXFP4 library (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxfp4 {

constexpr int kMaxStages = 8;
constexpr int kGemmThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2..5 quant + epilogue
constexpr int kTileN = 128;                // weight rows per MMA (the MMA's M)
constexpr int kAtomK = 256;                // K elements per pipeline step (128-byte rows)
constexpr int kMaxMTile = 256;             // tokens per tile (the MMA's N)
constexpr uint32_t kBStageBytes = kTileN * kAtomK / 2;   // 16 KB
constexpr uint32_t kSfChunk = 512;         // 128 rows x 4 scale bytes
constexpr size_t kSmemLimit = 227 * 1024;
// Split-K arrival counters live in a fixed region at the start of every workspace and are
// used for nothing else, so whatever plan ran before, a completed call leaves them all at 0.
constexpr int kMaxCounters = 16384;
constexpr size_t kCounterBytes = kMaxCounters * sizeof(uint32_t);

// Two-level tiling of one mxfp4_gemm call.
struct GemmPlan {
    int path;          // 1: A quantized by the GEMM's producer warps; 2: standalone quantize first
    int splits;        // K slices per output tile
    int m_tile;        // tokens per tile = MMA N (multiple of 16, <= 256)
    int nmc;           // 128-row scale chunks per token tile
    int m_tiles, n_tiles;
    int k_atoms;       // ceil(K / 256)
    int groups;        // scale-factor 4-block groups per row, padded to 2 per atom
    int atoms_max;     // most atoms any split gets
    int stages;
    int ctas;
    uint32_t off_a, off_sfb, off_sfa, off_bar;  // shared-memory layout (bytes from a 1 KB base)
    size_t smem_bytes;
    uint32_t tmem_cols;
    // workspace layout (bytes)
    size_t ws_aq, ws_sfa, ws_part, ws_ctr, ws_total;
};

struct GemmArgs {
    const uint16_t* a;    // bf16 A (fused path)
    int64_t lda;
    const uint8_t* sfa;   // A scale chunks (two-kernel path)
    const uint8_t* sfb;   // B scale chunks (packed B)
    uint16_t* c;
    int64_t ldc;
    float* part;          // split-K partial tiles
    uint32_t* ctr;        // split-K arrival counters, one per output tile
    uint32_t* status;     // device error word
    int M, N, K;
    int m_tile, nmc, m_tiles, n_tiles, splits, k_atoms, groups, stages;
    uint32_t off_a, off_sfb, off_sfa, off_bar;
    uint32_t tmem_cols;
    int fused;
    uint64_t wait_limit_ns;
};

// Device properties the planner needs (cached per device).
struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;
    uint32_t* status;     // address of the device error word on this device
};

int device_info(DeviceInfo* out);                 // MXFP4_OK or an error status
size_t packed_sf_offset(int64_t N, int64_t K);
int make_plan(int64_t M, int64_t N, int64_t K, int path_req, int splits_req, int sm_count, GemmPlan* plan);

// Kernel launchers (return cudaError_t).
// chunk_rows > 0: scales go to the tensor-core chunk layout covering chunk_rows rows (a
// multiple of 128) and `groups` 4-block groups, padding zeroed; 0: natural [rows, K/32].
cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* q,
                            uint8_t* scales, int64_t chunk_rows, int groups, cudaStream_t s);
cudaError_t launch_prepack_sf(const uint8_t* bs, int64_t N, int64_t K, uint8_t* sf_out, int groups,
                              cudaStream_t s);
cudaError_t launch_gemm(const GemmPlan& plan, const CUtensorMap& tmap_b, const CUtensorMap& tmap_a,
                        const GemmArgs& args, cudaStream_t s);
cudaError_t launch_timeout_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s);

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
