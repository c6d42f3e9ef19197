// C ABI of the MXFP4 library: argument checks, the GEMM plan (tiling, split-K, path), the TMA
// tensor maps and the launches. See include/mxfp4_gb300.h for the contract of each call.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/mxfp4_gb300.h"
#include "internal.h"

namespace mxfp4 {

__device__ uint32_t g_device_status;   // bit 0: a bounded wait gave up

static thread_local int t_last_cuda_error = 0;

static int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return MXFP4_ERR_CUDA;
}

// ------------------------------------------------------------------ device properties

int device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return MXFP4_ERR_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d = {};
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return cuda_fail(e);
        int optin = 0;
        if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return cuda_fail(e);
        d.smem_optin = static_cast<size_t>(optin);
        if (d.cc_major == 10 && d.cc_minor == 3) {
            void* sym = nullptr;
            if ((e = cudaGetSymbolAddress(&sym, g_device_status)) != cudaSuccess) return cuda_fail(e);
            d.status = static_cast<uint32_t*>(sym);
        }
        cache[dev] = d;
        have[dev] = true;
    }
    *out = cache[dev];
    if (out->cc_major != 10 || out->cc_minor != 3) return MXFP4_ERR_ARCH;
    return MXFP4_OK;
}

// ------------------------------------------------------------------ layout helpers

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t packed_sf_offset(int64_t N, int64_t K) { return align_up(static_cast<size_t>(N) * (K / 2), 1024); }

static size_t packed_sf_bytes(int64_t N, int64_t K) {
    return static_cast<size_t>(cdiv(N, kTileN)) * static_cast<size_t>(2 * cdiv(K, kAtomK)) * kSfChunk;
}

// ------------------------------------------------------------------ the GEMM plan

int make_plan(int64_t M, int64_t N, int64_t K, int path_req, int splits_req, int sm_count, GemmPlan* P) {
    GemmPlan p = {};
    if (M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_SHAPE;
    p.m_tile = M <= kMaxMTile ? static_cast<int>(cdiv(M, 16) * 16) : kMaxMTile;
    p.nmc = (p.m_tile + 127) / 128;
    p.m_tiles = static_cast<int>(cdiv(M, p.m_tile));
    p.n_tiles = static_cast<int>(cdiv(N, kTileN));
    p.k_atoms = static_cast<int>(cdiv(K, kAtomK));
    p.groups = 2 * p.k_atoms;
    const int64_t units = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    if (units > (1 << 24)) return MXFP4_ERR_SHAPE;
    // Fused quantization repeats A's quantization once per weight tile; keep it where A is
    // small next to the weight stream (M <= 32, the pages' small-M split), else quantize once.
    p.path = path_req ? path_req : (M <= 32 ? 1 : 2);
    if (p.path != 1 && p.path != 2) return MXFP4_ERR_ARG;
    int splits = splits_req;
    if (splits <= 0) {
        const int64_t fill = std::max<int64_t>(1, sm_count / std::max<int64_t>(1, units));
        splits = static_cast<int>(std::min<int64_t>(fill, p.k_atoms));
    }
    p.splits = std::max(1, std::min(splits, p.k_atoms));
    if (units > kMaxCounters) p.splits = 1;     // more tiles than counters: no split-K
    p.atoms_max = static_cast<int>(cdiv(p.k_atoms, p.splits));

    const uint32_t a_bytes = static_cast<uint32_t>(p.m_tile) * 128u;
    const uint32_t sfa_bytes = static_cast<uint32_t>(p.nmc) * 1024u;
    const size_t bar_bytes = 256;
    const size_t budget = kSmemLimit - 1024 - bar_bytes;
    size_t fixed = 0, per_stage = kBStageBytes + 1024;
    if (p.path == 1) fixed = static_cast<size_t>(p.atoms_max) * (a_bytes + sfa_bytes);
    else per_stage += a_bytes + sfa_bytes;
    if (fixed + per_stage > budget) {
        if (path_req == 1) return MXFP4_ERR_SHAPE;   // fused slice does not fit shared memory
        return make_plan(M, N, K, 2, splits_req, sm_count, P);
    }
    p.stages = static_cast<int>(std::min<size_t>({static_cast<size_t>(kMaxStages), static_cast<size_t>(p.atoms_max),
                                                  (budget - fixed) / per_stage}));
    p.off_a = static_cast<uint32_t>(p.stages) * kBStageBytes;
    const int a_slots = p.path == 1 ? p.atoms_max : p.stages;
    p.off_sfb = p.off_a + static_cast<uint32_t>(a_slots) * a_bytes;
    p.off_sfa = p.off_sfb + static_cast<uint32_t>(p.stages) * 1024u;
    p.off_bar = p.off_sfa + static_cast<uint32_t>(a_slots) * sfa_bytes;
    p.smem_bytes = p.off_bar + bar_bytes + 1024;
    const uint32_t cols = static_cast<uint32_t>(p.m_tile) + static_cast<uint32_t>(p.stages) * 8u * (1u + p.nmc);
    p.tmem_cols = 32;
    while (p.tmem_cols < cols) p.tmem_cols <<= 1;
    p.ctas = static_cast<int>(units * p.splits);

    // workspace: [counters (fixed 64 KB) | A e2m1 | A scale chunks | split-K partials]
    size_t off = 0;
    p.ws_ctr = off;
    off += kCounterBytes;
    p.ws_aq = off;
    if (p.path == 2) off += align_up(static_cast<size_t>(M) * (K / 2), 1024);
    p.ws_sfa = off;
    if (p.path == 2) {
        const size_t rows_cover = align_up(static_cast<size_t>(p.m_tiles) * p.m_tile, 128);
        off += align_up(rows_cover / 128 * p.groups * kSfChunk, 1024);
    }
    p.ws_part = off;
    if (p.splits > 1) off += align_up(static_cast<size_t>(units) * p.splits * kTileN * p.m_tile * sizeof(float), 1024);
    if (p.path == 1 && p.splits == 1) off = 0;     // nothing to keep: no workspace needed
    p.ws_total = off;
    *P = p;
    return MXFP4_OK;
}

// ------------------------------------------------------------------ tensor maps

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D uint8 map over [rows, row_bytes] with a (128 bytes x box_rows) box, 128-byte swizzle.
static int make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return cuda_fail(cudaErrorNotSupported);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return MXFP4_OK;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static uint64_t g_wait_limit_ns = 1000000000ull;   // 1 s per bounded wait

}  // namespace mxfp4

using namespace mxfp4;

// ====================================================================== C ABI

extern "C" {

const char* mxfp4_status_string(int status) {
    switch (status) {
        case MXFP4_OK: return "MXFP4_OK";
        case MXFP4_ERR_ARG: return "MXFP4_ERR_ARG";
        case MXFP4_ERR_SHAPE: return "MXFP4_ERR_SHAPE";
        case MXFP4_ERR_ALIGN: return "MXFP4_ERR_ALIGN";
        case MXFP4_ERR_ARCH: return "MXFP4_ERR_ARCH";
        case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA";
        case MXFP4_ERR_TIMEOUT: return "MXFP4_ERR_TIMEOUT";
        case MXFP4_ERR_WORKSPACE: return "MXFP4_ERR_WORKSPACE";
        default: return "MXFP4_ERR_UNKNOWN";
    }
}

int mxfp4_last_cuda_error(void) { return t_last_cuda_error; }

int mxfp4_version(void) { return 100; }

int mxfp4_quantize(const void* x, int64_t rows, int64_t K, int64_t ld, void* q, void* scales, void* stream) {
    if (rows < 0 || K < 0) return MXFP4_ERR_ARG;
    if (K % 32 != 0) return MXFP4_ERR_SHAPE;
    if (rows == 0 || K == 0) return MXFP4_OK;
    if (ld < K) return MXFP4_ERR_SHAPE;
    if (!x || !q || !scales) return MXFP4_ERR_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || ld % 8 != 0) return MXFP4_ERR_ALIGN;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    cudaError_t e = launch_quantize(static_cast<const uint16_t*>(x), rows, K, ld, static_cast<uint8_t*>(q),
                                    static_cast<uint8_t*>(scales), 0, 0, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

size_t mxfp4_prepack_b_size(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % 64 != 0) return 0;
    return packed_sf_offset(N, K) + packed_sf_bytes(N, K);
}

int mxfp4_prepack_b(const void* bq, const void* bs, int64_t N, int64_t K, void* packed, void* stream) {
    if (N <= 0 || K <= 0) return MXFP4_ERR_ARG;
    if (K % 64 != 0) return MXFP4_ERR_SHAPE;
    if (!bq || !bs || !packed) return MXFP4_ERR_ARG;
    if (!aligned(bq, 16) || !aligned(packed, 1024)) return MXFP4_ERR_ALIGN;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    auto s = static_cast<cudaStream_t>(stream);
    uint8_t* out = static_cast<uint8_t*>(packed);
    cudaError_t e = cudaMemcpyAsync(out, bq, static_cast<size_t>(N) * (K / 2), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_prepack_sf(static_cast<const uint8_t*>(bs), N, K, out + packed_sf_offset(N, K),
                          static_cast<int>(2 * cdiv(K, kAtomK)), s);
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

size_t mxfp4_gemm_workspace_size_ex(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options* opts) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 64 != 0) return 0;
    DeviceInfo di;
    if (device_info(&di) != MXFP4_OK) return 0;
    GemmPlan plan;
    if (make_plan(M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, di.sm_count, &plan) != MXFP4_OK) return 0;
    return plan.ws_total;
}

size_t mxfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    return mxfp4_gemm_workspace_size_ex(M, N, K, nullptr);
}

int mxfp4_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
    if (ws_bytes == 0) return MXFP4_OK;
    if (!workspace) return MXFP4_ERR_ARG;
    cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

int mxfp4_gemm_plan(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options* opts, int* path, int* splits,
                    int* m_tile, int* ctas, int* stages) {
    if (M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_ARG;
    if (K % 64 != 0) return MXFP4_ERR_SHAPE;
    if (opts && (opts->path < 0 || opts->path > 2 || opts->splits < 0)) return MXFP4_ERR_ARG;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    GemmPlan plan;
    st = make_plan(M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, di.sm_count, &plan);
    if (st != MXFP4_OK) return st;
    if (path) *path = plan.path;
    if (splits) *splits = plan.splits;
    if (m_tile) *m_tile = plan.m_tile;
    if (ctas) *ctas = plan.ctas;
    if (stages) *stages = plan.stages;
    return MXFP4_OK;
}

int mxfp4_gemm_ex(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N, void* c,
                  int64_t ldc, void* workspace, size_t ws_bytes, const mxfp4_gemm_options* opts, void* stream) {
    if (M < 0 || N < 0 || K < 0) return MXFP4_ERR_ARG;
    if (opts && (opts->path < 0 || opts->path > 2 || opts->splits < 0)) return MXFP4_ERR_ARG;
    if (K == 0 || K % 64 != 0) return MXFP4_ERR_SHAPE;
    if (M == 0 || N == 0) return MXFP4_OK;
    if (lda < K || ldc < N) return MXFP4_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 30)) return MXFP4_ERR_SHAPE;
    if (!a || !packed_b || !c) return MXFP4_ERR_ARG;
    if (!aligned(a, 16) || lda % 8 != 0 || !aligned(packed_b, 1024) || !aligned(c, 2)) return MXFP4_ERR_ALIGN;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    GemmPlan plan;
    st = make_plan(M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, di.sm_count, &plan);
    if (st != MXFP4_OK) return st;
    if (plan.ws_total > 0) {
        if (!workspace || ws_bytes < plan.ws_total) return MXFP4_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return MXFP4_ERR_ALIGN;
    }
    auto s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* pb = static_cast<const uint8_t*>(packed_b);

    CUtensorMap tmap_b, tmap_a;
    st = make_map(&tmap_b, pb, N, K / 2, kTileN);
    if (st != MXFP4_OK) return st;
    tmap_a = tmap_b;
    if (plan.path == 2) {
        st = make_map(&tmap_a, ws + plan.ws_aq, M, K / 2, plan.m_tile);
        if (st != MXFP4_OK) return st;
        const int64_t rows_cover = static_cast<int64_t>(align_up(static_cast<size_t>(plan.m_tiles) * plan.m_tile, 128));
        cudaError_t e = launch_quantize(static_cast<const uint16_t*>(a), M, K, lda, ws + plan.ws_aq, ws + plan.ws_sfa,
                                        rows_cover, plan.groups, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    GemmArgs g = {};
    g.a = static_cast<const uint16_t*>(a);
    g.lda = lda;
    g.sfa = ws ? ws + plan.ws_sfa : nullptr;
    g.sfb = pb + packed_sf_offset(N, K);
    g.c = static_cast<uint16_t*>(c);
    g.ldc = ldc;
    g.part = plan.splits > 1 ? reinterpret_cast<float*>(ws + plan.ws_part) : nullptr;
    g.ctr = plan.splits > 1 ? reinterpret_cast<uint32_t*>(ws + plan.ws_ctr) : nullptr;
    g.status = di.status;
    g.M = static_cast<int>(M);
    g.N = static_cast<int>(N);
    g.K = static_cast<int>(K);
    g.m_tile = plan.m_tile;
    g.nmc = plan.nmc;
    g.m_tiles = plan.m_tiles;
    g.n_tiles = plan.n_tiles;
    g.splits = plan.splits;
    g.k_atoms = plan.k_atoms;
    g.groups = plan.groups;
    g.stages = plan.stages;
    g.off_a = plan.off_a;
    g.off_sfb = plan.off_sfb;
    g.off_sfa = plan.off_sfa;
    g.off_bar = plan.off_bar;
    g.tmem_cols = plan.tmem_cols;
    g.fused = plan.path == 1 ? 1 : 0;
    g.wait_limit_ns = g_wait_limit_ns;
    cudaError_t e = launch_gemm(plan, tmap_b, tmap_a, g, s);
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

int mxfp4_gemm(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N, void* c,
               int64_t ldc, void* workspace, size_t ws_bytes, void* stream) {
    return mxfp4_gemm_ex(a, M, K, lda, packed_b, N, c, ldc, workspace, ws_bytes, nullptr, stream);
}

int mxfp4_device_status(void* stream) {
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t v = 0, zero = 0;
    if ((e = cudaMemcpy(&v, di.status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemcpy(di.status, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess) return cuda_fail(e);
    return v ? MXFP4_ERR_TIMEOUT : MXFP4_OK;
}

int mxfp4_selftest_timeout(int limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return MXFP4_ERR_ARG;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    cudaError_t e = launch_timeout_selftest(di.status, static_cast<uint64_t>(limit_us) * 1000ull,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

}  // extern "C"

// ====================================================================== no-allocation variant
//
// mxfp4_gemm_noalloc: the same launches as mxfp4_gemm_ex, with the workspace replaced by
// the file-scope array below. Host code must not use the array's name as a device pointer
// (on the host it only names a stand-in); its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.

namespace mxfp4 {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MXFP4_NOALLOC_SCRATCH_BYTES];

static int noalloc_scratch(int device, uint8_t** out) {
    static std::mutex mu;
    static uint8_t* addr[64] = {};
    if (device < 0 || device >= 64) return MXFP4_ERR_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        addr[device] = static_cast<uint8_t*>(p);
    }
    *out = addr[device];
    return MXFP4_OK;
}

}  // namespace mxfp4

extern "C" int mxfp4_gemm_noalloc(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N,
                                  void* c, int64_t ldc, void* stream) {
    if (M < 0 || N < 0 || K < 0) return MXFP4_ERR_ARG;
    if (K == 0 || K % 64 != 0) return MXFP4_ERR_SHAPE;
    if (M == 0 || N == 0) return MXFP4_OK;
    if (lda < K || ldc < N) return MXFP4_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 30)) return MXFP4_ERR_SHAPE;
    if (!a || !packed_b || !c) return MXFP4_ERR_ARG;
    if (!aligned(a, 16) || lda % 8 != 0 || !aligned(packed_b, 1024) || !aligned(c, 2)) return MXFP4_ERR_ALIGN;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    // the automatic plan; fewer K slices while its scratch does not fit the array
    GemmPlan plan;
    st = make_plan(M, N, K, 0, 0, di.sm_count, &plan);
    if (st != MXFP4_OK) return st;
    while (plan.ws_total > MXFP4_NOALLOC_SCRATCH_BYTES && plan.splits > 1) {
        st = make_plan(M, N, K, plan.path, plan.splits / 2, di.sm_count, &plan);
        if (st != MXFP4_OK) return st;
    }
    if (plan.ws_total > MXFP4_NOALLOC_SCRATCH_BYTES) return MXFP4_ERR_WORKSPACE;
    uint8_t* ws = nullptr;
    st = noalloc_scratch(di.device, &ws);
    if (st != MXFP4_OK) return st;
    auto s = static_cast<cudaStream_t>(stream);
    const uint8_t* pb = static_cast<const uint8_t*>(packed_b);
    CUtensorMap tmap_b, tmap_a;
    st = make_map(&tmap_b, pb, N, K / 2, kTileN);
    if (st != MXFP4_OK) return st;
    tmap_a = tmap_b;
    if (plan.path == 2) {
        st = make_map(&tmap_a, ws + plan.ws_aq, M, K / 2, plan.m_tile);
        if (st != MXFP4_OK) return st;
    }
    if (plan.splits > 1) {   // the array keeps the last call's contents: start the counters at zero
        cudaError_t e = cudaMemsetAsync(ws + plan.ws_ctr, 0,
                                        static_cast<size_t>(plan.m_tiles) * plan.n_tiles * sizeof(uint32_t), s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (plan.path == 2) {
        const int64_t rows_cover = static_cast<int64_t>(align_up(static_cast<size_t>(plan.m_tiles) * plan.m_tile, 128));
        cudaError_t e = launch_quantize(static_cast<const uint16_t*>(a), M, K, lda, ws + plan.ws_aq, ws + plan.ws_sfa,
                                        rows_cover, plan.groups, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    GemmArgs g = {};
    g.a = static_cast<const uint16_t*>(a);
    g.lda = lda;
    g.sfa = ws + plan.ws_sfa;
    g.sfb = pb + packed_sf_offset(N, K);
    g.c = static_cast<uint16_t*>(c);
    g.ldc = ldc;
    g.part = plan.splits > 1 ? reinterpret_cast<float*>(ws + plan.ws_part) : nullptr;
    g.ctr = plan.splits > 1 ? reinterpret_cast<uint32_t*>(ws + plan.ws_ctr) : nullptr;
    g.status = di.status;
    g.M = static_cast<int>(M);
    g.N = static_cast<int>(N);
    g.K = static_cast<int>(K);
    g.m_tile = plan.m_tile;
    g.nmc = plan.nmc;
    g.m_tiles = plan.m_tiles;
    g.n_tiles = plan.n_tiles;
    g.splits = plan.splits;
    g.k_atoms = plan.k_atoms;
    g.groups = plan.groups;
    g.stages = plan.stages;
    g.off_a = plan.off_a;
    g.off_sfb = plan.off_sfb;
    g.off_sfa = plan.off_sfa;
    g.off_bar = plan.off_bar;
    g.tmem_cols = plan.tmem_cols;
    g.fused = plan.path == 1 ? 1 : 0;
    g.wait_limit_ns = g_wait_limit_ns;
    cudaError_t e = launch_gemm(plan, tmap_b, tmap_a, g, s);
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}
