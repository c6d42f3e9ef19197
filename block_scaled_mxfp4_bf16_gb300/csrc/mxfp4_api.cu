// C ABI of the MXFP4 library: argument checks, the GEMM plan (tiling, split-K, path) and the
// launches. See include/mxfp4_gb300.h for the contract of each call.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>

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
static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t packed_b_bytes(int64_t N, int64_t K) {
    return static_cast<size_t>(cdiv(N, kTileN)) * static_cast<size_t>(cdiv(K, kAtomK)) * kWBlock;
}

// ------------------------------------------------------------------ the GEMM plan

// Shared-memory layout, tensor-memory columns and workspace of a plan whose tiling, path and
// split count are set. MXFP4_ERR_SHAPE if it does not fit.
static int plan_layout(GemmPlan& p, int max_stages) {
    p.atoms_max = static_cast<int>(cdiv(p.k_atoms, p.splits));
    const size_t bar_bytes = 256;
    const size_t budget = kSmemLimit - 1024 - bar_bytes;
    // fused: every atom's token block and the bf16 A slice of the real rows stay resident
    const size_t raw_bytes = p.path == 1 ? static_cast<size_t>(p.raw_rows) * raw_pitch(p.atoms_max) : 0;
    size_t fixed = raw_bytes, per_stage = kWBlock;
    if (p.path == 1) fixed += static_cast<size_t>(p.atoms_max) * p.a_block;
    else per_stage += p.a_block;
    if (fixed + per_stage > budget) return MXFP4_ERR_SHAPE;
    p.stages = static_cast<int>(std::min<size_t>({static_cast<size_t>(max_stages), static_cast<size_t>(p.atoms_max),
                                                  (budget - fixed) / per_stage}));
    // Two MMA issuers (one accumulator each, alternate steps) while their columns fit. On the
    // two-kernel path, when every step has a stage of its own (no refills), an epilogue warp
    // (idle during the MMAs there) is a third issuer: the issue chain is then the whole MMA phase
    // (64x7168x2048 1.32 -> 1.02 us); with refills the ring's round trip is the limit and a third
    // issuer gained nothing (256x4096x7168). A tile of more than 128 tokens has two issuers that
    // each take one part of every step's tokens (the first 128, the rest), with scale columns of
    // their own and one accumulator between them: one thread's ten tcgen05 instructions per step,
    // not the tensor core, set the pace there.
    const bool wide = p.m_tile > 128;
    p.issuers = wide ? 2 : std::min(2, p.atoms_max);
    if (p.path == 2 && !wide && p.atoms_max >= 3 && p.stages == p.atoms_max) p.issuers = 3;
    auto halves = [&]() { return wide && p.issuers == 2; };
    auto sf_cols = [&]() {
        return halves() ? static_cast<uint32_t>(p.stages) * 32u : static_cast<uint32_t>(p.stages) * 8u * (1u + p.nmc);
    };
    auto acc_cols = [&]() { return static_cast<uint32_t>(halves() ? p.m_tile : p.issuers * p.m_tile); };
    while (p.issuers > 1 && acc_cols() + sf_cols() > 512u) --p.issuers;
    // An issuer tells a stage's fills apart only by the parity of its full barrier, so it must
    // never wait for a stage's next fill before the previous fill of that stage has landed. That
    // holds when each stage has a single consumer (stages a multiple of the issuers, each issuer
    // taking every issuers-th step) or when no stage is refilled. Otherwise drop stages to a
    // multiple of the issuers, or issuers to a divisor of the stages.
    // (In halves every issuer consumes every fill, and a stage is refilled only once both
    // have released it.)
    if (!halves() && p.atoms_max > p.stages && p.stages % p.issuers != 0) {
        if (p.stages >= 2 * p.issuers) p.stages -= p.stages % p.issuers;
        else
            while (p.stages % p.issuers != 0) --p.issuers;
    }
    // Scale factors written into tensor memory by epilogue warps, so that the tensor pipe runs
    // MMAs only, where that pipe is the limit: two issuers sharing every step, or a ring that
    // refills (256x4096x7168 11.92 -> 11.74 us, 2048x4096x7168 36.4 -> 34.3). Plans whose steps
    // all have stages of their own are faster with the copies (64x7168x2048 4.82 against 4.85).
    p.sf_stores = p.path == 2 && (halves() || p.atoms_max > p.stages) ? 1 : 0;
    p.off_a = static_cast<uint32_t>(p.stages) * kWBlock;
    const int a_slots = p.path == 1 ? p.atoms_max : p.stages;
    p.off_araw = p.off_a + static_cast<uint32_t>(a_slots) * p.a_block;
    size_t end = align_up(p.off_araw + raw_bytes, 1024);
    const uint32_t cols = acc_cols() + sf_cols();
    p.tmem_cols = 32;
    while (p.tmem_cols < cols) p.tmem_cols <<= 1;
    // CTAs of this kernel that may share an SM: as many as tensor memory holds without any
    // allocation having to wait (at most 2). Shared memory then keeps more from landing on one SM.
    const int per_sm = std::max(1, std::min(2, static_cast<int>(512u / p.tmem_cols)));
    const size_t sm_smem = 233472;   // shared memory per SM; each CTA also reserves 1 KB
    auto fits = [&](size_t end, int n) { return n * (end + bar_bytes + 1024 + 1024) <= sm_smem; };
    // reduction receive buffer: [source rank][weight row][padded run of owned rows] fp32
    const size_t recv_bytes = p.splits > 1 ? red_recv_floats(red_rows_per(p.m_tile, p.splits), p.splits) * sizeof(float)
                                           : static_cast<size_t>(p.m_tile) * kTileN * sizeof(float);
    const size_t end_dedicated = align_up(end + recv_bytes, 1024);
    const size_t end_shared = std::max(end, align_up(recv_bytes, 1024));
    // a dedicated buffer saves a cluster barrier; giving up a co-resident CTA costs more
    const size_t pipe_end = end;   // pipeline buffers (and the fused path's A) end here
    if (p.splits > 1 && end_dedicated <= budget && (fits(end_dedicated, per_sm) || !fits(end_shared, per_sm))) {
        p.recv_dedicated = 1;       // peers may post while this CTA still runs MMAs
        p.off_recv = static_cast<uint32_t>(end);
        end = end_dedicated;
    } else {
        p.recv_dedicated = 0;       // over the pipeline buffers, written once every MMA is done
        p.off_recv = 0;
        end = end_shared;
    }
    // Long runs of owned rows (the row form) go as one bulk copy per owner from a staged tile;
    // the tile [m_tile][128] fp32 sits in the pipeline buffers, after the receive buffer when
    // that shares them.
    p.red_bulk = 0;
    p.off_stage = 0;
    if (p.splits > 1 && red_rows_per(p.m_tile, p.splits) > kRedVecMaxRows) {
        const size_t stage_bytes = static_cast<size_t>(p.m_tile) * kTileN * sizeof(float);
        const size_t at = p.recv_dedicated ? 0 : align_up(recv_bytes, 1024);
        if (at + stage_bytes <= pipe_end) {
            p.red_bulk = 1;
            p.off_stage = static_cast<uint32_t>(at);
        }
    }
    // no more CTAs per SM than tensor memory serves: pad shared memory so a further one cannot fit
    const size_t floor_bytes = sm_smem / (per_sm + 1) + 1;
    if (end + bar_bytes + 1024 + 1024 < floor_bytes) end = align_up(floor_bytes - bar_bytes - 1024 - 1024, 1024);
    p.off_bar = static_cast<uint32_t>(end);
    p.smem_bytes = p.off_bar + bar_bytes + 1024;
    if (p.smem_bytes > kSmemLimit) return MXFP4_ERR_SHAPE;
    p.ctas = p.m_tiles * p.n_tiles * p.splits;
    p.ws_total = p.path == 2 ? static_cast<size_t>(p.m_tiles) * p.k_atoms * p.a_block : 0;
    return MXFP4_OK;
}

// Clusters of a given size and shared memory resident at once on the current device (cached).
static int active_clusters(int device, int size, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(device, size, smem);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const int n = max_active_clusters(size, smem);
    cache[key] = n;
    return n;
}

static int active_clusters_resident(int device, int size, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(device, size, smem);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const int n = max_active_clusters_resident(size, smem);
    cache[key] = n;
    return n;
}

// Shared memory, tensor memory and limits of a weight-resident plan whose token tile and split
// count are set. one_per_sm pads shared memory so that no second CTA fits on an SM; otherwise a
// CTA of the next call can start beside one of this call (and request its weights early).
// MXFP4_ERR_SHAPE if the slice does not fit the kernel.
// max_items: 1x32 blocks of A a quantizing thread may take (kResManyItemsPerThread only on plans
// that read A before the dependency wait).
static int plan_resident_layout(GemmPlan& p, bool one_per_sm, int max_items = kResMaxItemsPerThread) {
    p.atoms_max = static_cast<int>(cdiv(p.k_atoms, p.splits));
    if (p.atoms_max > kResMaxAtoms) return MXFP4_ERR_SHAPE;
    const int64_t blocks = static_cast<int64_t>(p.raw_rows) * p.atoms_max * 8;
    if (blocks > static_cast<int64_t>(kResQuantThreads) * max_items) return MXFP4_ERR_SHAPE;
    p.many_items = blocks > static_cast<int64_t>(kResQuantThreads) * kResMaxItemsPerThread ? 1 : 0;
    p.nmc = 1;
    p.a_block = static_cast<uint32_t>(p.m_tile) * 128u + 2u * kSfChunk;
    p.stages = p.atoms_max;
    p.issuers = p.m_tile == 16 && p.atoms_max >= 3 ? 3 : 2;
    p.off_a = static_cast<uint32_t>(p.atoms_max) * kWBlock;
    p.off_araw = 0;
    p.off_recv = p.off_a + static_cast<uint32_t>(p.atoms_max) * p.a_block;
    const size_t recv_bytes = p.splits > 1 ? static_cast<size_t>(p.splits) * res_rows_per_owner(p.splits) *
                                                 res_row_words(p.m_tile) * sizeof(float)
                                           : 0;
    p.off_bar = static_cast<uint32_t>(align_up(p.off_recv + recv_bytes, 16));
    size_t end = p.off_bar + static_cast<size_t>(kResMaxAtoms + 3) * 8 + 8;
    // one CTA per SM: pad so that a second one cannot fit next to it
    const size_t sm_smem = 233472, one_only = sm_smem / 2 + 1;
    if (one_per_sm && end + 2048 < one_only) end = one_only - 2048;
    p.smem_bytes = align_up(end, 16) + 1024;      // + the 1 KB alignment of the base
    if (p.smem_bytes > kSmemLimit) return MXFP4_ERR_SHAPE;
    const uint32_t cols = static_cast<uint32_t>(p.issuers * p.m_tile) + 16u * static_cast<uint32_t>(p.atoms_max);
    p.tmem_cols = 32;
    while (p.tmem_cols < cols) p.tmem_cols <<= 1;
    p.recv_dedicated = p.splits > 1 ? 1 : 0;
    p.red_bulk = 0;
    p.off_stage = 0;
    p.ctas = p.m_tiles * p.n_tiles * p.splits;
    p.ws_total = 0;
    return MXFP4_OK;
}

// The weight-resident plan (rules from same-box measurements of the small-M workloads):
//   * token tile 16 for M <= 16; for 17..32 tokens two 16-token tiles when K is at most two
//     256-K steps (twice the CTAs for a launch that is all latency), one 32-token tile otherwise;
//   * the most K slices, up to the portable cluster size, that keep at least two 256-K steps per
//     slice, one wave of CTAs and every cluster resident with one CTA per SM (a one-step slice
//     costs more in the reduction than it saves: 32x4096x512 2.38 us unsplit, 3.34 us in two);
//   * with split-K, shared memory is not padded, so the next call's CTAs start beside this
//     call's and request their weights early (8x2112x7168: 4.00 -> 3.70 us); without it one CTA
//     per SM measured faster (32x4096x512: 2.50 -> 2.38 us, 4x2880x512: 2.04 -> 1.91 us).
// Whether the quantizing warps may load A before the dependency wait (a caller that declared A
// ready): when two CTAs share an SM and their shared memory leaves the L1 cache less than a
// 196 KB carve-out would, the early loads measured slower (8x2112x7168, six 112 KB slices:
// 3.39 -> 3.74 us per call; 8x2112x5120, six 91 KB slices: 3.06 -> 2.91, but 3.14 -> 3.28 with
// the same slices padded to 112 KB); with one CTA per SM they measured faster (the six 112 KB
// slices padded past half the SM: 3.74 -> 3.50).
static bool res_early_ok(const GemmPlan& q) {
    const size_t per_cta = q.smem_bytes + 1024, sm_smem = 233472;
    return 2 * per_cta > sm_smem || 2 * per_cta <= 196u * 1024u;
}

static int make_resident_plan(int64_t M, int64_t N, int64_t K, int splits_req, int mtile_req, int sm_count,
                              GemmPlan* P, const int* cluster_caps, bool a_ready) {
    GemmPlan p = {};
    p.path = 3;
    if (mtile_req != 0 && mtile_req != 16 && mtile_req != 32) return MXFP4_ERR_ARG;
    p.k_atoms = static_cast<int>(cdiv(K, kAtomK));
    p.m_tile = M <= 16 || p.k_atoms <= 2 ? 16 : kResMaxMTile;
    if (mtile_req) p.m_tile = mtile_req;
    p.m_tiles = static_cast<int>(cdiv(M, p.m_tile));
    p.n_tiles = static_cast<int>(cdiv(N, kTileN));
    p.raw_rows = static_cast<int>(std::min<int64_t>(M, p.m_tile));
    const int64_t units = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    if (units * kMaxSplits > (int64_t(1) << 31) - 1) return MXFP4_ERR_SHAPE;
    if (splits_req > 0) {
        p.splits = std::max(1, std::min({splits_req, p.k_atoms, kMaxSplits}));
        int st = plan_resident_layout(p, p.splits == 1);
        // a slice with more of A than two blocks per quantizing thread: the kernel variant that
        // takes up to kResManyItemsPerThread (chosen automatically only where A is read early)
        if (st != MXFP4_OK) st = plan_resident_layout(p, p.splits == 1, kResManyItemsPerThread);
        if (st != MXFP4_OK) return st;
        p.a_early = a_ready && res_early_ok(p) ? 1 : 0;
        *P = p;
        return MXFP4_OK;
    }
    int dev = 0;
    if (!cluster_caps && cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const int s_max = static_cast<int>(std::min<int64_t>({static_cast<int64_t>(kAutoMaxSplits),
                                                          std::max(1, p.k_atoms / 2),
                                                          std::max<int64_t>(1, sm_count / std::max<int64_t>(1, units))}));
    // A declared ready but the flagless plan leaves no room to read it early (or there is no
    // flagless plan): the most slices whose CTAs fill at most half the SMs, one per SM, so that
    // the next call's CTAs start on the other half, take their weights and quantize their A while
    // this call runs (8x2112x7168: six slices 3.39 us per call, four slices on 68 SMs 2.83;
    // 4x2112x7168 3.08 -> 2.82). Its A phase overlaps the call ahead, so a quantizing thread may
    // take up to kResManyItemsPerThread blocks.
    auto side_by_side = [&](int s_below, GemmPlan* out) {
        const int s_half = static_cast<int>(std::min<int64_t>(
            {static_cast<int64_t>(kAutoMaxSplits), std::max(1, p.k_atoms / 2),
             std::max<int64_t>(1, sm_count / 2 / std::max<int64_t>(1, units))}));
        if (units * 2 > sm_count) return false;
        for (int s2 = std::min(s_half, s_below); s2 >= 1; --s2) {
            GemmPlan h = p;
            h.splits = s2;
            if (plan_resident_layout(h, true, kResManyItemsPerThread) != MXFP4_OK) return false;
            const int res2 = cluster_caps ? cluster_caps[s2] : active_clusters_resident(dev, s2, h.smem_bytes);
            if (s2 == 1 || units <= res2) {
                h.a_early = 1;
                *out = h;
                return true;
            }
        }
        return false;
    };
    int last = MXFP4_ERR_SHAPE;
    for (int s = s_max; s >= 1; --s) {
        GemmPlan q = p;
        q.splits = s;
        last = plan_resident_layout(q, true);     // residency judged with one CTA per SM
        if (last != MXFP4_OK) break;              // fewer slices only make each one larger
        const int resident = cluster_caps ? cluster_caps[s] : active_clusters_resident(dev, s, q.smem_bytes);
        if (s == 1 || units <= resident) {
            if (s > 1 && (last = plan_resident_layout(q, false)) != MXFP4_OK) break;
            q.a_early = a_ready && res_early_ok(q) ? 1 : 0;
            if (a_ready && !q.a_early && side_by_side(s - 1, P)) return MXFP4_OK;
            *P = q;
            return MXFP4_OK;
        }
    }
    if (a_ready && side_by_side(s_max, P)) return MXFP4_OK;
    return last;
}

// Token tile of the streaming kernel's plans (and of the public token-block layout) for M tokens
// of depth K: the request (a multiple of 16, at most kMaxMTile) cut to M rounded up to 16, or
// the planner's own choice when mtile_req is 0.
static int token_tile(int64_t M, int64_t K, int mtile_req) {
    if (mtile_req > 0) return static_cast<int>(std::min<int64_t>(cdiv(M, 16) * 16, mtile_req));
    // 17..32 tokens with at most two 256-K steps: two 16-token tiles, twice the CTAs for a launch
    // that is all latency (32x4096x512: 3.65 -> 3.51 us, 32x2880x512: 3.60 -> 3.53 us; 64 tokens
    // at K = 2048 measured slower split)
    if (M > 16 && M <= 32 && cdiv(K, kAtomK) <= 2) return 16;
    // all of M up to 128; 128 up to M = 512 (half the A traffic and reduction per CTA of a 256
    // tile, measured faster on 256x4096x7168); 256 beyond
    return M <= 128 ? static_cast<int>(cdiv(M, 16) * 16) : (M <= 512 ? 128 : kMaxMTile);
}

int make_plan(int64_t M, int64_t N, int64_t K, int path_req, int splits_req, int mtile_req, int sm_count,
              GemmPlan* P, const int* cluster_caps, bool a_ready) {
    GemmPlan p = {};
    if (M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_SHAPE;
    if (mtile_req < 0 || mtile_req > kMaxMTile || mtile_req % 16 != 0) return MXFP4_ERR_ARG;
    if (path_req == 3) return make_resident_plan(M, N, K, splits_req, mtile_req, sm_count, P, cluster_caps, a_ready);
    p.m_tile = token_tile(M, K, mtile_req);
    p.nmc = (p.m_tile + 127) / 128;
    p.m_tiles = static_cast<int>(cdiv(M, p.m_tile));
    p.n_tiles = static_cast<int>(cdiv(N, kTileN));
    p.k_atoms = static_cast<int>(cdiv(K, kAtomK));
    p.a_block = static_cast<uint32_t>(p.m_tile) * 128u + static_cast<uint32_t>(p.nmc) * 2u * kSfChunk;
    p.raw_rows = static_cast<int>(std::min<int64_t>(M, p.m_tile));
    const int64_t units = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    if (units * kMaxSplits > (int64_t(1) << 31) - 1) return MXFP4_ERR_SHAPE;
    // Up to 32 tokens the weight-resident kernel is the automatic choice wherever its K slices
    // fit (it measured faster than both other paths on every such workload).
    if (path_req == 0 && M <= 32 && mtile_req == 0 &&
        make_resident_plan(M, N, K, splits_req, 0, sm_count, P, cluster_caps, a_ready) == MXFP4_OK)
        return MXFP4_OK;
    // Fused quantization puts A's load and quantization on the GEMM's critical path (behind the
    // dependency wait), while the two-kernel path overlaps them with the weight prologue but adds
    // a kernel and a dependency hop; the fused path wins for small token counts (below).
    p.path = path_req ? path_req : (M <= 32 ? 1 : 2);
    if (p.path != 1 && p.path != 2) return MXFP4_ERR_ARG;
    int dev = 0;
    if (!cluster_caps && cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    auto layout_once = [&](GemmPlan& q) { return plan_layout(q, kMaxStages); };
    auto layout = [&](GemmPlan& q) {
        int st = layout_once(q);
        if (st != MXFP4_OK && q.path == 1 && path_req == 0) {   // fused slice too big: two-kernel path
            q.path = 2;
            st = layout_once(q);
        }
        return st;
    };
    // 129..512 tokens: 64-token tiles instead of 128 when that is still one wave of CTAs, unsplit,
    // with every 256-K step in a stage of its own. Twice the CTAs share the 128-token MMAs' tensor
    // time; past one wave, or with a refilled ring (long K), the 128-token plan stays faster.
    // Same-box graph replay, 128 -> 64: 256x3072x1536 5.85 -> 5.36 us, 256x2048x1024 6.72 -> 4.60,
    // 512x2048x2048 6.97 -> 6.73, 200x4096x512 4.48 -> 4.23, 384x2880x1024 5.50 -> 5.47; against:
    // 160x7168x2048 (168 CTAs) 7.03 -> 9.41, 256x4096x7168 (28 steps) 11.92 -> 12.69.
    if (path_req != 1 && splits_req == 0 && mtile_req == 0 && p.path == 2 && M > 128 && M <= 512) {
        GemmPlan q = p;
        q.m_tile = 64;
        q.nmc = 1;
        q.m_tiles = static_cast<int>(cdiv(M, q.m_tile));
        q.a_block = static_cast<uint32_t>(q.m_tile) * 128u + 2u * kSfChunk;
        q.raw_rows = q.m_tile;
        q.splits = 1;
        if (static_cast<int64_t>(q.m_tiles) * q.n_tiles <= sm_count && layout_once(q) == MXFP4_OK &&
            q.stages == q.atoms_max) {
            *P = q;
            return MXFP4_OK;
        }
    }
    if (splits_req > 0) {
        p.splits = std::max(1, std::min({splits_req, p.k_atoms, kMaxSplits}));
        const int st = layout(p);
        if (st != MXFP4_OK) return st;
        *P = p;
        return MXFP4_OK;
    }
    // Automatic path for up to 32 tokens: the fused plan in 16-token tiles, while its in-kernel
    // quantization is at most one 1x32 block per thread and its CTAs fit in one wave. Measured:
    // 16x2112x7168 (two blocks per thread) fused 5.40 us, two-kernel 5.09 us; 32x4096x512 fused in
    // 16-token tiles 3.25 us, two-kernel 3.57 us; 32x2880x512 3.18 vs 3.46 us.
    if (path_req == 0 && p.path == 1) {
        GemmPlan f;
        if (make_plan(M, N, K, 1, 0, mtile_req ? mtile_req : 16, sm_count, &f, cluster_caps) == MXFP4_OK &&
            static_cast<int64_t>(f.raw_rows) * 8 * f.atoms_max <= kGemmThreads && f.ctas <= sm_count) {
            *P = f;
            return MXFP4_OK;
        }
        p.path = 2;
    }
    // Automatic: as many K slices as fill the SMs (within the portable cluster size), fewer if
    // that many clusters would not all be resident at once.
    // A split must buy more than its reduction costs: with few output tiles (under a quarter of
    // the SMs) each slice keeps at least two 256-K steps, otherwise at least eight (measured on
    // the 32x4096x512, 64x7168x2048 and 256x4096x7168 workloads).
    const int64_t fill = std::max<int64_t>(1, sm_count / std::max<int64_t>(1, units));
    const int64_t by_atoms = units * 4 < sm_count ? p.k_atoms / 2 : p.k_atoms / 8;
    const int s_cap = p.path == 2 ? kAutoMaxSplitsTwoKernel : kAutoMaxSplits;
    const int s_max = static_cast<int>(std::min<int64_t>({fill, std::max<int64_t>(1, by_atoms),
                                                          static_cast<int64_t>(s_cap)}));
    for (int s = s_max; s >= 1; --s) {
        GemmPlan q = p;
        q.splits = s;
        const int st = layout(q);
        if (st != MXFP4_OK) return st;
        const int resident = cluster_caps ? cluster_caps[s] : active_clusters(dev, s, q.smem_bytes);
        if (s == 1 || units <= resident) {
            *P = q;
            return MXFP4_OK;
        }
    }
    return MXFP4_ERR_SHAPE;
}

// The plan of (device, M, N, K, options) never changes within a process (it depends on the
// device's SM count and cluster residency, both fixed), so the entry points keep the last few in
// a small per-thread table instead of running the planner on every call (about 0.5 us of host
// time a call on the benchmark's workloads).
static int cached_plan(const DeviceInfo& di, int64_t M, int64_t N, int64_t K, int path_req, int splits_req,
                       int mtile_req, GemmPlan* P, bool a_ready = false) {
    struct Entry {
        int device, path, splits, mtile;
        bool a_ready;
        int64_t M, N, K;
        GemmPlan plan;
        bool used;
    };
    constexpr int kEntries = 16;
    static thread_local Entry table[kEntries] = {};
    static thread_local int next = 0;
    for (int i = 0; i < kEntries; ++i) {
        const Entry& e = table[i];
        if (e.used && e.M == M && e.N == N && e.K == K && e.device == di.device && e.path == path_req &&
            e.splits == splits_req && e.mtile == mtile_req && e.a_ready == a_ready) {
            *P = e.plan;
            return MXFP4_OK;
        }
    }
    const int st = make_plan(M, N, K, path_req, splits_req, mtile_req, di.sm_count, P, nullptr, a_ready);
    if (st != MXFP4_OK) return st;
    Entry& e = table[next];
    next = (next + 1) % kEntries;
    e = Entry{di.device, path_req, splits_req, mtile_req, a_ready, M, N, K, *P, true};
    return MXFP4_OK;
}

static uint64_t g_wait_limit_ns = 1000000000ull;   // 1 s per bounded wait

#ifdef MXFP4_TEST_HOOKS
static void* g_token_dump = nullptr;   // test build only: see mxfp4_test_token_dump
#endif

// Argument checks shared by the GEMM entry points.
static int check_gemm_args(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N,
                           const void* c, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return MXFP4_ERR_ARG;
    if (K == 0 || K % 8 != 0) return MXFP4_ERR_SHAPE;
    if (M == 0 || N == 0) return MXFP4_OK;
    if (lda < K || ldc < N) return MXFP4_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 30)) return MXFP4_ERR_SHAPE;
    if (!a || !packed_b || !c) return MXFP4_ERR_ARG;
    if (!aligned(a, 16) || lda % 8 != 0 || !aligned(packed_b, 1024) || !aligned(c, 2)) return MXFP4_ERR_ALIGN;
    return MXFP4_OK;
}

// Enqueue one planned GEMM: the quantize kernel into `ws` for the two-kernel path, then the GEMM.
// quantize_a = false: the two-kernel plan's token blocks are already in `ws` (the GEMM alone).
static int run_gemm(const GemmPlan& plan, const DeviceInfo& di, const void* a, int64_t M, int64_t K, int64_t lda,
                    const void* packed_b, int64_t N, void* c, int64_t ldc, uint8_t* ws, cudaStream_t s,
                    bool quantize_a = true, bool a_ready = false) {
    if (plan.path == 3) {
        ResidentArgs r = {};
        r.a = static_cast<const uint16_t*>(a);
        r.lda = lda;
        r.bblk = static_cast<const uint8_t*>(packed_b);
        r.c = static_cast<uint16_t*>(c);
        r.ldc = ldc;
        r.status = di.status;
        r.M = static_cast<int>(M);
        r.N = static_cast<int>(N);
        r.K = static_cast<int>(K);
        r.m_tile = plan.m_tile;
        r.m_tiles = plan.m_tiles;
        r.n_tiles = plan.n_tiles;
        r.splits = plan.splits;
        r.k_atoms = plan.k_atoms;
        r.issuers = plan.issuers;
        r.a_early = plan.a_early;
        r.a_block = plan.a_block;
        r.off_a = plan.off_a;
        r.off_recv = plan.off_recv;
        r.off_bar = plan.off_bar;
        r.tmem_cols = plan.tmem_cols;
        r.wait_limit_ns = g_wait_limit_ns;
#ifdef MXFP4_TEST_HOOKS
        r.token_dump = static_cast<uint8_t*>(g_token_dump);
#endif
        cudaError_t e = launch_gemm_resident(plan, r, s);
        return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
    }
    if (plan.path == 2 && quantize_a) {
        cudaError_t e = launch_quantize_blocks(static_cast<const uint16_t*>(a), M, K, lda, ws, plan.m_tile,
                                               plan.m_tiles, plan.k_atoms, plan.a_block, a_ready, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    GemmArgs g = {};
    g.a = static_cast<const uint16_t*>(a);
    g.lda = lda;
    g.ablk = ws;
    g.bblk = static_cast<const uint8_t*>(packed_b);
    g.c = static_cast<uint16_t*>(c);
    g.ldc = ldc;
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
    g.stages = plan.stages;
    g.atoms_max = plan.atoms_max;
    g.issuers = plan.issuers;
    g.a_block = plan.a_block;
    g.off_a = plan.off_a;
    g.off_araw = plan.off_araw;
    g.red_bulk = plan.red_bulk;
    g.off_stage = plan.off_stage;
    g.off_recv = plan.off_recv;
    g.recv_dedicated = plan.recv_dedicated;
    g.off_bar = plan.off_bar;
    g.tmem_cols = plan.tmem_cols;
    g.fused = plan.path == 1 ? 1 : 0;
    g.sf_stores = plan.sf_stores;
    g.a_ready = a_ready ? 1 : 0;
    g.c_vec4 = (ldc % 4 == 0 && aligned(c, 8)) ? 1 : 0;
    g.wait_limit_ns = g_wait_limit_ns;
#ifdef MXFP4_TEST_HOOKS
    g.token_dump = static_cast<uint8_t*>(g_token_dump);
#endif
    cudaError_t e = launch_gemm(plan, g, s);
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

}  // namespace mxfp4

using namespace mxfp4;

// ====================================================================== C ABI

// Options a call may not take: a negative override, a path out of range, or a flag bit other
// than MXFP4_GEMM_A_READY.
static bool bad_options(const mxfp4_gemm_options* o) {
    return o && (o->path < 0 || o->path > 3 || o->splits < 0 || o->m_tile < 0 ||
                 (o->flags & ~MXFP4_GEMM_A_READY) != 0);
}

static bool options_a_ready(const mxfp4_gemm_options* o) {
    return o && (o->flags & MXFP4_GEMM_A_READY) != 0;
}

// The planner's decisions as the public mxfp4_plan_info.
static void fill_plan_info(const mxfp4::GemmPlan& plan, mxfp4_plan_info* info) {
    using namespace mxfp4;
    mxfp4_plan_info out = {};
    out.path = plan.path;
    out.splits = plan.splits;
    out.m_tile = plan.m_tile;
    out.ctas = plan.ctas;
    out.stages = plan.stages;
    out.issuers = plan.issuers;
    // the form every CTA of a full token tile uses (a ragged last tile may post short runs)
    out.reduction = plan.splits == 1 ? 0
                    : plan.path == 3 ? 4
                    : plan.red_bulk ? 3
                    : (red_rows_per(plan.m_tile, plan.splits) <= kRedVecMaxRows ? 2 : 1);
    out.recv_dedicated = plan.splits > 1 ? plan.recv_dedicated : 0;
    out.smem_bytes = static_cast<int>(plan.smem_bytes);
    out.tmem_cols = static_cast<int>(plan.tmem_cols);
    out.scale_stores = plan.sf_stores;
    out.a_early = plan.a_early;
    *info = out;
}

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

int mxfp4_version(void) { return 204; }

int mxfp4_quantize(const void* x, int64_t rows, int64_t K, int64_t ld, void* q, void* scales, void* stream) {
    if (rows < 0 || K < 0) return MXFP4_ERR_ARG;
    if (K % 8 != 0) return MXFP4_ERR_SHAPE;
    if (rows == 0 || K == 0) return MXFP4_OK;
    if (ld < K) return MXFP4_ERR_SHAPE;
    if (!x || !q || !scales) return MXFP4_ERR_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || ld % 8 != 0) return MXFP4_ERR_ALIGN;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    cudaError_t e = launch_quantize(static_cast<const uint16_t*>(x), rows, K, ld, static_cast<uint8_t*>(q),
                                    static_cast<uint8_t*>(scales), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

// The largest weight matrix the GEMM takes (its own check below); prepacking a larger one
// would only build a buffer that no GEMM call accepts.
static bool weight_dims_fit(int64_t N, int64_t K) {
    return N <= (int64_t(1) << 31) - 1 && K <= (int64_t(1) << 30);
}

size_t mxfp4_prepack_b_size(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % 8 != 0 || !weight_dims_fit(N, K)) return 0;
    return packed_b_bytes(N, K);
}

int mxfp4_prepack_b(const void* bq, const void* bs, int64_t N, int64_t K, void* packed, void* stream) {
    if (N <= 0 || K <= 0) return MXFP4_ERR_ARG;
    if (K % 8 != 0 || !weight_dims_fit(N, K)) return MXFP4_ERR_SHAPE;
    if (!bq || !bs || !packed) return MXFP4_ERR_ARG;
    if (!aligned(bq, 16) || !aligned(packed, 1024)) return MXFP4_ERR_ALIGN;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    cudaError_t e = launch_prepack(static_cast<const uint8_t*>(bq), static_cast<const uint8_t*>(bs), N, K,
                                   static_cast<uint8_t*>(packed), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

size_t mxfp4_gemm_workspace_size_ex(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options* opts) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 8 != 0 || bad_options(opts)) return 0;
    DeviceInfo di;
    if (device_info(&di) != MXFP4_OK) return 0;
    GemmPlan plan;
    if (cached_plan(di, M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, opts ? opts->m_tile : 0, &plan,
                    options_a_ready(opts)) != MXFP4_OK)
        return 0;
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
    if (K % 8 != 0) return MXFP4_ERR_SHAPE;
    if (bad_options(opts)) return MXFP4_ERR_ARG;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    GemmPlan plan;
    st = cached_plan(di, M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, opts ? opts->m_tile : 0, &plan,
                    options_a_ready(opts));
    if (st != MXFP4_OK) return st;
    if (path) *path = plan.path;
    if (splits) *splits = plan.splits;
    if (m_tile) *m_tile = plan.m_tile;
    if (ctas) *ctas = plan.ctas;
    if (stages) *stages = plan.stages;
    return MXFP4_OK;
}

int mxfp4_gemm_plan_info(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options* opts, mxfp4_plan_info* info) {
    if (!info) return MXFP4_ERR_ARG;
    if (M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_ARG;
    if (K % 8 != 0) return MXFP4_ERR_SHAPE;
    if (bad_options(opts)) return MXFP4_ERR_ARG;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    GemmPlan plan;
    st = cached_plan(di, M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, opts ? opts->m_tile : 0, &plan,
                    options_a_ready(opts));
    if (st != MXFP4_OK) return st;
    fill_plan_info(plan, info);
    return MXFP4_OK;
}

int mxfp4_gemm_plan_model(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options* opts, int sm_count,
                          const int* cluster_caps, mxfp4_plan_info* info) {
    if (!info || sm_count < 1) return MXFP4_ERR_ARG;
    if (M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_ARG;
    if (K % 8 != 0) return MXFP4_ERR_SHAPE;
    if (bad_options(opts)) return MXFP4_ERR_ARG;
    int caps[kMaxSplits + 1];
    for (int s = 0; s <= kMaxSplits; ++s) caps[s] = cluster_caps ? cluster_caps[s] : (1 << 30);
    GemmPlan plan;
    const int st = make_plan(M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, opts ? opts->m_tile : 0,
                             sm_count, &plan, caps, options_a_ready(opts));
    if (st != MXFP4_OK) return st;
    fill_plan_info(plan, info);
    return MXFP4_OK;
}

}  // extern "C"

// A call with everything checked and resolved: the plan, the device, and for host buffers where
// A comes from and where C goes. mxfp4_gemm_ex / mxfp4_gemm_host resolve one per call; a
// prepared call (mxfp4_call_create*) keeps one and only enqueues at each run.
struct mxfp4_call {
    mxfp4::DeviceInfo di;
    mxfp4::GemmPlan plan;
    bool empty;              // M == 0 or N == 0: nothing to enqueue
    bool a_ready;            // MXFP4_GEMM_A_READY
    // the GEMM itself
    const void* a;           // the device A the GEMM reads (a_dev for host buffers)
    int64_t M, K, lda, N;
    const void* packed_b;
    void* c;                 // where the GEMM stores C: the caller's C, mapped c_host, or c_dev
    int64_t ldc;
    uint8_t* ws;
    // host buffers: A arrives from a_host (mapped: staged by a kernel), C leaves to c_host
    bool host;
    const void* a_host;
    const void* a_mapped;    // device address of mapped page-locked a_host, or null (copied)
    bool a_early;            // a_host is written by the host only: staged without waiting first
    int64_t a_host_ld;
    void* a_dev;
    void* c_host;            // copy-out target when C goes through c_dev (else null)
    int64_t c_host_ld;
    void* c_dev;
};

namespace mxfp4 {

// mxfp4_gemm_ex's checks and plan, into `call`.
static int resolve_device_call(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N,
                               void* c, int64_t ldc, void* workspace, size_t ws_bytes,
                               const mxfp4_gemm_options* opts, mxfp4_call* call) {
    if (bad_options(opts)) return MXFP4_ERR_ARG;
    *call = mxfp4_call{};
    call->a_ready = opts && (opts->flags & MXFP4_GEMM_A_READY) != 0;
    int st = check_gemm_args(a, M, K, lda, packed_b, N, c, ldc);
    if (st != MXFP4_OK) return st;
    call->empty = M == 0 || N == 0;
    if (call->empty) return MXFP4_OK;
    st = device_info(&call->di);
    if (st != MXFP4_OK) return st;
    st = cached_plan(call->di, M, N, K, opts ? opts->path : 0, opts ? opts->splits : 0, opts ? opts->m_tile : 0,
                     &call->plan, call->a_ready);
    if (st != MXFP4_OK) return st;
    if (call->plan.ws_total > 0) {
        if (!workspace || ws_bytes < call->plan.ws_total) return MXFP4_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return MXFP4_ERR_ALIGN;
    }
    call->a = a;
    call->M = M;
    call->K = K;
    call->lda = lda;
    call->packed_b = packed_b;
    call->N = N;
    call->c = c;
    call->ldc = ldc;
    call->ws = static_cast<uint8_t*>(workspace);
    return MXFP4_OK;
}

// mxfp4_gemm_host's checks and plan, and where A comes from and C goes, into `call`.
static int resolve_host_call(const void* a_host, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N,
                             void* c_host, int64_t ldc, void* a_dev, void* c_dev, void* workspace, size_t ws_bytes,
                             unsigned flags, mxfp4_call* call) {
    if (flags & ~static_cast<unsigned>(MXFP4_CALL_A_HOST_WRITTEN)) return MXFP4_ERR_ARG;
    // everything the device-side call checks is checked first, so nothing is copied on an error
    int st = resolve_device_call(a_dev, M, K, K, packed_b, N, c_dev, N, workspace, ws_bytes, nullptr, call);
    if (st != MXFP4_OK || call->empty) return st;
    if (!a_host || !c_host) return MXFP4_ERR_ARG;
    if (lda < K || ldc < N) return MXFP4_ERR_SHAPE;
    call->host = true;
    call->a_host = a_host;
    call->a_host_ld = lda;
    call->a_dev = a_dev;
    call->c_dev = c_dev;
    // A: page-locked host memory mapped into the device's address space (16-byte aligned rows)
    // is staged by a kernel that reads it in place, so the launch chain from the previous call's
    // GEMM to this one is never broken by a copy-engine transfer; anything else is copied.
    cudaPointerAttributes a_attr = {};
    if (cudaPointerGetAttributes(&a_attr, a_host) == cudaSuccess && a_attr.type == cudaMemoryTypeHost)
        call->a_mapped = a_attr.devicePointer;
    else
        cudaGetLastError();   // clear the error an unregistered pointer leaves behind
    if (call->a_mapped && !(aligned(call->a_mapped, 16) && lda % 8 == 0)) call->a_mapped = nullptr;
    call->a_early = (flags & MXFP4_CALL_A_HOST_WRITTEN) != 0;
    // Page-locked host memory mapped into the device's address space takes C straight from the
    // epilogue's stores (no separate device -> host copy) when it is aligned for bf16 stores;
    // anything else goes through c_dev.
    cudaPointerAttributes attr = {};
    void* c_mapped = nullptr;
    if (cudaPointerGetAttributes(&attr, c_host) == cudaSuccess && attr.type == cudaMemoryTypeHost)
        c_mapped = attr.devicePointer;
    else
        cudaGetLastError();   // clear the error an unregistered pointer leaves behind
    if (c_mapped && aligned(c_mapped, 2)) {
        call->c = c_mapped;
        call->ldc = ldc;
    } else {
        call->c_host = c_host;
        call->c_host_ld = ldc;
    }
    return MXFP4_OK;
}

// Enqueue a resolved call on `s`.
static int run_call(const mxfp4_call& call, cudaStream_t s) {
    if (call.empty) return MXFP4_OK;
    const size_t a_row = static_cast<size_t>(call.K) * 2, c_row = static_cast<size_t>(call.N) * 2;
    cudaError_t e;
    if (call.host) {
        if (call.a_mapped)
            e = launch_stage_rows(call.a_mapped, call.a_host_ld, call.a_dev, call.M, call.K, call.a_early, s);
        else   // one linear copy when the host rows are contiguous, a strided one otherwise
            e = call.a_host_ld == call.K
                    ? cudaMemcpyAsync(call.a_dev, call.a_host, a_row * call.M, cudaMemcpyHostToDevice, s)
                    : cudaMemcpy2DAsync(call.a_dev, a_row, call.a_host, static_cast<size_t>(call.a_host_ld) * 2,
                                        a_row, static_cast<size_t>(call.M), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    const int st = run_gemm(call.plan, call.di, call.a, call.M, call.K, call.lda, call.packed_b, call.N, call.c,
                            call.ldc, call.ws, s, true, call.a_ready);
    if (st != MXFP4_OK || !call.c_host) return st;
    e = call.c_host_ld == call.N
            ? cudaMemcpyAsync(call.c_host, call.c_dev, c_row * call.M, cudaMemcpyDeviceToHost, s)
            : cudaMemcpy2DAsync(call.c_host, static_cast<size_t>(call.c_host_ld) * 2, call.c_dev, c_row, c_row,
                                static_cast<size_t>(call.M), cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

}  // namespace mxfp4

extern "C" {

int mxfp4_gemm_ex(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N, void* c,
                  int64_t ldc, void* workspace, size_t ws_bytes, const mxfp4_gemm_options* opts, void* stream) {
    mxfp4_call call;
    const int st = resolve_device_call(a, M, K, lda, packed_b, N, c, ldc, workspace, ws_bytes, opts, &call);
    return st != MXFP4_OK ? st : run_call(call, static_cast<cudaStream_t>(stream));
}

int mxfp4_gemm(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N, void* c,
               int64_t ldc, void* workspace, size_t ws_bytes, void* stream) {
    return mxfp4_gemm_ex(a, M, K, lda, packed_b, N, c, ldc, workspace, ws_bytes, nullptr, stream);
}

int mxfp4_gemm_host(const void* a_host, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N,
                    void* c_host, int64_t ldc, void* a_dev, void* c_dev, void* workspace, size_t ws_bytes,
                    void* stream) {
    mxfp4_call call;
    const int st = resolve_host_call(a_host, M, K, lda, packed_b, N, c_host, ldc, a_dev, c_dev, workspace, ws_bytes,
                                     0u, &call);
    return st != MXFP4_OK ? st : run_call(call, static_cast<cudaStream_t>(stream));
}

size_t mxfp4_gemm_unpacked_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 8 != 0 || !weight_dims_fit(N, K)) return 0;
    return align_up(packed_b_bytes(N, K), 1024) + mxfp4_gemm_workspace_size(M, N, K);
}

int mxfp4_gemm_unpacked(const void* a, int64_t M, int64_t K, int64_t lda, const void* bq, const void* bs,
                        int64_t N, void* c, int64_t ldc, void* workspace, size_t ws_bytes, void* stream) {
    // B's packed image goes to the start of the workspace, the GEMM's own workspace after it
    if (M < 0 || N < 0 || K < 0) return MXFP4_ERR_ARG;
    if (K == 0 || K % 8 != 0 || (N > 0 && !weight_dims_fit(N, K))) return MXFP4_ERR_SHAPE;
    const size_t pb = N > 0 ? align_up(packed_b_bytes(N, K), 1024) : 0;
    const bool empty = M == 0 || N == 0;
    if (!empty) {
        if (!bq || !bs) return MXFP4_ERR_ARG;
        if (!aligned(bq, 16)) return MXFP4_ERR_ALIGN;
        if (!workspace || ws_bytes < pb) return MXFP4_ERR_WORKSPACE;
        if (!aligned(workspace, 1024)) return MXFP4_ERR_ALIGN;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    mxfp4_call call;
    const int st = resolve_device_call(a, M, K, lda, empty ? bq : ws, N, c, ldc, empty ? nullptr : ws + pb,
                                       empty ? 0 : ws_bytes - pb, nullptr, &call);
    if (st != MXFP4_OK || call.empty) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the prepack kernel never lets dependents start early, so the GEMM's early weight requests
    // see its whole image (see mxfp4_gemm); the next call's prepack waits for this GEMM
    const cudaError_t e = launch_prepack(static_cast<const uint8_t*>(bq), static_cast<const uint8_t*>(bs), N, K, ws, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return run_call(call, s);
}

int mxfp4_call_create(const void* a, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N, void* c,
                      int64_t ldc, void* workspace, size_t ws_bytes, const mxfp4_gemm_options* opts,
                      mxfp4_call** out) {
    if (!out) return MXFP4_ERR_ARG;
    *out = nullptr;
    mxfp4_call call;
    const int st = resolve_device_call(a, M, K, lda, packed_b, N, c, ldc, workspace, ws_bytes, opts, &call);
    if (st != MXFP4_OK) return st;
    *out = new (std::nothrow) mxfp4_call(call);
    return *out ? MXFP4_OK : MXFP4_ERR_ARG;
}

int mxfp4_call_create_host(const void* a_host, int64_t M, int64_t K, int64_t lda, const void* packed_b, int64_t N,
                           void* c_host, int64_t ldc, void* a_dev, void* c_dev, void* workspace, size_t ws_bytes,
                           unsigned flags, mxfp4_call** out) {
    if (!out) return MXFP4_ERR_ARG;
    *out = nullptr;
    mxfp4_call call;
    const int st = resolve_host_call(a_host, M, K, lda, packed_b, N, c_host, ldc, a_dev, c_dev, workspace, ws_bytes,
                                     flags, &call);
    if (st != MXFP4_OK) return st;
    *out = new (std::nothrow) mxfp4_call(call);
    return *out ? MXFP4_OK : MXFP4_ERR_ARG;
}

int mxfp4_call_run(const mxfp4_call* call, void* stream) {
    if (!call) return MXFP4_ERR_ARG;
    if (!call->empty) {   // a call runs on the device it was prepared on
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev != call->di.device) return MXFP4_ERR_ARG;
    }
    return run_call(*call, static_cast<cudaStream_t>(stream));
}

void mxfp4_call_destroy(mxfp4_call* call) { delete call; }

// Token-block layout of M tokens of depth K in tiles of m_tile tokens: (tiles, bytes).
static bool token_blocks_layout(int64_t M, int64_t K, int m_tile, int* m_tile_out, size_t* bytes) {
    if (M <= 0 || M > (int64_t(1) << 31) - 1 || K <= 0 || K % 8 != 0 || K > (int64_t(1) << 30)) return false;
    if (m_tile < 0 || m_tile > kMaxMTile || m_tile % 16 != 0) return false;
    const int mt = token_tile(M, K, m_tile);
    const int64_t nmc = (mt + 127) / 128;
    const size_t a_block = static_cast<size_t>(mt) * 128u + static_cast<size_t>(nmc) * 2u * kSfChunk;
    *m_tile_out = mt;
    *bytes = static_cast<size_t>(cdiv(M, mt)) * static_cast<size_t>(cdiv(K, kAtomK)) * a_block;
    return true;
}

int mxfp4_token_tile(int64_t M, int64_t K, int m_tile) {
    int mt = 0;
    size_t bytes = 0;
    return token_blocks_layout(M, K, m_tile, &mt, &bytes) ? mt : 0;
}

size_t mxfp4_token_blocks_size(int64_t M, int64_t K, int m_tile) {
    int mt = 0;
    size_t bytes = 0;
    return token_blocks_layout(M, K, m_tile, &mt, &bytes) ? bytes : 0;
}

int mxfp4_quantize_tokens(const void* a, int64_t M, int64_t K, int64_t lda, int m_tile, void* blocks,
                          size_t blocks_bytes, void* stream) {
    if (M < 0 || K < 0 || m_tile < 0) return MXFP4_ERR_ARG;
    if (K == 0 || K % 8 != 0) return MXFP4_ERR_SHAPE;
    if (M == 0) return MXFP4_OK;
    int mt = 0;
    size_t need = 0;
    if (m_tile > kMaxMTile || m_tile % 16 != 0) return MXFP4_ERR_ARG;
    if (lda < K || !token_blocks_layout(M, K, m_tile, &mt, &need)) return MXFP4_ERR_SHAPE;
    if (!a || !blocks) return MXFP4_ERR_ARG;
    if (!aligned(a, 16) || lda % 8 != 0 || !aligned(blocks, 256)) return MXFP4_ERR_ALIGN;
    if (blocks_bytes < need) return MXFP4_ERR_WORKSPACE;
    DeviceInfo di;
    int st = device_info(&di);
    if (st != MXFP4_OK) return st;
    const int nmc = (mt + 127) / 128;
    const uint32_t a_block = static_cast<uint32_t>(mt) * 128u + static_cast<uint32_t>(nmc) * 2u * kSfChunk;
    cudaError_t e = launch_quantize_blocks(static_cast<const uint16_t*>(a), M, K, lda, static_cast<uint8_t*>(blocks),
                                           mt, static_cast<int>(cdiv(M, mt)), static_cast<int>(cdiv(K, kAtomK)),
                                           a_block, false, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP4_OK : cuda_fail(e);
}

int mxfp4_gemm_tokens(const void* blocks, size_t blocks_bytes, int64_t M, int64_t K, int m_tile,
                      const void* packed_b, int64_t N, void* c, int64_t ldc, int splits, void* stream) {
    if (m_tile < 0 || splits < 0) return MXFP4_ERR_ARG;
    if (m_tile > kMaxMTile || m_tile % 16 != 0) return MXFP4_ERR_ARG;
    // the GEMM's checks, with the token blocks standing where A's rows would be checked
    int st = check_gemm_args(blocks, M, K, K, packed_b, N, c, ldc);
    if (st != MXFP4_OK || M == 0 || N == 0) return st;
    int mt = 0;
    size_t need = 0;
    if (!token_blocks_layout(M, K, m_tile, &mt, &need)) return MXFP4_ERR_SHAPE;
    if (!aligned(blocks, 256)) return MXFP4_ERR_ALIGN;
    if (blocks_bytes < need) return MXFP4_ERR_WORKSPACE;
    DeviceInfo di;
    st = device_info(&di);
    if (st != MXFP4_OK) return st;
    GemmPlan plan;
    st = cached_plan(di, M, N, K, 2, splits, mt, &plan);
    if (st != MXFP4_OK) return st;
    if (plan.path != 2 || plan.m_tile != mt || plan.ws_total != need) return MXFP4_ERR_SHAPE;   // never expected
    return run_gemm(plan, di, nullptr, M, K, K, packed_b, N, c, ldc,
                    static_cast<uint8_t*>(const_cast<void*>(blocks)), static_cast<cudaStream_t>(stream), false);
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

#ifdef MXFP4_TEST_HOOKS
// Test build only (-DMXFP4_TEST_HOOKS, never the product library): the CTAs of weight tile 0 of
// a plan that quantizes A inside the GEMM (fused or weight-resident) copy the token blocks they
// quantized to `dump` ([m_tiles][k_atoms][token block bytes], device memory, large enough), so a
// test can compare the GEMM's own quantization of A byte for byte. NULL turns it off.
void mxfp4_test_token_dump(void* dump) { g_token_dump = dump; }
#endif

}  // extern "C"

// ====================================================================== no-allocation variant
//
// mxfp4_gemm_noalloc: mxfp4_gemm with the workspace replaced by the file-scope array below.
// Host code must not use the array's name as a device pointer (on the host it only names a
// stand-in); its device address comes from cudaGetSymbolAddress, looked up once per device
// with that device current.

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
    int st = check_gemm_args(a, M, K, lda, packed_b, N, c, ldc);
    if (st != MXFP4_OK || M == 0 || N == 0) return st;
    DeviceInfo di;
    st = device_info(&di);
    if (st != MXFP4_OK) return st;
    // the automatic plan, whose scratch must fit the array
    GemmPlan plan;
    st = cached_plan(di, M, N, K, 0, 0, 0, &plan);
    if (st != MXFP4_OK) return st;
    if (plan.ws_total > MXFP4_NOALLOC_SCRATCH_BYTES) return MXFP4_ERR_WORKSPACE;
    uint8_t* ws = nullptr;
    st = noalloc_scratch(di.device, &ws);
    if (st != MXFP4_OK) return st;
    // nothing in the array has to start at zero: the quantize kernel rewrites every byte the
    // GEMM reads, padding included
    return run_gemm(plan, di, a, M, K, lda, packed_b, N, c, ldc, ws, static_cast<cudaStream_t>(stream));
}
