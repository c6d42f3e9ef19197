// Weight-resident block-scaled MXFP4 GEMM for small token counts: the weight-streaming shapes
// (M up to a few tens of tokens) where a call is a chain of latencies rather than a stream of
// bandwidth.
//
// One CTA = one (128-row weight tile, token tile of at most 32, K slice of at most eight 256-K
// steps); the K slices of a tile form one thread-block cluster. Shared memory holds the whole
// slice, so the CTA asks for all of its weight blocks (the prepacked shared-memory images, one
// bulk copy each) the moment it starts, before it waits for the previous grid: the weights
// never depend on it. After that wait:
//   warps 0, 3..11: each thread loads its 1x32 blocks of bf16 A straight from global memory
//                   into registers (the addresses are computed, and on short slices the lines
//                   prefetched into L2, before the wait; when the caller declared A ready and
//                   the plan allows it, the loads themselves go first), quantizes them (the pages' in-register A
//                   quantization, submission 711914 `mxfp4_gemm_fused_k512_kernel` with
//                   `_mxfp4_quant_tile`) and writes the token blocks into shared memory;
//   warps 1, 2:     warp 1 allocates tensor memory; lane 0 of each copies its 256-K steps' weight
//                   scale factors into it as they land, then, once A is quantized, issues those
//                   steps' block-scaled MMAs into an accumulator of its own (tcgen05.mma
//                   kind::mxf4, D = C^T: one weight row per lane, one token per column);
//                   warp 3 joins as a third issuer, once it has quantized its share of A, for
//                   16-token tiles of three or more steps;
//   warps 4..7:     add the accumulators (one lane quadrant each) and reduce the K slices: rank o
//                   of the cluster owns weight rows [o*R, (o+1)*R) of the tile and every CTA
//                   sends it those rows as 16-byte st.async stores counted on the owner's
//                   mbarrier; the owner adds the slices in rank order (run-to-run identical)
//                   and stores bf16 C.
// Every wait is bounded: on timeout the kernel records an error in the device status word,
// skips the work that depended on the wait, drains its own copies and frees tensor memory.
#include <cuda_bf16.h>

#include <atomic>
#include <initializer_list>
#include <mutex>

#include "internal.h"
#include "mma_desc.cuh"
#include "ptx.cuh"
#include "quant_device.cuh"

// Phase stamps of a timing build (-DMXFP4_TRACE): each CTA takes its own row of the trace buffer
// (in start order, so consecutive launches stay apart) and records its grid id, block index and
// SM, the global timer and the SM clock at its start and end (slots 0/10 and 13/11), and the SM
// clock at each phase; a product build compiles them to nothing.
#ifdef MXFP4_TRACE
#define RES_PHASE(slot) (::mxfp4::trace_buffer[trace_row][(slot)] = ::mxfp4::sm_clock())
#else
#define RES_PHASE(slot) ((void)0)
#endif

namespace mxfp4 {

namespace {

__device__ __forceinline__ void res_fail(const ResidentArgs& p, volatile uint32_t* abort_flag) {
    atomicOr(p.status, 1u);
    *abort_flag = 1u;
}

// 32 bf16 of A from `src` with `avail` elements left in the row (a multiple of 8, > 0): the
// 16-byte pieces at or past the row's end are not read and count as zeros. Loads bypass L1
// (the lines were prefetched into L2, and A may have been written by the previous grid).
__device__ __forceinline__ void load_a_block(const uint16_t* src, int avail, uint32_t (&w)[16]) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = 8 * i < avail ? __ldcg(p + i) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
}

// One 1x32 block of A owned by a quantizing thread.
struct AItem {
    const uint16_t* src;   // first element
    int avail;             // elements of the row from src on (<= 0: past K, zero codes)
    uint32_t codes;        // byte offset of its 16 code bytes from the token blocks' base
    uint32_t sf;           // byte offset of its scale byte
    bool valid;            // the item exists
};

__device__ __forceinline__ AItem make_item(const ResidentArgs& p, int idx, int items, int nb8, int m0, int a0,
                                           uint32_t a_rows) {
    AItem it;
    it.valid = idx < items;
    const int r = it.valid ? idx / nb8 : 0;      // token row within the tile
    const int kb = it.valid ? idx - r * nb8 : 0; // 1x32 block within the slice
    const int k = a0 * kAtomK + kb * 32;
    it.avail = p.K - k;
    it.src = p.a + static_cast<int64_t>(m0 + r) * p.lda + k;
    const uint32_t blk = static_cast<uint32_t>(kb >> 3) * p.a_block;
    const uint32_t c = static_cast<uint32_t>(kb & 7);
    it.codes = blk + swz_chunk_offset(static_cast<uint32_t>(r), c);
    it.sf = blk + a_rows + block_sf_offset(static_cast<uint32_t>(r), c);
    return it;
}

__device__ __forceinline__ void quantize_item(const AItem& it, const uint32_t (&w)[16], uint8_t* sA) {
    if (!it.valid) return;
    uint32_t out[4] = {0u, 0u, 0u, 0u};
    uint32_t sbyte = 0u;
    if (it.avail > 0) sbyte = quantize_block32(w, out);
    *reinterpret_cast<uint4*>(sA + it.codes) = make_uint4(out[0], out[1], out[2], out[3]);
    sA[it.sf] = static_cast<uint8_t>(sbyte);
}

}  // namespace

// kMany: up to kResManyItemsPerThread blocks of A per quantizing thread, loaded three at a time
// (plans that read A before the dependency wait); otherwise at most two, all loaded at once.
template <bool kMany>
__global__ void __launch_bounds__(kResThreads, 1)
mxfp4_gemm_resident_kernel(const ResidentArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* sB = smem;                               // weight blocks, one per 256-K step
    uint8_t* sA = smem + p.off_a;                     // token blocks, one per 256-K step
    float* sRecv = reinterpret_cast<float*>(smem + p.off_recv);   // [source][owned row][words]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);   // [kResMaxAtoms]
    uint64_t* a_ready = full + kResMaxAtoms;          // token blocks written (one arrival per warp)
    uint64_t* acc_full = a_ready + 1;                 // accumulator complete
    uint64_t* red_bar = acc_full + 1;                 // the peers' rows have landed here
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_bar + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    // warp index from lane 0: provably warp-uniform for the role branches and tcgen05 operands
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    // ---- work unit: (token tile, weight tile, K slice)
    const int S = p.splits;
    const int split = blockIdx.x % S;                 // = rank in the cluster
    const int tile = blockIdx.x / S;
    const int nt = tile % p.n_tiles;
    const int mt = tile / p.n_tiles;
    const int n0 = nt * kTileN;
    const int m0 = mt * p.m_tile;
    const int base = p.k_atoms / S, rem = p.k_atoms % S;
    const int a0 = split * base + (split < rem ? split : rem);
    const int na = base + (split < rem ? 1 : 0);
    const int atoms_max = base + (rem > 0 ? 1 : 0);
    const int m_valid = (p.M - m0) < p.m_tile ? (p.M - m0) : p.m_tile;
    const uint64_t lim = p.wait_limit_ns;
    const int R = res_rows_per_owner(S);              // weight rows each rank owns
    const int words = res_row_words(m_valid);         // fp32 per owned row per source
    const int own0 = split * R;
    const int own_rows = max(0, min(R, kTileN - own0));

#ifdef MXFP4_TRACE
    __shared__ unsigned int trace_row_s;
    if (threadIdx.x == 0) {
        const unsigned int row = atomicAdd(&trace_counter, 1u) & 4095u;
        trace_row_s = row;
        trace_buffer[row][10] = sm_clock();
        trace_buffer[row][0] = global_timer_ns();
        trace_buffer[row][12] = sm_id();
        trace_buffer[row][14] = grid_id();
        trace_buffer[row][15] = blockIdx.x;
    }
    __syncthreads();
    const unsigned int trace_row = trace_row_s;
#endif
    if (threadIdx.x == 0) {
        for (int j = 0; j < na; ++j) mbar_init(&full[j], 1);
        mbar_init(a_ready, kResQuantThreads / 32);
        mbar_init(acc_full, static_cast<uint32_t>(p.issuers));   // one commit per MMA issuer
        mbar_init(red_bar, 1);
        if (S > 1 && own_rows > 0)    // (S - 1) peers x owned rows x words
            mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>((S - 1) * own_rows * words) * 4u);
        abort_flag[0] = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    // Split-K: every CTA arrives once its barriers exist; a warp waits before its first post.
    if (S > 1) cluster_arrive_relaxed();
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        // the whole K slice of weights, requested before anything else
        const uint8_t* bsrc = p.bblk + (static_cast<size_t>(nt) * p.k_atoms + a0) * kWBlock;
        const uint64_t pol = policy_evict_first();
        for (int j = 0; j < na; ++j) {
            mbar_arrive_expect_tx(&full[j], kWBlock);
            bulk_load(sB + j * kWBlock, bsrc + static_cast<size_t>(j) * kWBlock, kWBlock, &full[j], pol);
        }
    }

    // ------------------------------------------------------------ A quantization (10 warps)
    if (warp != 1 && warp != 2) {
        const int qt = warp == 0 ? lane : static_cast<int>(threadIdx.x) - 64;
        const int nb8 = na * 8;                       // 1x32 blocks of the slice per token row
        const int items = m_valid * nb8;
        const uint32_t a_rows = static_cast<uint32_t>(p.m_tile) * 128u;
        if constexpr (kMany) {
            // every block of the slice from this CTA's A rows, three per thread at a time
            if (!p.a_early) pdl_wait_prior_grid();   // (the planner pairs kMany with a_early)
            if (threadIdx.x == 0) RES_PHASE(2);
            for (int b = qt; b < items; b += 3 * kResQuantThreads) {
                const AItem i0 = make_item(p, b, items, nb8, m0, a0, a_rows);
                const AItem i1 = make_item(p, b + kResQuantThreads, items, nb8, m0, a0, a_rows);
                const AItem i2 = make_item(p, b + 2 * kResQuantThreads, items, nb8, m0, a0, a_rows);
                uint32_t w0[16], w1[16], w2[16];
                if (i0.valid && i0.avail > 0) load_a_block(i0.src, i0.avail, w0);
                if (i1.valid && i1.avail > 0) load_a_block(i1.src, i1.avail, w1);
                if (i2.valid && i2.avail > 0) load_a_block(i2.src, i2.avail, w2);
                quantize_item(i0, w0, sA);
                quantize_item(i1, w1, sA);
                quantize_item(i2, w2, sA);
            }
            if (threadIdx.x == 0) RES_PHASE(3);
        } else {
        const AItem it0 = make_item(p, qt, items, nb8, m0, a0, a_rows);
        const AItem it1 = make_item(p, qt + kResQuantThreads, items, nb8, m0, a0, a_rows);
        // warm L2 with this thread's A while the previous grid finishes (see prefetch_l2), on
        // slices of at most two 256-K steps: longer slices' weight requests are in flight then
        // too, and the prefetches measured no faster there (8x2112x7168 3.351 us with, 3.295
        // without; 32x4096x512 2.389 with, 2.539 without)
        if (na <= 2) {
            if (it0.valid && it0.avail > 0) prefetch_l2(it0.src);
            if (it1.valid && it1.avail > 0) prefetch_l2(it1.src);
        }
        // A may be written by the previous grid, unless the caller declared it ready before the
        // launch and the plan reads it early (a_early; the token blocks go to this CTA's shared
        // memory only, and C is written after warp 1's wait)
        if (!p.a_early) pdl_wait_prior_grid();
        if (threadIdx.x == 0) RES_PHASE(2);
        uint32_t w0[16], w1[16];
        if (it0.valid && it0.avail > 0) load_a_block(it0.src, it0.avail, w0);
        if (it1.valid && it1.avail > 0) load_a_block(it1.src, it1.avail, w1);
        quantize_item(it0, w0, sA);
        if (threadIdx.x == 0) RES_PHASE(3);
        quantize_item(it1, w1, sA);
        }
#ifdef MXFP4_TEST_HOOKS
        // test build: the token blocks of weight tile 0's CTAs, as quantized, to the dump buffer
        // [m_tiles][k_atoms][a_block]
        named_barrier(5, kResQuantThreads);
        if (nt == 0 && p.token_dump) {
            uint8_t* dump = p.token_dump + (static_cast<size_t>(mt) * p.k_atoms + a0) * p.a_block;
            const int words = na * static_cast<int>(p.a_block) / 16;
            for (int i = qt; i < words; i += kResQuantThreads)
                reinterpret_cast<uint4*>(dump)[i] = reinterpret_cast<const uint4*>(sA)[i];
        }
#endif
        fence_proxy_async_smem();                     // the MMAs read the token blocks (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(a_ready);
        if (threadIdx.x == 0) RES_PHASE(4);
    }
    const int NI = p.issuers;
    if (warp == 1 || warp == 2 || (warp == 3 && NI == 3)) {
        // ------------------------------------------------ tensor memory and the MMAs (2-3 warps)
        // Warp 1 allocates the columns once the previous grid has finished (so a CTA never holds
        // columns that a CTA of the previous grid still waits for) and publishes them to the other
        // issuing warps and the epilogue. Lane 0 of each issuing warp issues the MMAs of every
        // NI-th 256-K step into an accumulator of its own: one thread's tcgen05 issue chain is the
        // limit of this phase. Warps 1-2 issue from the start; with a third issuer, warp 3 joins
        // once it has quantized its share of A.
        const int issuer = warp - 1;
        if (warp == 1) {
            pdl_wait_prior_grid();
            tmem_alloc(const_cast<uint32_t*>(tmem_slot), p.tmem_cols);
            tmem_relinquish();
            tc_fence_before_sync();
            named_barrier_arrive(4, 64);              // to warp 2
            if (NI == 3) named_barrier_arrive(6, 64); // to warp 3
            named_barrier_arrive(1, 32 + 128);        // to the epilogue
            __syncwarp();
        } else if (warp == 2) {
            named_barrier(4, 64);
        } else {
            named_barrier(6, 64);
        }
        tc_fence_after_sync();
        const uint32_t tmem_base = *tmem_slot;
        if (lane == 0) {
            // columns: accumulators [0, NI*m_tile), weight scales 8 per step, token scales 8 per step
            const uint32_t t_acc = tmem_base + static_cast<uint32_t>(issuer * p.m_tile);
            const uint32_t t_sfw = tmem_base + static_cast<uint32_t>(NI * p.m_tile);
            const uint32_t t_sft = t_sfw + 8u * static_cast<uint32_t>(atoms_max);
            const uint32_t a_rows = static_cast<uint32_t>(p.m_tile) * 128u;
            const uint32_t idesc0 = idesc_mxf4(static_cast<uint32_t>(p.m_tile));
            const uint32_t idesc1 = idesc0 | (2u << 29) | (2u << 4);         // scale bytes {2,3}
            const uint64_t w_desc0 = desc_sw128(smem_addr(sB));
            const uint64_t t_desc0 = desc_sw128(smem_addr(sA));
            const uint64_t sfw_desc0 = desc_sf(smem_addr(sB + kBRowsBytes));
            const uint64_t sft_desc0 = desc_sf(smem_addr(sA + a_rows));
            const uint32_t w_step = kWBlock >> 4, t_step = p.a_block >> 4, chunk_step = kSfChunk >> 4;
            bool ok = true;
            // While A is being quantized, copy the scale factors of this issuer's weight steps
            // that have landed; afterwards each step's MMAs go out as soon as that step is in.
            int wsf = issuer;                         // next of this issuer's steps without scales
            {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_test_wait(a_ready, 0)) {
                    if (wsf < na && mbar_test_wait(&full[wsf], 0)) {
                        tc_fence_after_sync();
                        const uint64_t sd = sfw_desc0 + static_cast<uint32_t>(wsf) * w_step;
                        tc_copy_sf(t_sfw + 8u * wsf, sd);
                        tc_copy_sf(t_sfw + 8u * wsf + 4u, sd + chunk_step);
                        wsf += NI;
                    } else if (global_timer_ns() - t0 > lim) {
                        ok = false;
                        break;
                    }
                }
            }
            if (threadIdx.x == 32) RES_PHASE(5);
            if (ok) {
                tc_fence_after_sync();
#pragma unroll 1
                for (int j = issuer; j < na; j += NI) {
                    const uint32_t sfw = t_sfw + 8u * j, sft = t_sft + 8u * j;
                    if (j >= wsf) {
                        if (!mbar_wait(&full[j], 0, lim)) { ok = false; break; }
                        tc_fence_after_sync();
                        const uint64_t sd = sfw_desc0 + static_cast<uint32_t>(j) * w_step;
                        tc_copy_sf(sfw, sd);
                        tc_copy_sf(sfw + 4u, sd + chunk_step);
                    }
                    const uint64_t sd = sft_desc0 + static_cast<uint32_t>(j) * t_step;
                    tc_copy_sf(sft, sd);
                    tc_copy_sf(sft + 4u, sd + chunk_step);
                    const uint64_t wd = w_desc0 + static_cast<uint32_t>(j) * w_step;
                    const uint64_t td = t_desc0 + static_cast<uint32_t>(j) * t_step;
                    // K step kk of the 256: +32 bytes in both operands (descriptor +2)
                    mma_mxf4(t_acc, wd + 0, td + 0, idesc0, sfw, sft, j != issuer);
                    mma_mxf4(t_acc, wd + 2, td + 2, idesc1, sfw, sft, 1);
                    mma_mxf4(t_acc, wd + 4, td + 4, idesc0, sfw + 4u, sft + 4u, 1);
                    mma_mxf4(t_acc, wd + 6, td + 6, idesc1, sfw + 4u, sft + 4u, 1);
                }
            }
            if (!ok) res_fail(p, abort_flag);
            tc_commit(acc_full);                      // one arrival per issuer
            if (threadIdx.x == 32) RES_PHASE(6);
            // never leave copies in flight into shared memory that is about to be freed
            for (int j = issuer; j < na; j += NI) mbar_wait(&full[j], 0, lim);
        }
        __syncwarp();
        if (S > 1) cluster_wait();
        if (warp == 1) {
            named_barrier(2, 32 + 128);               // the epilogue has read the accumulators
            tc_fence_after_sync();
            tmem_dealloc(tmem_base, p.tmem_cols);
        }
        return;
    }
    // The owner's sum over the K slices: thread t of `sum_threads` sums owned row t % own_rows,
    // tokens 4g..4g+3 with g = t / own_rows, over the sources in rank order (consecutive threads:
    // consecutive rows, contiguous in C). Always waited for (bounded) before leaving: peers may
    // still be posting into this CTA. Warps 8..11, done with A, join the epilogue warps in it when
    // the owned (row, group) pairs outnumber the epilogue's 128 threads.
    const int G = words / 4;                          // groups of 4 tokens
    const bool sum_helpers = S > 1 && own_rows * G > 128;
    const int sum_threads = sum_helpers ? 256 : 128;
    auto owner_sum = [&](const int t0, const bool ok_in) {
        const bool got = mbar_wait_cluster(red_bar, 0, lim);
        if (!got) res_fail(p, abort_flag);
        if (threadIdx.x == 128) RES_PHASE(9);
        if (got && ok_in) {
            const float4* rv = reinterpret_cast<const float4*>(sRecv);
            for (int t = t0; t < own_rows * G; t += sum_threads) {
                const int g = t / own_rows;
                const int r = t - g * own_rows;
                const int n = n0 + own0 + r;
                float4 acc = rv[g * R + r];
                for (int s0 = 1; s0 < S; s0 += 8) {
                    float4 x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (s0 + i < S) x[i] = rv[((s0 + i) * G + g) * R + r];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (s0 + i < S) {
                            acc.x += x[i].x;
                            acc.y += x[i].y;
                            acc.z += x[i].z;
                            acc.w += x[i].w;
                        }
                    }
                }
                if (n < p.N) {
                    uint16_t* cp = p.c + static_cast<int64_t>(m0 + 4 * g) * p.ldc + n;
                    const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (4 * g + i < m_valid) *cp = __bfloat16_as_ushort(__float2bfloat16_rn(vals[i]));
                        cp += p.ldc;
                    }
                }
            }
        }
    };
    if (warp >= 8 && sum_helpers) {
        cluster_wait();
        named_barrier(3, 256);                        // the epilogue has put this rank's own rows in place
        if (own_rows > 0) owner_sum(128 + static_cast<int>(threadIdx.x) - 256, abort_flag[0] == 0u);
        return;
    }
    if (warp < 4 || warp >= 8) {
        if (S > 1) cluster_wait();
        return;
    }

    // ------------------------------------------------------------ epilogue (warps 4..7)
    named_barrier(1, 32 + 128);                       // the column base, published by warp 1
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // every peer's barriers exist (long since): settled here, while the MMAs run, with the
    // destinations of this thread's split-K posts
    const int q = warp & 3;                           // lane quadrant this warp may read
    const int nl = q * 32 + lane;                     // weight row of the tile
    uint32_t dst = 0u, bar = 0u;
    int owner = 0;
    if (S > 1) {
        cluster_wait();
        owner = nl / R;
        const int rl = nl - owner * R;
        // receive buffer [source][token group][owned row][4 floats]: the owner's summing
        // threads read consecutive rows, 16 bytes apart
        const uint32_t off = static_cast<uint32_t>(split * G * R + rl) * 16u;
        dst = map_to_rank(smem_addr(sRecv) + off, static_cast<uint32_t>(owner));
        bar = map_to_rank(smem_addr(red_bar), static_cast<uint32_t>(owner));
    }
    const bool waited = mbar_wait(acc_full, 0, lim);
    tc_fence_after_sync();
    if (!waited) res_fail(p, abort_flag);
    if (threadIdx.x == 128) RES_PHASE(7);
    // one decision per warp (tcgen05.ld is warp-collective)
    const bool ok = !__any_sync(0xffffffffu, !waited || abort_flag[0] != 0u);
    uint32_t v[32];
    if (ok) {
        // the two issuers' accumulators, added (the second holds data from two steps on)
        const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t acc2 = static_cast<uint32_t>(p.m_tile);
        tmem_load_16(trow, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
        if (p.m_tile > 16) tmem_load_16(trow + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
        if (na >= 2) {
            uint32_t u[32];
            tmem_load_16(trow + acc2, *reinterpret_cast<uint32_t(*)[16]>(&u[0]));
            if (p.m_tile > 16) tmem_load_16(trow + acc2 + 16, *reinterpret_cast<uint32_t(*)[16]>(&u[16]));
            tmem_load_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(u[i]));
            if (NI == 3 && na >= 3) {   // a third issuer only with 16-token tiles
                tmem_load_16(trow + 2u * acc2, *reinterpret_cast<uint32_t(*)[16]>(&u[0]));
                tmem_load_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(u[i]));
            }
        } else {
            tmem_load_wait();
        }
    }
    if (threadIdx.x == 128) RES_PHASE(1);
    tc_fence_before_sync();
    named_barrier_arrive(2, 32 + 128);                // warp 1 may free tensor memory now

    if (S == 1) {
        // one K slice: accumulator -> bf16 C, one output column per thread
        if (ok && n0 + nl < p.N) {
            uint16_t* cp = p.c + static_cast<int64_t>(m0) * p.ldc + n0 + nl;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (i < m_valid) *cp = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i])));
                cp += p.ldc;
            }
        }
#ifdef MXFP4_TRACE
        if (threadIdx.x == 128) {
            trace_buffer[trace_row][11] = sm_clock();
            trace_buffer[trace_row][13] = global_timer_ns();
        }
#endif
        return;
    }

    // K slices > 1: every weight row goes to its owner's receive buffer, slot = this rank
    if (ok) {
        const uint32_t gstep = static_cast<uint32_t>(R) * 16u;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            if (g < G) {
                if (owner == split)
                    st_cluster_v4(dst + gstep * g, v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                else
                    st_async_v4(dst + gstep * g, v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3], bar);
            }
        }
    }
    if (threadIdx.x == 128) RES_PHASE(8);
    named_barrier(3, sum_helpers ? 256 : 128);        // this rank's own rows are in place
    if (own_rows > 0) owner_sum(static_cast<int>(threadIdx.x) - 128, ok);
#ifdef MXFP4_TRACE
    if (threadIdx.x == 128) {
        trace_buffer[trace_row][11] = sm_clock();
        trace_buffer[trace_row][13] = global_timer_ns();
    }
#endif
}

static cudaError_t set_resident_attributes() {
    static std::mutex mu;
    static std::atomic<bool> attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        for (const void* fn : {reinterpret_cast<const void*>(mxfp4_gemm_resident_kernel<false>),
                               reinterpret_cast<const void*>(mxfp4_gemm_resident_kernel<true>)}) {
            cudaFuncAttributes fa = {};
            e = cudaFuncGetAttributes(&fa, fn);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemLimit - fa.sharedSizeBytes));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        attr_set[dev].store(true, std::memory_order_release);
    }
    return cudaSuccess;
}

int max_active_clusters_resident(int cluster_size, size_t smem_bytes) {
    if (set_resident_attributes() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster_size);
    cfg.blockDim = dim3(kResThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mxfp4_gemm_resident_kernel<false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_gemm_resident(const GemmPlan& plan, const ResidentArgs& args, cudaStream_t s) {
    cudaError_t e = set_resident_attributes();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.ctas);
    cfg.blockDim = dim3(kResThreads);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(plan.splits);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plan.splits > 1 ? 2 : 1;
    if (plan.many_items) return cudaLaunchKernelEx(&cfg, mxfp4_gemm_resident_kernel<true>, args);
    return cudaLaunchKernelEx(&cfg, mxfp4_gemm_resident_kernel<false>, args);
}

}  // namespace mxfp4

#ifdef MXFP4_TRACE
extern "C" int mxfp4_trace_read_resident(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, mxfp4::trace_buffer, bytes));
}
#endif
