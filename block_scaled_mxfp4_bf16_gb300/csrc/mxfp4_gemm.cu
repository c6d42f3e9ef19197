// Block-scaled MXFP4 GEMM on the sm_103a tensor cores: tcgen05.mma kind::mxf4 with e8m0 scale
// factors in tensor memory, bulk-copy-fed shared-memory pipelines, a split-K reduction through
// distributed shared memory and a bf16 epilogue.
//
// Orientation. The weights B[N,K] are the MMA's 128-row "A" operand and the tokens A[M,K] the
// MMA's "B" operand (N_mma = token tile, 16..256), so the small-M shapes still fill the 128-row
// MMA and D = C^T sits in tensor memory with one weight row per lane.
//
// Operands arrive as "blocks" (internal.h): every (tile, 256-K atom) is stored as the exact
// swizzled shared-memory image the MMA reads, scale factors included, so one contiguous
// cp.async.bulk fills a stage and the weight stream reads DRAM sequentially.
//
// One CTA = one (weight tile of 128 rows, token tile, K slice); the K slices of one output tile
// form one thread-block cluster. Warp roles:
//   warp 0    : copy producer -- weight blocks (17 KB), the fused path's bf16 A slice (one
//               bulk copy per row) or the two-kernel path's token blocks. The first weight
//               stages are requested before the CTA waits on the previous grid (the weights never
//               depend on it); when the caller declared A ready, the fused path's A rows too.
//   warps 1-2 : tensor-memory allocation (warp 1) and two MMA-issuing threads (alternate 256-K
//               steps, two accumulators; on tiles of more than 128 tokens each takes part of
//               every step's tokens, one accumulator between them): per 256-K step a thread
//               copies the scale factors into tensor memory (tcgen05.cp) and issues four
//               128 x N x 64 block-scaled MMAs.
//   warps 3-10: the epilogue: they move the accumulators out of tensor memory. In the fused path
//               they first warm L2 with the CTA's A rows while the previous grid finishes and
//               zero the staged bytes past K of a 1x32 block that K cuts. On the two-kernel path,
//               when every step has a stage of its own, warp 3 is a third MMA issuer first; when
//               the ring refills (or steps are shared), warps 4-7 first write each stage's scale
//               factors into tensor memory (tcgen05.st), so the MMA threads issue MMAs only.
// In the fused path every warp first quantizes the staged slice into the token-block layout (the
// pages' in-register A quantization, submission 711914 `mxfp4_gemm_fused_k512_kernel`): the copy
// and MMA warps have nothing else to do until those blocks exist.
// Reduction: each output row has an owner CTA in the cluster; the K slices send their fp32 rows
// into the owner's shared memory -- short runs as st.async stores, long runs as bulk copies of
// four rows each, both counted on the owner's mbarrier (where neither fits, posted stores and a cluster
// barrier) -- and the owner sums them in slice order (run-to-run identical) and stores bf16 C.
// Every wait on an mbarrier is bounded; on timeout the kernel records an error in the device
// status word and unwinds (outputs undefined, no hang, tensor memory released).
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "mma_desc.cuh"
#include "ptx.cuh"
#include "quant_device.cuh"

namespace mxfp4 {

// A timing build (-DMXFP4_TRACE) gives each CTA its own row of the trace buffer (in start order,
// so consecutive launches stay apart): grid id, block index, SM, the global timer and the SM
// clock at its start (slots 0/10) and where it stores C (slots 13/11), and the SM clock at each
// other phase.
#ifdef MXFP4_TRACE
static __shared__ unsigned int g_trace_row;
// Per-step stamps of the same row (SM clock): [j] when step j's stage was seen full by its MMA
// thread, [32 + j] when the copy thread saw the stage it refills for step j released (j < 32).
static __device__ unsigned long long ring_buffer[4096][64];
__device__ __forceinline__ void trace_phase(int slot) {
    const unsigned int row = g_trace_row;
    if (slot == 0 || slot == 10 || slot == 13 || slot == 12) return;
    if (slot == 11) {
        trace_buffer[row][11] = sm_clock();
        trace_buffer[row][13] = global_timer_ns();
        return;
    }
    trace_buffer[row][slot] = sm_clock();
}
#undef MXFP4_PHASE
#define MXFP4_PHASE(slot) ::mxfp4::trace_phase(slot)
#endif

__device__ __forceinline__ bool et_first_lane(int warp, int lane) { return warp == 3 && lane == 0; }

// 32 accumulator columns of this thread's lane (the second 16 only if `upper`), plus the
// matching columns of the second accumulator `acc2` columns further when `two`.
__device__ __forceinline__ void load_acc32(uint32_t taddr, bool upper, int nacc, uint32_t acc2, uint32_t (&r)[32]) {
    tmem_load_16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
    if (upper) tmem_load_16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
    if (nacc >= 2) {
        uint32_t q[32];
        tmem_load_16(taddr + acc2, *reinterpret_cast<uint32_t(*)[16]>(&q[0]));
        if (upper) tmem_load_16(taddr + acc2 + 16, *reinterpret_cast<uint32_t(*)[16]>(&q[16]));
        tmem_load_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(q[i]));
        if (nacc >= 3) {   // the third issuer's accumulator, added last
            tmem_load_16(taddr + 2u * acc2, *reinterpret_cast<uint32_t(*)[16]>(&q[0]));
            if (upper) tmem_load_16(taddr + 2u * acc2 + 16, *reinterpret_cast<uint32_t(*)[16]>(&q[16]));
            tmem_load_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(q[i]));
        }
    } else {
        tmem_load_wait();
    }
}

__device__ __forceinline__ void fail(const GemmArgs& p, volatile uint32_t* abort_flag) {
    atomicOr(p.status, 1u);
    *abort_flag = 1u;
}

// Fused path: what the CTA's threads need to quantize its staged bf16 A slice.
struct QuantSlice {
    const uint8_t* raw;    // staged rows, raw_row bytes apart
    uint8_t* blocks;       // token blocks, one per 256-K step
    uint32_t raw_row, a_block, a_rows;
    int m_valid, nblk, kblk;
    uint64_t* a_raw;       // the staged rows have landed
    uint64_t* a_full;      // the token blocks are written (one arrival per warp)
    uint64_t lim;
#ifdef MXFP4_TEST_HOOKS
    uint8_t* dump;         // test build only: where this CTA's token blocks go (null: nowhere)
#endif
};

// Every thread of the CTA takes part (the copy and MMA warps have nothing else to do until the
// token blocks exist): one 1x32 block per item, items dealt round-robin over the CTA, one per
// thread per pass; K past the end becomes zero codes and scales.
// (In a last block cut by K the epilogue warps have zeroed the staged bytes past K.)
// Rows past M are left as they are: a token row only feeds its own accumulator column, and
// columns past M are never stored.
__device__ __forceinline__ void quantize_slice(const QuantSlice& q, int qt, const GemmArgs& p,
                                               volatile uint32_t* abort_flag) {
    const int lane = qt & 31;
    // idx / m_valid as a multiply-high (exact for idx < 2^16, m_valid <= 256), set up off the path
    const uint32_t magic = 0xFFFFFFFFu / static_cast<uint32_t>(q.m_valid) + 1u;
    const bool one_row = q.m_valid == 1;
    const bool got = mbar_wait(q.a_raw, 0, q.lim);
    if (qt == 96) MXFP4_PHASE(10);
    if (!got) fail(p, abort_flag);
    const int total = got ? q.m_valid * q.nblk : 0;
    constexpr int nq = kGemmThreads;
    // one item per thread per pass: the automatic plan keeps the fused path at one 1x32 block
    // per thread, and a single item keeps the code the CTA fetches small
    for (int idx = qt; idx < total; idx += nq) {
        uint32_t w[16], out[4];
        // rows run fastest: eight consecutive items read eight rows (distinct banks) and
        // write eight rows of one chunk column (distinct swizzled chunks)
        const int kq = one_row ? idx : static_cast<int>(__umulhi(static_cast<uint32_t>(idx), magic));
        const int rr = idx - kq * q.m_valid;
        uint32_t sbyte = 0u;
        out[0] = out[1] = out[2] = out[3] = 0u;
        if (kq < q.kblk) {
            const uint4* src = reinterpret_cast<const uint4*>(q.raw + rr * q.raw_row + kq * 64);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = src[i];
                w[4 * i + 0] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
            sbyte = quantize_block32(w, out);
        }
        const uint32_t c = static_cast<uint32_t>(kq & 7);
        uint8_t* blk = q.blocks + (kq >> 3) * q.a_block;
        *reinterpret_cast<uint4*>(blk + swz_chunk_offset(static_cast<uint32_t>(rr), c)) =
            make_uint4(out[0], out[1], out[2], out[3]);
        blk[q.a_rows + block_sf_offset(static_cast<uint32_t>(rr), c)] = static_cast<uint8_t>(sbyte);
    }
    if (qt == 96) MXFP4_PHASE(13);
#ifdef MXFP4_TEST_HOOKS
    // test build: the token blocks of weight tile 0's CTAs, as quantized, to the dump buffer
    // [m_tiles][k_atoms][a_block] (every thread of the CTA runs this function)
    __syncthreads();
    if (q.dump) {
        const int words = q.nblk / 8 * static_cast<int>(q.a_block) / 16;
        for (int i = qt; i < words; i += kGemmThreads)
            reinterpret_cast<uint4*>(q.dump)[i] = reinterpret_cast<const uint4*>(q.blocks)[i];
    }
#endif
    fence_proxy_async_smem();   // the MMAs read the token blocks through the async proxy
    __syncwarp();
    if (lane == 0) mbar_arrive(q.a_full);   // one arrival per warp
}

// kTwoKernel: an instantiation that only runs the two-kernel path (no quantizer code in it),
// kWide (with it): its tiles of more than 128 tokens, two issuers sharing every step (below),
// kSfStores (with it): scale factors written into tensor memory by epilogue warps (below);
// the other instantiation takes the path and the issue scheme from its arguments.
template <bool kTwoKernel, bool kWide, bool kSfStores>
__global__ void __launch_bounds__(kGemmThreads, 1)
mxfp4_gemm_kernel(const GemmArgs p) {
    static_assert(kTwoKernel || (!kWide && !kSfStores), "the fused path copies its own scale factors");
    const bool fused = kTwoKernel ? false : p.fused != 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* sB = smem;                           // stages x kWBlock
    uint8_t* sA = smem + p.off_a;                 // token blocks: stages (two-kernel) or atoms (fused)
    float* sRecv = reinterpret_cast<float*>(smem + p.off_recv);   // fp32 rows this CTA reduces / stages
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* empty = full + kMaxStages;
    uint64_t* a_full = empty + kMaxStages;
    uint64_t* acc_full = a_full + 1;
    uint64_t* a_raw = acc_full + 1;
    uint64_t* red_bar = a_raw + 1;                // split-K: the peers' rows have landed here
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_bar + 1);
    volatile uint32_t* flags = tmem_slot + 1;    // [0] abort
    uint64_t* sf_full = red_bar + 2;              // [kMaxStages] a stage's scale factors in tensor memory

    // The warp index broadcast from lane 0, so the compiler treats it (and the MMA operands
    // derived from it) as warp-uniform: tcgen05 instructions take their operands from uniform
    // registers, and operands it cannot prove uniform cost extra instructions at every issue.
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    // ---- work unit: (token tile, weight tile, K slice)
    const int S = p.splits;
    const int split = blockIdx.x % S;              // = rank in the cluster
    const int tile = blockIdx.x / S;
    const int nt = tile % p.n_tiles;
    const int mt = tile / p.n_tiles;
    const int n0 = nt * kTileN;
    const int m0 = mt * p.m_tile;
    const int base = p.k_atoms / S, rem = p.k_atoms % S;
    const int a0 = split * base + (split < rem ? split : rem);
    const int na = base + (split < rem ? 1 : 0);
    const int m_valid = (p.M - m0) < p.m_tile ? (p.M - m0) : p.m_tile;
    const int stages = p.stages;
    // Tiles of more than 128 tokens with two issuers ("halves"): the first issuer takes tokens
    // 0..127 of every step, the second the rest, each into its columns of one accumulator; both
    // release every stage.
    const bool halves = kTwoKernel ? kWide : (p.m_tile > 128 && p.issuers == 2);
    // kSfStores: epilogue warps 4..7 (one per lane quarter) write each stage's scale factors
    // into tensor memory (tcgen05.st) and the MMA threads wait for that instead of the stage
    // itself, so the tensor pipe runs MMAs only (no tcgen05.cp); scale columns then hold one copy
    // per stage shared by every issuer. The planner takes it where the pipe is the limit.
    constexpr bool sf_st = kSfStores;
    const uint32_t sf_col0 = static_cast<uint32_t>(halves ? p.m_tile : p.issuers * p.m_tile);   // first scale column
    const uint32_t a_block = p.a_block;
    const uint32_t a_rows = static_cast<uint32_t>(p.m_tile) * 128u;
    const uint64_t lim = p.wait_limit_ns;
    // rows of the output tile reduced (and stored) by CTA `rank` of the cluster
    const int rows_per = red_rows_per(m_valid, S);   // multiple of 4
    const int r0 = min(m_valid, split * rows_per);
    const int r1 = min(m_valid, r0 + rows_per);
    const bool vec = rows_per <= kRedVecMaxRows;   // short runs: 16-byte stores of four tokens
    // fused path: this CTA's bf16 A slice, rows of kslice elements
    const int kslice = min(na * kAtomK, p.K - a0 * kAtomK);
    const uint32_t raw_row = raw_pitch(p.atoms_max);   // bytes from one staged row to the next
    QuantSlice qs;
    qs.raw = smem + p.off_araw;
    qs.blocks = sA;
    qs.raw_row = raw_row;
    qs.a_block = a_block;
    qs.a_rows = a_rows;
    qs.m_valid = m_valid;
    qs.nblk = na * (kAtomK / 32);
    qs.kblk = (kslice + 31) / 32;            // blocks of this slice inside K
    qs.a_raw = a_raw;
    qs.a_full = a_full;
    qs.lim = lim;
#ifdef MXFP4_TEST_HOOKS
    qs.dump = (nt == 0 && p.token_dump) ? p.token_dump + (static_cast<size_t>(mt) * p.k_atoms + a0) * a_block : nullptr;
#endif

#ifdef MXFP4_TRACE
    if (threadIdx.x == 0) {
        const unsigned int row = atomicAdd(&trace_counter, 1u) & 4095u;
        g_trace_row = row;
        trace_buffer[row][10] = sm_clock();
        trace_buffer[row][0] = global_timer_ns();
        trace_buffer[row][12] = sm_id();
        trace_buffer[row][14] = grid_id();
        trace_buffer[row][15] = blockIdx.x;
    }
    __syncthreads();
#endif
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], halves ? 2 : 1);   // halves: both issuers release every stage
        }
        mbar_init(a_full, kGemmThreads / 32);
        mbar_init(acc_full, static_cast<uint32_t>(p.issuers));
        mbar_init(a_raw, 1 + kEpiWarps);   // the copy thread + the epilogue warps (tail zeroing)
        mbar_init(red_bar, 1);
        if (sf_st)
            for (int s = 0; s < stages; ++s) mbar_init(&sf_full[s], 4);   // one arrival per writing warp
        if (S > 1 && p.red_bulk && r1 > r0)   // (S - 1) peers x owned rows x 512 bytes
            mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>((S - 1) * (r1 - r0)) * kTileN * 4u);
        else if (S > 1 && vec && r1 > r0)     // (S - 1) peers x 128 weight rows x 16 bytes per 4 rows
            mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>((S - 1) * ((r1 - r0 + 3) / 4)) * kTileN * 16u);
        flags[0] = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    // Split-K by st.async or bulk copies: every CTA arrives here once its barriers exist, and each
    // warp waits (cluster_wait) at a point of its own off the critical path, before any post.
    const bool cluster_posts = S > 1 && (p.red_bulk || vec);
    if (cluster_posts) cluster_arrive_relaxed();
    pdl_launch_dependents();
    uint32_t tmem_base = 0;
    bool ok = true;

    const uint8_t* bsrc = p.bblk + (static_cast<size_t>(nt) * p.k_atoms + a0) * kWBlock;
    const uint8_t* asrc = p.ablk + (static_cast<size_t>(mt) * p.k_atoms + a0) * a_block;
    const uint32_t tx_bytes = kWBlock + (fused ? 0u : a_block);
    const int npro = na < stages ? na : stages;
    // One MMA-issuing thread: the MMAs of every issuers-th 256-K step into an accumulator of its
    // own (or, in halves, of every step for its tokens), each step's stage released with a
    // commit, then one commit on acc_full.
    auto issue_mmas = [&](const int issuer) {
        // The issue loop is kept to integer adds: a shared-memory descriptor's start-address
        // field (bits 0..13, address / 16) moves by (bytes / 16) from one buffer to the next.
        const uint32_t t_acc = tmem_base + static_cast<uint32_t>(issuer * (halves ? 128 : p.m_tile));
        // scale columns: per issuer in halves (weights, then its tokens), else shared per stage
        const uint32_t t_sfb0 = sf_st ? tmem_base + sf_col0
                                : halves ? tmem_base + static_cast<uint32_t>(p.m_tile + issuer * 16 * stages)
                                         : tmem_base + static_cast<uint32_t>(p.issuers * p.m_tile);
        const uint32_t t_sfa0 = t_sfb0 + static_cast<uint32_t>(stages) * 8u;
        const uint32_t mc = halves && !sf_st ? 1u : static_cast<uint32_t>(p.nmc);  // token row blocks per copy
        const uint32_t sfa_step = 8u * mc;                                // columns per stage
        // shared scale columns (sf_st): a token row block's 4 columns sit at 4 * block, so the
        // second issuer of halves starts 4 columns in (its K groups 8 columns apart, as for N = 256)
        const uint32_t tok_col = sf_st && halves ? 4u * static_cast<uint32_t>(issuer) : 0u;
        // halves: the first issuer's MMAs take tokens 0..127, the second's the rest of the tile
        const uint32_t n_mma = halves ? (issuer == 0 ? 128u : static_cast<uint32_t>(p.m_tile - 128))
                                      : static_cast<uint32_t>(p.m_tile);
        const uint32_t idesc0 = idesc_mxf4(n_mma);
        const uint32_t idesc1 = idesc0 | (2u << 29) | (2u << 4);         // scale bytes {2,3}
        const uint64_t b_desc0 = desc_sw128(smem_addr(sB));
        // halves: token rows 128h.. start 128 rows (16 KB, a whole number of swizzle atoms) in,
        // their scale chunks are (h, 0) and (h, 1)
        const uint32_t half = halves ? static_cast<uint32_t>(issuer) : 0u;
        const uint64_t a_desc0 = desc_sw128(smem_addr(sA)) + half * ((128u * 128u) >> 4);
        const uint64_t sfb_desc0 = desc_sf(smem_addr(sB + kBRowsBytes));
        const uint64_t sfa_desc0 = desc_sf(smem_addr(sA + a_rows)) + half * 2u * (kSfChunk >> 4);
        const uint32_t b_step = kWBlock >> 4, a_step = a_block >> 4, chunk_step = kSfChunk >> 4;
        const bool two_chunks = mc == 2;
        const int first = halves ? 0 : issuer, stride = halves ? 1 : p.issuers;
        bool mok = true;
        if (fused) mok = mbar_wait(a_full, 0, lim);
        if (issuer == 0) MXFP4_PHASE(3);
        tc_fence_after_sync();
        int s = first;
        uint32_t phase = 0;
        while (s >= stages) { s -= stages; phase ^= 1u; }
#pragma unroll 1
        for (int j = first; mok && j < na; j += stride) {
            if (!mbar_wait(sf_st ? &sf_full[s] : &full[s], phase, lim)) { mok = false; break; }
#ifdef MXFP4_TRACE
            if (j < 32) ring_buffer[g_trace_row][j] = sm_clock();
#endif
            if (j == 0) MXFP4_PHASE(4);
            if (j == na - 1) MXFP4_PHASE(5);
            tc_fence_after_sync();
            const uint32_t slot = static_cast<uint32_t>(fused ? j : s);
            const uint64_t bd = b_desc0 + static_cast<uint32_t>(s) * b_step;
            const uint64_t ad = a_desc0 + slot * a_step;
            const uint64_t sfbd = sfb_desc0 + static_cast<uint32_t>(s) * b_step;
            const uint64_t sfad = sfa_desc0 + slot * a_step;
            const uint32_t sfb_cols = t_sfb0 + static_cast<uint32_t>(s) * 8u;
            const uint32_t sfa_cols = t_sfa0 + static_cast<uint32_t>(s) * sfa_step + tok_col;
            // scale factors: weight groups 2j, 2j+1 -> 4 columns each; token chunks likewise
            if (!sf_st) {
                tc_copy_sf(sfb_cols, sfbd);
                tc_copy_sf(sfb_cols + 4u, sfbd + chunk_step);
                if (!two_chunks) {
                    tc_copy_sf(sfa_cols, sfad);
                    tc_copy_sf(sfa_cols + 4u, sfad + chunk_step);
                } else {   // 256 tokens: chunks (c, g) at 512 * (2c + g), columns 4 * (2g + c)
                    tc_copy_sf(sfa_cols, sfad);
                    tc_copy_sf(sfa_cols + 4u, sfad + 2 * chunk_step);
                    tc_copy_sf(sfa_cols + 8u, sfad + chunk_step);
                    tc_copy_sf(sfa_cols + 12u, sfad + 3 * chunk_step);
                }
            }
            const uint32_t sfa_g1 = sfa_cols + 4u * mc;
            // K step kk of the atom: +32 bytes in both operands (descriptor +2)
            mma_mxf4(t_acc, bd + 0, ad + 0, idesc0, sfb_cols, sfa_cols, j != first);
            mma_mxf4(t_acc, bd + 2, ad + 2, idesc1, sfb_cols, sfa_cols, 1);
            mma_mxf4(t_acc, bd + 4, ad + 4, idesc0, sfb_cols + 4u, sfa_g1, 1);
            mma_mxf4(t_acc, bd + 6, ad + 6, idesc1, sfb_cols + 4u, sfa_g1, 1);
            tc_commit(&empty[s]);
            s += stride;
            while (s >= stages) { s -= stages; phase ^= 1u; }
        }
        if (!mok) fail(p, flags);
        tc_commit(acc_full);
    };
    // ------------------------------------------------------------------------ set-up
    if (warp == 0) {
        // The weight ring's first stages go before the dependency wait (the weights never depend
        // on the previous grid). In the fused path only two: the A slice is the first thing the
        // CTA needs once the wait returns, and copies leave in issue order. When the caller has
        // declared A ready before the launch (a_ready), the fused path requests the A slice first
        // and the whole prologue before the wait.
        const uint64_t pol_b = policy_evict_first();
        const bool a_early = fused && p.a_ready;
        auto load_a_slice = [&]() {
            // the whole bf16 slice A[m0 .. m0+m_valid, a0*256 .. +kslice] in one round trip, one
            // row per lane so that the rows' copies are issued together
            const uint32_t row_bytes = static_cast<uint32_t>(kslice) * 2u;
            const uint16_t* arow = p.a + static_cast<int64_t>(m0) * p.lda + a0 * kAtomK;
            if (lane == 0) mbar_arrive_expect_tx(a_raw, row_bytes * static_cast<uint32_t>(m_valid));
            __syncwarp();
            for (int r = lane; r < m_valid; r += 32)
                bulk_load(smem + p.off_araw + r * raw_row, arow + r * p.lda, row_bytes, a_raw, policy_evict_last());
            __syncwarp();
        };
        if (a_early) load_a_slice();
        const int nfirst = fused && !a_early ? min(npro, 2) : npro;
        if (lane == 0) {
            for (int j = 0; j < nfirst; ++j) {
                mbar_arrive_expect_tx(&full[j], tx_bytes);
                bulk_load(sB + j * kWBlock, bsrc + static_cast<size_t>(j) * kWBlock, kWBlock, &full[j], pol_b);
            }
        }
        MXFP4_PHASE(1);
        pdl_wait_prior_grid();   // A and the token blocks may be written by the previous grid
        MXFP4_PHASE(2);
        if (fused) {
            if (!a_early) load_a_slice();
            if (lane == 0) {
                for (int j = nfirst; j < npro; ++j) {
                    mbar_arrive_expect_tx(&full[j], tx_bytes);
                    bulk_load(sB + j * kWBlock, bsrc + static_cast<size_t>(j) * kWBlock, kWBlock, &full[j], pol_b);
                }
            }
        } else if (lane == 0) {
            for (int j = 0; j < npro; ++j)
                bulk_load(sA + j * a_block, asrc + static_cast<size_t>(j) * a_block, a_block, &full[j],
                          policy_evict_last());
        }
    } else if (warp == 1) {
        // Columns are allocated only after the previous grid has finished, so a CTA of this
        // grid never holds columns a CTA of the previous grid is still waiting for.
        pdl_wait_prior_grid();
        tmem_alloc(const_cast<uint32_t*>(tmem_slot), p.tmem_cols);
        tmem_relinquish();
        tc_fence_before_sync();
        // publish the column base: to warp 2 now (barrier 3), to the epilogue warps once they
        // are done with the A slice (barrier 1)
        named_barrier_arrive(3, 64);
        named_barrier_arrive(1, 32 + kEpiThreads);
    } else if (warp == 2) {
        named_barrier(3, 64);
    } else if (fused) {
        // Warm L2 with the CTA's A rows while the previous grid finishes (plain prefetches from
        // the idle epilogue warps: they do not queue in front of the bulk copies).
        const int lines = (kslice * 2 + 127) / 128;
        const uint16_t* arow = p.a + static_cast<int64_t>(m0) * p.lda + a0 * kAtomK;
        for (int i = threadIdx.x - 96; i < m_valid * lines; i += kEpiThreads) {
            const int r = i / lines;
            prefetch_l2(arow + static_cast<int64_t>(r) * p.lda + (i - r * lines) * 64);
        }
        // K cuts the slice's last 1x32 block when kslice % 32 != 0: the copies stop at K, so the
        // rest of that block in every staged row is zeroed here (elements past K count as zeros).
        // Disjoint from the bytes the copies write; published by each warp's arrival on a_raw,
        // which the quantizing threads acquire with the copies. (Placed here, in warps that are
        // idle until then, it measured free; in the copy thread it slowed the fused path.)
        const uint32_t from = static_cast<uint32_t>(kslice) * 2u;
        const uint32_t end = static_cast<uint32_t>((kslice + 31) / 32) * 64u;
        const int per_row = static_cast<int>((end - from) / 16u);
        for (int i = threadIdx.x - 96; i < m_valid * per_row; i += kEpiThreads) {
            const int r = i / per_row;
            *reinterpret_cast<uint4*>(smem + p.off_araw + r * raw_row + from + (i - r * per_row) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(a_raw);
    }
    __syncwarp();
    // Fused path: every warp quantizes (one call site, so the quantizer is inlined once).
    if (fused) quantize_slice(qs, threadIdx.x, p, flags);

    if (warp == 0) {
        // -------------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_b = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            int issued = npro;
            for (int j = npro; j < na; ++j) {
                const int s = j % stages;
                if (!mbar_wait(&empty[s], ((j / stages) - 1) & 1, lim)) { fail(p, flags); break; }
#ifdef MXFP4_TRACE
                if (j < 32) ring_buffer[g_trace_row][32 + j] = sm_clock();
#endif
                mbar_arrive_expect_tx(&full[s], tx_bytes);
                bulk_load(sB + s * kWBlock, bsrc + static_cast<size_t>(j) * kWBlock, kWBlock, &full[s], pol_b);
                if (!fused)
                    bulk_load(sA + s * a_block, asrc + static_cast<size_t>(j) * a_block, a_block, &full[s], pol_a);
                issued = j + 1;
            }
            // never leave copies in flight into shared memory that is about to be reused or freed
            for (int j = (issued > stages ? issued - stages : 0); j < issued; ++j)
                mbar_wait(&full[j % stages], (j / stages) & 1, lim);
            if (fused) mbar_wait(a_raw, 0, lim);
        }
        __syncwarp();
        if (cluster_posts) cluster_wait();
    } else if (warp <= 2) {
        // ------------------------------------------------------------------- MMA issuers
        // Warp 1 allocates tensor memory; warps 1 and 2 (one thread each) issue the MMAs of
        // alternate 256-K steps into two accumulators, which halves the serial issue chain
        // (the epilogue adds them). With one issuer warp 2 only waits.
        const int issuer = warp - 1;
        tc_fence_after_sync();
        tmem_base = *tmem_slot;
        if (lane == 0 && issuer < p.issuers) issue_mmas(issuer);
        __syncwarp();
        if (cluster_posts) cluster_wait();
    } else {
        // -------------------------------------------------------------------- warps 3..10
        const int et = threadIdx.x - 96;
        named_barrier(1, 32 + kEpiThreads);       // the column base, published by warp 1 long ago
        tmem_base = *tmem_slot;
        if (cluster_posts) cluster_wait();         // every peer's red_bar exists (long since)
        // A third issuer on the two-kernel path: warp 3, idle there until the accumulators are
        // ready, takes every third step (its own accumulator), then joins the epilogue.
        if (warp == 3 && p.issuers == 3) {
            tc_fence_after_sync();
            if (lane == 0) issue_mmas(2);
            __syncwarp();
        }
        if (sf_st && warp >= 4 && warp < 8) {
            // Each stage's scale factors into its columns, every lane quarter the same words (what
            // a 32x128b.warpx4 copy writes): lane r of a 512-byte chunk holds the 4 K blocks of
            // rows r, 32 + r, 64 + r, 96 + r, one column each. Weights: 2 chunks -> 8 columns;
            // tokens: 2 chunks, or 4 for 256-token tiles ((c, g) at 512 * (2c + g) -> columns
            // 4 * (2g + c)).
            const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const uint32_t t_sfb0 = tmem_base + lane_base + sf_col0;
            const uint32_t t_sfa0 = t_sfb0 + static_cast<uint32_t>(stages) * 8u;
            const uint32_t sfa_step = 8u * static_cast<uint32_t>(p.nmc);
            int s = 0;
            uint32_t phase = 0;
#pragma unroll 1
            for (int j = 0; j < na; ++j) {
                if (!mbar_wait(&full[s], phase, lim)) { fail(p, flags); break; }
                const uint8_t* wsf = sB + s * kWBlock + kBRowsBytes + lane * 16;
                const uint4 w0 = *reinterpret_cast<const uint4*>(wsf);
                const uint4 w1 = *reinterpret_cast<const uint4*>(wsf + kSfChunk);
                const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                tmem_store_8(t_sfb0 + static_cast<uint32_t>(s) * 8u, wv);
                const uint8_t* tsf = sA + s * a_block + a_rows + lane * 16;
                const uint4 t0 = *reinterpret_cast<const uint4*>(tsf);
                const uint4 t1 = *reinterpret_cast<const uint4*>(tsf + kSfChunk);
                if (p.nmc == 1) {
                    const uint32_t tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                    tmem_store_8(t_sfa0 + static_cast<uint32_t>(s) * sfa_step, tv);
                } else {
                    const uint4 t2 = *reinterpret_cast<const uint4*>(tsf + 2 * kSfChunk);
                    const uint4 t3 = *reinterpret_cast<const uint4*>(tsf + 3 * kSfChunk);
                    const uint32_t tv[16] = {t0.x, t0.y, t0.z, t0.w, t2.x, t2.y, t2.z, t2.w,
                                             t1.x, t1.y, t1.z, t1.w, t3.x, t3.y, t3.z, t3.w};
                    tmem_store_16(t_sfa0 + static_cast<uint32_t>(s) * sfa_step, tv);
                }
                tmem_store_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_full[s]);
                if (++s == stages) { s = 0; phase ^= 1u; }
            }
        }
        const bool waited = mbar_wait(acc_full, 0, lim);
        tc_fence_after_sync();
        if (et == 0) MXFP4_PHASE(6);
        if (!waited) fail(p, flags);
        // one decision per warp (tcgen05.ld is warp-collective)
        ok = !__any_sync(0xffffffffu, !waited || flags[0] != 0u);
    }

    // ------------------------------------------------------------------------ output
    // Accumulator D = C^T: tensor-memory lane = weight row n, column = token m. Epilogue warp w
    // reads the lanes of quadrant w % 4 and every other 32-column chunk (two warps per quadrant).
    const int half = ((warp - 3) >> 2) & 1;
    const int nacc = halves ? 1 : min(p.issuers, na);   // accumulators that hold data
    const uint32_t acc2 = static_cast<uint32_t>(p.m_tile);
    const int nl = (warp & 3) * 32 + lane;
    const int n = n0 + nl;
    const uint32_t trow = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    __syncwarp();
    if (S == 1) {
        // one K slice: tensor memory -> bf16 C directly, one output column per thread
        if (warp >= 3 && ok) {
            for (int cb = half * 32; cb < m_valid; cb += 64) {
                uint32_t r[32];
                load_acc32(trow + cb, cb + 16 < m_valid, nacc, acc2, r);
                if (n < p.N) {
                    uint16_t* cp = p.c + static_cast<int64_t>(m0 + cb) * p.ldc + n;
                    const int cnt = min(32, m_valid - cb);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (i < cnt) *cp = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[i])));
                        cp += p.ldc;
                    }
                }
            }
            if (et_first_lane(warp, lane)) MXFP4_PHASE(11);
        }
        tc_fence_before_sync();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after_sync();
            tmem_dealloc(tmem_base, p.tmem_cols);
        }
        return;
    }

    // K slices > 1. Runs of rows_per rows of the tile belong to successive CTAs of the cluster
    // (the owners); every CTA sends its fp32 accumulator rows to their owners' receive buffers
    // (slot = source rank) in one of three forms below, and each owner sums its rows over the
    // sources in rank order (run-to-run identical) and stores bf16. Without a dedicated receive
    // buffer a cluster barrier first makes sure every peer's MMAs are done before its pipeline
    // buffers are overwritten.
    if (p.red_bulk) {
        // Long runs: every CTA stages its fp32 tile [row][n] in its own shared memory, then one
        // bulk copy per owner moves that owner's rows into the owner's receive buffer, counted
        // on the owner's red_bar. An owner sums its own staged rows and the received ones in
        // rank order; a last cluster barrier (reached by owners only once their rows are in)
        // keeps every CTA resident until no copy reads or writes its shared memory.
        float* sStage = reinterpret_cast<float*>(smem + p.off_stage);
        if (threadIdx.x == 96) MXFP4_PHASE(7);
        if (warp >= 3 && ok) {
            for (int cb = half * 32; cb < m_valid; cb += 64) {
                uint32_t r[32];
                load_acc32(trow + cb, cb + 16 < m_valid, nacc, acc2, r);
                const int cnt = min(32, m_valid - cb);
                float* dst = sStage + cb * kTileN + nl;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < cnt) dst[i * kTileN] = __uint_as_float(r[i]);
            }
            fence_proxy_async_smem();   // the copies read the staged tile through the async proxy
        }
        if (threadIdx.x == 96) MXFP4_PHASE(8);
        __syncwarp();
        if (!p.recv_dedicated) cluster_sync();     // every peer is done with the buffers it receives in
        tc_fence_before_sync();
        __syncthreads();                           // the staged tile is complete; TMEM reads done
        if (warp == 1) {
            tc_fence_after_sync();
            tmem_dealloc(tmem_base, p.tmem_cols);
        }
        if (warp == 3 && ok) {
            // one copy per 4 rows, issued by the lanes of warp 3 side by side
            const uint32_t slot_off = smem_addr(sRecv) + static_cast<uint32_t>(split * rows_per) * kTileN * 4u;
            for (int o = 0; o < S; ++o) {
                const int o0 = min(m_valid, o * rows_per), o1 = min(m_valid, o0 + rows_per);
                if (o == split || o1 <= o0) continue;
                const uint32_t dst = map_to_rank(slot_off, static_cast<uint32_t>(o));
                const uint32_t bar = map_to_rank(smem_addr(red_bar), static_cast<uint32_t>(o));
                for (int r = o0 + 4 * lane; r < o1; r += 128) {
                    const int rows = min(4, o1 - r);
                    bulk_copy_to_peer(dst + static_cast<uint32_t>(r - o0) * kTileN * 4u, sStage + r * kTileN,
                                      static_cast<uint32_t>(rows) * kTileN * 4u, bar);
                }
            }
        }
        // An owner whose rows did not all arrive in time skips its sum and stores (the status
        // word reports it). The bytes it still lacks belong to a peer that failed before posting:
        // a peer that posted has its copy land well within the limit.
        const bool owner = warp >= 3 && r1 > r0;
        const bool got = !owner || mbar_wait_cluster(red_bar, 0, lim);
        if (!got) fail(p, flags);
        __syncwarp();
        cluster_arrive();
        if (threadIdx.x == 96) MXFP4_PHASE(9);
        if (owner && got) {
            // a thread sums 4 consecutive columns of rows lm, lm+8, lm+16, lm+24 over the sources
            // in rank order; the four rows' values of a source are loaded before any is added
            // (one row at a time, each iteration waited on its loads and its store: ~200 ns a row)
            const int et = threadIdx.x - 96;
            const int nrows = r1 - r0;
            const int nl4 = (et & 31) * 4;
            const int n4 = n0 + nl4;
            const bool v4 = p.c_vec4 && n4 + 3 < p.N;
            constexpr int kRows = 4;
            for (int lm0 = et >> 5; lm0 < nrows; lm0 += kRows * kEpiWarps) {
                float4 acc[kRows];
                for (int src = 0; src < S; ++src) {
                    const float* base = src == split ? sStage + r0 * kTileN : sRecv + src * rows_per * kTileN;
                    float4 v[kRows];
#pragma unroll
                    for (int u = 0; u < kRows; ++u) {
                        const int lm = lm0 + u * kEpiWarps;
                        v[u] = lm < nrows ? *reinterpret_cast<const float4*>(base + lm * kTileN + nl4)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < kRows; ++u) {
                        if (src == 0) {
                            acc[u] = v[u];
                        } else {
                            acc[u].x += v[u].x;
                            acc[u].y += v[u].y;
                            acc[u].z += v[u].z;
                            acc[u].w += v[u].w;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kRows; ++u) {
                    const int lm = lm0 + u * kEpiWarps;
                    if (lm >= nrows) break;
                    uint16_t* crow = p.c + static_cast<int64_t>(m0 + r0 + lm) * p.ldc;
                    const uint32_t lo = pack_bf16x2(acc[u].x, acc[u].y), hi = pack_bf16x2(acc[u].z, acc[u].w);
                    if (v4) {
                        *reinterpret_cast<uint2*>(crow + n4) = make_uint2(lo, hi);
                    } else {
                        const uint16_t h[4] = {static_cast<uint16_t>(lo), static_cast<uint16_t>(lo >> 16),
                                               static_cast<uint16_t>(hi), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            if (n4 + t < p.N) crow[n4 + t] = h[t];
                    }
                }
            }
            if (et == 0) MXFP4_PHASE(11);
        }
        __syncwarp();
        cluster_wait();
        return;
    }

    const int stride = red_stride(rows_per);
    if (vec) {
        // Short runs: each source posts its rows as 16-byte st.async stores into the owners'
        // transposed receive buffers ([source][n][stride]), counted on the owner's red_bar (its
        // own rows as plain stores). An owner sums as soon as all its bytes are in; no CTA waits
        // for the others to finish, since only owners receive and they wait for every byte.
        if (!p.recv_dedicated) cluster_sync();     // every peer is done with the buffers it receives in
        if (threadIdx.x == 96) MXFP4_PHASE(7);
        if (warp >= 3 && ok) {
            const uint32_t recv_addr = smem_addr(sRecv);
            const uint32_t bar_addr = smem_addr(red_bar);
            const uint32_t own_off = static_cast<uint32_t>((split * kTileN + nl) * stride) * 4u;
            for (int cb = half * 32; cb < m_valid; cb += 64) {
                // destinations first: their division and address mapping overlap the loads below
                int owner = cb / rows_per;
                int lm = cb - owner * rows_per;
                uint32_t peer = map_to_rank(recv_addr, static_cast<uint32_t>(owner)) + own_off +
                                static_cast<uint32_t>(lm) * 4u;
                uint32_t peer_bar = map_to_rank(bar_addr, static_cast<uint32_t>(owner));
                uint32_t r[32];
                load_acc32(trow + cb, cb + 16 < m_valid, nacc, acc2, r);
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    if (cb + i < m_valid) {   // rows past M in this group of 4 carry padding, never stored
                        if (owner == split) st_cluster_v4(peer, r[i], r[i + 1], r[i + 2], r[i + 3]);
                        else st_async_v4(peer, r[i], r[i + 1], r[i + 2], r[i + 3], peer_bar);
                        peer += 16u;
                        lm += 4;
                        if (lm == rows_per) {
                            lm = 0;
                            ++owner;
                            if (owner < S) {
                                peer = map_to_rank(recv_addr, static_cast<uint32_t>(owner)) + own_off;
                                peer_bar = map_to_rank(bar_addr, static_cast<uint32_t>(owner));
                            }
                        }
                    }
                }
            }
        }
        if (threadIdx.x == 96) MXFP4_PHASE(8);
        __syncwarp();
        tc_fence_before_sync();
        __syncthreads();                           // own rows visible; TMEM reads done
        if (warp == 1) {
            tc_fence_after_sync();
            tmem_dealloc(tmem_base, p.tmem_cols);
        }
        if (warp >= 3 && r1 > r0) {
            if (!mbar_wait_cluster(red_bar, 0, lim)) {   // rows missing: no sum, no stores
                fail(p, flags);
                return;
            }
            if (threadIdx.x == 96) MXFP4_PHASE(9);
            // owner: a thread sums 4 consecutive rows of one column over the sources in rank order
            const int et = threadIdx.x - 96;
            const int nrows = r1 - r0;
            const int cn = et & (kTileN - 1);
            const int nn = n0 + cn;
            if (nn < p.N) {
                for (int lm = (et / kTileN) * 4; lm < nrows; lm += 4 * (kEpiThreads / kTileN)) {
                    float4 acc = *reinterpret_cast<const float4*>(sRecv + cn * stride + lm);
                    for (int src = 1; src < S; ++src) {
                        const float4 v = *reinterpret_cast<const float4*>(sRecv + (src * kTileN + cn) * stride + lm);
                        acc.x += v.x;
                        acc.y += v.y;
                        acc.z += v.z;
                        acc.w += v.w;
                    }
                    uint16_t* cp = p.c + static_cast<int64_t>(m0 + r0 + lm) * p.ldc + nn;
                    const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (lm + k < nrows) *cp = __bfloat16_as_ushort(__float2bfloat16_rn(vals[k]));
                        cp += p.ldc;
                    }
                }
            }
            if (et == 0) MXFP4_PHASE(11);
        }
        return;
    }

    // Long runs that the bulk form could not stage: posted 4-byte stores along contiguous rows
    // ([source][row][n], one 128-byte segment per warp store), then one cluster barrier.
    if (!p.recv_dedicated) cluster_sync();
    if (threadIdx.x == 96) MXFP4_PHASE(7);
    if (warp >= 3 && ok) {
        const uint32_t recv_addr = smem_addr(sRecv);
        const uint32_t own_off = static_cast<uint32_t>(split * rows_per * kTileN + nl) * 4u;
        for (int cb = half * 32; cb < m_valid; cb += 64) {
            // destinations first: their division and address mapping overlap the loads below
            int owner = cb / rows_per;
            int lm = cb - owner * rows_per;
            uint32_t peer = map_to_rank(recv_addr, static_cast<uint32_t>(owner)) + own_off +
                            static_cast<uint32_t>(lm) * kTileN * 4u;
            uint32_t r[32];
            load_acc32(trow + cb, cb + 16 < m_valid, nacc, acc2, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (cb + i < m_valid) {
                    st_cluster_f32(peer, __uint_as_float(r[i]));
                    peer += kTileN * 4u;
                    if (++lm == rows_per) {
                        lm = 0;
                        ++owner;
                        if (owner < S) peer = map_to_rank(recv_addr, static_cast<uint32_t>(owner)) + own_off;
                    }
                }
            }
        }
    }
    if (threadIdx.x == 96) MXFP4_PHASE(8);
    __syncwarp();
    tc_fence_before_sync();
    cluster_sync();
    if (threadIdx.x == 96) MXFP4_PHASE(9);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
    if (warp >= 3) {
        // owner: a thread sums 4 consecutive columns of one row over the sources in rank order
        const int et = threadIdx.x - 96;
        const int nrows = r1 - r0;
        const int nl4 = (et & 31) * 4;
        const int n4 = n0 + nl4;
        const bool v4 = p.c_vec4 && n4 + 3 < p.N;
        for (int lm = et >> 5; lm < nrows; lm += kEpiWarps) {
            float4 acc = *reinterpret_cast<const float4*>(sRecv + lm * kTileN + nl4);
            for (int src = 1; src < S; ++src) {
                const float4 v = *reinterpret_cast<const float4*>(sRecv + (src * rows_per + lm) * kTileN + nl4);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            uint16_t* crow = p.c + static_cast<int64_t>(m0 + r0 + lm) * p.ldc;
            const uint32_t lo = pack_bf16x2(acc.x, acc.y), hi = pack_bf16x2(acc.z, acc.w);
            if (v4) {
                *reinterpret_cast<uint2*>(crow + n4) = make_uint2(lo, hi);
            } else {
                const uint16_t h[4] = {static_cast<uint16_t>(lo), static_cast<uint16_t>(lo >> 16),
                                       static_cast<uint16_t>(hi), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    if (n4 + t < p.N) crow[n4 + t] = h[t];
            }
        }
        if (et == 0) MXFP4_PHASE(11);
    }
}

// Self-test of the failure path: wait on an mbarrier that nothing ever arrives on.
__global__ void timeout_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(status, 1u);
    }
}

static cudaError_t set_kernel_attributes() {
    static std::mutex mu;
    static std::atomic<bool> attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        for (auto* kernel : {mxfp4_gemm_kernel<false, false, false>, mxfp4_gemm_kernel<true, false, false>,
                             mxfp4_gemm_kernel<true, false, true>, mxfp4_gemm_kernel<true, true, true>}) {
            cudaFuncAttributes fa = {};
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemLimit - fa.sharedSizeBytes));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        attr_set[dev].store(true, std::memory_order_release);
    }
    return cudaSuccess;
}

int max_active_clusters(int cluster_size, size_t smem_bytes) {
    if (set_kernel_attributes() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster_size);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int best = -1;   // the same resources in every instantiation; the smallest count if they ever differ
    for (auto* kernel : {mxfp4_gemm_kernel<false, false, false>, mxfp4_gemm_kernel<true, false, false>,
                         mxfp4_gemm_kernel<true, false, true>, mxfp4_gemm_kernel<true, true, true>}) {
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        best = best < 0 || n < best ? n : best;
    }
    return best;
}

cudaError_t launch_gemm(const GemmPlan& plan, const GemmArgs& args, cudaStream_t s) {
    cudaError_t e = set_kernel_attributes();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.ctas);
    cfg.blockDim = dim3(kGemmThreads);
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
    if (args.fused) return cudaLaunchKernelEx(&cfg, mxfp4_gemm_kernel<false, false, false>, args);
    if (args.m_tile > 128 && args.issuers == 2) return cudaLaunchKernelEx(&cfg, mxfp4_gemm_kernel<true, true, true>, args);
    return args.sf_stores ? cudaLaunchKernelEx(&cfg, mxfp4_gemm_kernel<true, false, true>, args)
                          : cudaLaunchKernelEx(&cfg, mxfp4_gemm_kernel<true, false, false>, args);
}

cudaError_t launch_timeout_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    timeout_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mxfp4

#ifdef MXFP4_TRACE
extern "C" int mxfp4_trace_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, mxfp4::trace_buffer, bytes));
}
extern "C" int mxfp4_ring_read(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, mxfp4::ring_buffer, bytes));
}
extern "C" int mxfp4_trace_clusters(int size, size_t smem) { return mxfp4::max_active_clusters(size, smem); }
#endif
