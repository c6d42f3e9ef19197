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
//   warp 0    : copy producer -- weight blocks (17 KB) and, in the two-kernel path, token
//               blocks. The first stages are requested before the CTA waits on the previous
//               grid (the weights never depend on it).
//   warp 1    : tensor-memory allocation and the single MMA-issuing thread: per 256-K step it
//               copies the scale factors into tensor memory (tcgen05.cp) and issues four
//               128 x N x 64 block-scaled MMAs.
//   warps 2-5 : in the fused path they first quantize the CTA's token slice from bf16 straight
//               into the token-block layout in shared memory (the pages' in-register A
//               quantization, submission 711914 `mxfp4_gemm_fused_k512_kernel`); then they move
//               the accumulator to an fp32 tile in shared memory.
// Reduction: after a cluster barrier each CTA of the cluster sums its share of the tile's rows
// over all K slices through distributed shared memory, in slice order (run-to-run identical),
// and stores bf16 C.
// Every wait on an mbarrier is bounded; on timeout the kernel records an error in the device
// status word and unwinds (outputs undefined, no hang, tensor memory released).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_device.cuh"

namespace mxfp4 {

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) { return smem_desc(addr, 16, 1024, 2); }
__device__ __forceinline__ uint64_t desc_sf(uint32_t addr) { return smem_desc(addr, 0, 128, 0); }

// Instruction descriptor, kind::mxf4: e2m1 x e2m1, both K-major, UE8M0 scales, M = 128.
__device__ __forceinline__ uint32_t idesc_mxf4(uint32_t n_mma) {
    return (1u << 7)                        // A format: e2m1
         | (1u << 10)                       // B format: e2m1
         | ((n_mma >> 3) << 17)             // N / 8
         | (1u << 23)                       // scale factor type UE8M0
         | ((uint32_t(kTileN) >> 4) << 24); // M / 16
}

// OR of a predicate over the 128 threads of warps 2..5 (named barrier 2).
__device__ __forceinline__ bool any_of_128(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred p, 2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

__device__ __forceinline__ void fail(const GemmArgs& p, volatile uint32_t* abort_flag) {
    atomicOr(p.status, 1u);
    *abort_flag = 1u;
}

constexpr int kRedBatch = 8;   // output items a thread reduces at once (loads in flight per source)

__global__ void __launch_bounds__(kGemmThreads, 1)
mxfp4_gemm_kernel(const GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* sB = smem;                           // stages x kWBlock
    uint8_t* sA = smem + p.off_a;                 // token blocks: stages (two-kernel) or atoms (fused)
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* empty = full + kMaxStages;
    uint64_t* a_full = empty + kMaxStages;
    uint64_t* acc_full = a_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile uint32_t* flags = tmem_slot + 1;    // [0] abort
    float* sC = reinterpret_cast<float*>(smem);   // fp32 output tile [token][row], over the idle pipeline

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: (token tile, weight tile, K slice)
    const int split = blockIdx.x % p.splits;      // = rank in the cluster
    const int tile = blockIdx.x / p.splits;
    const int nt = tile % p.n_tiles;
    const int mt = tile / p.n_tiles;
    const int n0 = nt * kTileN;
    const int m0 = mt * p.m_tile;
    const int base = p.k_atoms / p.splits, rem = p.k_atoms % p.splits;
    const int a0 = split * base + (split < rem ? split : rem);
    const int na = base + (split < rem ? 1 : 0);
    const int m_valid = (p.M - m0) < p.m_tile ? (p.M - m0) : p.m_tile;
    const int stages = p.stages;
    const uint32_t a_block = p.a_block;
    const uint32_t a_rows = static_cast<uint32_t>(p.m_tile) * 128u;
    const uint64_t lim = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(a_full, 128);
        mbar_init(acc_full, 1);
        flags[0] = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------------------- producer
            const uint8_t* bsrc = p.bblk + (static_cast<size_t>(nt) * p.k_atoms + a0) * kWBlock;
            const uint8_t* asrc = p.ablk + (static_cast<size_t>(mt) * p.k_atoms + a0) * a_block;
            const uint32_t tx_bytes = kWBlock + (p.fused ? 0u : a_block);
            const uint64_t pol_b = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            const int npro = na < stages ? na : stages;
            for (int j = 0; j < npro; ++j) {
                mbar_arrive_expect_tx(&full[j], tx_bytes);
                bulk_load(sB + j * kWBlock, bsrc + static_cast<size_t>(j) * kWBlock, kWBlock, &full[j], pol_b);
            }
            pdl_wait_prior_grid();   // token blocks are written by the previous grid
            if (!p.fused)
                for (int j = 0; j < npro; ++j)
                    bulk_load(sA + j * a_block, asrc + static_cast<size_t>(j) * a_block, a_block, &full[j], pol_a);
            int issued = npro;
            for (int j = npro; j < na; ++j) {
                const int s = j % stages;
                if (!mbar_wait(&empty[s], ((j / stages) - 1) & 1, lim)) { fail(p, flags); break; }
                mbar_arrive_expect_tx(&full[s], tx_bytes);
                bulk_load(sB + s * kWBlock, bsrc + static_cast<size_t>(j) * kWBlock, kWBlock, &full[s], pol_b);
                if (!p.fused)
                    bulk_load(sA + s * a_block, asrc + static_cast<size_t>(j) * a_block, a_block, &full[s], pol_a);
                issued = j + 1;
            }
            // never leave copies in flight into shared memory that is about to be reused or freed
            for (int j = (issued > stages ? issued - stages : 0); j < issued; ++j)
                mbar_wait(&full[j % stages], (j / stages) & 1, lim);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------------- MMA issuer
        // Columns are allocated only after the previous grid has finished, so a CTA of this
        // grid never holds columns a CTA of the previous grid is still waiting for.
        pdl_wait_prior_grid();
        tmem_alloc(const_cast<uint32_t*>(tmem_slot), p.tmem_cols);
        tmem_relinquish();
        tc_fence_before_sync();
        named_barrier_arrive(1, 160);             // publish the column base to warps 2..5
        __syncwarp();
        tc_fence_after_sync();
        const uint32_t tmem_base = *tmem_slot;
        if (lane == 0) {
            const uint32_t t_acc = tmem_base;
            const uint32_t t_sfb = tmem_base + static_cast<uint32_t>(p.m_tile);
            const uint32_t t_sfa = t_sfb + static_cast<uint32_t>(stages) * 8u;
            const uint32_t idesc0 = idesc_mxf4(static_cast<uint32_t>(p.m_tile));
            bool ok = true;
            if (p.fused) ok = mbar_wait(a_full, 0, lim);
            tc_fence_after_sync();
            for (int j = 0; ok && j < na; ++j) {
                const int s = j % stages;
                if (!mbar_wait(&full[s], (j / stages) & 1, lim)) { ok = false; break; }
                tc_fence_after_sync();
                const uint8_t* bb = sB + s * kWBlock;
                const uint8_t* ab = sA + (p.fused ? j : s) * a_block;
                const uint32_t sfb_cols = t_sfb + static_cast<uint32_t>(s) * 8u;
                const uint32_t sfa_cols = t_sfa + static_cast<uint32_t>(s) * 8u * p.nmc;
                for (int g = 0; g < 2; ++g) {
                    tc_copy_sf(sfb_cols + 4u * g, desc_sf(smem_addr(bb + kBRowsBytes + kSfChunk * g)));
                    for (int c = 0; c < p.nmc; ++c)
                        tc_copy_sf(sfa_cols + 4u * (g * p.nmc + c),
                                   desc_sf(smem_addr(ab + a_rows + kSfChunk * (2 * c + g))));
                }
                const uint32_t b_addr = smem_addr(bb);
                const uint32_t a_addr = smem_addr(ab);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t g = kk >> 1;
                    const uint32_t sf_id = (kk & 1) * 2u;   // scale bytes {0,1} or {2,3} of the column
                    const uint32_t idesc = idesc0 | (sf_id << 29) | (sf_id << 4);
                    mma_mxf4(t_acc, desc_sw128(b_addr + 32u * kk), desc_sw128(a_addr + 32u * kk), idesc,
                             sfb_cols + 4u * g, sfa_cols + 4u * g * p.nmc, (j | kk) != 0);
                }
                tc_commit(&empty[s]);
            }
            if (!ok) fail(p, flags);
            tc_commit(acc_full);
        }
    } else {
        // -------------------------------------------------------------------- warps 2..5
        const int et = threadIdx.x - 64;
        pdl_wait_prior_grid();   // A may come from the previous grid; C may still be read by it
        if (p.fused) {
            // Quantize this CTA's token rows of its K slice into token blocks in shared memory,
            // one 1x32 block per item; two items' loads are issued before either is converted.
            const int nblk = na * (kAtomK / 32);
            const int total = p.m_tile * nblk;   // rows past M are written as zeros
            for (int first = et; first < total; first += 256) {
                uint32_t w[2][16];
                int rr[2], kk[2];
                bool live[2], inside[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int idx = first + 128 * u;
                    live[u] = idx < total;
                    rr[u] = live[u] ? idx / nblk : 0;
                    kk[u] = live[u] ? idx - rr[u] * nblk : 0;
                    const int gk = (a0 + (kk[u] >> 3)) * kAtomK + (kk[u] & 7) * 32;
                    inside[u] = live[u] && rr[u] < m_valid && gk < p.K;
                    if (inside[u]) load_block32(p.a + static_cast<int64_t>(m0 + rr[u]) * p.lda + gk, w[u]);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (!live[u]) continue;
                    uint32_t out[4] = {0u, 0u, 0u, 0u};
                    const uint32_t sbyte = inside[u] ? quantize_block32(w[u], out) : 0u;
                    const uint32_t r = static_cast<uint32_t>(rr[u]), c = static_cast<uint32_t>(kk[u] & 7);
                    uint8_t* blk = sA + (kk[u] >> 3) * a_block;
                    *reinterpret_cast<uint4*>(blk + swz_chunk_offset(r, c)) = make_uint4(out[0], out[1], out[2], out[3]);
                    blk[a_rows + block_sf_offset(r, c)] = static_cast<uint8_t>(sbyte);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(a_full);
        }
        const bool waited = mbar_wait(acc_full, 0, lim);
        named_barrier(1, 160);                    // the column base from warp 1
        tc_fence_after_sync();
        if (!waited) fail(p, flags);
        // one decision for all 128 threads (tcgen05.ld is warp-collective)
        const bool ok = !any_of_128(!waited || flags[0] != 0u);
        if (ok) {
            // accumulator D = C^T (lane = weight row, column = token) -> fp32 tile [token][row]
            const int q = warp & 3;               // this warp's 32-lane slice of tensor memory
            const int nl = q * 32 + lane;
            const uint32_t trow = *tmem_slot + (static_cast<uint32_t>(q * 32) << 16);
            for (int cb = 0; cb < m_valid; cb += 32) {
                uint32_t r[32];
                tmem_load_16(trow + cb, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
                if (cb + 16 < m_valid) tmem_load_16(trow + cb + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
                tmem_load_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (cb + i < m_valid) sC[(cb + i) * kTileN + nl] = __uint_as_float(r[i]);
            }
        }
    }

    // ------------------------------------------------------------------------ tile reduction
    __syncwarp();
    tc_fence_before_sync();
    if (p.splits > 1) cluster_sync();
    else __syncthreads();
    if (warp >= 2) {
        const int et = threadIdx.x - 64;
        const int S = p.splits;
        const int rows_per = (m_valid + S - 1) / S;
        const int r0 = split * rows_per;
        const int r1 = min(m_valid, r0 + rows_per);
        const int items = r1 > r0 ? (r1 - r0) * (kTileN / 4) : 0;   // 4 output columns per item
        const uint32_t sC_addr = smem_addr(sC);
        for (int first = et; first < items; first += 128 * kRedBatch) {
            float4 acc[kRedBatch];
            uint32_t off[kRedBatch];
#pragma unroll
            for (int u = 0; u < kRedBatch; ++u) {
                const int i = first + 128 * u;
                const int m = r0 + i / (kTileN / 4);
                off[u] = static_cast<uint32_t>(m * kTileN + (i % (kTileN / 4)) * 4) * 4u;
                acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            // slice order 0, 1, ..., S-1: the same sum whichever CTA finished first
            for (int src = 0; src < S; ++src) {
                const uint32_t peer = S == 1 ? sC_addr : map_to_rank(sC_addr, static_cast<uint32_t>(src));
                float4 v[kRedBatch];
#pragma unroll
                for (int u = 0; u < kRedBatch; ++u) {
                    if (first + 128 * u >= items) continue;
                    if (S == 1) v[u] = *reinterpret_cast<const float4*>(reinterpret_cast<const uint8_t*>(sC) + off[u]);
                    else v[u] = ld_cluster_f32x4(peer + off[u]);
                }
#pragma unroll
                for (int u = 0; u < kRedBatch; ++u) {
                    if (first + 128 * u < items) {
                        acc[u].x += v[u].x;
                        acc[u].y += v[u].y;
                        acc[u].z += v[u].z;
                        acc[u].w += v[u].w;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kRedBatch; ++u) {
                const int i = first + 128 * u;
                if (i >= items) continue;
                const int m = r0 + i / (kTileN / 4);
                const int n = n0 + (i % (kTileN / 4)) * 4;
                uint16_t* crow = p.c + static_cast<int64_t>(m0 + m) * p.ldc;
                const uint32_t lo = pack_bf16x2(acc[u].x, acc[u].y), hi = pack_bf16x2(acc[u].z, acc[u].w);
                if (p.c_vec4 && n + 3 < p.N) {
                    *reinterpret_cast<uint2*>(crow + n) = make_uint2(lo, hi);
                } else {
                    const uint16_t h[4] = {static_cast<uint16_t>(lo), static_cast<uint16_t>(lo >> 16),
                                           static_cast<uint16_t>(hi), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (n + t < p.N) crow[n + t] = h[t];
                }
            }
        }
    }
    __syncwarp();
    if (p.splits > 1) cluster_sync();   // keep this CTA's staged tile alive until every peer read it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(*tmem_slot, p.tmem_cols);
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
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(mxfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLimit));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(mxfp4_gemm_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
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
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mxfp4_gemm_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
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
    return cudaLaunchKernelEx(&cfg, mxfp4_gemm_kernel, args);
}

cudaError_t launch_timeout_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    timeout_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mxfp4
