// Block-scaled MXFP4 GEMM on the sm_103a tensor cores: tcgen05.mma kind::mxf4 with e8m0
// scale factors in tensor memory, TMA-fed shared-memory pipelines and a bf16 epilogue.
//
// Orientation. The weights B[N,K] are the MMA's 128-row "A" operand and the tokens A[M,K]
// the MMA's "B" operand (N_mma = token tile, 16..256), so the small-M shapes still fill the
// 128-row MMA and D = C^T sits in tensor memory with one weight row per lane.
//
// One CTA = one (weight tile of 128 rows, token tile, K slice). Warp roles:
//   warp 0    : TMA producer -- weight tiles (128 rows x 256 K = 16 KB, 128-byte swizzle)
//               and their scale chunks; in the two-kernel path also the pre-quantized
//               token tile and its scale chunks. The first stages are issued before the
//               CTA waits on the previous grid (weights never depend on it).
//   warp 1    : tensor-memory allocation and the single MMA-issuing thread: per 256-K
//               step it copies the scale factors into tensor memory (tcgen05.cp) and issues
//               four 128 x N x 64 block-scaled MMAs.
//   warps 2-5 : in the fused path they first quantize the CTA's token slice from bf16
//               straight into the swizzled shared-memory layout the MMA reads (the pages'
//               in-register A quantization, submission 711914 `mxfp4_gemm_fused_k512_kernel`);
//               then the epilogue: tensor memory -> registers -> bf16 C, or, with split-K,
//               fp32 partial tiles whose last-arriving CTA sums all slices in slice order.
// Every wait on an mbarrier is bounded; on timeout the kernel records an error in the
// device status word and unwinds (outputs undefined, no hang, tensor memory released).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_device.cuh"

namespace mxfp4 {

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) { return smem_desc(addr, 16, 1024, 2); }
__device__ __forceinline__ uint64_t desc_sf(uint32_t addr) { return smem_desc(addr, 0, 128, 0); }

// Instruction descriptor, kind::mxf4: e2m1 x e2m1, both K-major, UE8M0 scales, M = 128.
__device__ __forceinline__ uint32_t idesc_mxf4(uint32_t n_mma) {
    return (1u << 7)                      // A format: e2m1
         | (1u << 10)                     // B format: e2m1
         | ((n_mma >> 3) << 17)           // N / 8
         | (1u << 23)                     // scale factor type UE8M0
         | ((uint32_t(kTileN) >> 4) << 24);   // M / 16
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

__device__ __forceinline__ void fail(const GemmArgs& p, volatile uint32_t* abort_flag) {
    atomicOr(p.status, 1u);
    *abort_flag = 1u;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
mxfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_a,
                  const GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* sB = smem;
    uint8_t* sA = smem + p.off_a;
    uint8_t* sSFB = smem + p.off_sfb;
    uint8_t* sSFA = smem + p.off_sfa;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* empty = full + kMaxStages;
    uint64_t* a_full = empty + kMaxStages;
    uint64_t* acc_full = a_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile uint32_t* flags = tmem_slot + 1;   // [0] abort, [1] this CTA reduces the tile

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: (token tile, weight tile, K slice)
    const int split = blockIdx.x % p.splits;
    const int tile = blockIdx.x / p.splits;
    const int nt = tile % p.n_tiles;
    const int mt = tile / p.n_tiles;
    const int n0 = nt * kTileN;
    const int m0 = mt * p.m_tile;
    const int base = p.k_atoms / p.splits, rem = p.k_atoms % p.splits;
    const int a0 = split * base + (split < rem ? split : rem);
    const int na = base + (split < rem ? 1 : 0);
    const int stages = p.stages;
    const uint32_t a_bytes = static_cast<uint32_t>(p.m_tile) * 128u;
    const uint32_t sfa_bytes = static_cast<uint32_t>(p.nmc) * 1024u;
    const uint32_t tx_bytes = kBStageBytes + 1024u + (p.fused ? 0u : a_bytes + sfa_bytes);

    auto issue_b = [&](int j, int s, uint64_t pol) {
        tma_load_2d(sB + s * kBStageBytes, &tmap_b, (a0 + j) * (kAtomK / 2), n0, &full[s], pol);
        bulk_load(sSFB + s * 1024, p.sfb + (static_cast<size_t>(nt) * p.groups + 2 * (a0 + j)) * kSfChunk, 1024u,
                  &full[s], pol);
    };
    auto issue_a = [&](int j, int s, uint64_t pol) {
        tma_load_2d(sA + s * a_bytes, &tmap_a, (a0 + j) * (kAtomK / 2), m0, &full[s], pol);
        for (int c = 0; c < p.nmc; ++c)
            bulk_load(sSFA + s * sfa_bytes + c * 1024,
                      p.sfa + (static_cast<size_t>(m0 / 128 + c) * p.groups + 2 * (a0 + j)) * kSfChunk, 1024u,
                      &full[s], pol);
    };

    int issued[kMaxStages];
    const int npro = na < stages ? na : stages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            issued[s] = 0;
        }
        mbar_init(a_full, 128);
        mbar_init(acc_full, 1);
        flags[0] = 0u;
        flags[1] = 0u;
        fence_mbar_init();
        prefetch_tensormap(&tmap_b);
        if (!p.fused) prefetch_tensormap(&tmap_a);
        // weights never depend on the previous grid: start streaming them right away
        const uint64_t pol_b = policy_evict_first();
        for (int j = 0; j < npro; ++j) {
            mbar_arrive_expect_tx(&full[j], tx_bytes);
            issue_b(j, j, pol_b);
            issued[j] = 1;
        }
    }
    pdl_launch_dependents();
    // Everything below may read what the previous grid wrote or write what it reads; tensor
    // memory is also allocated only after it has finished (so a CTA of this grid never holds
    // columns a CTA of the previous grid is still waiting for).
    pdl_wait_prior_grid();
    if (warp == 1) {
        tmem_alloc(const_cast<uint32_t*>(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t t_acc = tmem_base;
    const uint32_t t_sfb = tmem_base + static_cast<uint32_t>(p.m_tile);
    const uint32_t t_sfa = t_sfb + static_cast<uint32_t>(stages) * 8u;
    const uint64_t lim = p.wait_limit_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------------------- producer
            const uint64_t pol_b = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            if (!p.fused)
                for (int j = 0; j < npro; ++j) issue_a(j, j, pol_a);
            for (int j = npro; j < na; ++j) {
                const int s = j % stages;
                if (!mbar_wait(&empty[s], ((j / stages) - 1) & 1, lim)) { fail(p, flags); break; }
                mbar_arrive_expect_tx(&full[s], tx_bytes);
                issue_b(j, s, pol_b);
                if (!p.fused) issue_a(j, s, pol_a);
                ++issued[s];
            }
            // never leave copies in flight into shared memory that is about to be released
            for (int s = 0; s < stages; ++s)
                if (issued[s] > 0) mbar_wait(&full[s], (issued[s] - 1) & 1, lim);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------------------- MMA issuer
            const uint32_t idesc0 = idesc_mxf4(static_cast<uint32_t>(p.m_tile));
            bool ok = true;
            if (p.fused) ok = mbar_wait(a_full, 0, lim);
            tc_fence_after_sync();
            for (int j = 0; ok && j < na; ++j) {
                const int s = j % stages;
                if (!mbar_wait(&full[s], (j / stages) & 1, lim)) { ok = false; break; }
                tc_fence_after_sync();
                const uint8_t* a_src = sA + (p.fused ? j : s) * a_bytes;
                const uint8_t* sfa_src = sSFA + (p.fused ? j : s) * sfa_bytes;
                const uint32_t sfb_cols = t_sfb + static_cast<uint32_t>(s) * 8u;
                const uint32_t sfa_cols = t_sfa + static_cast<uint32_t>(s) * 8u * p.nmc;
                for (int g = 0; g < 2; ++g) {
                    tc_copy_sf(sfb_cols + 4u * g, desc_sf(smem_addr(sSFB + s * 1024 + 512 * g)));
                    for (int c = 0; c < p.nmc; ++c)
                        tc_copy_sf(sfa_cols + 4u * (g * p.nmc + c), desc_sf(smem_addr(sfa_src + c * 1024 + 512 * g)));
                }
                const uint32_t b_addr = smem_addr(sB + s * kBStageBytes);
                const uint32_t a_addr = smem_addr(a_src);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t g = kk >> 1;
                    const uint32_t sf_id = (kk & 1) * 2u;     // scale bytes {0,1} or {2,3} of the column
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
        if (p.fused) {
            // quantize rows m0 .. m0+m_tile of this K slice into the swizzled MMA layout
            const int nblk = na * (kAtomK / 32);
            const int total = p.m_tile * nblk;
            for (int idx = et; idx < total; idx += 128) {
                const int r = idx / nblk;
                const int kb = idx - r * nblk;
                const int atom = kb >> 3, c = kb & 7;
                const int gk = (a0 + atom) * kAtomK + c * 32;
                const int m = m0 + r;
                uint32_t out[4] = {0u, 0u, 0u, 0u};
                uint32_t sbyte = 0u;
                if (m < p.M && gk < p.K) {
                    uint32_t w[16];
                    load_block32(p.a + static_cast<int64_t>(m) * p.lda + gk, w);
                    sbyte = quantize_block32(w, out);
                }
                uint8_t* dst = sA + atom * a_bytes + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
                sSFA[atom * sfa_bytes + sf_chunk_offset(static_cast<uint32_t>(r), static_cast<uint32_t>(c), 2u)] =
                    static_cast<uint8_t>(sbyte);
            }
            fence_proxy_async_smem();
            mbar_arrive(a_full);
        }
        const bool waited = mbar_wait(acc_full, 0, lim);
        tc_fence_after_sync();
        if (!waited) fail(p, flags);
        // one decision for all 128 threads, so the named barriers below are always matched
        const bool ok = !any_of_128(!waited || flags[0] != 0u);
        const int q = warp & 3;                    // this warp's 32-lane slice of tensor memory
        const int nl = q * 32 + lane;              // weight row within the tile
        const int n = n0 + nl;
        const uint32_t trow = t_acc + (static_cast<uint32_t>(q * 32) << 16);
        const int m_valid = (p.M - m0) < p.m_tile ? (p.M - m0) : p.m_tile;
        if (ok) {
            if (p.splits == 1) {
                for (int cb = 0; cb < m_valid; cb += 16) {
                    uint32_t r[16];
                    tmem_load_16(trow + cb, r);
                    tmem_load_wait();
                    if (n < p.N) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (cb + i < m_valid)
                                p.c[static_cast<int64_t>(m0 + cb + i) * p.ldc + n] =
                                    __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[i])));
                    }
                }
            } else {
                float* mine = p.part + (static_cast<size_t>(tile) * p.splits + split) * (kTileN * p.m_tile);
                for (int cb = 0; cb < m_valid; cb += 16) {
                    uint32_t r[16];
                    tmem_load_16(trow + cb, r);
                    tmem_load_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (cb + i < m_valid) mine[(cb + i) * kTileN + nl] = __uint_as_float(r[i]);
                }
                __threadfence();
                named_barrier(1, 128);
                if (et == 0) {
                    const uint32_t prev = atomicAdd(&p.ctr[tile], 1u);
                    flags[1] = (prev == static_cast<uint32_t>(p.splits - 1)) ? 1u : 0u;
                }
                named_barrier(1, 128);
                if (flags[1]) {
                    __threadfence();
                    if (et == 0) p.ctr[tile] = 0u;    // leave the counter ready for the next call
                    const float* tp = p.part + static_cast<size_t>(tile) * p.splits * (kTileN * p.m_tile);
                    if (n < p.N) {
                        for (int m = 0; m < m_valid; ++m) {
                            float acc = 0.0f;
                            for (int sp = 0; sp < p.splits; ++sp)
                                acc += __ldcg(tp + (static_cast<size_t>(sp) * p.m_tile + m) * kTileN + nl);
                            p.c[static_cast<int64_t>(m0 + m) * p.ldc + n] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(acc));
                        }
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, p.tmem_cols);
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

cudaError_t launch_gemm(const GemmPlan& plan, const CUtensorMap& tmap_b, const CUtensorMap& tmap_a,
                        const GemmArgs& args, cudaStream_t s) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(mxfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLimit));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return launch_pdl(mxfp4_gemm_kernel, dim3(plan.ctas), dim3(kGemmThreads), plan.smem_bytes, s, tmap_b, tmap_a,
                      args);
}

cudaError_t launch_timeout_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    timeout_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mxfp4
