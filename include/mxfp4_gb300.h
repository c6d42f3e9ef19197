/*
 * mxfp4_gb300.h -- C ABI of the GB300 (sm_103a) block-scaled MXFP4 GEMM library.
 *
 *   C[M,N] (bf16) = MXFP4(A[M,K] bf16) . MXFP4(B[N,K])^T
 *
 * MXFP4 here is the format the "amd-mxfp4-mm" leaderboard submissions compute (submission
 * 711914, `_mxfp4_quant_tile`; submission 608632, `_hw_mxfp4_quant_op`): along K, every
 * block of 32 consecutive elements of a row shares one e8m0 scale byte; each element is a
 * 4-bit e2m1 code (bit 3 sign, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) and two codes share a
 * byte, the even-indexed element in the low nibble.
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers (cudaMalloc'd or equivalent) unless stated.
 *     The caller owns every buffer; the library never allocates, frees or synchronizes
 *     (except mxfp4_device_status, which synchronizes the given stream by design).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Work is
 *     enqueued asynchronously on it.
 *   - Matrices are row-major with the K dimension contiguous. Sizes are element counts.
 *   - Return value: an mxfp4_status. Arguments are validated before anything is enqueued;
 *     on an error nothing is written. MXFP4_ERR_CUDA reports a launch failure (see
 *     mxfp4_last_cuda_error). Kernel-side failures (a bounded wait that ran out) are not
 *     visible in the return value of the asynchronous call; read them with
 *     mxfp4_device_status.
 *   - Inputs must be finite; NaN or Inf in A or B gives unspecified (but memory-safe)
 *     results. Scale bytes of 255 (e8m0 NaN) in B likewise.
 *   - K is a positive multiple of 8 (bf16 rows move in 16-byte pieces). A row has
 *     nblk = ceil(K/32) blocks; when K % 32 != 0 the last block is cut by K and its elements
 *     past K count as zeros, as submission 711914's `_standalone_quant_kernel` loads A under
 *     the mask offs_k < K with 0 as the fill value: they do not change the block's scale and
 *     are stored as zero codes. The natural packed layout keeps whole blocks: codes
 *     [rows, nblk*16] bytes, scales [rows, nblk] bytes.
 *   - Size limits of the GEMM and the weight prepack: M and N below 2^31, K at most 2^30
 *     (MXFP4_ERR_SHAPE beyond; mxfp4_prepack_b_size returns 0).
 *   - The library targets compute capability 10.3 (GB300) only; other devices give
 *     MXFP4_ERR_ARCH.
 */
#ifndef MXFP4_GB300_H
#define MXFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MXFP4_OK = 0,
    MXFP4_ERR_ARG = 1,       /* null pointer, negative size, bad option value */
    MXFP4_ERR_SHAPE = 2,     /* K not a positive multiple of 8, ld smaller than K, too large */
    MXFP4_ERR_ALIGN = 3,     /* pointer or leading dimension misaligned (see each call) */
    MXFP4_ERR_ARCH = 4,      /* current device is not compute capability 10.3 */
    MXFP4_ERR_CUDA = 5,      /* a CUDA runtime/driver call or a launch failed */
    MXFP4_ERR_TIMEOUT = 6,   /* a device-side bounded wait ran out (from mxfp4_device_status) */
    MXFP4_ERR_WORKSPACE = 7  /* workspace missing or smaller than mxfp4_gemm_workspace_size */
} mxfp4_status;

/* Human-readable name of a status code (static string). */
const char *mxfp4_status_string(int status);

/* Last CUDA error code (cudaError_t as int) recorded by a call that returned MXFP4_ERR_CUDA
 * on this host thread, 0 if none. */
int mxfp4_last_cuda_error(void);

/* Library ABI version (major*100 + minor). 2.01: K any multiple of 8 (was a multiple of 64).
 * 2.02: token-block entry points (mxfp4_quantize_tokens, mxfp4_gemm_tokens). 2.03: prepared
 * calls (mxfp4_call_create, mxfp4_call_create_host, mxfp4_call_run, mxfp4_call_destroy), the
 * scale_stores field of mxfp4_plan_info, mxfp4_gemm_unpacked. 2.04: mxfp4_gemm_options.flags
 * (MXFP4_GEMM_A_READY) and mxfp4_plan_info.a_early. */
int mxfp4_version(void);

/*
 * mxfp4_quantize -- quantize a bf16 matrix to MXFP4 (one e8m0 scale per 1x32 block).
 * Follows submission 711914, `_mxfp4_quant_tile`: amax = max|x| of the block in fp32; the
 * amax bit pattern plus 0x200000, masked with 0xFF800000, rounds it to a power of two;
 * s = clamp(floor(log2(amax_r)) - 2, -127, 127); scale byte = s + 127; each element
 * x * 2^-s is rounded to the nearest e2m1 value (ties to even, saturating at 6, the sign
 * kept even when the value rounds to zero) and packed even-low / odd-high.
 *   x       : bf16 [rows, K], row stride `ld` elements (ld >= K). 16-byte aligned, ld % 8 == 0.
 *   q       : out, uint8 [rows, nblk*16] (nblk = ceil(K/32)), row stride nblk*16 bytes
 *             (K/2 when K % 32 == 0). 16-byte aligned. Codes past K are zero.
 *   scales  : out, uint8 [rows, nblk], row stride nblk bytes (no alignment requirement).
 *   K       : multiple of 8.  rows == 0 or K == 0 is a no-op.
 * Bytes are bit-identical to the CPU oracle.
 */
int mxfp4_quantize(const void *x, int64_t rows, int64_t K, int64_t ld,
                   void *q, void *scales, void *stream);

/*
 * mxfp4_prepack_b_size -- bytes of the packed-B buffer mxfp4_prepack_b writes for an
 * [N, K] weight matrix. Its counterpart in the pages is the shuffled weight buffer their
 * harness builds once before timing (submission 608632, `_new_generate_input`: B quantized,
 * then `shuffle_weight` and `e8m0_shuffle` for the MFMA layout). Here the buffer is
 * ceil(N/128) x ceil(K/256) blocks of 17408 bytes, one per 128-row
 * tile and 256-element K step, each holding that piece's e2m1 rows (16 KB, swizzled the
 * way the tensor cores read shared memory) and its e8m0 scales (1 KB, in the tensor-memory
 * scale-factor layout). Rows past N and K past the last multiple of 256 are zero padding.
 * 0 for invalid sizes (including N >= 2^31 or K > 2^30).
 */
size_t mxfp4_prepack_b_size(int64_t N, int64_t K);

/*
 * mxfp4_prepack_b -- one-time relayout of a pre-quantized weight matrix B for mxfp4_gemm.
 * The pages prepare B outside the timed call too (their harness shuffles B and its scales
 * for the MFMA layout, submission 608632 `_new_generate_input`); here every (128-row tile,
 * 256-K step) becomes one contiguous block that is the exact shared-memory image the tcgen05
 * block-scaled MMA reads, so the GEMM streams the weights with one bulk copy per step.
 *   bq     : uint8 [N, nblk*16] packed e2m1 (even element low nibble), nblk = ceil(K/32),
 *            row stride nblk*16 bytes (the layout mxfp4_quantize writes). 16-byte aligned.
 *            Codes past K only ever meet A's zero codes, so their value does not matter.
 *   bs     : uint8 [N, nblk] e8m0 scales (as written by mxfp4_quantize).
 *   K      : positive multiple of 8.  N >= 1. K and ceil(K/32)*32 give the same buffer.
 *   packed : out, mxfp4_prepack_b_size(N, K) bytes, 1024-byte aligned. Must not overlap
 *            bq or bs.
 */
int mxfp4_prepack_b(const void *bq, const void *bs, int64_t N, int64_t K,
                    void *packed, void *stream);

/*
 * mxfp4_gemm_workspace_size -- bytes of device workspace mxfp4_gemm needs for this shape
 * on the CURRENT device (the plan depends on its SM count). Its counterpart in the pages is
 * the per-shape buffer cache of submission 711914 (`_quant_buffers`: the quantized A and its
 * scales, kept between calls of one shape), here owned by the caller. The workspace holds the
 * quantized A (as token blocks) of the two-kernel path; plans that quantize A inside the
 * GEMM (the automatic plan for small M, see mxfp4_gemm_plan_info) need none and return 0.
 * Split-K partial sums never leave the chip.
 */
size_t mxfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * mxfp4_workspace_init -- zero-fill a workspace (cudaMemsetAsync on `stream`). Optional:
 * the GEMM never depends on the workspace's previous contents.
 */
int mxfp4_workspace_init(void *workspace, size_t ws_bytes, void *stream);

/*
 * mxfp4_gemm -- C = MXFP4(A) . MXFP4(B)^T in bf16, A quantized inside the call.
 * Defined by the pages' GEMM kernels, for example submission 711914's
 * `mxfp4_gemm_fused_k512_kernel`: A quantized per 1x32 block (`_mxfp4_quant_tile`), then
 * `tl.dot_scaled(a_fp4, a_scales, "e2m1", b, b_scales, "e2m1")` accumulated in fp32 over K and cast
 * to bf16; the entry point there is `custom_kernel`, which takes A, the pre-quantized B and
 * its scales and returns C.
 * The products of e2m1 values and e8m0 scales are accumulated in fp32 on the tensor cores
 * (tcgen05.mma kind::mxf4, block size 32) and rounded once to bf16 (round to nearest even).
 *   a        : bf16 [M, K], row stride lda elements (lda >= K, lda % 8 == 0), 16-byte aligned.
 *   packed_b : buffer written by mxfp4_prepack_b for the same N and K.
 *   c        : out, bf16 [M, N], row stride ldc elements (ldc >= N), 2-byte aligned.
 *   workspace: ws_bytes >= mxfp4_gemm_workspace_size(M, N, K), 256-byte aligned; may be
 *              NULL when that size is 0. Calls sharing a workspace must be ordered (same
 *              stream, or synchronized); overlapping calls on one workspace race.
 *   K        : positive multiple of 8.  M == 0 or N == 0 is a no-op.
 * Ordering: the call waits for the work before it on `stream` before it reads A or writes C.
 * The weights in packed_b are requested before that wait (they are meant to be constant), so
 * packed_b must not be written by a kernel that is still running when the call is enqueued and
 * that lets dependent launches start early (programmatic dependent launch). Ordinary kernels and
 * copies never let them; this library's kernels do, but none of them writes packed_b that way
 * (mxfp4_prepack_b's kernel does not let dependents start early).
 * A is quantized exactly like mxfp4_quantize (bit-identical codes and scales). With split-K
 * the K slices of an output tile run as one thread-block cluster and their fp32 partial
 * sums are added in slice order through distributed shared memory, so results are
 * run-to-run identical.
 */
int mxfp4_gemm(const void *a, int64_t M, int64_t K, int64_t lda,
               const void *packed_b, int64_t N,
               void *c, int64_t ldc,
               void *workspace, size_t ws_bytes, void *stream);

/* Plan overrides for mxfp4_gemm_ex (tests and measurement). Zero-initialise, then set. */
typedef struct {
    int path;    /* 0 = automatic, 1 = A quantized inside the GEMM's producer warps (fused),
                    2 = standalone quantize kernel into the workspace, then the GEMM */
    int splits;  /* 0 = automatic, else the number of K slices per output tile (>= 1) */
    int m_tile;  /* 0 = automatic, else tokens per tile: a multiple of 16 in [16, 256] */
    int flags;   /* 0, or MXFP4_GEMM_A_READY (below); other bits: MXFP4_ERR_ARG */
    int reserved[4];
} mxfp4_gemm_options;

/* MXFP4_GEMM_A_READY -- the caller guarantees that every write to A was made by work that had
 * finished before the operation enqueued just before this call on the stream began to run. The
 * call's kernels may start as soon as that operation starts (they are launched as programmatic
 * dependents, and the calls of this library let their dependents start early), so A must not be
 * written by that operation nor by anything still running when it starts. Typical use: the
 * second and later of several calls that read the same A (projections of one activation,
 * experts on one gathered batch), when the first of them follows A's producer and that producer
 * is an ordinary kernel or copy. Not valid for A written by the call just before, nor for the C
 * of a call of this library whose successor is the first reader. With the flag the call loads
 * and quantizes A as soon as its kernels start, overlapping the work before it; it still writes
 * nothing (C, workspace) before that work has finished. With an explicit plan (path and splits
 * given) the results are the same bits either way. The automatic plan may differ with the flag
 * (mxfp4_plan_info.a_early): up to 32 tokens, fewer K slices whose CTAs fill at most half the
 * SMs, when the flagless weight-resident plan leaves no room to read A early or none fits (the
 * flagless call then runs the two-kernel path); C then differs from the flagless call's only by
 * the order of the split-K sum, within the same tolerance. */
#define MXFP4_GEMM_A_READY 1

/* mxfp4_gemm with an explicit plan. The workspace must be at least
 * mxfp4_gemm_workspace_size_ex(M, N, K, opts). opts == NULL is the automatic plan. */
int mxfp4_gemm_ex(const void *a, int64_t M, int64_t K, int64_t lda,
                  const void *packed_b, int64_t N,
                  void *c, int64_t ldc,
                  void *workspace, size_t ws_bytes,
                  const mxfp4_gemm_options *opts, void *stream);
size_t mxfp4_gemm_workspace_size_ex(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options *opts);

/* The plan mxfp4_gemm_ex would run on the current device: path (1 fused / 2 two-kernel),
 * splits, M tile, number of CTAs, pipeline stages (NULL outputs are skipped). Returns MXFP4_OK,
 * an argument or shape error, or MXFP4_ERR_ARCH / MXFP4_ERR_CUDA from the device query. */
int mxfp4_gemm_plan(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options *opts,
                    int *path, int *splits, int *m_tile, int *ctas, int *stages);

/*
 * mxfp4_gemm_unpacked -- mxfp4_gemm for B as mxfp4_quantize writes it: packed e2m1 nibbles
 * bq [N, nblk*16] and e8m0 scales bs [N, nblk] (nblk = ceil(K/32)), the two arrays the pages'
 * `custom_kernel` receives with A. The call first writes B's prepacked image (mxfp4_prepack_b)
 * into the workspace, then runs mxfp4_gemm on it: the same C, bit for bit, at the cost of the
 * prepack on every call. For weights used more than once, prepack them once and call mxfp4_gemm.
 *   a, c, M, K, lda, ldc, N: as for mxfp4_gemm.  bq, bs: as for mxfp4_prepack_b.
 *   workspace: ws_bytes >= mxfp4_gemm_unpacked_workspace_size(M, N, K), 1024-byte aligned:
 *              B's image first (mxfp4_prepack_b_size rounded up to 1 KB), then mxfp4_gemm's
 *              workspace. Calls sharing a workspace must be ordered, as for mxfp4_gemm (a call's
 *              prepack waits for the work before it on `stream`).
 * Errors: those of mxfp4_gemm and mxfp4_prepack_b, checked before anything is enqueued.
 * mxfp4_gemm_unpacked_workspace_size returns 0 for invalid sizes.
 */
size_t mxfp4_gemm_unpacked_workspace_size(int64_t M, int64_t N, int64_t K);
int mxfp4_gemm_unpacked(const void *a, int64_t M, int64_t K, int64_t lda, const void *bq, const void *bs,
                        int64_t N, void *c, int64_t ldc, void *workspace, size_t ws_bytes, void *stream);

/*
 * mxfp4_gemm_host -- mxfp4_gemm for A and C in host memory: on `stream`, move A (rows of K
 * elements, row stride lda) into the caller's device buffer a_dev, run mxfp4_gemm, and deliver C
 * into c_host (row stride ldc): page-locked host memory mapped into the device's address space
 * (cudaHostAlloc / cudaHostRegister), 2-byte aligned, receives C straight from the GEMM's stores;
 * any other host memory receives it by a copy from the caller's device buffer c_dev. Likewise A: from mapped
 * page-locked memory with 16-byte aligned rows (lda % 8 == 0) a small kernel reads it in place
 * and writes a_dev (it chains with the GEMMs by programmatic dependent launch, so back-to-back
 * calls overlap; it still reads A only after the work before it on `stream` has finished, so A
 * may be the C of a previous call); from any other host memory it is copied. The call is
 * asynchronous like mxfp4_gemm: c_host is valid once `stream` has completed, and a_host /
 * c_host must stay valid until then (page-locked host memory lets the copies overlap other
 * work; pageable memory works but the copies then block the host).
 *   a_host : bf16 [M, K], row stride lda (lda >= K); a_dev: device bf16 [M, K] packed
 *            (row stride K), 16-byte aligned; c_dev: device bf16 [M, N] packed (row stride N),
 *            2-byte aligned, required (and checked) even where C goes straight to c_host;
 *   packed_b, workspace: as for mxfp4_gemm.
 * Errors: as mxfp4_gemm, checked before any copy; MXFP4_ERR_CUDA if a copy fails to enqueue.
 */
int mxfp4_gemm_host(const void *a_host, int64_t M, int64_t K, int64_t lda, const void *packed_b, int64_t N,
                    void *c_host, int64_t ldc, void *a_dev, void *c_dev, void *workspace, size_t ws_bytes,
                    void *stream);

/*
 * Prepared calls -- for a serving loop whose buffers stay the same from one call to the next.
 * mxfp4_call_create (the arguments of mxfp4_gemm_ex) and mxfp4_call_create_host (those of
 * mxfp4_gemm_host) do all of that call's checks, its planning and, for host buffers, the queries
 * of where A comes from and where C goes, once, on the current device; each mxfp4_call_run then
 * only enqueues the call's kernels and copies on `stream`: exactly what the unprepared call would
 * enqueue with the same arguments (same results, bit for bit).
 *   out    : receives a handle owned by the caller, released with mxfp4_call_destroy (NULL is a
 *            no-op there); a run keeps nothing of it, so it may be destroyed as soon as its last
 *            run has been enqueued. On an error *out is NULL and nothing is allocated.
 *   Buffers: every pointer given at creation must stay valid, with the same size and (for host
 *            memory) the same page-locked / mapped state, until the last run has completed on
 *            its stream; their contents may change freely between runs.
 * Runs of one call share its workspace (and a_dev / c_dev): order them (one stream, or events),
 * as for repeated unprepared calls. mxfp4_call_run must be made on the device the call was
 * created on (MXFP4_ERR_ARG otherwise) and returns MXFP4_OK or MXFP4_ERR_CUDA if a launch or copy
 * fails to enqueue.
 * Errors at creation: those of mxfp4_gemm_ex / mxfp4_gemm_host; MXFP4_ERR_ARG also if `out` is
 * NULL or the handle cannot be allocated.
 */
typedef struct mxfp4_call mxfp4_call;
int mxfp4_call_create(const void *a, int64_t M, int64_t K, int64_t lda, const void *packed_b, int64_t N,
                      void *c, int64_t ldc, void *workspace, size_t ws_bytes, const mxfp4_gemm_options *opts,
                      mxfp4_call **out);
/* flags: 0, or MXFP4_CALL_A_HOST_WRITTEN -- the caller guarantees that a_host is written by the
 * host only, never by device work (in particular it is not the C of an earlier call, and no
 * device-to-host copy into it is pending). A staged from mapped page-locked a_host is then read
 * over the link as soon as the call's first kernel starts, while the work before it on the
 * stream still runs, instead of after that work; as always, the host must have written A
 * before the run is enqueued. Without the flag (and in mxfp4_gemm_host) A is read only once
 * the work before it has completed. Other bits: MXFP4_ERR_ARG. */
#define MXFP4_CALL_A_HOST_WRITTEN 1u
int mxfp4_call_create_host(const void *a_host, int64_t M, int64_t K, int64_t lda, const void *packed_b,
                           int64_t N, void *c_host, int64_t ldc, void *a_dev, void *c_dev, void *workspace,
                           size_t ws_bytes, unsigned flags, mxfp4_call **out);
int mxfp4_call_run(const mxfp4_call *call, void *stream);
void mxfp4_call_destroy(mxfp4_call *call);

/*
 * Token blocks: A quantized once into the layout the GEMM's tensor cores read, for callers that
 * feed the same activation to several GEMMs or keep it between calls. The pages do this for their
 * large-M path (submission 711914, `_run_aiter_large_m_gemm`: `_fast_mxfp4_quant` writes the e2m1
 * codes and a pre-shuffled scale buffer once, and the GEMM takes them as they are); the GEMM's
 * two-kernel plan uses the same layout in its workspace.
 *
 * Layout: the M tokens in tiles of m_tile rows, K in steps of 256; tile t, step j is one block of
 * m_tile*128 + ceil(m_tile/128)*1024 bytes at offset (t*ceil(K/256) + j) * that size. In a block,
 * row r's 128 code bytes (the step's 256 e2m1 values, even element in the low nibble) start at
 * r*128, its eight 16-byte chunks stored at chunk (c ^ r%8) (the 128-byte swizzle of the MMA's
 * shared-memory operand); then per 128 rows two 512-byte scale chunks, the scale of 1x32 block b
 * (0..7) of row r at m_tile*128 + (r/128*2 + b/4)*512 + (r%32)*16 + (r/32%4)*4 + b%4 (in a tile
 * of under 128 rows the scale slots of the rows it lacks are not part of the layout: never
 * written, never read). Rows past M and K past the end hold zero codes and zero scale bytes.
 * Codes and scales are bit-identical to mxfp4_quantize's.
 *
 * m_tile arguments: 0 = a default from M and K alone (M rounded up to 16 up to 128 tokens, 128 up
 * to 512, 256 beyond; 16 for 17..32 tokens of at most two 256-K steps), else a multiple of 16 in
 * [16, 256]; either way cut to M rounded up to 16 (mxfp4_token_tile returns the result). The
 * GEMM's own two-kernel plan may pick another tile (it also weighs N and the SM count: see
 * mxfp4_gemm_plan_info).
 * Blocks written with one (M, K, m_tile) must be read with the same.
 */

/* The token tile of the layout for (M, K, m_tile); 0 for invalid arguments (M < 1, K not a
 * positive multiple of 8, m_tile not 0 or a multiple of 16 up to 256, or a size limit). */
int mxfp4_token_tile(int64_t M, int64_t K, int m_tile);

/* Bytes of the token blocks of M tokens of depth K; 0 for invalid arguments. */
size_t mxfp4_token_blocks_size(int64_t M, int64_t K, int m_tile);

/*
 * mxfp4_quantize_tokens -- quantize A into token blocks (the quantization of mxfp4_quantize).
 *   a      : bf16 [M, K], row stride lda (lda >= K, lda % 8 == 0), 16-byte aligned.
 *   blocks : out, blocks_bytes >= mxfp4_token_blocks_size(M, K, m_tile), 256-byte aligned. Every
 *            byte of the layout is written (padding included).
 * M == 0 is a no-op. Ordering as mxfp4_gemm: A is read, and the blocks written, only after the
 * work before it on `stream` has finished. MXFP4_ERR_WORKSPACE if blocks_bytes is too small.
 */
int mxfp4_quantize_tokens(const void *a, int64_t M, int64_t K, int64_t lda, int m_tile,
                          void *blocks, size_t blocks_bytes, void *stream);

/*
 * mxfp4_gemm_tokens -- C = A . MXFP4(B)^T for A already in token blocks: the GEMM of the
 * two-kernel plan alone (mxfp4_gemm with the option path = 2 runs mxfp4_quantize_tokens and then
 * this; the results are bit-identical).
 *   blocks   : written by mxfp4_quantize_tokens for the same M, K and m_tile; blocks_bytes its
 *              size (checked against mxfp4_token_blocks_size); 256-byte aligned.
 *   packed_b, N, c, ldc: as for mxfp4_gemm.
 *   splits   : 0 = automatic, else the number of K slices per output tile (as in
 *              mxfp4_gemm_options).
 * No workspace is needed. Ordering as mxfp4_gemm (the blocks are read after the work before it on
 * `stream` has finished). Errors: as mxfp4_gemm; MXFP4_ERR_WORKSPACE if blocks_bytes is too small.
 */
int mxfp4_gemm_tokens(const void *blocks, size_t blocks_bytes, int64_t M, int64_t K, int m_tile,
                      const void *packed_b, int64_t N, void *c, int64_t ldc, int splits, void *stream);

/* Everything the planner decided for one call. */
typedef struct mxfp4_plan_info {
    int path;            /* 1: A quantized inside the GEMM; 2: standalone quantize, then the GEMM */
    int splits;          /* K slices per output tile (= thread-block cluster size) */
    int m_tile;          /* tokens per tile (the MMA's N) */
    int ctas;            /* CTAs of the GEMM launch */
    int stages;          /* weight pipeline stages per CTA */
    int issuers;         /* MMA-issuing threads per CTA, one tensor-memory accumulator each */
    int reduction;       /* split-K form: 0 none (one slice); 1 posted 4-byte rows + cluster
                            barrier; 2 16-byte st.async posts counted on the owner's mbarrier;
                            3 one bulk shared-memory copy per owner */
    int recv_dedicated;  /* 1: the receive buffer has shared memory of its own; 0: it lies over
                            the pipeline buffers (one more cluster barrier before the posts) */
    int smem_bytes;      /* dynamic shared memory per CTA */
    int tmem_cols;       /* tensor-memory columns allocated per CTA */
    int scale_stores;    /* 1: epilogue warps write each stage's scale factors into tensor memory
                            (the tensor pipe then runs MMAs only); 0: the MMA threads copy them */
    int a_early;         /* 1: the weight-resident kernel loads and quantizes A before waiting for
                            the work ahead of it (only with MXFP4_GEMM_A_READY, on plans whose
                            shared memory leaves the SM room for it) */
    int reserved[4];
} mxfp4_plan_info;

/* The full plan mxfp4_gemm_ex would run on the current device (superset of mxfp4_gemm_plan).
 * `info` must not be NULL. Returns MXFP4_OK, an argument / shape error, or MXFP4_ERR_ARCH /
 * MXFP4_ERR_CUDA from the device query. */
int mxfp4_gemm_plan_info(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options *opts, mxfp4_plan_info *info);

/*
 * mxfp4_gemm_plan_model -- the planner alone, for a device described by its SM count and, for
 * every cluster size s = 1..16, how many clusters of s CTAs can be resident at once
 * (cluster_caps[s]; cluster_caps[0] is ignored; NULL means no limit). Makes no CUDA call, so it
 * works without a GPU. On a device with those properties the plan equals mxfp4_gemm_plan_info's
 * (the device query there also accounts for each plan's shared memory; on sm_103a the count did
 * not depend on it). Returns MXFP4_OK or an argument / shape error.
 */
int mxfp4_gemm_plan_model(int64_t M, int64_t N, int64_t K, const mxfp4_gemm_options *opts, int sm_count,
                          const int *cluster_caps, mxfp4_plan_info *info);

/*
 * mxfp4_device_status -- synchronize `stream`, then read and clear the library's device
 * error word for the current device: MXFP4_OK, or MXFP4_ERR_TIMEOUT if a kernel gave up a
 * bounded wait (the kernel then skipped its remaining work and released its resources;
 * its outputs are undefined). Returns MXFP4_ERR_CUDA if the synchronization or the read
 * failed, MXFP4_ERR_ARCH on a device other than compute capability 10.3.
 * There is one error word per device, shared by every stream. Only `stream` is synchronized:
 * a kernel still running on another stream may set the word after it is read, and a timeout
 * it set before is reported (and cleared) here. To attribute a timeout to one stream's work,
 * synchronize the device (or every stream using the library) first, or pass NULL with the
 * legacy default stream ordering every other blocking stream.
 */
int mxfp4_device_status(void *stream);

/*
 * mxfp4_selftest_timeout -- launch one CTA that waits on a barrier nothing ever signals,
 * with a wait limit of `limit_us` microseconds (1..1000000). The kernel gives up, records
 * MXFP4_ERR_TIMEOUT in the device error word and exits normally, so a following
 * mxfp4_device_status returns MXFP4_ERR_TIMEOUT. Exercises the failure path without a fault.
 */
int mxfp4_selftest_timeout(int limit_us, void *stream);

/*
 * mxfp4_gemm_noalloc -- mxfp4_gemm for callers that cannot allocate device memory.
 * (No counterpart in the pages: it exists for callers, not for the method.)
 *
 * Some callers have no way to hand the library a workspace: a plugin running inside an
 * inference engine whose host owns the whole device-memory plan and forbids allocation once
 * it runs, or a latency-critical serving loop that must never call cudaMalloc/cudaFree
 * because those can synchronize the whole device. This entry point needs no workspace
 * argument: its scratch (the quantized A that the two-kernel path -- M > 32, or a small M
 * that the planner does not fuse -- hands from its quantize kernel to the GEMM kernel) lives
 * in one statically sized array inside the library, which every GPU that loads the library
 * keeps for the life of the process.
 *
 *   Arguments and results are those of mxfp4_gemm without `workspace` / `ws_bytes`; it runs
 *   the same plan, so the output is the same.
 *   Scratch limit: MXFP4_NOALLOC_SCRATCH_BYTES. A shape whose scratch does not fit (about
 *   M*K/2 bytes plus M*K/32 of scales, rounded up to whole tiles) returns
 *   MXFP4_ERR_WORKSPACE before anything is enqueued.
 *   No allocation: the call never calls cudaMalloc, cudaFree or any allocating routine.
 *   First call per device: it looks up the array's device address (cudaGetSymbolAddress)
 *   with that device current; make that first call before any stream capture. The address
 *   is kept for the life of the process: after cudaDeviceReset on a device the library must
 *   not be called on that device again in the same process (the same holds for every entry
 *   point, which keep the device's error-word address the same way).
 *   Sharing: all calls on a device share the one array and it keeps the previous call's
 *   contents; nothing in it has to start at zero (each call rewrites every byte it reads).
 *   Calls that can overlap on the GPU (different streams without ordering, or several host
 *   threads) race on the array and give wrong results: order them.
 */
#define MXFP4_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int mxfp4_gemm_noalloc(const void *a, int64_t M, int64_t K, int64_t lda,
                       const void *packed_b, int64_t N,
                       void *c, int64_t ldc, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GB300_H */
