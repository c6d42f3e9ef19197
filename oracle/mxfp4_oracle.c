/*
 * MXFP4 oracle: a plain, slow, CPU-only restatement of what the MXFP4 GEMM computes.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or calls this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * What it follows (the pages are three diffs of the "amd-mxfp4-mm" leaderboard
 * submissions 608632, 610679 and 711914):
 *   - block scale: submission 711914, `_mxfp4_quant_tile` (amax over a 1x32 block, the
 *     +0x200000 / &0xFF800000 rounding, floor(log2)-2 clamped to [-127,127], +127 bias);
 *     cross-checked against submission 608632, `_hw_mxfp4_quant_op` step 1 (direct
 *     exponent form).
 *   - element encode: submission 711914, `_mxfp4_quant_tile` (three-way saturate /
 *     sub-one / normal branch, round to nearest even, sign in bit 3).
 *   - packing: even element in the low nibble, odd element in the high nibble
 *     (submission 608632, `_hw_mxfp4_quant_op` step 3).
 *   - GEMM: C = dequant(A) . dequant(B)^T accumulated in fp64, rounded once to bf16.
 *
 * Readings taken where the pages are silent or inconsistent are listed in the design
 * notes; the two that change bytes are: an amax that rounds to +inf gives scale byte 254
 * (log2 form), and a negative value that rounds to zero keeps its sign (code 0x8).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -fopenmp (no -ffast-math: fp32 products must be
 * IEEE round-to-nearest with subnormals honoured).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float f32_of(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* bf16 -> fp32 is exact: a bf16 is the top half of an fp32. */
float oracle_bf16_to_f32(uint16_t h) { return f32_of((uint32_t)h << 16); }

/* ---------------------------------------------------------------------------------------
 * Block scale (submission 711914, `_mxfp4_quant_tile`, the amax / scale_ub lines)
 * ------------------------------------------------------------------------------------- */

/* Round the block amax to a power of two: add 2^21 to the fp32 bit pattern (a quarter of
 * the 23-bit mantissa range) and clear the mantissa. Mantissas >= 0.75 carry into the
 * exponent. Result bits are 0, a power of two, or +inf (0x7F800000). */
uint32_t oracle_round_amax_bits(float amax)
{
    uint32_t u = bits_of(amax) + 0x200000u;
    return u & 0xFF800000u;
}

/* Unbiased scale exponent s = clamp(floor(log2(amax_r)) - 2, -127, 127).
 * amax_r is 0, an exact power of two or +inf, so floor(log2) is taken exactly from the
 * exponent field: log2(0) = -inf and log2(+inf) = +inf both land on the clamp. The "-2"
 * maps the largest e2m1 magnitude 6 = 1.5 * 2^2 onto the top binade. */
int oracle_scale_exponent(uint32_t amax_r_bits)
{
    long e;
    if (amax_r_bits == 0u) return -127;            /* floor(log2(0)) = -inf */
    if (amax_r_bits >= 0x7F800000u) return 127;    /* floor(log2(+inf)) = +inf */
    e = (long)(amax_r_bits >> 23) - 127;           /* exact for a power of two */
    e -= 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (int)e;
}

/* e8m0 byte: biased by 127, so the byte is in [0, 254] and 255 (NaN) never occurs. */
uint8_t oracle_scale_byte(int s) { return (uint8_t)(s + 127); }

/* ---------------------------------------------------------------------------------------
 * Element encode (submission 711914, `_mxfp4_quant_tile`, the sat / den / nor branch)
 * ------------------------------------------------------------------------------------- */

/* Encode one already-scaled fp32 value qx as an e2m1 code (bit 3 sign, bits 2..1
 * exponent with bias 1, bit 0 mantissa), round to nearest even, saturating at 6. */
uint8_t oracle_e2m1_encode(float qx)
{
    uint32_t u = bits_of(qx);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u ^ sign;             /* |qx| as bits */
    float a = f32_of(mag);
    uint8_t code;

    if (a >= 6.0f) {
        code = 7;                        /* saturate to 6.0 */
    } else if (a < 1.0f) {
        /* Sub-one range: the e2m1 grid is 0, 0.5 (and 1.0 by rounding up). Adding 2^22
         * puts the fp32 ulp at 0.5, so the fp32 add itself rounds a to the nearest
         * multiple of 0.5 with ties to even; the mantissa field then holds 2*round(a). */
        float t = a + 4194304.0f;
        code = (uint8_t)(bits_of(t) - (149u << 23));
    } else {
        /* [1, 6): move the exponent bias from 127 to 1 (subtract 126 from the exponent
         * field), then round the 23-bit mantissa to its top bit, ties to even; a carry
         * out of the mantissa bumps the exponent, which is the correct next code. */
        uint32_t rebased = mag - (126u << 23);
        uint32_t keep = (rebased >> 22) & 1u;      /* lsb that survives */
        uint32_t rounded = rebased + 0x1FFFFFu + keep;
        code = (uint8_t)(rounded >> 22);
    }
    return (uint8_t)(code | (sign >> 28));   /* sign into bit 3, also for values that round to 0 */
}

/* e2m1 decode from the bit fields of the format: exponent bias 1, one mantissa bit,
 * exponent 0 is the subnormal binade with step 0.5. */
double oracle_e2m1_decode(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Independent encoder for cross-checking oracle_e2m1_encode: search the eight decoded
 * magnitudes for the nearest one, ties to the even code; finite values past 6 saturate by
 * being nearest to 6. Sign copied from the input's sign bit. Distances are compared
 * exactly: a is nearer to g2 than to g1 < g2 iff a is above their midpoint, and the
 * midpoint of two grid values is exact in double. */
uint8_t oracle_e2m1_encode_nearest(float v)
{
    double grid[8];
    double a = fabs((double)v);
    int best = 0, c;
    for (c = 0; c < 8; ++c) grid[c] = oracle_e2m1_decode((uint8_t)c);
    for (c = 1; c < 8; ++c) {
        double lo = grid[best] < grid[c] ? grid[best] : grid[c];
        double hi = grid[best] < grid[c] ? grid[c] : grid[best];
        double mid = 0.5 * (lo + hi);
        int c_nearer = (grid[c] == hi) ? (a > mid) : (a < mid);
        int tie = (a == mid);
        if (c_nearer || (tie && (c & 1) == 0 && (best & 1) == 1)) best = c;
    }
    return (uint8_t)(best | (signbit(v) ? 8 : 0));
}

/* ---------------------------------------------------------------------------------------
 * Quantizer: bf16 rows -> packed e2m1 [rows, K/2] + e8m0 [rows, K/32]
 * ------------------------------------------------------------------------------------- */
void oracle_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                     uint8_t *q, uint8_t *scales)
{
    int64_t nb = K / 32;
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t j;
        for (j = 0; j < nb; ++j) {
            float xs[32];
            float amax = 0.0f;
            uint8_t codes[32];
            int i, s;
            float mul;
            for (i = 0; i < 32; ++i) {
                xs[i] = oracle_bf16_to_f32(x[r * ld + j * 32 + i]);
                amax = fmaxf(amax, fabsf(xs[i]));
            }
            s = oracle_scale_exponent(oracle_round_amax_bits(amax));
            scales[r * nb + j] = oracle_scale_byte(s);
            mul = ldexpf(1.0f, -s);                    /* 2^-s exactly, subnormal when s = 127 */
            for (i = 0; i < 32; ++i)
                codes[i] = oracle_e2m1_encode(xs[i] * mul);   /* one fp32 multiply, RNE */
            for (i = 0; i < 16; ++i)
                q[r * (K / 2) + j * 16 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
        }
    }
}

/* ---------------------------------------------------------------------------------------
 * Dequantize and the fp64 GEMM
 * ------------------------------------------------------------------------------------- */

/* value of element k of a packed row: low nibble for even k, high nibble for odd k */
static double elem(const uint8_t *qrow, const uint8_t *srow, int64_t k)
{
    uint8_t byte = qrow[k / 2];
    uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
    return oracle_e2m1_decode(code) * ldexp(1.0, (int)srow[k / 32] - 127);
}

void oracle_dequantize(const uint8_t *q, const uint8_t *scales, int64_t rows, int64_t K,
                       double *out)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t k;
        for (k = 0; k < K; ++k)
            out[r * K + k] = elem(q + r * (K / 2), scales + r * (K / 32), k);
    }
}

/* C[m,n] = sum_k A[m,k] * B[n,k] over dequantized fp64 operands (A [M,K], B [N,K] row-major).
 * Every product of two MXFP4 values is exact in fp64; only the running sum rounds. */
void oracle_gemm_f64(const double *a, const double *b, int64_t M, int64_t N, int64_t K, double *c)
{
    int64_t mn;
#pragma omp parallel for schedule(static)
    for (mn = 0; mn < M * N; ++mn) {
        int64_t m = mn / N, n = mn % N, k;
        double acc = 0.0;
        for (k = 0; k < K; ++k) acc += a[m * K + k] * b[n * K + k];
        c[mn] = acc;
    }
}

/* Selected entries C[idx_m[i], idx_n[i]] straight from the packed operands, for checking
 * sampled outputs of problems too large for the full fp64 GEMM. */
void oracle_gemm_entries(const uint8_t *aq, const uint8_t *as, const uint8_t *bq, const uint8_t *bs,
                         int64_t K, const int64_t *idx_m, const int64_t *idx_n, int64_t count,
                         double *out)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < count; ++i) {
        const uint8_t *qa = aq + idx_m[i] * (K / 2), *sa = as + idx_m[i] * (K / 32);
        const uint8_t *qb = bq + idx_n[i] * (K / 2), *sb = bs + idx_n[i] * (K / 32);
        double acc = 0.0;
        int64_t k;
        for (k = 0; k < K; ++k) acc += elem(qa, sa, k) * elem(qb, sb, k);
        out[i] = acc;
    }
}

/* fp64 -> bf16, round to nearest even, in one rounding: first round to fp32 with
 * round-to-odd (truncate, then force the last bit to 1 if anything was lost), which keeps
 * 16 more bits than bf16 so the second, nearest-even rounding cannot double-round. */
uint16_t oracle_f64_to_bf16(double d)
{
    float f = (float)d;
    uint32_t u;
    if (isnan(d)) return 0x7FC0;
    if ((double)f != d && !isinf(f)) {
        if (fabs((double)f) > fabs(d)) f = nextafterf(f, 0.0f);   /* truncate toward zero */
        u = bits_of(f) | 1u;                                       /* sticky: inexact */
    } else {
        u = bits_of(f);
    }
    if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16);  /* inf */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void oracle_f64_to_bf16_array(const double *in, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(in[i]);
}

/* ---------------------------------------------------------------------------------------
 * Exhaustive self-check: compare oracle_e2m1_encode with oracle_e2m1_encode_nearest over
 * every fp32 bit pattern in [lo, hi) (both signs). Returns the mismatch count and the
 * first mismatching pattern through *first (0xFFFFFFFF if none).
 * ------------------------------------------------------------------------------------- */
int64_t oracle_encode_selfcheck(uint32_t lo, uint32_t hi, uint32_t step, uint32_t *first)
{
    int64_t bad = 0;
    uint32_t first_bad = 0xFFFFFFFFu;
    int64_t i, n = ((int64_t)hi - (int64_t)lo + step - 1) / step;
#pragma omp parallel for schedule(static) reduction(+ : bad)
    for (i = 0; i < n; ++i) {
        uint32_t u = lo + (uint32_t)i * step;
        int sgn;
        for (sgn = 0; sgn < 2; ++sgn) {
            float v = f32_of(u | (sgn ? 0x80000000u : 0u));
            if (oracle_e2m1_encode(v) != oracle_e2m1_encode_nearest(v)) {
                ++bad;
#pragma omp critical
                if (u < first_bad) first_bad = u;
            }
        }
    }
    if (first) *first = first_bad;
    return bad;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the parallel loops use from now on (n >= 1); for timing the oracle on one core. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
