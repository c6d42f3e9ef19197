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
 *   - element encode: what submission 711914's `_mxfp4_quant_tile` computes for each
 *     scaled element, written from the e2m1 definition: the nearest grid value, ties to
 *     even, saturating at 6, sign in bit 3.
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
 * Element encode: round an already-scaled fp32 value onto the e2m1 grid
 * ------------------------------------------------------------------------------------- */

/* e2m1 decode from the bit fields of the format: exponent bias 1, one mantissa bit,
 * exponent 0 is the subnormal binade with step 0.5. */
double oracle_e2m1_decode(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * (double)(1 << (e - 1));
    return s ? -v : v;
}

/* The e2m1 code of qx, from the definition of the element step in submission 711914's
 * `_mxfp4_quant_tile` (its saturate / sub-one / normal branches): the grid magnitude
 * nearest to |qx|, a tie going to the code whose mantissa bit is 0 (round to nearest even),
 * finite magnitudes past 6 saturating to 6 (6 is the nearest grid value to them), and the
 * sign of qx in bit 3 even when the magnitude rounds to 0 (reading Q6).
 * The eight codes are scanned keeping the nearest so far. Distances are compared through
 * midpoints, which is exact: two grid values are short dyadic fractions, so their midpoint
 * is exact in double, and a float converts to double exactly. */
uint8_t oracle_e2m1_encode(float qx)
{
    double a = fabs((double)qx);
    int best = 0, c;
    for (c = 1; c < 8; ++c) {
        double g_best = oracle_e2m1_decode((uint8_t)best), g_c = oracle_e2m1_decode((uint8_t)c);
        double mid = 0.5 * (g_best + g_c);
        int c_nearer = (g_c > g_best) ? (a > mid) : (a < mid);
        int tie_to_even = (a == mid) && (c & 1) == 0 && (best & 1) == 1;
        if (c_nearer || tie_to_even) best = c;
    }
    return (uint8_t)(best | (signbit(qx) ? 8 : 0));
}

/* A second, independently built encoder for the exhaustive self-check below: the grid
 * ascends with the code, so the code of |v| is the number of the seven midpoints between
 * neighbouring grid values that |v| lies above, plus one when |v| sits exactly on a
 * midpoint whose upper neighbour has the even code. Sign from v's sign bit. */
uint8_t oracle_e2m1_encode_count(float v)
{
    double a = fabs((double)v);
    int code = 0, c;
    for (c = 0; c < 7; ++c) {
        double mid = 0.5 * (oracle_e2m1_decode((uint8_t)c) + oracle_e2m1_decode((uint8_t)(c + 1)));
        if (a > mid) code += 1;
        else if (a == mid && ((c + 1) & 1) == 0) code += 1;
    }
    return (uint8_t)(code | (signbit(v) ? 8 : 0));
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
 * Exhaustive self-check: compare oracle_e2m1_encode with oracle_e2m1_encode_count over
 * every step-th fp32 bit pattern in [lo, hi) (both signs). Returns the mismatch count and the
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
            if (oracle_e2m1_encode(v) != oracle_e2m1_encode_count(v)) {
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
