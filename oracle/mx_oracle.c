/*
 * CPU oracle for the MXFP4 / NVFP4 block-scaled GEMM and its BF16 quantize
 * pre-pass.  TEST INFRASTRUCTURE ONLY: nothing on the product path may link,
 * load or call this file.  Only the test suite, the smoke check of the entry
 * module and the CPU-baseline leg of the benchmark use it.
 *
 * Plain, slow, obviously-correct C99 (+ optional OpenMP over independent
 * rows).  It shares no code, header, table or helper with the CUDA library.
 * Build with -ffp-contract=off: the NVFP4 quantizer is defined by a fixed
 * sequence of binary32 operations and must not be fused into FMAs.
 *
 * Where each definition comes from (pages cited by title and section):
 *  - "Integrate MXFP4 hipblaslt GEMM support" (ROCm/TransformerEngine #697),
 *    Description/Changes: the operand type is FP4 E2M1, the scales are UE8M0
 *    with one scale per 32 elements along K ("FP4xFP4 + UE8M0 block-32"), the
 *    GEMM is TN with BF16/FP32 output, K % 256 == 0, M and N % 32 == 0,
 *    beta == 0, no bias or GELU; the test checks the GEMM against a reference
 *    built by CPU-dequantizing the same operands (that is oracle_block_gemm).
 *  - "feat(ck-tile): aquant GEMM TE to dispatcher bridge" (ROCm/rocm-libraries
 *    #9980), pk_int4 fix: packed 4-bit storage holds two elements per byte.
 *  - NVIDIA/TransformerEngine #3809 (CuTeDSL NVFP4 quantize kernels), commit
 *    messages: NVFP4 = E2M1 codes with E4M3 scales per 16 elements and an
 *    FP32 per-tensor amax; round-to-nearest output is byte-identical across
 *    implementations.
 *  - The E2M1 value set, the UE8M0 decode 2^(e-127), the E4M3 grid and the
 *    shared-exponent rule floor(log2 amax) - emax(E2M1) are those of the OCP
 *    Microscaling (MX) v1.0 and OCP FP8 formats named by the pages' type
 *    names; the pages do not print them.  Readings where the pages are silent:
 *      * nibble order: element 2t in the low nibble, 2t+1 in the high nibble;
 *      * an all-zero MX block gets scale byte 0 (exponent clamped to -127);
 *      * a value that rounds to zero keeps its sign (code 0x8 for negative);
 *      * |y| above 6 saturates to 6;
 *      * NVFP4: s_t = amax_t / 2688 (2688 = 6 * 448), block scale
 *        sb = E4M3_RNE_satfinite(amax_b / (6 * s_t)), code =
 *        E2M1_RNE(x / (E4M3(sb) * s_t)), every step one binary32 RN op;
 *        when s_t == 0 or sb == 0 the codes of the block are 0x0;
 *      * NVFP4 stochastic rounding (the pages: one Philox4x32 draw per
 *        output block, keyed by block coordinates and direction, with a
 *        configurable round count): counter (block column j, row r,
 *        direction, 0), key (seed low, seed high), byte i of the draw for
 *        element i, round up iff u / 256 < p (oracle_e2m1_encode_sr); the
 *        scales stay round-to-nearest.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Element and scale codecs                                            */
/* ------------------------------------------------------------------ */

/* E2M1 magnitudes of codes 0..7 (1 sign bit, 2 exponent bits with bias 1,
 * 1 mantissa bit; code 1 is the subnormal 0.5).  Bit 3 is the sign. */
static const double k_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_decode(uint32_t code)
{
    double m = k_e2m1_mag[code & 7u];
    return (code & 8u) ? -m : m;
}

/* Round y to the nearest E2M1 value; a tie goes to the code whose mantissa
 * bit (bit 0) is 0; magnitudes beyond 6 saturate to 6; the sign of y is kept
 * even when the magnitude rounds to 0. */
uint32_t oracle_e2m1_encode(double y)
{
    uint32_t sign = signbit(y) ? 8u : 0u;
    double a = fabs(y);
    if (a >= 6.0)
        return 7u | sign;
    uint32_t best = 0;
    double best_d = a;
    for (uint32_t c = 1; c < 8; ++c) {
        double d = fabs(a - k_e2m1_mag[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best | sign;
}

/* BF16 is the upper half of a binary32. */
float oracle_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* floor(log2 |x|) of a non-zero finite BF16, from its bits, in integers:
 * normal numbers have it in the biased exponent field (bias 127); a
 * subnormal m * 2^-133 has it at the position of m's leading one. */
int oracle_bf16_floor_log2(uint16_t b)
{
    int e = (b >> 7) & 0xFF;
    int m = b & 0x7F;
    if (e != 0)
        return e - 127;
    int p = 6;
    while (p > 0 && !((m >> p) & 1))
        --p;
    return p - 133;
}

/* UE8M0 scale byte e -> 2^(e-127).  (0xFF is NaN in the format; the
 * quantizer never produces it.) */
double oracle_ue8m0_decode(uint32_t e)
{
    return ldexp(1.0, (int)(e & 0xFF) - 127);
}

/* E4M3 (OCP FP8 E4M3FN): 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, 0x7F/0xFF are NaN, largest finite 448. */
double oracle_e4m3_decode(uint32_t byte)
{
    uint32_t e = (byte >> 3) & 0xF, m = byte & 7u;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), (int)e - 10);
    return (byte & 0x80u) ? -v : v;
}

/* Round a non-negative value to the nearest finite E4M3 value, a tie going
 * to the even code, values beyond 448 saturating to 448 (satfinite). */
uint32_t oracle_e4m3_encode(double v)
{
    if (!(v > 0.0))
        return 0;
    if (v >= 448.0)
        return 0x7E;
    uint32_t best = 0;
    double best_d = v;
    for (uint32_t c = 1; c <= 0x7E; ++c) {
        double d = fabs(v - oracle_e4m3_decode(c));
        if (d < best_d || (d == best_d && (c & 1u) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* Round a double to the nearest BF16 (ties to even), directly (no detour
 * through binary32, which would round twice).  Returns the BF16 bits. */
uint16_t oracle_round_bf16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
    double q;
    int shift;
    if (ex - 1 >= -126) {
        shift = 8 - ex; /* 8 significant bits */
    } else {
        shift = 133; /* subnormal grid 2^-133 */
    }
    q = rint(ldexp(a, shift));
    double r = ldexp(q, -shift);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80u; /* overflow to infinity */
    float f = (float)r;    /* exact: r is a BF16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFFu);
}

/* oracle_round_bf16 over an array. */
void oracle_round_bf16_array(const double *x, int64_t n, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_round_bf16(x[i]);
}

/* ------------------------------------------------------------------ */
/* Quantizers                                                          */
/* ------------------------------------------------------------------ */

static void put_nibble(uint8_t *row_codes, int64_t col, uint32_t code)
{
    uint8_t *p = row_codes + col / 2;
    if (col % 2 == 0)
        *p = (uint8_t)((*p & 0xF0u) | (code & 0xFu));
    else
        *p = (uint8_t)((*p & 0x0Fu) | ((code & 0xFu) << 4));
}

/* BF16 [rows, cols] (row stride ld elements) -> MXFP4.
 * codes: [rows, cols/2] bytes; scales: [rows, cols/32] UE8M0 bytes (plain).
 * Per row and per block of 32 consecutive elements:
 *   amax = max |x|;  e = clamp(floor(log2 amax) - 2, -127, 127)
 *   (e = -127 when amax == 0);  scale byte = e + 127;
 *   code_i = E2M1_RNE_sat(x_i * 2^-e)  (exact scaling in binary64). */
void oracle_mx_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                        uint8_t *codes, uint8_t *scales)
{
    const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        uint8_t *row_codes = codes + r * (cols / 2);
        for (int64_t j = 0; j < nb; ++j) {
            const uint16_t *blk = x + r * ld + j * 32;
            double amax = 0.0;
            uint16_t amax_bits = 0;
            for (int i = 0; i < 32; ++i) {
                double v = fabs((double)oracle_bf16_to_float(blk[i]));
                if (v > amax) {
                    amax = v;
                    amax_bits = (uint16_t)(blk[i] & 0x7FFFu);
                }
            }
            int e = -127;
            if (amax > 0.0) {
                e = oracle_bf16_floor_log2(amax_bits) - 2;
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            scales[r * nb + j] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) {
                double y = ldexp((double)oracle_bf16_to_float(blk[i]), -e);
                put_nibble(row_codes, j * 32 + i, oracle_e2m1_encode(y));
            }
        }
    }
}

/* Per-tensor amax of a BF16 matrix (binary32, exact). */
float oracle_bf16_amax(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float v = fabsf(oracle_bf16_to_float(x[r * ld + c]));
            if (v > amax)
                amax = v;
        }
    return amax;
}

/* BF16 [rows, cols] -> NVFP4.
 * codes: [rows, cols/2]; scales: [rows, cols/16] E4M3 bytes (plain);
 * *tensor_scale = s_t.  Steps, each a binary32 round-to-nearest operation:
 *   s_t   = amax_t / 2688
 *   t     = 6 * s_t
 *   sb    = E4M3_RNE_satfinite(amax_b / t)
 *   den   = E4M3(sb) * s_t
 *   code  = E2M1_RNE_sat(x / den)
 * with codes 0x0 for a block whose sb is 0 or when s_t is 0. */
void oracle_nvfp4_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                           uint8_t *codes, uint8_t *scales, float *tensor_scale)
{
    const int64_t nb = cols / 16;
    volatile float amax_t = oracle_bf16_amax(x, rows, cols, ld);
    volatile float s_t = amax_t / 2688.0f;
    *tensor_scale = s_t;
    const float s_t_v = s_t;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        uint8_t *row_codes = codes + r * (cols / 2);
        for (int64_t j = 0; j < nb; ++j) {
            const uint16_t *blk = x + r * ld + j * 16;
            float amax_b = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float v = fabsf(oracle_bf16_to_float(blk[i]));
                if (v > amax_b)
                    amax_b = v;
            }
            uint32_t sb = 0;
            if (s_t_v > 0.0f) {
                volatile float t = 6.0f * s_t_v;
                volatile float ratio = amax_b / t;
                sb = oracle_e4m3_encode((double)ratio);
            }
            scales[r * nb + j] = (uint8_t)sb;
            if (sb == 0) {
                for (int i = 0; i < 16; ++i)
                    put_nibble(row_codes, j * 16 + i, 0u);
                continue;
            }
            volatile float den = (float)oracle_e4m3_decode(sb) * s_t_v;
            for (int i = 0; i < 16; ++i) {
                volatile float y = oracle_bf16_to_float(blk[i]) / den;
                put_nibble(row_codes, j * 16 + i, oracle_e2m1_encode((double)y));
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Stochastic rounding (NVFP4)                                         */
/* ------------------------------------------------------------------ */

/* Philox4x32-R, the counter-based generator of Salmon, Moraes, Dror and
 * Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011), Philox
 * section: a 128-bit counter c0..c3 and a 64-bit key k0, k1.  One round
 * multiplies c0 and c2 by the constants 0xD2511F53 and 0xCD9E8D57 (full
 * 64-bit products), then forms
 *   (hi(c2 * M1) ^ c1 ^ k0,  lo(c2 * M1),  hi(c0 * M0) ^ c3 ^ k1,  lo(c0 * M0));
 * between rounds the key is bumped by the Weyl constants 0x9E3779B9 and
 * 0xBB67AE85 (the first round uses the key as given).  The output is the
 * counter after `rounds` rounds (10 is the published default).
 * NVIDIA/TransformerEngine #3809 (CuTeDSL NVFP4 kernels): each stochastic
 * rounding draw is plain Philox4x32 of a known counter, with a configurable
 * round count. */
void oracle_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds, uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int i = 0; i < rounds; ++i) {
        if (i > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Stochastic rounding of y to E2M1 with the uniform byte u (0..255): with
 * lo <= |y| < hi the two neighbouring E2M1 magnitudes and
 * p = (|y| - lo) / (hi - lo), the magnitude becomes hi when u / 256 < p, else
 * lo (so it is hi with probability ceil(256 p) / 256, and a value on the grid
 * never moves).  |y| >= 6 saturates to 6 and the sign of y is kept, as in
 * oracle_e2m1_encode.  Reading: the pages name stochastic rounding but not
 * its arithmetic; this is the textbook rule with 8 random bits per element,
 * the 128 bits of one Philox draw spread over a 16-element block. */
uint32_t oracle_e2m1_encode_sr(double y, uint32_t u)
{
    const uint32_t sign = signbit(y) ? 8u : 0u;
    const double a = fabs(y);
    if (a >= 6.0)
        return 7u | sign;
    uint32_t c = 0;
    while (c < 6 && k_e2m1_mag[c + 1] <= a)
        ++c;
    const double p = (a - k_e2m1_mag[c]) / (k_e2m1_mag[c + 1] - k_e2m1_mag[c]);
    return ((double)(u & 0xFFu) / 256.0 < p ? c + 1 : c) | sign;
}

/* As oracle_nvfp4_quantize (same s_t, same block scales, same quotient
 * x / den), with the quotient rounded stochastically instead of to nearest.
 * NVIDIA/TransformerEngine #3809 (CuTeDSL NVFP4 kernels): one Philox draw
 * per output block, keyed by the block's coordinates and direction.
 * Reading: block (r, j) (row r of the output, j-th 16-element block along
 * it) draws Philox4x32-`rounds` of counter (j, r, direction, 0) under the key
 * (low, high 32 bits of seed); element i of the block (0..15) takes byte
 * i % 4 (least significant first) of word i / 4 of the draw.  direction is
 * 0 for the rowwise output and 1 for the columnwise one (the quantize of
 * x^T, whose rows are the columns of x). */
void oracle_nvfp4_quantize_sr(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                              uint64_t seed, int rounds, uint32_t direction,
                              uint8_t *codes, uint8_t *scales, float *tensor_scale)
{
    const int64_t nb = cols / 16;
    volatile float amax_t = oracle_bf16_amax(x, rows, cols, ld);
    volatile float s_t = amax_t / 2688.0f;
    *tensor_scale = s_t;
    const float s_t_v = s_t;
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        uint8_t *row_codes = codes + r * (cols / 2);
        for (int64_t j = 0; j < nb; ++j) {
            const uint16_t *blk = x + r * ld + j * 16;
            float amax_b = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float v = fabsf(oracle_bf16_to_float(blk[i]));
                if (v > amax_b)
                    amax_b = v;
            }
            uint32_t sb = 0;
            if (s_t_v > 0.0f) {
                volatile float t = 6.0f * s_t_v;
                volatile float ratio = amax_b / t;
                sb = oracle_e4m3_encode((double)ratio);
            }
            scales[r * nb + j] = (uint8_t)sb;
            if (sb == 0) {
                for (int i = 0; i < 16; ++i)
                    put_nibble(row_codes, j * 16 + i, 0u);
                continue;
            }
            const uint32_t ctr[4] = {(uint32_t)j, (uint32_t)r, direction, 0u};
            uint32_t draw[4];
            oracle_philox4x32(ctr, key, rounds, draw);
            volatile float den = (float)oracle_e4m3_decode(sb) * s_t_v;
            for (int i = 0; i < 16; ++i) {
                volatile float y = oracle_bf16_to_float(blk[i]) / den;
                const uint32_t u = (draw[i / 4] >> (8 * (i % 4))) & 0xFFu;
                put_nibble(row_codes, j * 16 + i, oracle_e2m1_encode_sr((double)y, u));
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* GEMM epilogue: bias, GELU, beta                                      */
/* ------------------------------------------------------------------ */

/* GELU(y) = y * Phi(y), the Gaussian error linear unit in its defining form
 * (Phi the standard normal CDF), evaluated as Phi(y) = erfc(-y / sqrt(2)) / 2,
 * which equals (1 + erf(y / sqrt(2))) / 2 without its cancellation for
 * negative y. */
double oracle_gelu(double y)
{
    return 0.5 * y * erfc(-y / sqrt(2.0));
}

/* out[i, j] = act(d[i, j] + beta * c[i, j] + bias[j]) in binary64, where
 * act is GELU when gelu != 0 and the identity otherwise; bias (length n)
 * and c ([m, n]) may be NULL (no term).  "Integrate MXFP4 hipblaslt GEMM
 * support" (ROCm/TransformerEngine #697) names bias, GELU and beta != 0 as
 * what the block-scaled GEMM leaves out, and the AITER a4w4 bias as FP32;
 * the order (scale, then the C and bias terms, then the activation) is the
 * usual GEMM epilogue D = act(alpha A B^T + beta C + bias). */
void oracle_gemm_epilogue(const double *d, int64_t m, int64_t n, const float *bias, int gelu,
                          double beta, const double *c, double *out)
{
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double y = d[i * n + j];
            if (c)
                y += beta * c[i * n + j];
            if (bias)
                y += (double)bias[j];
            out[i * n + j] = gelu ? oracle_gelu(y) : y;
        }
    }
}

/* ------------------------------------------------------------------ */
/* GEMM                                                                */
/* ------------------------------------------------------------------ */

/* D[i, j] = sum_k a(row_i, k) * b(col_j, k) for the TN product of two
 * block-scaled FP4 matrices, in binary64:
 *   A codes [m, k/2], A scales [m, k/blk] (plain), likewise B [n, ...];
 *   block size blk = 32 with UE8M0 scales (format 0, MXFP4) or
 *   blk = 16 with E4M3 scales (format 1, NVFP4, then times s_tA * s_tB).
 * Per block: P = sum (2 a_code)(2 b_code) is an exact integer, and
 * P * sa * sb / 4 is exact in binary64; the blocks are summed in K order.
 * s_abs receives the same sum taken over |a||b|.
 * rows / cols select which outputs to compute (NULL = all, in order); the
 * outputs are [n_rows, n_cols] row-major. */
void oracle_block_gemm(int format, const uint8_t *a_codes, const uint8_t *a_scales,
                       const uint8_t *b_codes, const uint8_t *b_scales, int64_t m, int64_t n,
                       int64_t k, float a_tensor_scale, float b_tensor_scale,
                       const int64_t *rows, int64_t n_rows, const int64_t *cols,
                       int64_t n_cols, double *d, double *s_abs)
{
    const int blk = (format == 0) ? 32 : 16;
    const int64_t nb = k / blk;
    if (!rows)
        n_rows = m;
    if (!cols)
        n_cols = n;
    const double tensor = (format == 0) ? 1.0 : (double)a_tensor_scale * (double)b_tensor_scale;

    /* Decode B once: 2*value as small integers, and the block scales. */
    int8_t *b2 = (int8_t *)malloc((size_t)n_cols * (size_t)k);
    double *bs = (double *)malloc(sizeof(double) * (size_t)n_cols * (size_t)nb);
    for (int64_t jj = 0; jj < n_cols; ++jj) {
        int64_t c = cols ? cols[jj] : jj;
        for (int64_t kk = 0; kk < k; ++kk) {
            uint8_t byte = b_codes[c * (k / 2) + kk / 2];
            uint32_t code = (kk % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
            b2[jj * k + kk] = (int8_t)(2.0 * oracle_e2m1_decode(code));
        }
        for (int64_t t = 0; t < nb; ++t) {
            uint8_t s = b_scales[c * nb + t];
            bs[jj * nb + t] = (format == 0) ? oracle_ue8m0_decode(s) : oracle_e4m3_decode(s);
        }
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ii = 0; ii < n_rows; ++ii) {
        int64_t r = rows ? rows[ii] : ii;
        int8_t *a2 = (int8_t *)malloc((size_t)k);
        double *as = (double *)malloc(sizeof(double) * (size_t)nb);
        for (int64_t kk = 0; kk < k; ++kk) {
            uint8_t byte = a_codes[r * (k / 2) + kk / 2];
            uint32_t code = (kk % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
            a2[kk] = (int8_t)(2.0 * oracle_e2m1_decode(code));
        }
        for (int64_t t = 0; t < nb; ++t) {
            uint8_t s = a_scales[r * nb + t];
            as[t] = (format == 0) ? oracle_ue8m0_decode(s) : oracle_e4m3_decode(s);
        }
        for (int64_t jj = 0; jj < n_cols; ++jj) {
            const int8_t *bj = b2 + jj * k;
            const double *bsj = bs + jj * nb;
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t t = 0; t < nb; ++t) {
                int32_t p = 0, p_abs = 0;
                for (int i = 0; i < blk; ++i) {
                    int32_t prod = (int32_t)a2[t * blk + i] * (int32_t)bj[t * blk + i];
                    p += prod;
                    p_abs += prod < 0 ? -prod : prod;
                }
                double f = as[t] * bsj[t] * 0.25;
                acc += (double)p * f;
                acc_abs += (double)p_abs * f;
            }
            d[ii * n_cols + jj] = acc * tensor;
            s_abs[ii * n_cols + jj] = acc_abs * tensor;
        }
        free(a2);
        free(as);
    }
    free(b2);
    free(bs);
}

/* ------------------------------------------------------------------ */
/* Scale-factor tile order of the tensor-core block-scaled MMA          */
/* ------------------------------------------------------------------ */

/* Plain scales [rows, kb] (kb = K / block) -> the tiled order consumed by
 * the GPU GEMM: rows padded to a multiple of 128 and kb to a multiple of 4
 * with zero bytes; 512-byte atoms of 128 rows x 4 scale columns, ordered by
 * (row tile, column tile) with the column tile fastest; inside an atom the
 * byte of (row r, column c) sits at (r % 32) * 16 + (r / 32 % 4) * 4 + c % 4.
 * (This order is the one NVIDIA documents for tcgen05 block scaling; the
 * pages only say that scales come "plain" or "swizzled".) */
void oracle_scale_tile(const uint8_t *plain, int64_t rows, int64_t kb, uint8_t *tiled)
{
    const int64_t rows_pad = (rows + 127) / 128 * 128;
    const int64_t kb_pad = (kb + 3) / 4 * 4;
    const int64_t atoms_k = kb_pad / 4;
    memset(tiled, 0, (size_t)(rows_pad * kb_pad));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < kb; ++c) {
            int64_t atom = (r / 128) * atoms_k + c / 4;
            int64_t off = atom * 512 + (r % 32) * 16 + (r / 32 % 4) * 4 + c % 4;
            tiled[off] = plain[r * kb + c];
        }
}
