/*
 * gq_oracle.c -- the plain, slow CPU oracle for the quantized skinny MUL_MAT.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is used by the test-suite, by the smoke
 * check and by the benchmark's CPU-baseline leg; the product library never
 * links, loads or calls it, and it shares no code, header or table with the
 * CUDA sources.  It is scalar C with no SIMD, no threads and no blocking: every
 * function follows the definition it cites so that it can be checked by eye.
 *
 * What is computed (the llama.cpp MUL_MAT of the q_f32 and f16_f32 kinds):
 *     dst[m][n] = sum_k src0[n][k] * src1[m][k]
 * with src0 Q4_0, Q4_1, Q5_0 or Q8_0 block-quantized weights or F16 weights,
 * and src1 F32 activations.  For the Q4_0 kind, src1 is first quantized row by row into
 * Q8_0 blocks (the "wdata" buffer) and the product is taken as integer block
 * dot products scaled by the two block scales:
 *   - llama.cpp pull request #1632, "Introduction": the three MUL_MAT kinds
 *     (f32, f16_f32, q_f32 with src0 in Q4_0/Q4_1/...), each with an INIT stage
 *     that prepares the operands and a COMPUTE stage.
 *   - Arm China article on the NUMA patch for llama.cpp (PR #14232), section
 *     "MulMat 算子優化": src1 is quantized into a buffer named wdata and the
 *     operator computes dst = src0 * wdata; every worker reads all of wdata.
 *
 * The block formats are the common ggml ones; the pages name them (Q4_0, Q8_0)
 * without defining them, so this library reads them as follows:
 *   Q4_0 block (18 bytes): fp16 scale d, then 16 bytes of 4-bit codes.  For a
 *     block x[0..31]: m = the element of largest magnitude (first one wins on a
 *     tie), d = m / -8, q_j = clamp(round(x_j / d) + 8, 0, 15) (q_j = 8 when
 *     d == 0); byte i holds q_i in its low nibble and q_{i+16} in its high
 *     nibble; the weight is w_j = (q_j - 8) * fp16(d).
 *   Q8_0 block (34 bytes): fp16 scale d = amax / 127, then 32 int8 codes
 *     q_j = round(x_j / d) (0 when d == 0); the value is q_j * fp16(d).
 *   round() is C roundf (ties away from zero); x / d is an IEEE f32 division
 *   with the f32 d; fp16(d) is IEEE round-to-nearest-even and is the scale
 *   that is stored and used to de-quantize.
 *
 * The end of the file holds the INT8 KV cache (per-token, per-head scales) and
 * the decode attention over it; its own header there says what it follows.
 *
 * Floating point: the quantizers decide integer codes, so they work in f32 as
 * the kernels do (the operands are F32).  Everything that is a sum is formed
 * in f64: each term d4 * d8 * sumi is exact in f64 (11 + 11 + 16 bits), so the
 * Q4_0 result differs from the exact value of the de-quantized product only by
 * the f64 rounding of the running sum.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define QK 32            /* values per block */
#define Q4_0_BYTES 18    /* 2-byte scale + 16 bytes of nibbles */
#define Q8_0_BYTES 34    /* 2-byte scale + 32 int8 */
#define Q5_0_BYTES 22    /* 2-byte scale + 4 bytes of fifth bits + 16 bytes of nibbles */
#define Q4_1_BYTES 20    /* 2-byte scale + 2-byte minimum + 16 bytes of nibbles */

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16, written from the format's definition.
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   E in 1..30: value = (1024 + F) * 2^(E - 25);  E == 0: value = F * 2^-24.
 * Conversion from binary32 rounds to nearest, ties to even, with gradual
 * underflow; magnitudes that round beyond 65504 become infinity.
 * ------------------------------------------------------------------------- */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t exp = (u >> 23) & 0xffu;
    uint32_t frac = u & 0x7fffffu;

    if (exp == 0xffu)                       /* infinity or NaN */
        return frac ? (uint16_t)(sign | 0x7e00u) : (uint16_t)(sign | 0x7c00u);
    if (exp == 0 && frac == 0)              /* signed zero */
        return sign;

    /* value = sig * 2^e exactly, sig a 24-bit (or smaller) integer */
    uint32_t sig;
    int e;
    if (exp == 0) { sig = frac;             e = -149; }
    else          { sig = frac | 0x800000u; e = (int)exp - 150; }

    int lead = 31;                          /* position of the top set bit */
    while (!((sig >> lead) & 1u)) lead--;
    int top = lead + e;                     /* floor(log2(value)) */

    /* binary16 spacing at this magnitude: 2^(top-10), never below 2^-24 */
    int qexp = top - 10;
    if (qexp < -24) qexp = -24;

    uint32_t q;                             /* value / 2^qexp, rounded */
    int shift = qexp - e;
    if (shift <= 0) {
        q = sig << (-shift);                /* exact */
    } else if (shift > 30) {
        q = 0;                              /* below half the smallest step */
    } else {
        uint32_t rem = sig & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        q = sig >> shift;
        if (rem > half || (rem == half && (q & 1u))) q++;
    }
    if (q == 0) return sign;
    if (q >= 2048u) { q >>= 1; qexp++; }    /* rounding carried into a new bit */

    /* q in [1, 2047]; with qexp == -24 and q < 1024 this is a subnormal */
    int E = qexp + 25;                      /* biased exponent if normal */
    if (q < 1024u) return (uint16_t)(sign | q);
    if (E >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(((uint32_t)E << 10) | (q - 1024u)));
}

float oracle_f16_to_f32(uint16_t h)
{
    uint32_t E = (h >> 10) & 31u;
    uint32_t F = h & 1023u;
    float v;
    if (E == 0)       v = ldexpf((float)F, -24);
    else if (E == 31) v = F ? NAN : INFINITY;
    else              v = ldexpf((float)(1024u + F), (int)E - 25);
    return (h & 0x8000u) ? -v : v;
}

static void put_f16(uint8_t *p, uint16_t h) { p[0] = (uint8_t)(h & 0xffu); p[1] = (uint8_t)(h >> 8); }
static uint16_t get_f16(const uint8_t *p) { return (uint16_t)(p[0] | ((uint16_t)p[1] << 8)); }

/* ---------------------------------------------------------------------------
 * Q4_0 quantization of one block of 32 weights (the format stated at the top).
 * ------------------------------------------------------------------------- */
static void quantize_block_q4_0(const float *x, uint8_t *out)
{
    float amax = 0.0f, vmax = 0.0f;
    for (int j = 0; j < QK; j++) {
        float a = fabsf(x[j]);
        if (a > amax) { amax = a; vmax = x[j]; }   /* strict: the first wins */
    }
    float d = vmax / -8.0f;
    int q[QK];
    for (int j = 0; j < QK; j++) {
        if (d != 0.0f) {
            int v = (int)roundf(x[j] / d) + 8;
            q[j] = v < 0 ? 0 : (v > 15 ? 15 : v);
        } else {
            q[j] = 8;
        }
    }
    put_f16(out, oracle_f32_to_f16(d));
    for (int i = 0; i < QK / 2; i++)
        out[2 + i] = (uint8_t)(q[i] | (q[i + QK / 2] << 4));
}

/* w: f32 [N][K] row-major; out: canonical Q4_0 blocks [N][K/32] x 18 bytes. */
void oracle_quantize_q4_0(const float *w, uint8_t *out, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            quantize_block_q4_0(w + n * K + b * QK, out + (n * nb + b) * Q4_0_BYTES);
}

/* ---------------------------------------------------------------------------
 * Q8_0 quantization of one block of 32 activations: the INIT stage that turns
 * an F32 row of src1 into wdata.
 * ------------------------------------------------------------------------- */
static void quantize_block_q8_0(const float *x, uint8_t *out)
{
    float amax = 0.0f;
    for (int j = 0; j < QK; j++) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    put_f16(out, oracle_f32_to_f16(d));
    for (int j = 0; j < QK; j++) {
        int v = 0;
        if (d != 0.0f) {
            v = (int)roundf(x[j] / d);
            v = v < -127 ? -127 : (v > 127 ? 127 : v);
        }
        out[2 + j] = (uint8_t)(int8_t)v;
    }
}

/* x: f32 [M][K]; out: Q8_0 blocks [M][K/32] x 34 bytes. */
void oracle_quantize_q8_0(const float *x, uint8_t *out, int64_t M, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++)
            quantize_block_q8_0(x + m * K + b * QK, out + (m * nb + b) * Q8_0_BYTES);
}

/* ---------------------------------------------------------------------------
 * Q5_0 quantization of one block of 32 weights.  llama.cpp PR #1632, "Results":
 * Q5_0 is one of the three types measured on 7B; the pages do not define it,
 * and this library reads it as Q4_0 with five-bit codes: block (22 bytes) =
 * fp16 d, a little-endian 32-bit word qh whose bit j is bit 4 of q_j, then 16
 * bytes with the low four bits of q_i in the low nibble and those of q_{i+16}
 * in the high nibble of byte i.  m = the element of largest magnitude (the
 * first one wins), d = m / -16, q_j = clamp(round(x_j / d) + 16, 0, 31)
 * (q_j = 16 when d == 0); the weight is (q_j - 16) * fp16(d).
 * ------------------------------------------------------------------------- */
static void quantize_block_q5_0(const float *x, uint8_t *out)
{
    float amax = 0.0f, vmax = 0.0f;
    for (int j = 0; j < QK; j++) {
        float a = fabsf(x[j]);
        if (a > amax) { amax = a; vmax = x[j]; }   /* strict: the first wins */
    }
    float d = vmax / -16.0f;
    int q[QK];
    for (int j = 0; j < QK; j++) {
        if (d != 0.0f) {
            int v = (int)roundf(x[j] / d) + 16;
            q[j] = v < 0 ? 0 : (v > 31 ? 31 : v);
        } else {
            q[j] = 16;
        }
    }
    uint32_t qh = 0;
    for (int j = 0; j < QK; j++)
        qh |= (uint32_t)((q[j] >> 4) & 1) << j;
    put_f16(out, oracle_f32_to_f16(d));
    for (int k = 0; k < 4; k++)
        out[2 + k] = (uint8_t)(qh >> (8 * k));
    for (int i = 0; i < QK / 2; i++)
        out[6 + i] = (uint8_t)((q[i] & 0x0f) | ((q[i + QK / 2] & 0x0f) << 4));
}

/* w: f32 [N][K]; out: Q5_0 blocks [N][K/32] x 22 bytes. */
void oracle_quantize_q5_0(const float *w, uint8_t *out, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            quantize_block_q5_0(w + n * K + b * QK, out + (n * nb + b) * Q5_0_BYTES);
}

/* ---------------------------------------------------------------------------
 * Q4_1 quantization of one block of 32 weights.  llama.cpp PR #1632,
 * "Introduction": Q4_1 is named beside Q4_0 as a src0 type of the q_f32 kind;
 * the pages do not define it, and this library reads it as a scale and a
 * minimum per block: block (20 bytes) = fp16 d, fp16 m, then 16 bytes with q_i
 * in the low nibble and q_{i+16} in the high nibble of byte i.  lo, hi = the
 * smallest and largest element, d = (hi - lo) / 15, m = lo,
 * q_j = clamp(round((x_j - lo) / d), 0, 15) (q_j = 0 when d == 0), all in f32;
 * the weight is q_j * fp16(d) + fp16(m).
 * ------------------------------------------------------------------------- */
static void quantize_block_q4_1(const float *x, uint8_t *out)
{
    float lo = x[0], hi = x[0];
    for (int j = 1; j < QK; j++) {
        if (x[j] < lo) lo = x[j];
        if (x[j] > hi) hi = x[j];
    }
    float d = (hi - lo) / 15.0f;
    int q[QK];
    for (int j = 0; j < QK; j++) {
        if (d != 0.0f) {
            int v = (int)roundf((x[j] - lo) / d);
            q[j] = v < 0 ? 0 : (v > 15 ? 15 : v);
        } else {
            q[j] = 0;
        }
    }
    put_f16(out, oracle_f32_to_f16(d));
    put_f16(out + 2, oracle_f32_to_f16(lo));
    for (int i = 0; i < QK / 2; i++)
        out[4 + i] = (uint8_t)(q[i] | (q[i + QK / 2] << 4));
}

/* w: f32 [N][K]; out: Q4_1 blocks [N][K/32] x 20 bytes. */
void oracle_quantize_q4_1(const float *w, uint8_t *out, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            quantize_block_q4_1(w + n * K + b * QK, out + (n * nb + b) * Q4_1_BYTES);
}

/* ---------------------------------------------------------------------------
 * De-quantization (for the invariant checks): value = (q - 8) * d  (Q4_0),
 * value = (q - 16) * d (Q5_0), value = q * d + m (Q4_1), value = q * d (Q8_0),
 * in f64 (exact).
 * ------------------------------------------------------------------------- */
static int q4_code(const uint8_t *blk, int j)
{
    uint8_t byte = blk[2 + (j % (QK / 2))];
    return j < QK / 2 ? (byte & 0x0f) : (byte >> 4);
}

static int q8_code(const uint8_t *blk, int j) { return (int)(int8_t)blk[2 + j]; }

static int q5_code(const uint8_t *blk, int j)
{
    uint32_t qh = (uint32_t)blk[2] | ((uint32_t)blk[3] << 8) | ((uint32_t)blk[4] << 16) | ((uint32_t)blk[5] << 24);
    uint8_t byte = blk[6 + (j % (QK / 2))];
    int lo = j < QK / 2 ? (byte & 0x0f) : (byte >> 4);
    return lo | (int)(((qh >> j) & 1u) << 4);
}

static int q41_code(const uint8_t *blk, int j)
{
    uint8_t byte = blk[4 + (j % (QK / 2))];
    return j < QK / 2 ? (byte & 0x0f) : (byte >> 4);
}

void oracle_dequantize_q4_1(const uint8_t *q41, double *out, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = q41 + (n * nb + b) * Q4_1_BYTES;
            double d = (double)oracle_f16_to_f32(get_f16(blk));
            double m = (double)oracle_f16_to_f32(get_f16(blk + 2));
            for (int j = 0; j < QK; j++)
                out[n * K + b * QK + j] = (double)q41_code(blk, j) * d + m;
        }
}

void oracle_dequantize_q5_0(const uint8_t *q5, double *out, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = q5 + (n * nb + b) * Q5_0_BYTES;
            double d = (double)oracle_f16_to_f32(get_f16(blk));
            for (int j = 0; j < QK; j++)
                out[n * K + b * QK + j] = (double)(q5_code(blk, j) - 16) * d;
        }
}

void oracle_dequantize_q4_0(const uint8_t *q4, double *out, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = q4 + (n * nb + b) * Q4_0_BYTES;
            double d = (double)oracle_f16_to_f32(get_f16(blk));
            for (int j = 0; j < QK; j++)
                out[n * K + b * QK + j] = (double)(q4_code(blk, j) - 8) * d;
        }
}

void oracle_dequantize_q8_0(const uint8_t *q8, double *out, int64_t M, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = q8 + (m * nb + b) * Q8_0_BYTES;
            double d = (double)oracle_f16_to_f32(get_f16(blk));
            for (int j = 0; j < QK; j++)
                out[m * K + b * QK + j] = (double)q8_code(blk, j) * d;
        }
}

/* ---------------------------------------------------------------------------
 * The integer block dot of the COMPUTE stage:
 *     sumi = sum_{j<32} (q4_j - 8) * q8_j           (|sumi| <= 32*8*127)
 * ------------------------------------------------------------------------- */
static int32_t block_dot(const uint8_t *b4, const uint8_t *b8)
{
    int32_t s = 0;
    for (int j = 0; j < QK; j++)
        s += (int32_t)(q4_code(b4, j) - 8) * (int32_t)q8_code(b8, j);
    return s;
}

/* sumi: int32 [M][N][K/32] */
void oracle_block_dots(const uint8_t *q4, const uint8_t *q8, int32_t *sumi,
                       int64_t M, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            for (int64_t b = 0; b < nb; b++)
                sumi[(m * N + n) * nb + b] =
                    block_dot(q4 + (n * nb + b) * Q4_0_BYTES, q8 + (m * nb + b) * Q8_0_BYTES);
}

/* One output of the q_f32 kind from the quantized operands:
 *     dst = sum_b d4_b * d8_b * sumi_b               (f64)
 * and the error denominator of the de-quantized terms:
 *     T   = sum_b |d4_b| |d8_b| sum_j |q4_j - 8| |q8_j|
 */
static void dot_row_q4_0_q8_0(const uint8_t *row4, const uint8_t *row8, int64_t nb,
                              double *dst, double *T)
{
    double acc = 0.0, tacc = 0.0;
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *b4 = row4 + b * Q4_0_BYTES;
        const uint8_t *b8 = row8 + b * Q8_0_BYTES;
        double d4 = (double)oracle_f16_to_f32(get_f16(b4));
        double d8 = (double)oracle_f16_to_f32(get_f16(b8));
        acc += d4 * d8 * (double)block_dot(b4, b8);
        int64_t sabs = 0;
        for (int j = 0; j < QK; j++)
            sabs += (int64_t)abs(q4_code(b4, j) - 8) * (int64_t)abs(q8_code(b8, j));
        tacc += fabs(d4) * fabs(d8) * (double)sabs;
    }
    *dst = acc;
    *T = tacc;
}

/* Full q_f32 MUL_MAT for the output columns n in [n_begin, n_end):
 * INIT quantizes every row of src1 to Q8_0, COMPUTE forms the block dots.
 * q4: canonical Q4_0 [N][K/32]; src1: f32 [M][K]; dst, T: f64 [M][N]. */
int oracle_mul_mat_q4_0_f32(const uint8_t *q4, const float *src1, double *dst, double *T,
                            int64_t M, int64_t N, int64_t K, int64_t n_begin, int64_t n_end)
{
    int64_t nb = K / QK;
    uint8_t *wdata = (uint8_t *)malloc((size_t)(M * nb * Q8_0_BYTES) + 1);
    if (!wdata) return 1;
    oracle_quantize_q8_0(src1, wdata, M, K);
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = n_begin; n < n_end; n++)
            dot_row_q4_0_q8_0(q4 + n * nb * Q4_0_BYTES, wdata + m * nb * Q8_0_BYTES, nb,
                              &dst[m * N + n], &T[m * N + n]);
    free(wdata);
    return 0;
}

/* Selected outputs (ms[i], ns[i]) of the q_f32 kind from already quantized
 * operands (q8 from oracle_quantize_q8_0).  out, T: f64 [count]. */
void oracle_mul_mat_q4_0_q8_0_at(const uint8_t *q4, const uint8_t *q8, const int64_t *ms,
                                 const int64_t *ns, int64_t count, int64_t K,
                                 double *out, double *T)
{
    int64_t nb = K / QK;
    for (int64_t i = 0; i < count; i++)
        dot_row_q4_0_q8_0(q4 + ns[i] * nb * Q4_0_BYTES, q8 + ms[i] * nb * Q8_0_BYTES, nb,
                          &out[i], &T[i]);
}

/* ---------------------------------------------------------------------------
 * The q_f32 kind with Q8_0 weights.  llama.cpp pull request #1632,
 * "Introduction": src0 of the q_f32 kind may be any quantized type; "Results":
 * Q8_0 is one of the three types measured on 7B.  The weights use the Q8_0
 * block above (the activations' format), src1 is quantized to Q8_0 exactly as
 * for Q4_0, and the integer block dot has no offset:
 *     sumi = sum_{j<32} qw_j * qx_j                   (|sumi| <= 32*127*127)
 *     dst  = sum_b dw_b * dx_b * sumi_b               (f64; each term exact)
 *     T    = sum_b |dw_b| |dx_b| sum_j |qw_j| |qx_j|
 * ------------------------------------------------------------------------- */
static int32_t block_dot_q8_0(const uint8_t *bw, const uint8_t *bx)
{
    int32_t s = 0;
    for (int j = 0; j < QK; j++)
        s += (int32_t)q8_code(bw, j) * (int32_t)q8_code(bx, j);
    return s;
}

/* sumi: int32 [M][N][K/32] */
void oracle_block_dots_q8_0(const uint8_t *qw, const uint8_t *qx, int32_t *sumi,
                            int64_t M, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            for (int64_t b = 0; b < nb; b++)
                sumi[(m * N + n) * nb + b] =
                    block_dot_q8_0(qw + (n * nb + b) * Q8_0_BYTES, qx + (m * nb + b) * Q8_0_BYTES);
}

static void dot_row_q8_0_q8_0(const uint8_t *roww, const uint8_t *rowx, int64_t nb,
                              double *dst, double *T)
{
    double acc = 0.0, tacc = 0.0;
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *bw = roww + b * Q8_0_BYTES;
        const uint8_t *bx = rowx + b * Q8_0_BYTES;
        double dw = (double)oracle_f16_to_f32(get_f16(bw));
        double dx = (double)oracle_f16_to_f32(get_f16(bx));
        acc += dw * dx * (double)block_dot_q8_0(bw, bx);
        int64_t sabs = 0;
        for (int j = 0; j < QK; j++)
            sabs += (int64_t)abs(q8_code(bw, j)) * (int64_t)abs(q8_code(bx, j));
        tacc += fabs(dw) * fabs(dx) * (double)sabs;
    }
    *dst = acc;
    *T = tacc;
}

/* Full MUL_MAT with Q8_0 weights for the output columns n in [n_begin, n_end).
 * qw: Q8_0 [N][K/32]; src1: f32 [M][K]; dst, T: f64 [M][N]. */
int oracle_mul_mat_q8_0_f32(const uint8_t *qw, const float *src1, double *dst, double *T,
                            int64_t M, int64_t N, int64_t K, int64_t n_begin, int64_t n_end)
{
    int64_t nb = K / QK;
    uint8_t *wdata = (uint8_t *)malloc((size_t)(M * nb * Q8_0_BYTES) + 1);
    if (!wdata) return 1;
    oracle_quantize_q8_0(src1, wdata, M, K);
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = n_begin; n < n_end; n++)
            dot_row_q8_0_q8_0(qw + n * nb * Q8_0_BYTES, wdata + m * nb * Q8_0_BYTES, nb,
                              &dst[m * N + n], &T[m * N + n]);
    free(wdata);
    return 0;
}

/* Selected outputs (ms[i], ns[i]) with Q8_0 weights from quantized activations qx. */
void oracle_mul_mat_q8_0_q8_0_at(const uint8_t *qw, const uint8_t *qx, const int64_t *ms,
                                 const int64_t *ns, int64_t count, int64_t K,
                                 double *out, double *T)
{
    int64_t nb = K / QK;
    for (int64_t i = 0; i < count; i++)
        dot_row_q8_0_q8_0(qw + ns[i] * nb * Q8_0_BYTES, qx + ms[i] * nb * Q8_0_BYTES, nb,
                          &out[i], &T[i]);
}

/* ---------------------------------------------------------------------------
 * The q_f32 kind with Q5_0 weights (the format above), src1 in Q8_0 as for
 * Q4_0:  sumi = sum_{j<32} (q5_j - 16) * q8_j      (|sumi| <= 32*16*127)
 *        dst = sum_b d5_b * d8_b * sumi_b (f64),  T = sum_b |d5| |d8| sum_j |q5_j - 16| |q8_j|
 * ------------------------------------------------------------------------- */
static int32_t block_dot_q5_0(const uint8_t *b5, const uint8_t *b8)
{
    int32_t s = 0;
    for (int j = 0; j < QK; j++)
        s += (int32_t)(q5_code(b5, j) - 16) * (int32_t)q8_code(b8, j);
    return s;
}

/* sumi: int32 [M][N][K/32] */
void oracle_block_dots_q5_0(const uint8_t *q5, const uint8_t *q8, int32_t *sumi,
                            int64_t M, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            for (int64_t b = 0; b < nb; b++)
                sumi[(m * N + n) * nb + b] =
                    block_dot_q5_0(q5 + (n * nb + b) * Q5_0_BYTES, q8 + (m * nb + b) * Q8_0_BYTES);
}

static void dot_row_q5_0_q8_0(const uint8_t *row5, const uint8_t *row8, int64_t nb,
                              double *dst, double *T)
{
    double acc = 0.0, tacc = 0.0;
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *b5 = row5 + b * Q5_0_BYTES;
        const uint8_t *b8 = row8 + b * Q8_0_BYTES;
        double d5 = (double)oracle_f16_to_f32(get_f16(b5));
        double d8 = (double)oracle_f16_to_f32(get_f16(b8));
        acc += d5 * d8 * (double)block_dot_q5_0(b5, b8);
        int64_t sabs = 0;
        for (int j = 0; j < QK; j++)
            sabs += (int64_t)abs(q5_code(b5, j) - 16) * (int64_t)abs(q8_code(b8, j));
        tacc += fabs(d5) * fabs(d8) * (double)sabs;
    }
    *dst = acc;
    *T = tacc;
}

int oracle_mul_mat_q5_0_f32(const uint8_t *q5, const float *src1, double *dst, double *T,
                            int64_t M, int64_t N, int64_t K, int64_t n_begin, int64_t n_end)
{
    int64_t nb = K / QK;
    uint8_t *wdata = (uint8_t *)malloc((size_t)(M * nb * Q8_0_BYTES) + 1);
    if (!wdata) return 1;
    oracle_quantize_q8_0(src1, wdata, M, K);
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = n_begin; n < n_end; n++)
            dot_row_q5_0_q8_0(q5 + n * nb * Q5_0_BYTES, wdata + m * nb * Q8_0_BYTES, nb,
                              &dst[m * N + n], &T[m * N + n]);
    free(wdata);
    return 0;
}

void oracle_mul_mat_q5_0_q8_0_at(const uint8_t *q5, const uint8_t *q8, const int64_t *ms,
                                 const int64_t *ns, int64_t count, int64_t K,
                                 double *out, double *T)
{
    int64_t nb = K / QK;
    for (int64_t i = 0; i < count; i++)
        dot_row_q5_0_q8_0(q5 + ns[i] * nb * Q5_0_BYTES, q8 + ms[i] * nb * Q8_0_BYTES, nb,
                          &out[i], &T[i]);
}

/* ---------------------------------------------------------------------------
 * The q_f32 kind with Q4_1 weights (the format above), src1 in Q8_0:
 *   sum_j (q_j d + m) (q8_j d8) = d d8 sumi + m d8 sx,  sumi = sum_j q_j q8_j,  sx = sum_j q8_j
 *   dst = sum_b (d_b d8_b sumi_b + m_b d8_b sx_b)   (f64; each product exact)
 *   T   = sum_b |d8_b| sum_j |q_j d_b + m_b| |q8_j|
 * ------------------------------------------------------------------------- */
/* sumi and sx of one block pair: out[0] = sum_j q_j q8_j, out[1] = sum_j q8_j */
static void block_sums_q4_1(const uint8_t *b41, const uint8_t *b8, int32_t out[2])
{
    int32_t s = 0, sx = 0;
    for (int j = 0; j < QK; j++) {
        s += (int32_t)q41_code(b41, j) * (int32_t)q8_code(b8, j);
        sx += (int32_t)q8_code(b8, j);
    }
    out[0] = s;
    out[1] = sx;
}

/* sums: int32 [M][N][K/32][2] */
void oracle_block_sums_q4_1(const uint8_t *q41, const uint8_t *q8, int32_t *sums,
                            int64_t M, int64_t N, int64_t K)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            for (int64_t b = 0; b < nb; b++)
                block_sums_q4_1(q41 + (n * nb + b) * Q4_1_BYTES, q8 + (m * nb + b) * Q8_0_BYTES,
                                sums + ((m * N + n) * nb + b) * 2);
}

static void dot_row_q4_1_q8_0(const uint8_t *row41, const uint8_t *row8, int64_t nb,
                              double *dst, double *T)
{
    double acc = 0.0, tacc = 0.0;
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *b41 = row41 + b * Q4_1_BYTES;
        const uint8_t *b8 = row8 + b * Q8_0_BYTES;
        double d = (double)oracle_f16_to_f32(get_f16(b41));
        double mn = (double)oracle_f16_to_f32(get_f16(b41 + 2));
        double d8 = (double)oracle_f16_to_f32(get_f16(b8));
        int32_t sums[2];
        block_sums_q4_1(b41, b8, sums);
        acc += d * d8 * (double)sums[0];
        acc += mn * d8 * (double)sums[1];
        double t = 0.0;
        for (int j = 0; j < QK; j++)
            t += fabs((double)q41_code(b41, j) * d + mn) * (double)abs(q8_code(b8, j));
        tacc += fabs(d8) * t;
    }
    *dst = acc;
    *T = tacc;
}

int oracle_mul_mat_q4_1_f32(const uint8_t *q41, const float *src1, double *dst, double *T,
                            int64_t M, int64_t N, int64_t K, int64_t n_begin, int64_t n_end)
{
    int64_t nb = K / QK;
    uint8_t *wdata = (uint8_t *)malloc((size_t)(M * nb * Q8_0_BYTES) + 1);
    if (!wdata) return 1;
    oracle_quantize_q8_0(src1, wdata, M, K);
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = n_begin; n < n_end; n++)
            dot_row_q4_1_q8_0(q41 + n * nb * Q4_1_BYTES, wdata + m * nb * Q8_0_BYTES, nb,
                              &dst[m * N + n], &T[m * N + n]);
    free(wdata);
    return 0;
}

void oracle_mul_mat_q4_1_q8_0_at(const uint8_t *q41, const uint8_t *q8, const int64_t *ms,
                                 const int64_t *ns, int64_t count, int64_t K,
                                 double *out, double *T)
{
    int64_t nb = K / QK;
    for (int64_t i = 0; i < count; i++)
        dot_row_q4_1_q8_0(q41 + ns[i] * nb * Q4_1_BYTES, q8 + ms[i] * nb * Q8_0_BYTES, nb,
                          &out[i], &T[i]);
}

/* ---------------------------------------------------------------------------
 * The f16_f32 kind: dst[m][n] = sum_k w16[n][k] * src1[m][k] in f64 with the
 * F32 activations taken as they are; T[m][n] = sum_k |w16[n][k] * src1[m][k]|.
 * ------------------------------------------------------------------------- */
static void dot_row_f16_f32(const uint16_t *w, const float *x, int64_t K, double *dst, double *T)
{
    double acc = 0.0, tacc = 0.0;
    for (int64_t k = 0; k < K; k++) {
        double p = (double)oracle_f16_to_f32(w[k]) * (double)x[k];
        acc += p;
        tacc += fabs(p);
    }
    *dst = acc;
    *T = tacc;
}

void oracle_mul_mat_f16_f32(const uint16_t *w16, const float *src1, double *dst, double *T,
                            int64_t M, int64_t N, int64_t K, int64_t n_begin, int64_t n_end)
{
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = n_begin; n < n_end; n++)
            dot_row_f16_f32(w16 + n * K, src1 + m * K, K, &dst[m * N + n], &T[m * N + n]);
}

void oracle_mul_mat_f16_f32_at(const uint16_t *w16, const float *src1, const int64_t *ms,
                               const int64_t *ns, int64_t count, int64_t K,
                               double *out, double *T)
{
    for (int64_t i = 0; i < count; i++)
        dot_row_f16_f32(w16 + ns[i] * K, src1 + ms[i] * K, K, &out[i], &T[i]);
}

/* Element-wise conversions, exported for the binary16 pins. */
void oracle_f32_to_f16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_f16(x[i]);
}

void oracle_f16_to_f32_array(const uint16_t *h, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f16_to_f32(h[i]);
}

/* ---------------------------------------------------------------------------
 * The INT8 KV cache and the decode attention that reads it.
 *
 * xFasterTransformer (arXiv 2407.07304), "2.2 Effective KV cache
 * Optimization": after the first token, attention over the cache is a pair of
 * memory-bound GEMVs; the cache is stored as INT8 with its own scale for each
 * token and each head, and the INT8 operand is widened to FP32 before the
 * multiply-add.  Section "2.1 LLM Optimization" (SlimAttention) fixes the
 * order for one query row: the whole row of scores first, then the softmax
 * over it, then the product of the softmax with the values.
 *
 * The page gives the granularity of the scale but not its formula.  This
 * library reads it like the Q8_0 scale above: for the D values x[0..D-1] of
 * one token and one head, s = amax / 127 in f32, q_j = round(x_j / s) (IEEE f32
 * division, ties away from zero; 0 when s == 0), and the cached value is
 * q_j * s.  Inputs must be finite.
 *
 * Layouts: codes int8 [B][Hkv][Tcap][D], scales f32 [B][Hkv][Tcap], queries
 * f32 [B][Hq][D] with Hq = G * Hkv (grouped queries: query head h reads KV
 * head h / G), lens int32 [B] with 0 <= lens[b] <= Tcap, output [B][Hq][D].
 * For query head h of sequence b, over the tokens t < lens[b]:
 *     score_t = c * ks_t * sum_j q_j * k_tj          (c: the softmax scale)
 *     p_t     = exp(score_t - max_u score_u) / sum_u exp(score_u - max_u score_u)
 *     out_j   = sum_t p_t * vs_t * v_tj
 * and an empty sequence gives out = 0.  Every sum is formed in f64 (each
 * product q_j * k_tj of an f32 and an int8 is exact there).  For error bounds
 * the oracle also returns E[b][h][j] = sum_t p_t * |vs_t * v_tj| and
 * S[b][h] = max_t |c * ks_t| * sum_j |q_j * k_tj|.
 * ------------------------------------------------------------------------- */
void oracle_kv_quantize_i8(const float *x, int8_t *q, float *scale, int64_t rows, int64_t D)
{
    for (int64_t r = 0; r < rows; r++) {
        const float *xr = x + r * D;
        float amax = 0.0f;
        for (int64_t j = 0; j < D; j++) {
            float a = fabsf(xr[j]);
            if (a > amax) amax = a;
        }
        float s = amax / 127.0f;
        scale[r] = s;
        for (int64_t j = 0; j < D; j++) {
            int v = 0;
            if (s != 0.0f) {
                v = (int)roundf(xr[j] / s);
                v = v < -127 ? -127 : (v > 127 ? 127 : v);
            }
            q[r * D + j] = (int8_t)v;
        }
    }
}

void oracle_kv_dequantize_i8(const int8_t *q, const float *scale, double *out, int64_t rows,
                             int64_t D)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t j = 0; j < D; j++)
            out[r * D + j] = (double)q[r * D + j] * (double)scale[r];
}

int oracle_attn_decode_i8(const float *q, const int8_t *k, const float *ks, const int8_t *v,
                          const float *vs, const int32_t *lens, double c, double *out,
                          double *E, double *S, int64_t B, int64_t Hq, int64_t Hkv,
                          int64_t Tcap, int64_t D)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    int64_t G = Hq / Hkv;
    double *p = (double *)malloc((size_t)(Tcap > 0 ? Tcap : 1) * sizeof(double));
    if (!p)
        return -2;
    for (int64_t b = 0; b < B; b++) {
        int64_t L = lens[b];
        if (L < 0 || L > Tcap) {
            free(p);
            return -1;
        }
        for (int64_t h = 0; h < Hq; h++) {
            int64_t hk = h / G;
            const float *qv = q + (b * Hq + h) * D;
            const int8_t *kb = k + (b * Hkv + hk) * Tcap * D;
            const int8_t *vb = v + (b * Hkv + hk) * Tcap * D;
            const float *ksb = ks + (b * Hkv + hk) * Tcap;
            const float *vsb = vs + (b * Hkv + hk) * Tcap;
            double *o = out + (b * Hq + h) * D;
            double *e = E + (b * Hq + h) * D;
            double smax = 0.0;
            /* the row of scores */
            for (int64_t t = 0; t < L; t++) {
                double dot = 0.0, adot = 0.0;
                for (int64_t j = 0; j < D; j++) {
                    double term = (double)qv[j] * (double)kb[t * D + j];
                    dot += term;
                    adot += fabs(term);
                }
                p[t] = c * (double)ksb[t] * dot;
                double a = fabs(c * (double)ksb[t]) * adot;
                if (a > smax) smax = a;
            }
            S[b * Hq + h] = smax;
            /* the softmax over it */
            double m = -INFINITY;
            for (int64_t t = 0; t < L; t++)
                if (p[t] > m) m = p[t];
            double l = 0.0;
            for (int64_t t = 0; t < L; t++) {
                p[t] = exp(p[t] - m);
                l += p[t];
            }
            for (int64_t t = 0; t < L; t++)
                p[t] /= l;
            /* its product with the values */
            for (int64_t j = 0; j < D; j++) {
                double acc = 0.0, eacc = 0.0;
                for (int64_t t = 0; t < L; t++) {
                    double term = p[t] * (double)vsb[t] * (double)vb[t * D + j];
                    acc += term;
                    eacc += fabs(term);
                }
                o[j] = acc;
                e[j] = eacc;
            }
        }
    }
    free(p);
    return 0;
}
