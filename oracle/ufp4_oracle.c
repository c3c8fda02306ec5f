/*
 * ufp4_oracle.c -- plain, slow, single-threaded CPU oracle for the UFP4
 * quantization hot path.  TEST INFRASTRUCTURE ONLY: nothing in the library
 * path may link or call this file; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant generator with the CUDA path.
 *
 * Sources (the three web pages on arXiv:2606.20381, "Rethinking Shrinkage
 * Bias in LLM FP4 Pretraining: Geometric Origin, Systemic Impact, and UFP4
 * Recipe"), cited below as:
 *   [ZC]  zhichai.net post "Shrinkage Bias: The Hidden Geometric Trap in FP4
 *         Training ... and the UFP4 Fix", section + bullet name;
 *   [AN]  autonainews.com article "UFP4 Eliminates Shrinkage Bias in FP4 LLM
 *         Pretraining, Ant Group Research Finds", section name;
 *   [HP]  hotpaper.ai card of the paper, section name.
 * Where the pages leave a step open (block size, scale format, RHT size and
 * normalisation, random-number generator, bit layouts) this file follows the
 * readings listed in the repository's design notes; each is marked READING.
 *
 * Parity status: every function here is pinned by the CPU tests
 * (tests/test_oracle_pins.py) except the SQNR *values* the pages print for
 * their real outlier tensor, which cannot be reproduced without it
 * (parity unpinned for those values; only their ranking is checked).
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -fPIC -shared.
 * -ffp-contract=off matters: every fl32() step below is one IEEE rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <float.h>

#define REF_E2M1 0
#define REF_E1M2 1
#define REF_E2M1C 2
#define REF_RTNE 0
#define REF_SR   1

/* ------------------------------------------------------------------------
 * Philox4x32-10.  Written from the algorithm of Salmon, Moraes, Dror and
 * Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of
 * the 4x32 S-box built from two 32x32->64 multiplications, with the key
 * advanced by the Weyl constants between rounds.  READING: the pages name
 * stochastic rounding but no generator; Philox is this library's choice.
 * ---------------------------------------------------------------------- */
static void philox_round(uint32_t c[4], const uint32_t k[2])
{
    const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k[0];
    const uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
}

void ref_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k[0] += 0x9E3779B9u; k[1] += 0xBB67AE85u; }
        philox_round(c, k);
    }
    memcpy(out, c, sizeof c);
}

/* ------------------------------------------------------------------------
 * RHT signs and the 16-point Hadamard matrix.
 * [ZC] Key points, "The RHT paradox"; [AN] "The UFP4 Recipe".
 * READING: one vector d of 16 random signs, drawn from the RHT seed, is shared
 * by every block of every tensor; d_j = -1 iff bit j of the first Philox word
 * for key = seed and counter 0 is set.
 * ---------------------------------------------------------------------- */
void ref_rht_signs(uint64_t seed, int32_t d[16])
{
    const uint32_t ctr[4] = {0, 0, 0, 0};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    ref_philox4x32_10(ctr, key, w);
    for (int j = 0; j < 16; ++j) d[j] = ((w[0] >> j) & 1u) ? -1 : 1;
}

/* Sylvester-ordered Hadamard entry H[i][j] = (-1)^popcount(i & j). */
int32_t ref_hadamard16(int32_t i, int32_t j)
{
    unsigned v = (unsigned)(i & j), pc = 0;
    while (v) { pc += v & 1u; v >>= 1; }
    return (pc & 1u) ? -1 : 1;
}

/* y = (1/4) * H * diag(d) * x for one 16-block, in fp64, rounded to fp32
 * once.  READING: the 1/4 normalisation makes the transform orthonormal, so
 * two operands rotated with the same d along K keep their inner products.
 * hd[i][j] = H[i][j] * d[j] (+-1), built once per tensor by rht16_matrix. */
static void rht16_matrix(const int32_t d[16], double hd[16][16])
{
    for (int i = 0; i < 16; ++i)
        for (int j = 0; j < 16; ++j) hd[i][j] = (double)ref_hadamard16(i, j) * (double)d[j];
}

static void rht16_forward(const float x[16], const double hd[16][16], float y[16])
{
    for (int i = 0; i < 16; ++i) {
        double s = 0.0;
        for (int j = 0; j < 16; ++j) s += hd[i][j] * (double)x[j];
        y[i] = (float)(0.25 * s);
    }
}

/* Inverse: x = diag(d) * (1/4) * H * y (H is symmetric and H*H = 16 I). */
static void rht16_inverse(const double y[16], const int32_t d[16], double x[16])
{
    for (int i = 0; i < 16; ++i) {
        double s = 0.0;
        for (int j = 0; j < 16; ++j) s += (double)ref_hadamard16(i, j) * y[j];
        x[i] = (double)d[i] * 0.25 * s;
    }
}

/* ------------------------------------------------------------------------
 * FP8 E4M3 (OCP 8-bit floating point specification): 1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits; subnormals for exponent field 0; S.1111.111
 * is NaN, so the largest finite magnitude is 448.  Used for the per-block
 * scale of the two-level (NVFP4-style) scaling the pages name as the E2M1
 * baseline ([ZC] Key points, "The symptom"; [HP] technical approach).
 * ---------------------------------------------------------------------- */
double ref_e4m3_decode(uint8_t c)
{
    const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even with saturation to +-448 (and +-inf to +-448):
 * brute force over the 127 finite non-negative codes; exact comparisons in
 * fp64; a tie picks the code with an even mantissa LSB. */
uint8_t ref_e4m3_encode(float v)
{
    if (isnan(v)) return 0x7F;
    const int neg = signbit(v) ? 1 : 0;
    const double a = fabs((double)v);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c < 0x7F; ++c) {
        const double err = fabs(a - ref_e4m3_decode((uint8_t)c));
        if (err < best_err || (err == best_err && (c & 1) == 0)) { best = c; best_err = err; }
    }
    if (a > 448.0) best = 0x7E;           /* satfinite */
    return (uint8_t)(best | (neg << 7));
}

/* ------------------------------------------------------------------------
 * The 4-bit grids.  [ZC] Key points, "The cause" (E2M1 values) and
 * "The fix -- UFP4" (E1M2 values).  Both grids carry a sign bit and use all
 * 16 codes.  The third is the ablation the pages report as failing: a
 * uniform grid emulated by clamping E2M1's range ([ZC] Key points,
 * "Validation results") -- READING: E2M1 restricted to its largest uniform
 * part {0, .5, 1, 1.5, 2} (codes 0..4 with sign), qmax = 2.
 * A code is (sign << 3) | m, m the magnitude index.
 * ---------------------------------------------------------------------- */
double ref_grid_value(int grid, int m)
{
    static const double e2m1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    if (grid == REF_E2M1 || grid == REF_E2M1C) return e2m1[m & 7];
    return 0.5 * (double)(m & 7);
}

double ref_grid_qmax(int grid) { return grid == REF_E2M1 ? 6.0 : (grid == REF_E1M2 ? 3.5 : 2.0); }

/* Number of magnitudes of the grid (8, or 5 for clamped E2M1). */
int ref_grid_levels(int grid) { return grid == REF_E2M1C ? 5 : 8; }

/* Round-to-nearest-even onto the grid: brute-force argmin over the grid's
 * magnitudes, ties to the even index (IEEE RNE for E2M1's bit layout; even
 * integer 2a for E1M2 and clamped E2M1).  a >= 0, already clamped to qmax. */
int ref_round_rtne(int grid, float a)
{
    int best = 0;
    double best_err = INFINITY;
    for (int m = 0; m < ref_grid_levels(grid); ++m) {
        const double err = fabs((double)a - ref_grid_value(grid, m));
        if (err < best_err || (err == best_err && (m & 1) == 0)) { best = m; best_err = err; }
    }
    return best;
}

/* Stochastic rounding ([ZC] "The fix -- UFP4"; [HP] key contributions: SR on
 * dY only): with lo <= a < hi the neighbouring grid points, round up with
 * probability p = (a - lo)/(hi - lo).  READING: the Bernoulli draw compares
 * a 16-bit uniform r (half of a Philox word, see ref_sr_bits) as
 * u = r * 2^-16 against p, both exact in fp32: the round-up probability is p
 * rounded up to a multiple of 2^-16, within 2^-16 of a grid step of the
 * unbiased draw.  Only the low 16 bits of r are used. */
int ref_round_sr(int grid, float a, uint32_t r)
{
    const int top = ref_grid_levels(grid) - 1;
    if ((double)a >= ref_grid_qmax(grid)) return top;
    int m = 0;
    while (m < top && ref_grid_value(grid, m + 1) <= (double)a) ++m;
    const float lo = (float)ref_grid_value(grid, m);
    const float hi = (float)ref_grid_value(grid, m + 1);
    const float p = (a - lo) / (hi - lo);
    const float u = (float)(r & 0xFFFFu) * 0x1p-16f;
    return (u < p) ? m + 1 : m;
}

/* The 16 random bits that drive SR for logical element index i of the
 * output code buffer: key = sr_seed, counter = (i / 8, sr_counter), and of
 * the four words the call returns, word (i mod 8) / 2, its low half for
 * even i and its high half for odd i. */
uint32_t ref_sr_bits(uint64_t sr_seed, uint64_t sr_counter, uint64_t i)
{
    const uint64_t q = i >> 3;
    const uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32),
                             (uint32_t)sr_counter, (uint32_t)(sr_counter >> 32)};
    const uint32_t key[2] = {(uint32_t)sr_seed, (uint32_t)(sr_seed >> 32)};
    uint32_t w[4];
    ref_philox4x32_10(ctr, key, w);
    return (w[(i >> 1) & 3] >> (16 * (unsigned)(i & 1))) & 0xFFFFu;
}

/* ------------------------------------------------------------------------
 * Block quantization of one rows x k matrix whose 16-blocks run along k.
 *
 *   y       : the rows x k input (row stride ld, fp32 values); with rht set
 *             each 16-block is rotated first, and the rotated values are
 *             written to y_out (may be NULL).
 *   A_t     : max |y| over the tensor, or *amax_in when given.
 *   S_enc   = fl32(448 qmax / A_t)  (clamped to FLT_MAX);  S_dec = fl32(A_t / (448 qmax));
 *             A_t == 0 gives S_enc = S_dec = 1.
 *   e_b     = E4M3(fl32(fl32(amax_b / qmax) * S_enc)).
 *   k_b     = fl32(S_enc / e_b) (clamped to FLT_MAX);  q = fl32(y k_b);
 *   a       = min(|q|, qmax);  code = signbit(q) << 3 | round(a).
 *   e_b == 0 gives all-zero codes for the block.
 * READING: the pages give the grids and the rounding modes; the two-level
 * scale (16-element blocks, E4M3 block scale, FP32 tensor scale) and the
 * order of operations above are this library's contract.
 *
 * Outputs: codes rows x k (one code per byte, unpacked), scales rows x k/16
 * (row-major E4M3 bytes), *tensor_scale = S_dec.  elem_base offsets the SR
 * element index (i = elem_base + r * k + j).
 * Returns 0, or -1 on k % 16 != 0.
 * ---------------------------------------------------------------------- */
int ref_quantize_strided(const float *x, int64_t rows, int64_t k, int64_t ld,
                         int grid, int rht, uint64_t rht_seed,
                         int round_mode, uint64_t sr_seed, uint64_t sr_counter,
                         uint64_t elem_base, uint64_t sr_row_stride, const float *amax_in,
                         uint8_t *codes, uint8_t *scales, float *tensor_scale,
                         float *y_out);

int ref_quantize(const float *x, int64_t rows, int64_t k, int64_t ld,
                 int grid, int rht, uint64_t rht_seed,
                 int round_mode, uint64_t sr_seed, uint64_t sr_counter,
                 uint64_t elem_base, const float *amax_in,
                 uint8_t *codes, uint8_t *scales, float *tensor_scale,
                 float *y_out)
{
    return ref_quantize_strided(x, rows, k, ld, grid, rht, rht_seed, round_mode, sr_seed,
                                sr_counter, elem_base, (uint64_t)k, amax_in, codes, scales,
                                tensor_scale, y_out);
}

/* As ref_quantize; the SR element index is elem_base + r * sr_row_stride + j
 * (a segment that is one piece of a larger output tensor uses that tensor's
 * row length, so its random words are those of its place in the whole). */
int ref_quantize_strided(const float *x, int64_t rows, int64_t k, int64_t ld,
                         int grid, int rht, uint64_t rht_seed,
                         int round_mode, uint64_t sr_seed, uint64_t sr_counter,
                         uint64_t elem_base, uint64_t sr_row_stride, const float *amax_in,
                         uint8_t *codes, uint8_t *scales, float *tensor_scale,
                         float *y_out)
{
    if (k % 16 != 0) return -1;
    const float qmax = (float)ref_grid_qmax(grid);
    const int64_t nb = k / 16;
    int32_t d[16];
    double hd[16][16];
    ref_rht_signs(rht_seed, d);
    rht16_matrix(d, hd);

    float *y = (float *)malloc(sizeof(float) * (size_t)(rows * k > 0 ? rows * k : 1));
    if (!y) return -2;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float *src = x + r * ld + b * 16;
            float *dst = y + r * k + b * 16;
            if (rht) rht16_forward(src, hd, dst);
            else memcpy(dst, src, 16 * sizeof(float));
        }

    float A_t = 0.0f;
    if (amax_in) A_t = *amax_in;
    else for (int64_t i = 0; i < rows * k; ++i) if (fabsf(y[i]) > A_t) A_t = fabsf(y[i]);

    float S_enc = 1.0f, S_dec = 1.0f;
    if (A_t > 0.0f) {
        const float num = 448.0f * qmax;
        S_enc = num / A_t;
        if (S_enc > FLT_MAX) S_enc = FLT_MAX;
        S_dec = A_t / num;
    }
    *tensor_scale = S_dec;

    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float *blk = y + r * k + b * 16;
            float amax_b = 0.0f;
            for (int j = 0; j < 16; ++j) if (fabsf(blk[j]) > amax_b) amax_b = fabsf(blk[j]);
            const float s1 = amax_b / qmax;
            const float s2 = s1 * S_enc;
            const uint8_t e_b = ref_e4m3_encode(s2);
            scales[r * nb + b] = e_b;
            uint8_t *out = codes + r * k + b * 16;
            if (e_b == 0) { memset(out, 0, 16); continue; }
            float kb = S_enc / (float)ref_e4m3_decode(e_b);
            if (kb > FLT_MAX) kb = FLT_MAX;
            for (int j = 0; j < 16; ++j) {
                const float q = blk[j] * kb;
                float a = fabsf(q);
                if (a > qmax) a = qmax;
                int m;
                if (round_mode == REF_SR) {
                    const uint64_t i = elem_base + (uint64_t)r * sr_row_stride + (uint64_t)(b * 16 + j);
                    m = ref_round_sr(grid, a, ref_sr_bits(sr_seed, sr_counter, i));
                } else {
                    m = ref_round_rtne(grid, a);
                }
                out[j] = (uint8_t)((signbit(q) ? 8 : 0) | m);
            }
        }
    if (y_out) memcpy(y_out, y, sizeof(float) * (size_t)(rows * k));
    free(y);
    return 0;
}

/* A_t = max |y| over a rows x k matrix (blocks along k), y the rotated blocks
 * when rht is set -- the tensor amax step of ref_quantize on its own, so a
 * sample of rows can be quantized against the whole tensor's scale. */
float ref_tensor_amax(const float *x, int64_t rows, int64_t k, int64_t ld, int rht, uint64_t rht_seed)
{
    int32_t d[16];
    double hd[16][16];
    ref_rht_signs(rht_seed, d);
    rht16_matrix(d, hd);
    float A_t = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < k / 16; ++b) {
            float y[16];
            const float *src = x + r * ld + b * 16;
            if (rht) rht16_forward(src, hd, y);
            else memcpy(y, src, sizeof y);
            for (int j = 0; j < 16; ++j) if (fabsf(y[j]) > A_t) A_t = fabsf(y[j]);
        }
    return A_t;
}

/* ------------------------------------------------------------------------
 * Dequantization: value = v(m) * e_b * S_dec, exact in fp64 (v * e_b has at
 * most 7 significant bits, S_dec 24).  With inverse_rht set, each 16-block is
 * rotated back: x = diag(d) (1/4) H y.  Output fp64, rows x k.
 * ---------------------------------------------------------------------- */
void ref_dequantize(const uint8_t *codes, const uint8_t *scales, float tensor_scale,
                    int64_t rows, int64_t k, int grid, int inverse_rht,
                    uint64_t rht_seed, double *out)
{
    const int64_t nb = k / 16;
    int32_t d[16];
    ref_rht_signs(rht_seed, d);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const double e = ref_e4m3_decode(scales[r * nb + b]);
            double blk[16];
            for (int j = 0; j < 16; ++j) {
                const uint8_t c = codes[r * k + b * 16 + j];
                const double v = ref_grid_value(grid, c & 7);
                blk[j] = ((c & 8) ? -v : v) * e * (double)tensor_scale;
            }
            if (inverse_rht) {
                double xb[16];
                rht16_inverse(blk, d, xb);
                memcpy(blk, xb, sizeof xb);
            }
            memcpy(out + r * k + b * 16, blk, sizeof blk);
        }
}

/* ------------------------------------------------------------------------
 * GEMM of two dequantized operands, both stored with K contiguous:
 * C[m][n] = sum_k A[m][k] * B[n][k] in fp64 ([ZC] "The fix -- UFP4": the
 * quantized operands feed fwd_y, bwd_dx and bwd_dw).
 * ---------------------------------------------------------------------- */
void ref_gemm_f64(const double *A, const double *B, int64_t M, int64_t N, int64_t K, double *C)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t kk = 0; kk < K; ++kk) s += A[m * K + kk] * B[n * K + kk];
            C[m * N + n] = s;
        }
}

/* Same, for a list of (m, n) entries only (sampled checks at large sizes). */
void ref_gemm_entries(const double *A, const double *B, int64_t K,
                      const int64_t *mi, const int64_t *ni, int64_t count, double *out)
{
    for (int64_t t = 0; t < count; ++t) {
        double s = 0.0;
        const double *a = A + mi[t] * K, *b = B + ni[t] * K;
        for (int64_t kk = 0; kk < K; ++kk) s += a[kk] * b[kk];
        out[t] = s;
    }
}

/* ------------------------------------------------------------------------
 * Quality statistics of one quantization ([ZC] Key points, "The cause",
 * "Compounding decay" and "The RHT paradox"):
 *   sum_aq = <deq, A>, sum_aa = <A, A>, sum_err2 = ||A - deq||^2,
 *   alpha  = sum_aq / sum_aa  (the shrinkage factor in Q(A) = alpha A + R_A),
 *   sqnr_db = 10 log10(sum_aa / sum_err2),
 *   mean_bias = mean over elements with a != 0 of (v(m) - a), in grid units
 *               (negative = pulled toward zero).
 * A is the tensor actually quantized (the rotated one when RHT is on).  The
 * grid-unit magnitude is a = min(|A| / (e_b S_dec), qmax) in fp64, formed
 * from the stored scales only (it equals the quantizer's min(|q|, qmax) up to
 * the rounding of S_enc and q).  Blocks with e_b == 0 are left out of the bias.
 * out = {alpha, sqnr_db, mean_bias, sum_aq, sum_aa, sum_err2, bias_count}.
 * ---------------------------------------------------------------------- */
void ref_stats(const float *A, const uint8_t *codes, const uint8_t *scales,
               float tensor_scale, int64_t rows, int64_t k, int grid, double out[7])
{
    const int64_t nb = k / 16;
    const double qmax = ref_grid_qmax(grid);
    double saq = 0, saa = 0, se2 = 0, bias = 0, cnt = 0;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const double e = ref_e4m3_decode(scales[r * nb + b]);
            for (int j = 0; j < 16; ++j) {
                const int64_t i = r * k + b * 16 + j;
                const uint8_t c = codes[i];
                const double v = ref_grid_value(grid, c & 7);
                const double dq = ((c & 8) ? -v : v) * e * (double)tensor_scale;
                const double a = (double)A[i];
                saq += dq * a; saa += a * a; se2 += (a - dq) * (a - dq);
                if (e > 0.0) {
                    double g = fabs(a) / (e * (double)tensor_scale);
                    if (g > qmax) g = qmax;
                    if (g != 0.0) { bias += v - g; cnt += 1.0; }
                }
            }
        }
    out[0] = saa > 0 ? saq / saa : 1.0;
    out[1] = se2 > 0 ? 10.0 * log10(saa / se2) : INFINITY;
    out[2] = cnt > 0 ? bias / cnt : 0.0;
    out[3] = saq; out[4] = saa; out[5] = se2; out[6] = cnt;
}

/* ------------------------------------------------------------------------
 * MXFP4, a comparison format of the pages ([HP] technical approach, the
 * "comparison formats" line: E2M1-based NVFP4 and MXFP4); the pages give no
 * details.  READING: the OCP Microscaling (MX) definition of MXFP4 --
 *   blocks of 32 elements along k share one E8M0 scale X = 2^s with
 *   s = floor(log2(max |y|)) - 2  (2 = the exponent of E2M1's largest
 *   normal, 6 = 1.5 * 2^2), clamped to the E8M0 range [-127, 127]; a block
 *   whose max is 0 stores s = -127;
 *   q = y / X (exact: a power-of-two scaling, rounded once to fp32);
 *   code = signbit(q) << 3 | E2M1 rounding of min(|q|, 6): RTNE, or SR with
 *   the same Philox words as ref_quantize;
 *   no tensor-level scale.
 * With rht set each 16-element half of a block is rotated as in
 * ref_quantize.  Outputs: codes rows x k (one code per byte), scales
 * rows x k/32 (biased exponent bytes s + 127).  SR element index r * k + j.
 * Returns 0, or -1 on k % 32 != 0.
 * ---------------------------------------------------------------------- */
double ref_e8m0_decode(uint8_t b)
{
    if (b == 255) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* floor(log2(a)) - 2 clamped to [-127, 127]; -127 for a == 0. */
int ref_mx_shared_exp(float a)
{
    if (!(a > 0.0f)) return -127;
    int e;
    frexp((double)a, &e);          /* a = f 2^e, f in [0.5, 1): floor(log2 a) = e - 1 */
    int s = (e - 1) - 2;
    if (s < -127) s = -127;
    if (s > 127) s = 127;
    return s;
}

int ref_quantize_mx(const float *x, int64_t rows, int64_t k, int64_t ld, int rht, uint64_t rht_seed,
                    int round_mode, uint64_t sr_seed, uint64_t sr_counter,
                    uint8_t *codes, uint8_t *scales, float *y_out)
{
    if (k % 32 != 0) return -1;
    const int64_t nb = k / 32;
    int32_t d[16];
    double hd[16][16];
    ref_rht_signs(rht_seed, d);
    rht16_matrix(d, hd);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            float blk[32];
            for (int h = 0; h < 2; ++h) {
                const float *src = x + r * ld + b * 32 + 16 * h;
                if (rht) rht16_forward(src, hd, blk + 16 * h);
                else memcpy(blk + 16 * h, src, 16 * sizeof(float));
            }
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) if (fabsf(blk[j]) > amax) amax = fabsf(blk[j]);
            const int s = ref_mx_shared_exp(amax);
            scales[r * nb + b] = (uint8_t)(s + 127);
            for (int j = 0; j < 32; ++j) {
                const float q = (float)ldexp((double)blk[j], -s);
                float a = fabsf(q);
                if (a > 6.0f) a = 6.0f;
                int m;
                if (round_mode == REF_SR) {
                    const uint64_t i = (uint64_t)r * (uint64_t)k + (uint64_t)(b * 32 + j);
                    m = ref_round_sr(REF_E2M1, a, ref_sr_bits(sr_seed, sr_counter, i));
                } else {
                    m = ref_round_rtne(REF_E2M1, a);
                }
                codes[r * k + b * 32 + j] = (uint8_t)((signbit(q) ? 8 : 0) | m);
            }
            if (y_out) memcpy(y_out + r * k + b * 32, blk, sizeof blk);
        }
    return 0;
}

/* MXFP4 dequantization: v(m) * 2^s, exact in fp64; inverse_rht rotates each
 * 16-element half back.  Output fp64 rows x k. */
void ref_dequantize_mx(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t k,
                       int inverse_rht, uint64_t rht_seed, double *out)
{
    const int64_t nb = k / 32;
    int32_t d[16];
    ref_rht_signs(rht_seed, d);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const double X = ref_e8m0_decode(scales[r * nb + b]);
            double blk[32];
            for (int j = 0; j < 32; ++j) {
                const uint8_t c = codes[r * k + b * 32 + j];
                const double v = ref_grid_value(REF_E2M1, c & 7);
                blk[j] = ((c & 8) ? -v : v) * X;
            }
            if (inverse_rht)
                for (int h = 0; h < 2; ++h) {
                    double xb[16];
                    rht16_inverse(blk + 16 * h, d, xb);
                    memcpy(blk + 16 * h, xb, sizeof xb);
                }
            memcpy(out + r * k + b * 32, blk, sizeof blk);
        }
}

/* ref_stats for MXFP4: the grid-unit magnitude is a = min(|A| / X, 6). */
void ref_stats_mx(const float *A, const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t k,
                  double out[7])
{
    const int64_t nb = k / 32;
    double saq = 0, saa = 0, se2 = 0, bias = 0, cnt = 0;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const double X = ref_e8m0_decode(scales[r * nb + b]);
            for (int j = 0; j < 32; ++j) {
                const int64_t i = r * k + b * 32 + j;
                const uint8_t c = codes[i];
                const double v = ref_grid_value(REF_E2M1, c & 7);
                const double dq = ((c & 8) ? -v : v) * X;
                const double a = (double)A[i];
                saq += dq * a; saa += a * a; se2 += (a - dq) * (a - dq);
                double g = fabs(a) / X;
                if (g > 6.0) g = 6.0;
                if (g != 0.0) { bias += v - g; cnt += 1.0; }
            }
        }
    out[0] = saa > 0 ? saq / saa : 1.0;
    out[1] = se2 > 0 ? 10.0 * log10(saa / se2) : INFINITY;
    out[2] = cnt > 0 ? bias / cnt : 0.0;
    out[3] = saq; out[4] = saa; out[5] = se2; out[6] = cnt;
}
