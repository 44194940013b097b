/*
 * hlq_oracle.c -- CPU oracle of the HLQ/HOT backward pass of one linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg call this file; the product library never links, loads or
 * calls it, and it shares no code, header or table with the CUDA sources.
 *
 * It is written to be checked by eye, not to be fast: explicit 16x16 Hadamard
 * matrices (no butterfly), exact multi-word accumulation for the transform,
 * scalar quantizers, an int64 GEMM and an fp64 dequant; one thread.
 *
 * What it computes (layer y = x . w^T, x [T,Cin], w [Cout,Cin], g_y [T,Cout]):
 *
 *  - "HLQ: Fast and Efficient Backpropagation via Hadamard Low-rank
 *    Quantization" (Kim & Park), TL;DR: g_x = g_y . w computed with 4-bit
 *    Hadamard quantization (HQ), and g_w = (1/B) gbar_y^T . xbar computed with
 *    the Hadamard low-rank approximation (HLA) and int8 arithmetic, with the
 *    stored activation compressed at forward time (ACBP).
 *  - "HOT: Hadamard-based Optimized Training" (atlas summary), Approach:
 *    int4 HQ on the activation-gradient path, HLA + int8 on the weight-gradient
 *    path, the saved activation compressed when the forward pass runs, a per-token
 *    vs per-tensor quantizer chosen per layer.
 *
 * Readings where the pages are silent (block 16, rank 8, int4 range [-7,7],
 * int8 range [-127,127], scale = RN(amax/qmax), Philox4x32-10 stochastic
 * rounding keyed on (seed, element index), lowest-sequency rows for HLA,
 * B = 16 = the Hadamard block, the transform result defined as the exact sum
 * rounded once to fp32) are the ones the design notes list.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_NONFINITE -2

/* ------------------------------------------------------------------------- */
/* Hadamard matrix H16 (Sylvester construction) and its sequency ordering.    */
/* "HLQ ..." section "Hadamard Transform"; the Walsh functions ordered by the  */
/* number of sign changes along a row.                                        */
/* ------------------------------------------------------------------------- */

/* H[i][j] = (-1)^(number of bits set in both i and j). */
static int hadamard_entry(int i, int j)
{
    int both = i & j, ones = 0;
    while (both) {
        ones += both & 1;
        both >>= 1;
    }
    return (ones % 2 == 0) ? 1 : -1;
}

int orc_hadamard16(int32_t *H)
{
    for (int i = 0; i < 16; ++i)
        for (int j = 0; j < 16; ++j)
            H[i * 16 + j] = hadamard_entry(i, j);
    return ORC_OK;
}

/* sigma[k] = the Sylvester row whose entries change sign exactly k times. */
int orc_sequency_order(int32_t *sigma)
{
    int seen[16] = {0};
    for (int i = 0; i < 16; ++i) {
        int changes = 0;
        for (int j = 1; j < 16; ++j)
            if (hadamard_entry(i, j) != hadamard_entry(i, j - 1))
                ++changes;
        if (seen[changes])
            return ORC_ERR_ARG;
        seen[changes] = 1;
        sigma[changes] = i;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Exact sum of +-fp32 values, rounded once to fp32 (nearest, ties to even).  */
/* Every finite fp32 value is m * 2^(pos-149) with m < 2^24 and pos >= 0; the */
/* sum is kept as a 320-bit integer in units of 2^-149 (a long accumulator).  */
/* ------------------------------------------------------------------------- */

#define NLIMB 10

typedef struct {
    uint64_t limb[NLIMB]; /* 32 payload bits per limb after normalisation */
} longacc;

static void decompose(float v, int *neg, uint32_t *m, int *pos)
{
    uint32_t b;
    memcpy(&b, &v, sizeof b);
    uint32_t e = (b >> 23) & 0xffu, frac = b & 0x7fffffu;
    *neg = (int)(b >> 31);
    if (e == 0) { /* zero or subnormal: frac * 2^-149 */
        *m = frac;
        *pos = 0;
    } else { /* normal: (2^23 + frac) * 2^(e-150) */
        *m = frac | 0x800000u;
        *pos = (int)e - 1;
    }
}

static int is_finite_f32(float v)
{
    uint32_t b;
    memcpy(&b, &v, sizeof b);
    return ((b >> 23) & 0xffu) != 0xffu;
}

static void acc_add(longacc *a, uint32_t m, int pos)
{
    int li = pos / 32, sh = pos % 32;
    uint64_t v = (uint64_t)m << sh; /* below 2^56 */
    a->limb[li] += v & 0xffffffffu;
    a->limb[li + 1] += v >> 32;
}

static void acc_normalise(longacc *a)
{
    uint64_t carry = 0;
    for (int i = 0; i < NLIMB; ++i) {
        uint64_t t = a->limb[i] + carry;
        a->limb[i] = t & 0xffffffffu;
        carry = t >> 32;
    }
}

static int acc_cmp(const longacc *a, const longacc *b)
{
    for (int i = NLIMB - 1; i >= 0; --i) {
        if (a->limb[i] > b->limb[i])
            return 1;
        if (a->limb[i] < b->limb[i])
            return -1;
    }
    return 0;
}

/* r = a - b for normalised a >= b */
static void acc_sub(longacc *r, const longacc *a, const longacc *b)
{
    int64_t borrow = 0;
    for (int i = 0; i < NLIMB; ++i) {
        int64_t t = (int64_t)a->limb[i] - (int64_t)b->limb[i] - borrow;
        borrow = 0;
        if (t < 0) {
            t += (int64_t)1 << 32;
            borrow = 1;
        }
        r->limb[i] = (uint64_t)t;
    }
}

static int acc_bit(const longacc *a, int i)
{
    return (int)((a->limb[i / 32] >> (i % 32)) & 1u);
}

static int acc_msb(const longacc *a)
{
    for (int i = NLIMB - 1; i >= 0; --i)
        if (a->limb[i])
            for (int b = 31; b >= 0; --b)
                if ((a->limb[i] >> b) & 1u)
                    return i * 32 + b;
    return -1;
}

/* any bit set strictly below position p */
static int acc_any_below(const longacc *a, int p)
{
    for (int i = 0; i < NLIMB && i * 32 < p; ++i) {
        int hi = p - i * 32; /* bits [0, hi) of this limb count */
        uint64_t mask = (hi >= 32) ? 0xffffffffu : (((uint64_t)1 << hi) - 1u);
        if (a->limb[i] & mask)
            return 1;
    }
    return 0;
}

/* Round magnitude*2^-149 to the nearest fp32, ties to even. */
static float acc_round(const longacc *mag, int neg)
{
    int p = acc_msb(mag);
    if (p < 0)
        return 0.0f; /* an exact zero sum is +0 */
    float r;
    if (p <= 23) {
        uint32_t v = 0;
        for (int b = p; b >= 0; --b)
            v = (v << 1) | (uint32_t)acc_bit(mag, b);
        r = ldexpf((float)v, -149); /* exact: v < 2^24 in units of 2^-149 */
    } else {
        int shift = p - 23;
        uint32_t keep = 0;
        for (int b = p; b >= shift; --b)
            keep = (keep << 1) | (uint32_t)acc_bit(mag, b);
        int half = acc_bit(mag, shift - 1);
        int sticky = acc_any_below(mag, shift - 1);
        if (half && (sticky || (keep & 1u)))
            ++keep;
        if (keep == (1u << 24)) {
            keep >>= 1;
            ++shift;
        }
        r = ldexpf((float)keep, shift - 149);
    }
    return neg ? -r : r;
}

/* RN_f32( sum_j h[j] * v[j*stride] ), h[j] in {+1,-1}, computed exactly. */
static float exact_signed_sum(const int32_t *h, const float *v, ptrdiff_t stride,
                              int n)
{
    longacc pos_part, neg_part, mag;
    memset(&pos_part, 0, sizeof pos_part);
    memset(&neg_part, 0, sizeof neg_part);
    for (int j = 0; j < n; ++j) {
        int neg, pos;
        uint32_t m;
        decompose(v[j * stride], &neg, &m, &pos);
        if (m == 0)
            continue;
        if (h[j] < 0)
            neg = !neg;
        acc_add(neg ? &neg_part : &pos_part, m, pos);
    }
    acc_normalise(&pos_part);
    acc_normalise(&neg_part);
    if (acc_cmp(&pos_part, &neg_part) >= 0) {
        acc_sub(&mag, &pos_part, &neg_part);
        return acc_round(&mag, 0);
    }
    acc_sub(&mag, &neg_part, &pos_part);
    return acc_round(&mag, 1);
}

/* Exposed for the tests: RN_f32 of the exact signed sum of n values. */
float orc_exact_sum_f32(const int32_t *h, const float *v, int n)
{
    return exact_signed_sum(h, v, 1, n);
}

/* ------------------------------------------------------------------------- */
/* Transforms.                                                                */
/* ------------------------------------------------------------------------- */

/*
 * HQ transform along the contraction dim Cout, in blocks of 16, rows of H in
 * Sylvester order ("HLQ ..." sections "Hadamard Transform" and "Alternative
 * Optimization Technique: Hadamard Quantization").
 *   axis 0: src [rows, cols] with the blocks along cols (g_y, [T, Cout]):
 *           Y[r, 16b+i] = RN_f32( sum_j H[i][j] src[r, 16b+j] )
 *   axis 1: src [rows, cols] with the blocks along rows (w, [Cout, Cin]):
 *           Y[16b+i, c] = RN_f32( sum_j H[i][j] src[16b+j, c] )
 * Y has the layout of src.
 */
int orc_hq_transform(const float *src, int64_t rows, int64_t cols, int axis,
                     float *Y)
{
    int32_t H[256];
    orc_hadamard16(H);
    if (axis == 0) {
        if (cols % 16)
            return ORC_ERR_ARG;
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t b = 0; b < cols / 16; ++b)
                for (int i = 0; i < 16; ++i)
                    Y[r * cols + 16 * b + i] = exact_signed_sum(
                        &H[i * 16], &src[r * cols + 16 * b], 1, 16);
    } else if (axis == 1) {
        if (rows % 16)
            return ORC_ERR_ARG;
        for (int64_t b = 0; b < rows / 16; ++b)
            for (int i = 0; i < 16; ++i)
                for (int64_t c = 0; c < cols; ++c)
                    Y[(16 * b + i) * cols + c] = exact_signed_sum(
                        &H[i * 16], &src[16 * b * cols + c], (ptrdiff_t)cols,
                        16);
    } else {
        return ORC_ERR_ARG;
    }
    return ORC_OK;
}

/*
 * HLA transform along the token dim ("HLQ ..." section "Analysis on Hadamard
 * Low-rank Approximation for Backpropagation"; HOT Approach): per block of 16
 * tokens keep the `rank` lowest-sequency Hadamard rows.
 *   src [T, C]  ->  out [C, T*rank/16] (token dim contiguous):
 *   out[c, rank*b + k] = RN_f32( sum_j H[sigma(k)][j] src[16b+j, c] ), k < rank
 */
int orc_hla_transform(const float *src, int64_t T, int64_t C, int rank,
                      float *out)
{
    int32_t H[256], sigma[16];
    if (T % 16 || rank < 1 || rank > 16)
        return ORC_ERR_ARG;
    orc_hadamard16(H);
    if (orc_sequency_order(sigma) != ORC_OK)
        return ORC_ERR_ARG;
    int64_t Tp = T / 16 * rank;
    for (int64_t b = 0; b < T / 16; ++b)
        for (int k = 0; k < rank; ++k)
            for (int64_t c = 0; c < C; ++c)
                out[c * Tp + rank * b + k] = exact_signed_sum(
                    &H[sigma[k] * 16], &src[16 * b * C + c], (ptrdiff_t)C, 16);
    return ORC_OK;
}

/* The same two transforms with plain fp64 accumulation and no rounding to
 * fp32: the "quantization off" pipeline used only by the closed-form checks. */
int orc_hq_transform_f64(const double *src, int64_t rows, int64_t cols,
                         int axis, double *Y)
{
    int32_t H[256];
    orc_hadamard16(H);
    if (axis == 0) {
        if (cols % 16)
            return ORC_ERR_ARG;
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t b = 0; b < cols / 16; ++b)
                for (int i = 0; i < 16; ++i) {
                    double s = 0.0;
                    for (int j = 0; j < 16; ++j)
                        s += H[i * 16 + j] * src[r * cols + 16 * b + j];
                    Y[r * cols + 16 * b + i] = s;
                }
    } else if (axis == 1) {
        if (rows % 16)
            return ORC_ERR_ARG;
        for (int64_t b = 0; b < rows / 16; ++b)
            for (int i = 0; i < 16; ++i)
                for (int64_t c = 0; c < cols; ++c) {
                    double s = 0.0;
                    for (int j = 0; j < 16; ++j)
                        s += H[i * 16 + j] * src[(16 * b + j) * cols + c];
                    Y[(16 * b + i) * cols + c] = s;
                }
    } else {
        return ORC_ERR_ARG;
    }
    return ORC_OK;
}

int orc_hla_transform_f64(const double *src, int64_t T, int64_t C, int rank,
                          double *out)
{
    int32_t H[256], sigma[16];
    if (T % 16 || rank < 1 || rank > 16)
        return ORC_ERR_ARG;
    orc_hadamard16(H);
    if (orc_sequency_order(sigma) != ORC_OK)
        return ORC_ERR_ARG;
    int64_t Tp = T / 16 * rank;
    for (int64_t b = 0; b < T / 16; ++b)
        for (int k = 0; k < rank; ++k)
            for (int64_t c = 0; c < C; ++c) {
                double s = 0.0;
                for (int j = 0; j < 16; ++j)
                    s += H[sigma[k] * 16 + j] * src[(16 * b + j) * C + c];
                out[c * Tp + rank * b + k] = s;
            }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel Random Numbers: As    */
/* Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies, with the */
/* two key words bumped by the Weyl constants between rounds.                 */
/* ------------------------------------------------------------------------- */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                       uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
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

/* The random word of element e in stream `stream`: word e%4 of the block at
 * counter (e/4 low, e/4 high, stream, 0) under key (seed low, seed high). */
uint32_t orc_philox_word(uint64_t seed, uint32_t stream, uint64_t e)
{
    uint32_t ctr[4] = {(uint32_t)(e / 4), (uint32_t)((e / 4) >> 32), stream, 0};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[e % 4];
}

/* ------------------------------------------------------------------------- */
/* Quantizers.                                                                */
/* ------------------------------------------------------------------------- */

#define ORC_RNE 0
#define ORC_SR 1

/* One code: x = RN_f32(y / s); round to an integer (ties to even, or
 * stochastically: floor(x) + [u < x - floor(x)] with u = (word >> 8) * 2^-24);
 * clamp to [-qmax, qmax].  s == 0 gives code 0. */
static int quant_one(float y, float s, int qmax, int rnd, uint32_t word)
{
    if (s == 0.0f)
        return 0;
    float x = y / s;
    float r;
    if (rnd == ORC_RNE) {
        r = rintf(x); /* default rounding mode: nearest, ties to even */
    } else {
        float f = floorf(x);
        float frac = x - f; /* fp32 difference (exact unless -2^-24 < x < 0) */
        float u = (float)(word >> 8) * 0x1p-24f;
        r = f + ((u < frac) ? 1.0f : 0.0f);
    }
    if (r > (float)qmax)
        r = (float)qmax;
    if (r < (float)-qmax)
        r = (float)-qmax;
    return (int)r;
}

/*
 * HQ int4 quantizer of the transformed tensor Y [rows, cols] (layer-wise
 * quantizer selection of HOT: gran 1 = one scale per row (per token),
 * gran 0 = one scale for the tensor).  s = RN_f32(amax / 7).  Element
 * (r, c) draws Philox word e = r*cols + c of `stream`.
 * codes [rows, cols] int8 in [-7, 7]; scales [rows] or [1].
 *
 * orc_hq_quantize_rows quantizes a subset of the rows of a larger tensor:
 * Y holds `nrows` rows whose row numbers in the full tensor are row_ids[],
 * and, for gran 0, tensor_amax is the max |Y| over the full tensor.
 */
int orc_hq_quantize_rows(const float *Y, int64_t nrows, int64_t cols,
                         const int64_t *row_ids, int gran, float tensor_amax,
                         int rnd, uint64_t seed, uint32_t stream,
                         int8_t *codes, float *scales)
{
    const int qmax = 7;
    for (int64_t i = 0; i < nrows * cols; ++i)
        if (!is_finite_f32(Y[i]))
            return ORC_ERR_NONFINITE;
    for (int64_t r = 0; r < nrows; ++r) {
        float amax = tensor_amax;
        if (gran == 1) {
            amax = 0.0f;
            for (int64_t c = 0; c < cols; ++c)
                if (fabsf(Y[r * cols + c]) > amax)
                    amax = fabsf(Y[r * cols + c]);
        }
        float s = amax / (float)qmax;
        if (gran == 1)
            scales[r] = s;
        else if (r == 0)
            scales[0] = s;
        int64_t row = row_ids ? row_ids[r] : r;
        for (int64_t c = 0; c < cols; ++c) {
            uint64_t e = (uint64_t)(row * cols + c);
            uint32_t word = (rnd == ORC_SR) ? orc_philox_word(seed, stream, e) : 0;
            codes[r * cols + c] =
                (int8_t)quant_one(Y[r * cols + c], s, qmax, rnd, word);
        }
    }
    return ORC_OK;
}

int orc_hq_quantize(const float *Y, int64_t rows, int64_t cols, int gran,
                    int rnd, uint64_t seed, uint32_t stream, int8_t *codes,
                    float *scales)
{
    float tensor_amax = 0.0f;
    for (int64_t i = 0; i < rows * cols; ++i) {
        if (!is_finite_f32(Y[i]))
            return ORC_ERR_NONFINITE;
        if (fabsf(Y[i]) > tensor_amax)
            tensor_amax = fabsf(Y[i]);
    }
    return orc_hq_quantize_rows(Y, rows, cols, NULL, gran, tensor_amax, rnd,
                                seed, stream, codes, scales);
}

/* Largest |v| of an fp32 array. */
float orc_amax(const float *v, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i)
        if (fabsf(v[i]) > amax)
            amax = fabsf(v[i]);
    return amax;
}

/* Round-to-nearest-even quantizer with one scale per tensor:
 * s = RN_f32(amax / qmax), codes clamp(rint(RN_f32(v / s)), -qmax, qmax).
 * qmax = 127 gives the int8 HLA operands; qmax = 7 the int4 form of the
 * stored activation (HLQ TL;DR: int4 activation compression). */
int orc_rne_quantize(const float *v, int64_t n, int qmax, int8_t *codes, float *scale)
{
    if (qmax != 7 && qmax != 127)
        return ORC_ERR_ARG;
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        if (!is_finite_f32(v[i]))
            return ORC_ERR_NONFINITE;
        if (fabsf(v[i]) > amax)
            amax = fabsf(v[i]);
    }
    float s = amax / (float)qmax;
    *scale = s;
    for (int64_t i = 0; i < n; ++i)
        codes[i] = (int8_t)quant_one(v[i], s, qmax, ORC_RNE, 0);
    return ORC_OK;
}

/* int8 quantizer of the HLA operands: orc_rne_quantize with qmax = 127. */
int orc_int8_quantize(const float *v, int64_t n, int8_t *codes, float *scale)
{
    return orc_rne_quantize(v, n, 127, codes, scale);
}

/* Nibble packing of int4 codes (two's complement; element 2k in the low
 * nibble, 2k+1 in the high nibble), for the compact storage format. */
int orc_pack_int4(const int8_t *codes, int64_t n, uint8_t *packed)
{
    if (n % 2)
        return ORC_ERR_ARG;
    for (int64_t k = 0; k < n / 2; ++k)
        packed[k] = (uint8_t)(((uint8_t)codes[2 * k] & 0x0fu) |
                              (((uint8_t)codes[2 * k + 1] & 0x0fu) << 4));
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Integer GEMM and dequantisation.                                           */
/* ------------------------------------------------------------------------- */

/* C[m, n] = sum_k A[m, k] * B[n, k]; A [M, K], B [N, K] int8; int64 sums. */
void orc_gemm_i64(const int8_t *A, const int8_t *B, int64_t M, int64_t N,
                  int64_t K, int64_t *C)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k)
                s += (int64_t)A[m * K + k] * (int64_t)B[n * K + k];
            C[m * N + n] = s;
        }
}

/* g_x[t, i] = acc[t, i] * s_gy[t or 0] * s_w / 16  (fp64).  The 1/16 undoes
 * H^T H = 16 I of the unnormalised transform applied to both operands. */
void orc_dequant_gx(const int64_t *acc, const float *s_gy, int gran_gy,
                    float s_w, int64_t T, int64_t Cin, double *g_x)
{
    for (int64_t t = 0; t < T; ++t) {
        double sg = (double)s_gy[gran_gy == 1 ? t : 0];
        for (int64_t i = 0; i < Cin; ++i)
            g_x[t * Cin + i] = (double)acc[t * Cin + i] * sg * (double)s_w / 16.0;
    }
}

/* g_w[o, i] = acc[o, i] * s_g * s_x / 16  (fp64): the 1/B of
 * g_w = (1/B) gbar_y^T xbar with B the Hadamard block size. */
void orc_dequant_gw(const int64_t *acc, float s_g, float s_x, int64_t Cout,
                    int64_t Cin, double *g_w)
{
    for (int64_t o = 0; o < Cout; ++o)
        for (int64_t i = 0; i < Cin; ++i)
            g_w[o * Cin + i] = (double)acc[o * Cin + i] * (double)s_g *
                               (double)s_x / 16.0;
}

/* Per-channel scales of the stored activation: g_w[o, i] = acc[o, i] * s_g *
 * s_x[i] / 16 (fp64).  A scale per input channel i is a scale per column of
 * g_w, so it factors out of the contraction over tokens exactly like the
 * per-tensor one. */
void orc_dequant_gw_cols(const int64_t *acc, float s_g, const float *s_x,
                         int64_t Cout, int64_t Cin, double *g_w)
{
    for (int64_t o = 0; o < Cout; ++o)
        for (int64_t i = 0; i < Cin; ++i)
            g_w[o * Cin + i] = (double)acc[o * Cin + i] * (double)s_g *
                               (double)s_x[i] / 16.0;
}
