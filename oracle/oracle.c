/*
 * CPU oracle for the quantized decode GEMV: block formats, quantizers,
 * dequantizers, fp64 GEMV and per-sub-block integer sums.
 *
 * TEST INFRASTRUCTURE.  Plain loops, no blocking, no SIMD, no reordering
 * beyond what the definitions state.  Block fields are read and written at
 * explicit byte offsets so the layout can be checked against the pages by eye.
 *
 * Precision: every decision that produces an integer code (a quantized value,
 * a 6-bit scale) is taken in fp32 with IEEE round-to-nearest operations and
 * no fused multiply-add (built with -ffp-contract=off), because that is the
 * precision the pages' kernels use; the GEMV itself is evaluated in fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdlib.h>
#include <string.h>

#include "qmv_oracle.h"

/* ------------------------------------------------------------------------
 * Block layouts.
 *
 * block_q4_0  (18 B, 32 weights)  "mul_mat_vec_q" page, section
 *   "权重的排法": half d at 0, qs[16] at 2.  Byte i holds element i in its
 *   low nibble and element i+16 in its high nibble (vec_dot_q4_0_q8_1 reads
 *   u[2i] = x[iqs+i], u[2i+1] = x[iqs+i+QI4_0]).  w = d*(q-8).
 * block_q4_K  (144 B, 256 weights) "GGUF 量化内幕 第16章" 16.1.2: half d at 0,
 *   half dmin at 2, scales[12] at 4, qs[128] at 16 (the order of the struct
 *   carrying the static_assert; the mul_mat_vec_q page prints another order
 *   and this reading takes the asserted one).  Element order from
 *   dequantize_row_q4_K (16.2.1): chunk c = 0..3 holds qs[32c..32c+31];
 *   low nibbles are elements 64c+l (sub-block 2c), high nibbles elements
 *   64c+32+l (sub-block 2c+1).  w = d*sc*q - dmin*m.
 * block_q6_K  (210 B, 256 weights) mul_mat_vec_q page (Q6_K snippet and the
 *   format table: 16 sub-blocks, low 4 bits in ql, high 2 bits in qh, value
 *   stored as 0..63 with offset 32).  Reading of the byte order: ql[128] at
 *   0, qh[64] at 128, int8 scales[16] at 192, half d at 208; element e with
 *   h = e/128, r = e%128, g = r/32, l = r%32 takes the (g>>1) nibble of
 *   ql[64h + 32(g&1) + l] and bits 2g..2g+1 of qh[32h + l]; sub-block e/16.
 *   w = d*sc*(v-32).
 * block_q8_1  (36 B, 32 values) mul_mat_vec_q page, section "激活的量化":
 *   half d at 0, half s at 2, int8 qs[32] at 4.
 * ---------------------------------------------------------------------- */

#define QK4_0 32
#define QK_K 256
#define QK8_1 32
#define ROW_PAD 512 /* MATRIX_ROW_PADDING */

#define Q4_0_BYTES 18
#define Q4_K_BYTES 144
#define Q6_K_BYTES 210
#define Q8_1_BYTES 36

_Static_assert(2 + QK4_0 / 2 == Q4_0_BYTES, "block_q4_0 is 18 bytes");
_Static_assert(2 * 2 + 12 + QK_K / 2 == Q4_K_BYTES, "block_q4_K is 144 bytes");
_Static_assert(QK_K / 2 + QK_K / 4 + QK_K / 16 + 2 == Q6_K_BYTES, "block_q6_K is 210 bytes");
_Static_assert(2 * 2 + QK8_1 == Q8_1_BYTES, "block_q8_1 is 36 bytes");

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }
static double h2d(const uint8_t *p) { return (double)oracle_f16_to_f32(rd16(p)); }

int64_t oracle_block_elems(int type)
{
    switch (type) {
    case ORACLE_Q4_0: return QK4_0;
    case ORACLE_Q4_K: return QK_K;
    case ORACLE_Q6_K: return QK_K;
    case ORACLE_Q8_1: return QK8_1;
    default: return 0;
    }
}

int64_t oracle_block_bytes(int type)
{
    switch (type) {
    case ORACLE_Q4_0: return Q4_0_BYTES;
    case ORACLE_Q4_K: return Q4_K_BYTES;
    case ORACLE_Q6_K: return Q6_K_BYTES;
    case ORACLE_Q8_1: return Q8_1_BYTES;
    default: return 0;
    }
}

int64_t oracle_row_bytes(int type, int64_t K)
{
    int64_t qk = oracle_block_elems(type);
    if (qk == 0) return -1;
    if (K <= 0 || K % qk) return -2;
    return K / qk * oracle_block_bytes(type);
}

int64_t oracle_q8_1_padded_k(int64_t K) { return (K + ROW_PAD - 1) / ROW_PAD * ROW_PAD; }

static int weight_type_ok(int t) { return t == ORACLE_Q4_0 || t == ORACLE_Q4_K || t == ORACLE_Q6_K; }

/* Clamp a rounded float into [lo, hi] and convert to int (inputs are finite
 * or +-inf; the comparisons keep the conversion defined). */
static int clamp_round(float z, float lo, float hi)
{
    float r = roundf(z); /* C roundf: halfway cases away from zero */
    if (r < lo) r = lo;
    if (r > hi) r = hi;
    return (int)r;
}

/* ------------------------------------------------------------------------
 * q8_1 activation quantization ("mul_mat_vec_q" page, quantize_q8_1 kernel).
 * Per 32-value block: amax = max|x|, d = amax/127 (fp32), q = round(x/d).
 * Values past K (the 512-padding) read as 0.
 * Readings:
 *   - s: the struct comment says s = d*sum(q) while the printed kernel stores
 *     the float sum of x; this oracle stores half(d * sum(q)) with d the fp32
 *     scale and sum(q) the exact integer sum.
 *   - the printed zero test is amax == 0; when amax is a subnormal so small
 *     that amax/127 underflows to 0 the printed division is undefined, so the
 *     test is taken on d == 0 instead, and q is clamped to [-127, 127] (only
 *     subnormal blocks can round past 127).  For every normal input both
 *     readings agree.
 * ---------------------------------------------------------------------- */
int oracle_quantize_q8_1(const float *x, int64_t K, int64_t ncols, int64_t ldx, uint8_t *xq)
{
    if (!x || !xq) return -3;
    if (K <= 0 || ncols <= 0 || ldx < K) return -2;
    int64_t kp = oracle_q8_1_padded_k(K);
    int64_t nb = kp / QK8_1;
    for (int64_t c = 0; c < ncols; ++c) {
        const float *xc = x + c * ldx;
        for (int64_t b = 0; b < nb; ++b) {
            uint8_t *blk = xq + (c * nb + b) * Q8_1_BYTES;
            float v[QK8_1];
            float amax = 0.0f;
            for (int i = 0; i < QK8_1; ++i) {
                int64_t k = b * QK8_1 + i;
                v[i] = k < K ? xc[k] : 0.0f;
                float a = fabsf(v[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int sum = 0;
            for (int i = 0; i < QK8_1; ++i) {
                int q = (d == 0.0f) ? 0 : clamp_round(v[i] / d, -127.0f, 127.0f);
                blk[4 + i] = (uint8_t)(int8_t)q;
                sum += q;
            }
            wr16(blk + 0, oracle_f32_to_f16(d));
            wr16(blk + 2, oracle_f32_to_f16(d * (float)sum));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Weight quantizers.
 * ---------------------------------------------------------------------- */

/* Q4_0: "解构LLM" page, section "量化格式": scale = max_abs/7,
 * q = round(v/scale) + 8 (clamped to the 4-bit range), d stored as half. */
static void quantize_block_q4_0(const float *v, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < QK4_0; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 7.0f;
    int q[QK4_0];
    for (int i = 0; i < QK4_0; ++i)
        q[i] = (d == 0.0f) ? 8 : clamp_round(v[i] / d, -8.0f, 7.0f) + 8;
    wr16(blk, oracle_f32_to_f16(d));
    for (int i = 0; i < QK4_0 / 2; ++i)
        blk[2 + i] = (uint8_t)(q[i] | (q[i + 16] << 4));
}

/* Q4_K 6-bit scale/min packing: the inverse of the unpack printed on the
 * mul_mat_vec_q page ("一次 vec_dot 的解剖"), which reads sub-block sb as
 *   sb < 4:  sc = s[sb] & 63,                         m = s[sb+4] & 63
 *   sb >= 4: sc = (s[sb+4] & 15) | ((s[sb-4] >> 6) << 4),
 *            m  = (s[sb+4] >> 4) | ((s[sb]   >> 6) << 4).                  */
static void pack_scales_q4_K(const int *sc, const int *m, uint8_t *s)
{
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
}

static void unpack_scale_min_q4_K(const uint8_t *s, int sb, int *sc, int *m)
{
    if (sb < 4) {
        *sc = s[sb] & 63;
        *m = s[sb + 4] & 63;
    } else {
        *sc = (s[sb + 4] & 15) | ((s[sb - 4] >> 6) << 4);
        *m = (s[sb + 4] >> 4) | ((s[sb] >> 6) << 4);
    }
}

/* Q4_K quantizer.  The pages give only "estimate sub-block scale/min,
 * quantize 4-bit codes" ("GGUF 量化内幕 第16章" 16.2.1), so this is a plain
 * reading: per 32-value sub-block lo = min(0, min x), step = (max x - lo)/15;
 * d = max step / 63 and dmin = max(-lo) / 63 stored as half; sc and m are the
 * rounded ratios to the stored halves (6-bit clamp); q = round((x + dmin*m) /
 * (d*sc)) clamped to 0..15, computed from the stored half values. */
static void quantize_block_q4_K(const float *v, uint8_t *blk)
{
    float step[8], neg[8];
    for (int sb = 0; sb < 8; ++sb) {
        const float *p = v + 32 * sb;
        float mn = p[0], mx = p[0];
        for (int i = 1; i < 32; ++i) {
            if (p[i] < mn) mn = p[i];
            if (p[i] > mx) mx = p[i];
        }
        float lo = (mn < 0.0f) ? mn : 0.0f;
        step[sb] = (mx - lo) / 15.0f;
        neg[sb] = (mn < 0.0f) ? -mn : 0.0f;
    }
    float smax = 0.0f, nmax = 0.0f;
    for (int sb = 0; sb < 8; ++sb) {
        if (step[sb] > smax) smax = step[sb];
        if (neg[sb] > nmax) nmax = neg[sb];
    }
    uint16_t dh = oracle_f32_to_f16(smax / 63.0f);
    uint16_t mh = oracle_f32_to_f16(nmax / 63.0f);
    float df = oracle_f16_to_f32(dh), mf = oracle_f16_to_f32(mh);
    int sc[8], m[8];
    for (int sb = 0; sb < 8; ++sb) {
        sc[sb] = (df > 0.0f) ? clamp_round(step[sb] / df, 0.0f, 63.0f) : 0;
        m[sb] = (mf > 0.0f) ? clamp_round(neg[sb] / mf, 0.0f, 63.0f) : 0;
    }
    wr16(blk + 0, dh);
    wr16(blk + 2, mh);
    pack_scales_q4_K(sc, m, blk + 4);
    uint8_t *qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        for (int l = 0; l < 32; ++l) {
            int q2[2];
            for (int half = 0; half < 2; ++half) {
                int e = 64 * c + 32 * half + l;
                int sb = 2 * c + half;
                float t = df * (float)sc[sb];
                float z = v[e] + mf * (float)m[sb];
                q2[half] = (t > 0.0f) ? clamp_round(z / t, 0.0f, 15.0f) : 0;
            }
            qs[32 * c + l] = (uint8_t)(q2[0] | (q2[1] << 4));
        }
    }
}

/* Q6_K quantizer.  Not printed on the pages; plain reading: per 16-value
 * sub-block s = max|x| / 31; d = max s / 127 stored as half; int8
 * sc = round(s/d); v = round(x / (d*sc)) clamped to -32..31, stored +32. */
static void quantize_block_q6_K(const float *v, uint8_t *blk)
{
    float s[16];
    for (int sb = 0; sb < 16; ++sb) {
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(v[16 * sb + i]);
            if (a > amax) amax = a;
        }
        s[sb] = amax / 31.0f;
    }
    float smax = 0.0f;
    for (int sb = 0; sb < 16; ++sb)
        if (s[sb] > smax) smax = s[sb];
    uint16_t dh = oracle_f32_to_f16(smax / 127.0f);
    float df = oracle_f16_to_f32(dh);
    int sc[16];
    for (int sb = 0; sb < 16; ++sb)
        sc[sb] = (df > 0.0f) ? clamp_round(s[sb] / df, -128.0f, 127.0f) : 0;
    uint8_t *ql = blk, *qh = blk + 128;
    memset(ql, 0, 128);
    memset(qh, 0, 64);
    for (int e = 0; e < QK_K; ++e) {
        int sb = e / 16;
        float t = df * (float)sc[sb];
        int q = (t != 0.0f) ? clamp_round(v[e] / t, -32.0f, 31.0f) + 32 : 32;
        int h = e / 128, r = e % 128, g = r / 32, l = r % 32;
        int qlb = 64 * h + 32 * (g & 1) + l;
        ql[qlb] |= (uint8_t)((q & 15) << (4 * (g >> 1)));
        qh[32 * h + l] |= (uint8_t)(((q >> 4) & 3) << (2 * g));
    }
    for (int sb = 0; sb < 16; ++sb) blk[192 + sb] = (uint8_t)(int8_t)sc[sb];
    wr16(blk + 208, dh);
}

int oracle_quantize_rows(int type, const float *w, int64_t M, int64_t K, int64_t ldw, uint8_t *W)
{
    if (!weight_type_ok(type)) return -1;
    if (!w || !W) return -3;
    int64_t rb = oracle_row_bytes(type, K);
    if (rb < 0 || M <= 0 || ldw < K) return -2;
    int64_t qk = oracle_block_elems(type), bs = oracle_block_bytes(type), nb = K / qk;
    for (int64_t r = 0; r < M; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float *v = w + r * ldw + b * qk;
            uint8_t *blk = W + r * rb + b * bs;
            if (type == ORACLE_Q4_0) quantize_block_q4_0(v, blk);
            else if (type == ORACLE_Q4_K) quantize_block_q4_K(v, blk);
            else quantize_block_q6_K(v, blk);
        }
    return 0;
}

/* ------------------------------------------------------------------------
 * Decoding: the code of element e of a block, and its scale fields.
 * ---------------------------------------------------------------------- */

/* Q4_0: raw nibble 0..15 of element e (0..31). */
static int q4_0_code(const uint8_t *blk, int e)
{
    const uint8_t *qs = blk + 2;
    return e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);
}

/* Q4_K: raw nibble of element e (0..255), per dequantize_row_q4_K. */
static int q4_K_code(const uint8_t *blk, int e)
{
    const uint8_t *qs = blk + 16;
    int c = e / 64, r = e % 64;
    return r < 32 ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);
}

/* Q6_K: stored 6-bit value v (0..63) of element e (0..255). */
static int q6_K_code(const uint8_t *blk, int e)
{
    const uint8_t *ql = blk, *qh = blk + 128;
    int h = e / 128, r = e % 128, g = r / 32, l = r % 32;
    int lo = (ql[64 * h + 32 * (g & 1) + l] >> (4 * (g >> 1))) & 15;
    int hi = (qh[32 * h + l] >> (2 * g)) & 3;
    return lo | (hi << 4);
}

static double dequant_elem(int type, const uint8_t *blk, int e)
{
    if (type == ORACLE_Q4_0) return h2d(blk) * (double)(q4_0_code(blk, e) - 8);
    if (type == ORACLE_Q4_K) {
        int sc, m;
        unpack_scale_min_q4_K(blk + 4, e / 32, &sc, &m);
        return h2d(blk) * sc * q4_K_code(blk, e) - h2d(blk + 2) * m;
    }
    int8_t sc = (int8_t)blk[192 + e / 16];
    return h2d(blk + 208) * sc * (double)(q6_K_code(blk, e) - 32);
}

int oracle_dequantize_rows(int type, const uint8_t *W, int64_t M, int64_t K, double *out)
{
    if (!weight_type_ok(type)) return -1;
    if (!W || !out) return -3;
    int64_t rb = oracle_row_bytes(type, K);
    if (rb < 0 || M <= 0) return -2;
    int64_t qk = oracle_block_elems(type), bs = oracle_block_bytes(type);
    for (int64_t r = 0; r < M; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = dequant_elem(type, W + r * rb + (k / qk) * bs, (int)(k % qk));
    return 0;
}

int oracle_dequantize_q8_1(const uint8_t *xq, int64_t K, int64_t ncols, double *out)
{
    if (!xq || !out) return -3;
    if (K <= 0 || ncols <= 0) return -2;
    int64_t nb = oracle_q8_1_padded_k(K) / QK8_1;
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t k = 0; k < K; ++k) {
            const uint8_t *blk = xq + (c * nb + k / QK8_1) * Q8_1_BYTES;
            out[c * K + k] = h2d(blk) * (double)(int8_t)blk[4 + k % QK8_1];
        }
    return 0;
}

/* Q4_K weights in fp32 ("GGUF 量化内幕 第16章", 16.2.1, the float decoder):
 * element e of a super-block belongs to 32-value sub-block e/32, whose 6-bit
 * scale sc and min m give the fp32 factors d*sc and dmin*m; the weight is
 * (d*sc)*code - dmin*m, each product and the difference rounded to fp32 in
 * that order (the oracle is built without contraction, so no fused
 * multiply-add merges them). */
int oracle_dequantize_row_q4_K_f32(const uint8_t *W, int64_t K, float *out)
{
    if (!W || !out) return -3;
    if (K <= 0 || K % QK_K) return -2;
    for (int64_t k = 0; k < K; ++k) {
        const uint8_t *blk = W + (k / QK_K) * Q4_K_BYTES;
        const int e = (int)(k % QK_K);
        int sc, m;
        unpack_scale_min_q4_K(blk + 4, e / 32, &sc, &m);
        const float scale = oracle_f16_to_f32(rd16(blk)) * (float)sc;
        const float offset = oracle_f16_to_f32(rd16(blk + 2)) * (float)m;
        const float scaled = scale * (float)q4_K_code(blk, e);
        out[k] = scaled - offset;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * GEMV.
 * ---------------------------------------------------------------------- */

static int gemv_args_ok(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                        int64_t ncols, const int64_t *rows, int64_t nrows)
{
    if (!weight_type_ok(type)) return -1;
    if (!W || !xq) return -3;
    if (oracle_row_bytes(type, K) < 0 || M <= 0 || ncols <= 0 || nrows < 0) return -2;
    if (!rows && nrows != M) return -2;
    if (rows)
        for (int64_t i = 0; i < nrows; ++i)
            if (rows[i] < 0 || rows[i] >= M) return -2;
    return 0;
}

/* Plain definition: y[c][r] = sum_k What[r][k] * xhat[c][k] in fp64, with
 * What the exact block value of the weight and xhat = d8 * q8. */
int oracle_gemv_plain(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                      int64_t ncols, const int64_t *rows, int64_t nrows, double *y)
{
    int rc = gemv_args_ok(type, W, M, K, xq, ncols, rows, nrows);
    if (rc) return rc;
    if (!y) return -3;
    double *wrow = malloc(sizeof(double) * K), *xh = malloc(sizeof(double) * K * ncols);
    if (!wrow || !xh) { free(wrow); free(xh); return -3; }
    oracle_dequantize_q8_1(xq, K, ncols, xh);
    int64_t rb = oracle_row_bytes(type, K);
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        oracle_dequantize_rows(type, W + r * rb, 1, K, wrow);
        for (int64_t c = 0; c < ncols; ++c) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += wrow[k] * xh[c * K + k];
            y[c * nrows + i] = acc;
        }
    }
    free(wrow);
    free(xh);
    return 0;
}

/* One row, one column, by the method's block formula ("mul_mat_vec_q" page):
 *   Q4_0: sum_b d4 * (d8*sumi - 8*s),  sumi = sum q*qy over the block
 *         (vec_dot_q4_0_q8_1_impl; the constant 8*vdr/QI4_0 per call adds
 *         up to 8 per block);
 *   Q4_K: sum_sb d*sc*d8*dot1 - dmin*m*d8*dot2, dot1 = sum q*qy,
 *         dot2 = sum qy (vec_dot_q4_K_q8_1_impl_vmmq);
 *   Q6_K: sum_sb d*sc*d8*sum (v-32)*qy over each 16-value sub-block.
 * All in fp64; l1 accumulates |term| for each term listed. */
static void formula_row(int type, const uint8_t *wrow, int64_t K, const uint8_t *xqc,
                        double *yo, double *l1o)
{
    double y = 0.0, l1 = 0.0;
    if (type == ORACLE_Q4_0) {
        for (int64_t b = 0; b < K / QK4_0; ++b) {
            const uint8_t *blk = wrow + b * Q4_0_BYTES;
            const uint8_t *xb = xqc + b * Q8_1_BYTES;
            long sumi = 0;
            for (int e = 0; e < 32; ++e) sumi += (long)q4_0_code(blk, e) * (int8_t)xb[4 + e];
            double d4 = h2d(blk), d8 = h2d(xb), s = h2d(xb + 2);
            double t1 = d4 * d8 * (double)sumi, t2 = 8.0 * d4 * s;
            y += t1 - t2;
            l1 += fabs(t1) + fabs(t2);
        }
    } else if (type == ORACLE_Q4_K) {
        for (int64_t b = 0; b < K / QK_K; ++b) {
            const uint8_t *blk = wrow + b * Q4_K_BYTES;
            double d = h2d(blk), dmin = h2d(blk + 2);
            for (int sb = 0; sb < 8; ++sb) {
                const uint8_t *xb = xqc + (b * 8 + sb) * Q8_1_BYTES;
                long dot1 = 0, dot2 = 0;
                for (int i = 0; i < 32; ++i) {
                    int qy = (int8_t)xb[4 + i];
                    dot1 += (long)q4_K_code(blk, 32 * sb + i) * qy;
                    dot2 += qy;
                }
                int sc, m;
                unpack_scale_min_q4_K(blk + 4, sb, &sc, &m);
                double d8 = h2d(xb);
                double t1 = d * sc * d8 * (double)dot1, t2 = dmin * m * d8 * (double)dot2;
                y += t1 - t2;
                l1 += fabs(t1) + fabs(t2);
            }
        }
    } else {
        for (int64_t b = 0; b < K / QK_K; ++b) {
            const uint8_t *blk = wrow + b * Q6_K_BYTES;
            double d = h2d(blk + 208);
            for (int sb = 0; sb < 16; ++sb) {
                const uint8_t *xb = xqc + (b * 8 + sb / 2) * Q8_1_BYTES;
                long sumi = 0;
                for (int i = 0; i < 16; ++i)
                    sumi += (long)(q6_K_code(blk, 16 * sb + i) - 32) * (int8_t)xb[4 + 16 * (sb % 2) + i];
                double t = d * (int8_t)blk[192 + sb] * h2d(xb) * (double)sumi;
                y += t;
                l1 += fabs(t);
            }
        }
    }
    *yo = y;
    if (l1o) *l1o = l1;
}

/* One row, one column, by the method's integer formula in fp32: exact int32
 * block sums, then the block scaling of formula_row evaluated in fp32 (each
 * product and sum rounded to fp32 in the order written), the way the method's
 * kernels scale their dp4a sums ("mul_mat_vec_q" page, vec_dot_q4_0_q8_1_impl,
 * vec_dot_q4_K_q8_1_impl_vmmq, the Q6_K vec_dot).  The CPU counterpart of the
 * GPU arithmetic, timed as a second CPU baseline. */
static float int_formula_row(int type, const uint8_t *wrow, int64_t K, const uint8_t *xqc)
{
    float y = 0.0f;
    if (type == ORACLE_Q4_0) {
        for (int64_t b = 0; b < K / QK4_0; ++b) {
            const uint8_t *blk = wrow + b * Q4_0_BYTES;
            const uint8_t *xb = xqc + b * Q8_1_BYTES;
            int32_t sumi = 0;
            for (int e = 0; e < 32; ++e) sumi += q4_0_code(blk, e) * (int8_t)xb[4 + e];
            const float d4 = oracle_f16_to_f32(rd16(blk)), d8 = oracle_f16_to_f32(rd16(xb));
            const float s = oracle_f16_to_f32(rd16(xb + 2));
            const float scaled = d8 * (float)sumi, corr = 8.0f * s;
            const float term = d4 * (scaled - corr);
            y += term;
        }
    } else if (type == ORACLE_Q4_K) {
        for (int64_t b = 0; b < K / QK_K; ++b) {
            const uint8_t *blk = wrow + b * Q4_K_BYTES;
            const float d = oracle_f16_to_f32(rd16(blk)), dmin = oracle_f16_to_f32(rd16(blk + 2));
            for (int sb = 0; sb < 8; ++sb) {
                const uint8_t *xb = xqc + (b * 8 + sb) * Q8_1_BYTES;
                int32_t dot1 = 0, dot2 = 0;
                for (int i = 0; i < 32; ++i) {
                    const int qy = (int8_t)xb[4 + i];
                    dot1 += q4_K_code(blk, 32 * sb + i) * qy;
                    dot2 += qy;
                }
                int sc, m;
                unpack_scale_min_q4_K(blk + 4, sb, &sc, &m);
                const float d8 = oracle_f16_to_f32(rd16(xb));
                const float t1 = (d * (float)sc) * (d8 * (float)dot1);
                const float t2 = (dmin * (float)m) * (d8 * (float)dot2);
                y += t1 - t2;
            }
        }
    } else {
        for (int64_t b = 0; b < K / QK_K; ++b) {
            const uint8_t *blk = wrow + b * Q6_K_BYTES;
            const float d = oracle_f16_to_f32(rd16(blk + 208));
            for (int sb = 0; sb < 16; ++sb) {
                const uint8_t *xb = xqc + (b * 8 + sb / 2) * Q8_1_BYTES;
                int32_t sumi = 0;
                for (int i = 0; i < 16; ++i)
                    sumi += (q6_K_code(blk, 16 * sb + i) - 32) * (int8_t)xb[4 + 16 * (sb % 2) + i];
                const float t = (d * (float)(int8_t)blk[192 + sb]) * (oracle_f16_to_f32(rd16(xb)) * (float)sumi);
                y += t;
            }
        }
    }
    return y;
}

int oracle_gemv_formula(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                        int64_t ncols, const int64_t *rows, int64_t nrows, double *y, double *l1)
{
    int rc = gemv_args_ok(type, W, M, K, xq, ncols, rows, nrows);
    if (rc) return rc;
    if (!y) return -3;
    int64_t rb = oracle_row_bytes(type, K);
    int64_t xstride = oracle_q8_1_padded_k(K) / QK8_1 * Q8_1_BYTES;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        for (int64_t c = 0; c < ncols; ++c)
            formula_row(type, W + r * rb, K, xq + c * xstride, &y[c * nrows + i],
                        l1 ? &l1[c * nrows + i] : NULL);
    }
    return 0;
}

/* Threaded variant for the timed CPU baseline: threads claim chunks of rows
 * from a shared atomic counter (the work-stealing shape of ggml's CPU
 * mul_mat, "解构LLM" page, "原子抢占").  Same arithmetic per row. */
typedef struct {
    int type;
    const uint8_t *W, *xq;
    int64_t M, K, ncols, rb, xstride;
    double *y, *l1;
    float *yf; /* set: the fp32 integer formula instead of the fp64 one */
    atomic_llong next;
} mt_job;

#define MT_CHUNK 16

static void *mt_worker(void *arg)
{
    mt_job *j = arg;
    for (;;) {
        long long r0 = atomic_fetch_add(&j->next, MT_CHUNK);
        if (r0 >= j->M) break;
        long long r1 = r0 + MT_CHUNK < j->M ? r0 + MT_CHUNK : j->M;
        for (long long r = r0; r < r1; ++r)
            for (int64_t c = 0; c < j->ncols; ++c) {
                if (j->yf)
                    j->yf[c * j->M + r] = int_formula_row(j->type, j->W + r * j->rb, j->K, j->xq + c * j->xstride);
                else
                    formula_row(j->type, j->W + r * j->rb, j->K, j->xq + c * j->xstride,
                                &j->y[c * j->M + r], j->l1 ? &j->l1[c * j->M + r] : NULL);
            }
    }
    return NULL;
}

static void run_mt(mt_job *job, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    atomic_init(&job->next, 0);
    pthread_t th[512];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[started], NULL, mt_worker, job) == 0) ++started;
    mt_worker(job);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

int oracle_gemv_formula_mt(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                           int64_t ncols, double *y, double *l1, int nthreads)
{
    int rc = gemv_args_ok(type, W, M, K, xq, ncols, NULL, M);
    if (rc) return rc;
    if (!y) return -3;
    mt_job job = {type, W, xq, M, K, ncols, oracle_row_bytes(type, K),
                  oracle_q8_1_padded_k(K) / QK8_1 * Q8_1_BYTES, y, l1, NULL, 0};
    run_mt(&job, nthreads);
    return 0;
}

int oracle_gemv_int_f32(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                        int64_t ncols, float *y, int nthreads)
{
    int rc = gemv_args_ok(type, W, M, K, xq, ncols, NULL, M);
    if (rc) return rc;
    if (!y) return -3;
    mt_job job = {type, W, xq, M, K, ncols, oracle_row_bytes(type, K),
                  oracle_q8_1_padded_k(K) / QK8_1 * Q8_1_BYTES, NULL, NULL, y, 0};
    run_mt(&job, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------
 * Per-sub-block integer sums (the exact int32 intermediates of the method).
 * ---------------------------------------------------------------------- */
int64_t oracle_subblock_count(int type, int64_t K)
{
    if (type == ORACLE_Q4_0) return K / 32;
    if (type == ORACLE_Q4_K) return K / 16; /* (dot1, dot2) per 32 */
    if (type == ORACLE_Q6_K) return K / 16;
    return -1;
}

int oracle_subblock_sums(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                         int64_t ncols, const int64_t *rows, int64_t nrows, int32_t *out)
{
    int rc = gemv_args_ok(type, W, M, K, xq, ncols, rows, nrows);
    if (rc) return rc;
    if (!out) return -3;
    int64_t rb = oracle_row_bytes(type, K);
    int64_t xstride = oracle_q8_1_padded_k(K) / QK8_1 * Q8_1_BYTES;
    int64_t n = oracle_subblock_count(type, K);
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t r = rows ? rows[i] : i;
            const uint8_t *wrow = W + r * rb, *xqc = xq + c * xstride;
            int32_t *o = out + (c * nrows + i) * n;
            if (type == ORACLE_Q4_0) {
                for (int64_t b = 0; b < K / 32; ++b) {
                    int32_t s = 0;
                    for (int e = 0; e < 32; ++e)
                        s += q4_0_code(wrow + b * Q4_0_BYTES, e) * (int8_t)xqc[b * Q8_1_BYTES + 4 + e];
                    o[b] = s;
                }
            } else if (type == ORACLE_Q4_K) {
                for (int64_t sb = 0; sb < K / 32; ++sb) {
                    const uint8_t *blk = wrow + (sb / 8) * Q4_K_BYTES;
                    int32_t d1 = 0, d2 = 0;
                    for (int i2 = 0; i2 < 32; ++i2) {
                        int qy = (int8_t)xqc[sb * Q8_1_BYTES + 4 + i2];
                        d1 += q4_K_code(blk, (int)(32 * (sb % 8) + i2)) * qy;
                        d2 += qy;
                    }
                    o[2 * sb] = d1;
                    o[2 * sb + 1] = d2;
                }
            } else {
                for (int64_t sb = 0; sb < K / 16; ++sb) {
                    const uint8_t *blk = wrow + (sb / 16) * Q6_K_BYTES;
                    int32_t s = 0;
                    for (int i2 = 0; i2 < 16; ++i2)
                        s += (q6_K_code(blk, (int)(16 * (sb % 16) + i2)) - 32) *
                             (int8_t)xqc[(sb / 2) * Q8_1_BYTES + 4 + 16 * (sb % 2) + i2];
                    o[sb] = s;
                }
            }
        }
    return 0;
}
