/*
 * CPU oracle for the quantized decode GEMV (test infrastructure only).
 *
 * Plain, slow, obviously-correct C.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg use it; the GPU library never links it and
 * shares no code, header or table with it.
 *
 * What it computes, and where each piece comes from (page titles as printed):
 *   - q8_1 activation quantization: "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q",
 *     section "激活的量化：为什么是 q8_1" (quantize_q8_1 kernel and block_q8_1).
 *   - Q4_0 quantization rule: "解构LLM：以llama.cpp分析模型推理过程", section
 *     "量化格式：用更少的位数表示权重" (scale = max_abs/7, q = round(v/scale)+8).
 *   - Q4_K decode: "GGUF 量化内幕 第16章", section 16.2.1 (dequantize_row_q4_K)
 *     and the 6-bit scale/min unpack of the mul_mat_vec_q page, section
 *     "一次 vec_dot 的解剖".
 *   - Q6_K decode: mul_mat_vec_q page, Q6_K vec_dot snippet and the format
 *     table (210 bytes, 16 sub-blocks, low-4/high-2 split).
 *   - Block dot formulas: mul_mat_vec_q page, vec_dot_q4_0_q8_1_impl,
 *     vec_dot_q4_K_q8_1_impl_vmmq and the Q6_K snippet.
 *   - GEMV: y[c][r] = sum_k What[r][k] * xhat[c][k] evaluated in fp64.
 *
 * Where the pages are silent or contradict themselves, the reading taken is
 * stated at the function it concerns, below.
 *
 * Parity pins: every function here is checked by the CPU test-suite against
 * closed forms, worked examples and brute force (tests/test_oracle_*.py),
 * except the Q6_K byte layout, whose GGUF compatibility is a reading of the
 * pages (parity unpinned with respect to GGUF files; pinned to the stated
 * layout).
 *
 * Return codes: 0 = ok, -1 = bad type, -2 = bad shape, -3 = null pointer.
 */
#ifndef QMV_ORACLE_H
#define QMV_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Type ids as ggml numbers them ("GGUF 量化内幕 第16章", 16.1.1). */
enum { ORACLE_Q4_0 = 2, ORACLE_Q8_1 = 9, ORACLE_Q4_K = 12, ORACLE_Q6_K = 14 };

/* ---- IEEE-754 binary16 ------------------------------------------------- */
uint16_t oracle_f32_to_f16(float f);          /* round to nearest, ties to even */
float    oracle_f16_to_f32(uint16_t h);       /* exact */
void     oracle_f32_to_f16_array(const float *in, uint16_t *out, int64_t n);
void     oracle_f16_to_f32_array(const uint16_t *in, float *out, int64_t n);

/* ---- sizes ------------------------------------------------------------- */
int64_t oracle_block_elems(int type);         /* 32 or 256; 0 for unknown */
int64_t oracle_block_bytes(int type);         /* 18, 144, 210, 36; 0 for unknown */
int64_t oracle_row_bytes(int type, int64_t K);/* K/qk * block bytes; -2 if K % qk */
int64_t oracle_q8_1_padded_k(int64_t K);      /* ceil(K/512)*512 */

/* ---- quantizers -------------------------------------------------------- */
/* x: ncols columns of K floats, column c at x + c*ldx.  xq: ncols rows of
 * padded_k/32 blocks of 36 bytes. */
int oracle_quantize_q8_1(const float *x, int64_t K, int64_t ncols, int64_t ldx, uint8_t *xq);
/* w: M rows of K floats, row r at w + r*ldw.  W: M rows of row_bytes. */
int oracle_quantize_rows(int type, const float *w, int64_t M, int64_t K, int64_t ldw, uint8_t *W);

/* ---- dequantizers (exact block values in fp64) -------------------------- */
int oracle_dequantize_rows(int type, const uint8_t *W, int64_t M, int64_t K, double *out);
int oracle_dequantize_q8_1(const uint8_t *xq, int64_t K, int64_t ncols, double *out);
/* Q4_K row decoded in fp32 the way the printed row function does it. */
int oracle_dequantize_row_q4_K_f32(const uint8_t *W, int64_t K, float *out);

/* ---- GEMV ---------------------------------------------------------------
 * rows: optional list of nrows row indices (NULL = all M rows, nrows = M).
 * Outputs are [ncols][nrows].
 *   plain:   y = sum_k What*xhat (dequantize, then dot) in fp64.
 *   formula: the method's per-block formula from the stored fields in fp64;
 *            l1 = sum over the row's scaled terms of |term|.
 */
int oracle_gemv_plain(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                      int64_t ncols, const int64_t *rows, int64_t nrows, double *y);
int oracle_gemv_formula(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                        int64_t ncols, const int64_t *rows, int64_t nrows, double *y, double *l1);
/* Same as oracle_gemv_formula over all rows, split over nthreads host threads
 * that claim row chunks from a shared counter (timed CPU baseline). */
int oracle_gemv_formula_mt(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                           int64_t ncols, double *y, double *l1, int nthreads);
/* The method's integer formula in fp32 over all rows (int32 block sums, fp32
 * block scaling): y [ncols][M] float; threaded like oracle_gemv_formula_mt.
 * A CPU baseline, agreeing with oracle_gemv_formula within fp32 rounding. */
int oracle_gemv_int_f32(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                        int64_t ncols, float *y, int nthreads);

/* Per-sub-block integer sums, [ncols][nrows][n] int32:
 *   Q4_0: n = K/32, sum over the block of q*qy with q the raw nibble 0..15;
 *   Q4_K: n = K/16, pairs (dot1, dot2) per 32-sub-block: dot1 = sum q*qy,
 *         dot2 = sum qy;
 *   Q6_K: n = K/16, per 16-sub-block sum (v-32)*qy.                         */
int64_t oracle_subblock_count(int type, int64_t K);
int oracle_subblock_sums(int type, const uint8_t *W, int64_t M, int64_t K, const uint8_t *xq,
                         int64_t ncols, const int64_t *rows, int64_t nrows, int32_t *out);

#ifdef __cplusplus
}
#endif
#endif
