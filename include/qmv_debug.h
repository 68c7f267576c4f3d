/*
 * libqmv test-only entry points: exact integer intermediates of the GEMV, a
 * way to make the library's one bounded wait run out on purpose, and a
 * per-CTA timeline of launches.  Not part of the compute API; they exist so
 * that tests can check the kernels bit for bit, exercise the fault path and
 * measure where a launch's time goes.  Conventions (ownership, asynchronous
 * execution on `stream`, host validation before any launch, status codes)
 * are those of qmv.h.
 *
 * The last two run instrumented twins of the streaming tile kernel: the same
 * code plus the timeline stores and the withheld share, which the ordinary
 * kernels do not carry.  Twins exist for the plain GEMV of one or two columns
 * and the fused gate/up GEMV of one column (4-row tiles, dp4a decode).
 */
#ifndef QMV_DEBUG_H
#define QMV_DEBUG_H

#include "qmv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The exact int32 intermediates of the block formulas ("sumi" of the page
 * "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q", section "一次 vec_dot 的解剖",
 * and dot1 / dot2 of vec_dot_q4_K_q8_1_impl_vmmq), computed by the same
 * device code as qmv_mul_mat_vec, for bit-exact parity tests.  out is
 * [ncols][M][n] int32 (device) with
 *   Q4_0: n = K/32, per block sum of code*qy (code = raw nibble 0..15);
 *   Q4_K: n = K/16, per 32-value sub-block the pair (dot1, dot2);
 *   Q6_K: n = K/16, per 16-value sub-block sum (v-32)*qy.
 * Arguments and limits as for qmv_mul_mat_vec.  out is cleared and written
 * asynchronously on stream. */
qmv_status qmv_debug_subblock_sums(int type, const void *W, int64_t M, int64_t K, const void *xq,
                                   int ncols, int32_t *out, void *stream);

/* qmv_mul_mat_vec_f32 (same arguments, limits and outputs), launched so that
 * the bounded wait of its activation exchange runs out: in every cluster of
 * CTAs that share the quantization of x, the CTA of rank 1 withholds its
 * share from the others, and the CTA of rank 0 waits at most wait_ns
 * nanoseconds for it (1 ns .. 1 s) before its warps give up.  Warps that gave
 * up record code 2 in the device fault word (qmv_device_fault) and write NaN
 * to the outputs of their rows; every other output is the value
 * qmv_mul_mat_vec_f32 computes.  The CTAs of rank 1 still receive rank 0's
 * share and finish normally, so nothing waits without a bound and no store
 * into a CTA arrives after it has exited.  Returns QMV_ERR_CONFIG, before
 * launching, if the launch would not use clusters of CTAs (the exchange then
 * does not exist) or without an instrumented twin (ncols > 2); the argument
 * errors of qmv_mul_mat_vec_f32 otherwise.  The
 * pages have no counterpart: it tests the library's own fault reporting. */
qmv_status qmv_debug_f32_withheld_share(int type, const void *W, int64_t M, int64_t K, const float *x,
                                        int64_t ldx, int ncols, float *y, uint64_t wait_ns, void *stream);

/* The same withheld share for qmv_mul_mat_vec_fused_q8_1 of one column
 * (plain, fp32 input x of K contiguous values, no biases; y optional, yq
 * required): the warps that give up write NaN to their rows of y, and every
 * q8_1 block holding one of those rows gets a NaN scale (half 0x7e00); every
 * other output is the value qmv_mul_mat_vec_fused_q8_1 computes.
 * QMV_ERR_CONFIG as above; the argument errors of qmv_mul_mat_vec_fused_q8_1
 * otherwise.  No counterpart in the pages. */
qmv_status qmv_debug_f32_withheld_share_q8_1(int type, const void *W, int64_t M, int64_t K, const float *x,
                                             float *y, void *yq, uint64_t wait_ns, void *stream);

/* Timeline of the streaming GEMV launches, for measuring where a launch's
 * time goes.  While enabled, each of the next `slots` launches that have an
 * instrumented twin (any call of qmv.h whose launch takes one; other launches
 * are not recorded and take no slot) runs the twin, which writes, per CTA b,
 * six globaltimer readings (ns) into buf + (k*1024 + b)*6, k = the launch's
 * index since this call: [0] the CTA's first instruction, [1] the return of the
 * wait for the previous kernel on the stream (programmatic dependent launch),
 * [2] its first activation loads returned (thread 0), [3] its own part of the
 * staging done (thread 0: fp32 input, its share quantized and sent to the
 * cluster; q8_1 input, the blocks repacked), [4] all activations in its shared
 * memory (after the CTA barrier and the partners' shares), [5] the last of its
 * warps done (an atomic max, so [5] must be zero beforehand).  [2] and [3]
 * stay zero where q8_1 input is not 16-byte aligned (another staging path).
 * buf: device memory of slots * 1024 * 6 * 8 bytes, 8-byte aligned; launches of more than 1024 CTAs
 * and launches past the slots are not recorded.  Under CUDA graph capture the
 * slot is fixed when the call is captured.  buf NULL or slots 0 disables it.
 * Costs nothing when disabled.  Not thread-safe with
 * concurrent launches from other host threads (the slot counter is shared).
 * The pages have no counterpart: a measurement aid of this library.
 * Returns QMV_ERR_SHAPE for slots < 0, QMV_ERR_ALIGN for a misaligned buf. */
qmv_status qmv_debug_trace(unsigned long long *buf, int64_t slots);

#ifdef __cplusplus
}
#endif
#endif /* QMV_DEBUG_H */
