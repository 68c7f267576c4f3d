/*
 * libqmv -- quantized decode GEMV for NVIDIA GB300 (sm_103a).
 *
 * Computes y = W . x for decode-time LLM inference, where W is stored in the
 * GGUF block formats Q4_0, Q4_K or Q6_K and x is first quantized to q8_1
 * blocks.  Each block product is an int8 dot product (dp4a) scaled by the
 * block scales.  The operation and the formats follow the page
 * "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q——解码时一条量化权重如何被 dp4a
 * 逐块点积" (sections "权重的排法", "激活的量化", "dp4a", "一次 vec_dot 的解剖",
 * "融合", "MoE") and "GGUF 量化内幕 第16章" (16.1.2 block structs,
 * 16.2.1 dequantize_row_q4_K).
 *
 * Conventions shared by every call:
 *   - Ownership: the caller allocates and owns every buffer; device pointers
 *     point to device memory.  The library allocates no memory and keeps no
 *     per-call state.
 *   - Execution: calls are asynchronous on `stream` (a cudaStream_t passed as
 *     void*, NULL for the legacy default stream).  Arguments are validated on
 *     the host before anything is launched; a failed validation launches
 *     nothing and returns the status below.  A failed launch returns
 *     QMV_ERR_CUDA.
 *   - Layouts: W is row-major, row r at W + r*qmv_row_bytes(type, K), blocks
 *     back to back within a row (GGUF order).  Activations are q8_1 rows of
 *     qmv_q8_1_padded_k(K)/32 blocks of 36 bytes, column c at
 *     xq + c*qmv_q8_1_bytes(K, 1), as written by qmv_quantize_q8_1.  Outputs
 *     are fp32, column-major over rows: y[c*M + r].
 *   - Limits: 1 <= ncols <= 8 (MMVQ_MAX_BATCH_SIZE on the page); K a
 *     positive multiple of the block size (32 for Q4_0, 256 for Q4_K/Q6_K);
 *     M >= 1.  W must be 2-byte aligned, xq 4-byte aligned, y 4-byte
 *     aligned.  Rows whose byte size is a multiple of 16 with a 16-byte
 *     aligned W take the streaming path; other shapes take a slower generic
 *     path with identical results.
 *   - Threads: calls are thread-safe; the tuning overrides below are
 *     process-wide.
 *   - Waits: weight copies (cp.async) complete in hardware and are awaited
 *     with cp.async.wait_group; CTAs synchronise with __syncwarp /
 *     __syncthreads, cluster barriers and the programmatic-dependent-launch
 *     wait on the previous grid.  The one spin-wait is bounded: the fp32-input
 *     plain and gate/up calls, whose clusters of CTAs share the quantization
 *     of the activations, wait on an mbarrier for the partners' shares for at
 *     most one second; past that each warp that gave up records code 2 in
 *     the sticky device fault word (qmv_device_fault), writes NaN to the
 *     outputs of its rows and returns instead of hanging.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Type ids, numbered as ggml numbers them ("GGUF 量化内幕 第16章", 16.1.1). */
typedef enum {
    QMV_TYPE_Q4_0 = 2,  /* 32 weights per 18-byte block: half d, 16 bytes of nibbles; w = d*(q-8) */
    QMV_TYPE_Q8_1 = 9,  /* 32 int8 activations per 36-byte block: half d, half s = d*sum(q) */
    QMV_TYPE_Q4_K = 12, /* 256 weights per 144-byte block: half d, half dmin, 12 bytes of 6-bit
                           scales/mins, 128 bytes of nibbles; w = d*sc*q - dmin*m */
    QMV_TYPE_Q6_K = 14  /* 256 weights per 210-byte block: ql[128], qh[64], int8 scales[16],
                           half d; w = d*sc*(v-32), v = 6-bit code */
} qmv_type;

typedef enum {
    QMV_OK = 0,
    QMV_ERR_NULL = 1,         /* a required pointer is NULL */
    QMV_ERR_TYPE = 2,         /* unsupported type id */
    QMV_ERR_SHAPE = 3,        /* M, K, ldx, n_expert, n_tokens or top_k out of range */
    QMV_ERR_NCOLS = 4,        /* ncols (or n_tokens for MoE) not in 1..8 */
    QMV_ERR_ALIGN = 5,        /* a pointer violates the alignment stated above */
    QMV_ERR_CUDA = 6,         /* a CUDA runtime call or launch failed */
    QMV_ERR_IDS = 7,          /* reserved: invalid expert ids are reported through dev_status */
    QMV_ERR_DEVICE_FAULT = 8, /* a kernel's bounded wait ran out (see qmv_device_fault) */
    QMV_ERR_RANGE = 9,        /* checked mode: an argument's byte range is not inside one device
                                 allocation (see qmv_set_checked) */
    QMV_ERR_CONFIG = 10       /* the QMV_GEOM environment override is malformed or out of range;
                                 or a test entry of qmv_debug.h has no launch of the form it needs */
} qmv_status;

/* Human-readable name of a status code (static storage). */
const char *qmv_status_str(int status);

/* Library version: major*10000 + minor*100 + patch. */
int qmv_version(void);

/* ---- sizes ---------------------------------------------------------------- */

/* Bytes of one weight row: (K / block elems) * block bytes; 0 if the type is
 * not a weight type or K is not a positive multiple of its block size.  The
 * block sizes are those of the block structs ("GGUF 量化内幕 第16章", 16.1.2,
 * whose static_asserts fix 18 / 144 / 210 bytes; the mul_mat_vec_q page,
 * section "权重的排法").  A size helper: no computation on the pages. */
size_t qmv_row_bytes(int type, int64_t K);

/* K rounded up to a multiple of 512: activations are quantized and strided
 * with this padded width (MATRIX_ROW_PADDING on the mul_mat_vec_q page,
 * section "激活的量化"); the padding quantizes to zero blocks. */
int64_t qmv_q8_1_padded_k(int64_t K);

/* Bytes of ncols q8_1 activation rows: ncols * padded_k/32 * 36, the 36-byte
 * block_q8_1 of the mul_mat_vec_q page, section "激活的量化".  A size helper:
 * no computation on the pages. */
size_t qmv_q8_1_bytes(int64_t K, int ncols);

/* ---- activation quantization -------------------------------------------------
 * q8_1 quantization of ncols fp32 columns (mul_mat_vec_q page, quantize_q8_1
 * kernel): per 32 values amax = max|x|, d = amax/127 in fp32, q = round(x/d)
 * (halfway cases away from zero), stored d and s = d*sum(q) as half.  Column c
 * is read from x + c*ldx (K floats, device); values past K quantize as zeros
 * up to the padded width.  xq receives qmv_q8_1_bytes(K, ncols) bytes.
 * Readings where the page is silent: s holds d*sum(q) (the struct comment)
 * rather than the float sum of x; a block whose amax/127 underflows to zero
 * quantizes to zero; codes are clamped to [-127, 127].
 * Inputs must be finite.  ncols may exceed 8 here (any ncols >= 1). */
qmv_status qmv_quantize_q8_1(const float *x, int64_t K, int ncols, int64_t ldx, void *xq, void *stream);

/* ---- weight quantization ------------------------------------------------------
 * Quantizes an fp32 matrix w (M rows of K floats, row r at w + r*ldw,
 * device) into blocks of `type` written to W (M * qmv_row_bytes bytes).
 * Q4_0 follows the rule on "解构LLM：以llama.cpp分析模型推理过程", section
 * "量化格式" (scale = max|x|/7, q = round(x/scale) + 8).  The Q4_K and Q6_K
 * quantizers are not printed on the pages; they are plain min/max (Q4_K) and
 * absmax (Q6_K) rules taken from the stored half scales.  Bit-identical to
 * the repository's CPU oracle.  Not performance-critical (a preparation step).
 * Inputs must be finite with |x| < 1e4. */
qmv_status qmv_quantize_weights(int type, const float *w, int64_t M, int64_t K, int64_t ldw, void *W,
                                void *stream);

/* ---- GEMV ---------------------------------------------------------------------
 * y[c*M + r] = sum over blocks of the block formula for row r and activation
 * column c, for c < ncols (mul_mat_vec_q page, vec_dot_q4_0_q8_1_impl,
 * vec_dot_q4_K_q8_1_impl_vmmq and the Q6_K vec_dot):
 *   Q4_0: sum_b d4 * (d8*sumi - 8*s)              sumi = sum of code*qy
 *   Q4_K: sum_sb d*sc*d8*dot1 - dmin*m*d8*dot2     dot1 = sum code*qy, dot2 = sum qy
 *   Q6_K: sum_sb d*sc*d8*sum((v-32)*qy)            per 16-value sub-block
 * accumulated in fp32.  W is read from HBM exactly once per call whatever
 * ncols is: each weight tile, staged in shared memory, serves every column
 * (the default decode unpacks it again per column; the opt-in tensor-core
 * decode, qmv_set_mma_min_cols, once for all columns). */
qmv_status qmv_mul_mat_vec(int type, const void *W, int64_t M, int64_t K, const void *xq, int ncols,
                           float *y, void *stream);

/* Fused gate/up GEMV with SwiGLU epilogue (mul_mat_vec_q page, section
 * "融合"): both products are accumulated in one pass over the shared q8_1
 * activations and y[c*M + r] = up * silu(gate), silu(g) = g/(1+exp(-g)).
 * W_gate and W_up have identical shape and type.  The page fuses only at a
 * single column; this call accepts 1 <= ncols <= 8. */
qmv_status qmv_mul_mat_vec_gate_up_swiglu(int type, const void *W_gate, const void *W_up, int64_t M,
                                          int64_t K, const void *xq, int ncols, float *y, void *stream);

/* Expert-indexed GEMV for mixture-of-experts (mul_mat_vec_q page, section
 * "MoE"): W holds n_expert matrices back to back (expert e at
 * W + e*M*row_bytes); xq holds one q8_1 row per token; ids (device, int32,
 * [n_tokens][top_k]) names the expert of each token slot.  Output
 * y[(t*top_k + k)*M + r] = (W[ids[t][k]] . x[t])[r].  Tokens routed to the
 * same expert share one pass over its weights; experts no token selects are
 * not read.  An id outside [0, n_expert) zero-fills that slot's output; if
 * dev_status is not NULL the kernel stores there the number of such slots
 * (0 when all ids are valid).  1 <= n_tokens <= 8, 1 <= top_k <= 32,
 * 1 <= n_expert <= 65534. */
qmv_status qmv_mul_mat_vec_id(int type, const void *W, int64_t n_expert, int64_t M, int64_t K,
                              const void *xq, const int32_t *ids, int n_tokens, int top_k, float *y,
                              int32_t *dev_status, void *stream);

/* ---- GEMV with the activation quantization fused in ---------------------------
 * The same products with fp32 activations: x holds ncols columns of K floats
 * (MoE: one column per token), column c at x + c*ldx (ldx >= K, x 4-byte
 * aligned; 16-byte alignment of x and of ldx*4 enables 128-bit loads).  Each
 * CTA quantizes x to q8_1 in shared memory with the arithmetic of
 * qmv_quantize_q8_1 (mul_mat_vec_q page, sections "激活的量化" and "PDL":
 * here the quantize pass is not a separate kernel at all), so y is
 * bit-identical to qmv_quantize_q8_1 followed by the q8_1-input call, with one
 * kernel launch instead of two.  Available for Q4_0 and Q4_K with K a
 * multiple of 256 and for Q6_K with K a multiple of 2048, W (and W_gate)
 * 16-byte aligned; otherwise returns QMV_ERR_SHAPE or QMV_ERR_ALIGN before
 * launching (QMV_ERR_TYPE for a type that is not a weight type), and the
 * q8_1-input calls apply.  Arguments, limits, outputs and error behaviour
 * are otherwise those of the calls above. */
qmv_status qmv_mul_mat_vec_f32(int type, const void *W, int64_t M, int64_t K, const float *x, int64_t ldx,
                               int ncols, float *y, void *stream);

qmv_status qmv_mul_mat_vec_gate_up_swiglu_f32(int type, const void *W_gate, const void *W_up, int64_t M,
                                              int64_t K, const float *x, int64_t ldx, int ncols, float *y,
                                              void *stream);

qmv_status qmv_mul_mat_vec_id_f32(int type, const void *W, int64_t n_expert, int64_t M, int64_t K,
                                  const float *x, int64_t ldx, const int32_t *ids, int n_tokens, int top_k,
                                  float *y, int32_t *dev_status, void *stream);

/* ---- fused epilogue extras -----------------------------------------------------
 * The mul_mat_vec_q page, section "融合:把 gate、bias 和 SwiGLU 塞进同一个 kernel",
 * lists what its fused launch can carry besides the gate matrix: a bias on
 * the up (x) output and one on the gate output, added before the GLU, and a
 * MoE shared expert served as one more slice of the same grid.
 *
 * qmv_mul_mat_vec_fused: y = W_up . x (+ bias) when W_gate is NULL, else
 *   y = (W_up . x + bias) * silu(W_gate . x + gate_bias), per column.
 *   Exactly one of xq (q8_1 activations, as for qmv_mul_mat_vec) and x
 *   (fp32 activations, column c at x + c*ldx, as for qmv_mul_mat_vec_f32;
 *   ldx is ignored for xq) is non-NULL.  bias and gate_bias are NULL or
 *   fp32 [M] (4-byte aligned), the same for every column; gate_bias needs
 *   W_gate.  The biases are read after the kernel has waited for the
 *   previous kernel on the stream (so earlier work on the stream may write
 *   them), through the read-only path: nothing may write them while the call
 *   runs.  With both biases NULL the result equals qmv_mul_mat_vec(_f32) or
 *   qmv_mul_mat_vec_gate_up_swiglu(_f32) bit for bit.  Shapes and alignment
 *   as for the _f32 calls (the streaming kernel only: Q4_0 / Q4_K with K a
 *   multiple of 256, Q6_K with K a multiple of 2048, W_up and W_gate 16-byte
 *   aligned).  Errors: QMV_ERR_NULL (no activations, y NULL), QMV_ERR_SHAPE
 *   (both activations given, gate_bias without W_gate, shape), QMV_ERR_ALIGN,
 *   QMV_ERR_NCOLS (ncols outside 1..8), QMV_ERR_TYPE; all before launching.
 *
 * qmv_mul_mat_vec_id_fused: qmv_mul_mat_vec_id(_f32) (one of xq / x, as
 *   above) with the MoE fusions of the same section:
 *   - W_gate (nullable): the experts' gate matrices, laid out like W_up
 *     ([n_expert][M][row bytes], 16-byte aligned).  With it, every routed
 *     slot gets y[t][k] = (W_up[e] . x_t) * silu(W_gate[e] . x_t),
 *     e = ids[t][k], in one pass over both matrices of each picked expert.
 *   - W_shared_up (nullable): a shared expert applied to every token,
 *     y_shared[t*M + r] = (W_shared_up . x_t)[r], or with a gate
 *     (W_shared_gate) (W_shared_up . x_t) * silu(W_shared_gate . x_t), for
 *     t < n_tokens; each one [M][row bytes] matrix (16-byte aligned) and
 *     y_shared fp32 [n_tokens][M].
 *   W_shared_up and y_shared are both NULL or both set, and a gated launch
 *   (W_gate set) with a shared expert needs W_shared_gate, a plain one must
 *   not pass it (QMV_ERR_NULL / QMV_ERR_SHAPE otherwise).  The routed
 *   outputs, invalid-id handling and dev_status are those of
 *   qmv_mul_mat_vec_id; one launch serves the routed and the shared
 *   experts. */
qmv_status qmv_mul_mat_vec_fused(int type, const void *W_up, const void *W_gate, int64_t M, int64_t K,
                                 const void *xq, const float *x, int64_t ldx, int ncols, const float *bias,
                                 const float *gate_bias, float *y, void *stream);

/* qmv_mul_mat_vec_fused_q8_1: qmv_mul_mat_vec_fused of one column (ncols
 * must be 1) whose result is also written as q8_1 blocks, ready to be the
 * activations of the next GEMV: yq receives qmv_q8_1_bytes(M, 1) bytes, the
 * blocks qmv_quantize_q8_1 would write for y with K = M (the 512-padding
 * included, as zero blocks), bit for bit.  The pages quantize each
 * activation vector in a pass of its own before the GEMV (mul_mat_vec_q
 * page, section "激活的量化"); here the producing GEMV does it in its
 * epilogue: every CTA owns whole 32-row blocks of y, keeps their values in
 * shared memory and quantizes them once its warps are done, so the consumer
 * reads 36 bytes per 32 values instead of 128 and needs no quantize pass.
 * y (fp32 [M]) is optional: NULL writes only yq; otherwise y equals
 * qmv_mul_mat_vec_fused's bit for bit.  yq must be 4-byte aligned; the other
 * arguments, shapes and errors are those of qmv_mul_mat_vec_fused
 * (QMV_ERR_NULL for yq NULL, QMV_ERR_NCOLS for ncols != 1).  A warp whose
 * wait for its cluster partner's share of x ran out (qmv_device_fault, code
 * 2) leaves NaN in its rows of y and a NaN scale in their blocks. */
qmv_status qmv_mul_mat_vec_fused_q8_1(int type, const void *W_up, const void *W_gate, int64_t M, int64_t K,
                                      const void *xq, const float *x, int64_t ldx, int ncols, const float *bias,
                                      const float *gate_bias, float *y, void *yq, void *stream);

qmv_status qmv_mul_mat_vec_id_fused(int type, const void *W_up, const void *W_gate, int64_t n_expert,
                                    int64_t M, int64_t K, const void *xq, const float *x, int64_t ldx,
                                    const int32_t *ids, int n_tokens, int top_k, float *y,
                                    const void *W_shared_up, const void *W_shared_gate, float *y_shared,
                                    int32_t *dev_status, void *stream);

/* ---- fault reporting -------------------------------------------------------- */

/* Reads and clears the sticky device fault word of the current device: 0 if
 * no kernel's bounded wait has run out since the last call, else the OR of
 * nonzero codes (2: a cluster partner's share of the staged fp32 activations
 * did not arrive within the wait limit).  A warp whose wait ran out computes
 * nothing: it writes NaN to every output of its rows and returns, so a bad
 * result cannot pass for a good one.  Callers of the fp32-input plain and
 * gate/up calls (and of qmv_mul_mat_vec_fused with fp32 x) should read this
 * word after synchronizing before they trust those outputs.  Synchronous
 * (waits for the device).  The pages have no counterpart: their kernels have
 * no spin-waits; this word is the library's own report of its one bounded
 * wait. */
qmv_status qmv_device_fault(unsigned int *code);

/* ---- tuning (process-wide) -----------------------------------------------------
 * Overrides the launch geometry the library picks for the streaming GEMV of
 * `type` (0 = keep the built-in choice for that field).  Meant for tuning
 * sweeps; results are identical for every setting.
 *   Q4_0 / Q4_K (tile kernel): threads = threads per CTA (multiple of 32,
 *     <= 384; all of them stage the activations, as many warps as the row
 *     groups and shared memory allow also stream weights); slice_units = units of 144 bytes per tile row (4, 8 or 16:
 *     tiles of 8, 4 or 2 rows; 8 and 2 only for one plain column);
 *     stages = tile buffers per warp (1..4); ctas_per_sm = CTAs per SM;
 *     smem_share = a CTA takes at most 1/smem_share of an SM's shared
 *     memory (1..4, default 2, which leaves room for the next kernel).
 *   Q6_K: the same tile kernel with tiles of 4 rows x 8 super-blocks
 *     (slice_units is ignored).
 *   cluster: CTAs per thread-block cluster for the fp32-input plain and
 *     gate/up calls (1..8; 1 = no cluster), which share the quantization of
 *     the activations among the cluster's CTAs (default 2).
 * Returns QMV_ERR_TYPE for a non-weight type, QMV_ERR_SHAPE for values out of
 * range. */
qmv_status qmv_set_tuning(int type, int threads, int slice_units, int stages, int ctas_per_sm, int smem_share,
                          int cluster);

/* Two more launch-geometry overrides of the streaming GEMV of `type`, for
 * sweeps (0 keeps the built-in choice; results are identical for every
 * setting): dec_warps = most warps per CTA that stream and decode weight tiles
 * (1..12); pre_tiles = tiles each of those warps requests before waiting for
 * the previous kernel on the stream (1..4, at most the ring's stages; the
 * rest of the ring is requested once the activations are staged).  Returns
 * QMV_ERR_TYPE for a non-weight type, QMV_ERR_SHAPE for values out of range. */
qmv_status qmv_set_stream_tuning(int type, int dec_warps, int pre_tiles);

/* How many of the decoding warps (the first ones) request their early tiles
 * before the dependency wait (1..12; 0 = all of them, the default); the
 * others request theirs after the activations are staged.  For sweeps of the
 * trade-off between weight bytes in flight across the kernel boundary and
 * the activation loads that queue behind them; results are identical for
 * every setting.  Returns QMV_ERR_TYPE / QMV_ERR_SHAPE as above. */
qmv_status qmv_set_early_warps(int type, int early_warps);

/* Delay, in ns, between the start of a CTA and its early weight requests, for
 * launches of `type` in which the next kernel's CTA fits beside this one on
 * the SM and either every warp requests all of its tiles before the
 * dependency wait (the 4096x4096 class of shapes) or the activations are fp32
 * (the _f32 and fused calls given x).  Such a CTA typically starts just as the
 * kernel beside it passes its own dependency wait; holding the requests back
 * lets that kernel's activation loads reach the memory system first, while
 * the tiles still land long before this launch needs them; fp32-input
 * launches so held back also request every warp's whole ring of tiles early.
 * ns: 1..100000 sets the delay, 0 restores the built-in defaults (400 ns for
 * q8_1 input, 700 ns for fp32 input, measured on GB300 with the library's
 * GEMVs back to back on one stream), -1 turns it off (fp32-input launches
 * then request one tile per warp early).  The hold-back pays only while the
 * kernel before this one on the stream still runs (another GEMV of this
 * library, which lets this launch start early); where the CTA's last warp
 * neither decodes nor requests tiles early, it waits for that kernel at once
 * and ends the hold-back as soon as the wait returns.  After a kernel
 * launched without programmatic dependent launch the CTAs start only once it
 * has finished, and what remains of the hold-back and the fuller early
 * requests still costs: measured on GB300, a Q4_K fp32-input GEMV right
 * after a PyTorch elementwise kernel took 11.14 instead of 10.22 us at
 * 12288x4096, 7.85 instead of 7.45 at 4096x4096 and 12.25 instead of 11.70
 * at 4096x11008 with the defaults (without the early end: 11.82, 8.55,
 * 12.81); back to back 7.28, 4.37 and 9.01 us instead of 7.34, 4.62 and
 * 8.88.  Turn it off where the GEMVs mostly follow other kernels.  Results
 * are identical for every setting.
 * Returns QMV_ERR_TYPE / QMV_ERR_SHAPE as above.  (A tuning entry point of
 * this library; the pages have no counterpart.) */
qmv_status qmv_set_early_delay(int type, int ns);

/* Column count from which the plain GEMV of `type` (qmv_mul_mat_vec, its
 * fp32-input and fused forms) decodes with the tensor cores instead of the
 * per-column dp4a: 8-row tiles multiplied by all columns at once with
 * mma.sync (fp16 operands holding the exact 4-bit and int8 codes, fp32
 * accumulators holding the exact integer block dots), then the same fp32
 * block scaling.  Q4_K only (other types ignore it).  min_cols: 1..8, 9 =
 * never, 0 = the built-in default (never: on GB300 this decode measured
 * slower than dp4a at every column count up to 8; it is kept for that
 * comparison and for other parts).  Results agree with the dp4a decode to
 * fp32 rounding of the scaled sums (not bit for bit); q8_1 and fp32 input
 * stay bit-identical to each other at every setting.  Returns QMV_ERR_TYPE for
 * a non-weight type, QMV_ERR_SHAPE for values out of range. */
qmv_status qmv_set_mma_min_cols(int type, int min_cols);

/* Diagnostic: reads every 16-byte piece of the device buffer buf (bytes, a
 * multiple of 16; buf 16-byte aligned) once, with the GEMV weight stream's
 * load width (128-bit loads cached in L2 only) over 4 CTAs per SM, so that
 * timing it gives this device's read-only streaming ceiling.  *sink (device,
 * 4 bytes) is written only in the practically impossible case that one
 * thread's XOR of the words it read equals 0x9E3779B9 (this keeps the loads
 * from being optimised away).  Asynchronous on stream. */
qmv_status qmv_read_bandwidth_probe(const void *buf, size_t bytes, unsigned int *sink, void *stream);

/* The launch the library would make for a plain (gate_up = 0) or fused
 * gate/up SwiGLU (gate_up = 1) GEMV of `type` with M rows, K columns and
 * ncols activation columns, from q8_1 (fp32_input = 0) or fp32 input
 * (fp32_input = 1), on the current device with the current tuning: weights
 * and activations are taken as 16-byte aligned.  Nothing is launched and no
 * memory is touched.  Fills *info; returns the status the GEMV call itself
 * would return for these shapes (QMV_ERR_NULL if info is NULL). */
typedef struct {
    int tile_kernel;    /* 1: the streaming tile kernel; 0: the generic kernel */
    int tensor_cores;   /* 1: the tensor-core decode (qmv_set_mma_min_cols) */
    int rows_per_tile;  /* weight rows per warp tile (tile kernel) */
    int grid;           /* CTAs */
    int block;          /* threads per CTA */
    int cluster;        /* CTAs per cluster (1: none) */
    int stages;         /* tile buffers per decoding warp (tile kernel) */
    int dec_warps;      /* warps per CTA that stream and decode (tile kernel) */
    int pre_tiles;      /* tiles per warp requested before the dependency wait */
    size_t smem;        /* dynamic shared bytes per CTA */
} qmv_launch_info;
qmv_status qmv_describe_gemv(int type, int gate_up, int64_t M, int64_t K, int ncols, int fp32_input,
                             qmv_launch_info *info);

/* Environment override of the geometry knobs above, for tuning runs:
 * QMV_GEOM="type:key=value,key=value;type:..." with type q4_0, q4_K or q6_K
 * and keys threads, slice_units, stages, ctas_per_sm, smem_share, cluster,
 * dec_warps, pre_tiles, early_warps, early_delay_ns and mma_min_cols (the
 * arguments of qmv_set_tuning, qmv_set_stream_tuning, qmv_set_early_warps,
 * qmv_set_early_delay and qmv_set_mma_min_cols, same ranges).  It is read
 * once, before the first GEMV-family call is planned, and applied through
 * those setters; later setter calls override it.  A malformed spec or an
 * out-of-range value makes every GEMV-family call return QMV_ERR_CONFIG
 * (nothing is launched) for the life of the process. */

/* Enables (1, default) or disables (0) programmatic dependent launch for the
 * library's q8_1 and GEMV kernels.  When enabled, a GEMV may start streaming
 * its weights while the kernel before it on the stream is still finishing,
 * and reads activations, ids and writes outputs only after that kernel has
 * completed.  The weights must therefore not be written by a kernel that
 * signals early completion (griddepcontrol.launch_dependents); ordinary
 * kernels and copies are waited for as usual, and the library's own kernels
 * never write weights except qmv_quantize_weights, which launches
 * ordinarily. */
qmv_status qmv_set_pdl(int enable);

/* Checked mode (process-wide; off by default, or on when the environment
 * variable QMV_CHECKED is set to anything but "0" before the first call).
 * When on, every call also checks on the host, before it launches, that the
 * whole byte range it will read or write through each pointer argument lies
 * inside one device allocation known to the CUDA driver (cuMemGetAddressRange):
 *   W (each weight matrix)   M * qmv_row_bytes(type, K) bytes, times n_expert
 *                            for the MoE calls
 *   xq                       qmv_q8_1_bytes(K, ncols or n_tokens)
 *   x                        ((ncols - 1) * ldx + K) * 4 bytes
 *   y                        ncols * M * 4 (MoE: n_tokens * top_k * M * 4)
 *   ids / dev_status         n_tokens * top_k * 4 / 4
 *   bias, gate_bias          M * 4;  y_shared  n_tokens * M * 4
 * A range that runs past its allocation, or a pointer outside every device
 * allocation the driver tracks (pageable host memory, a freed buffer),
 * returns QMV_ERR_RANGE and launches nothing.  The check works at the
 * granularity of driver allocations: a sub-allocator (PyTorch's caching
 * allocator, for one) hands out slices of larger allocations, and an overrun
 * that stays inside the same allocation is not seen.  It costs one driver
 * query per pointer, so it is meant for debugging and tests; under CUDA graph
 * capture it runs once, when the call is captured.  Returns QMV_OK. */
qmv_status qmv_set_checked(int enable);

#ifdef __cplusplus
}
#endif
#endif /* QMV_H */
