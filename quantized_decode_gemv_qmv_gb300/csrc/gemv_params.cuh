// Launch parameters shared by the GEMV kernels (tile kernel, generic kernel).
#pragma once

#include "common.cuh"

namespace qmv {

enum Mode { MODE_PLAIN = 0, MODE_GATE = 1, MODE_MOE = 2, MODE_DEBUG = 3, MODE_MOE_GATE = 4 };

struct GemvParams {
    const uint8_t *W;    // weights (MoE: expert 0); GATE: the up matrix
    const uint8_t *W2;   // GATE: the gate matrix; MOE, MOE_GATE: the shared expert's (up) matrix (nullable)
    const uint8_t *W3;   // MOE_GATE: the experts' gate matrices [n_expert][M][row_bytes]
    const uint8_t *W4;   // MOE_GATE with a shared expert: its gate matrix
    const uint8_t *xq;   // q8_1 activations, column c at xq + c*xq_col_bytes
    const float *xf;     // fp32 activations quantized in place (tile kernel), column c at xf + c*ldx; or null
    int64_t ldx;
    float *y;            // PLAIN/GATE: y[c*ldy + r] (nullable when yq is set); MOE: y[(t*top_k + k)*M + r]
    uint8_t *yq;         // PLAIN/GATE (tile kernel): y quantized to q8_1 as well, column c at yq + c*yq_col_bytes (nullable)
    int32_t *dbg;        // DEBUG: per-sub-block int sums
    const int32_t *ids;  // MOE: [n_tokens][top_k]
    int32_t *status;     // MOE: number of invalid ids (nullable)
    const float *bias;       // PLAIN/GATE: [M] added to every column's (up) output (nullable)
    const float *gate_bias;  // GATE: [M] added to the gate output before silu (nullable)
    float *y_shared;         // MOE with a shared expert (W2): y_shared[t*M + r] = (W2 x_t)[r]
    unsigned int *fault;     // sticky device word: kernels OR in a code when a bounded wait runs out
    int64_t M;
    int64_t ldy;
    int64_t row_bytes;
    int64_t xq_col_bytes;
    int64_t expert_bytes;
    int64_t yq_col_bytes;  // yq: bytes per column (yq_nb_pad blocks of 36 bytes)
    int64_t n_groups;    // tile kernel: ceil(M / rows per tile)
    int K;
    int ncols;           // active columns (PLAIN/GATE/DEBUG)
    int n_tokens, top_k, n_expert;
    int units_per_row;   // tile kernel: K / 256
    int stages;          // tile kernel: tile buffers per warp
    int dec_warps;       // tile kernel: warps that stream and decode (the first ones; the rest only stage)
    int pre_tiles;       // tile kernel: tiles per warp requested before the dependency wait (1..stages)
    int early_warps;     // tile kernel: warps that make those early requests (the first ones; >= dec_warps: all)
    int early_delay;     // tile kernel: SM clock cycles from the CTA's start to its early requests (0: none)
    uint32_t act_bytes;  // tile kernel: shared bytes of the activation area
    uint32_t raw_off;    // tile kernel: offset of the raw q8_1 copy inside the activation area (0: none)
    uint32_t ybuf_off;   // yq: offset of the CTA's fp32 rows of y inside the activation area
    int ybuf_rows;       // yq: rows of that buffer per column (whole 32-row blocks)
    int yq_nb_pad;       // yq: blocks per column, the 512-padding included
    unsigned long long *trace;  // diagnostics: per-CTA timestamps [entry, waited, staged, done] (nullable)
    int withhold;        // test only: the rank-1 CTA of each fp32-staging cluster keeps its share to itself
    unsigned long long withhold_wait_ns;  // test only: how long the rank-0 CTA then waits for that share
};

// SwiGLU's gate nonlinearity, silu(g) = g / (1 + e^-g) (CUDA expf).
__device__ __forceinline__ float silu_f32(float g)
{
    return g / (1.0f + expf(-g));
}

}  // namespace qmv
