// Warp-tile streaming GEMV for the 144-byte-unit formats (Q4_K super-blocks;
// Q4_0 in runs of 8 blocks), sm_103a.
//
// Method: "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q" (vec_dot_q4_0_q8_1_impl,
// vec_dot_q4_K_q8_1_impl_vmmq), evaluated per unit by unit_dot.
//
// Design (GB300-specific):
//   * Warp tiles of RW rows x UW = 32/RW units (4,608 bytes: one unit per
//     lane).  Each lane copies 9 of the tile's 288 16-byte pieces with
//     cp.async; every warp-wide copy instruction covers 512 contiguous bytes
//     of one row segment, so DRAM and L2 see whole sectors, and the data never
//     occupies registers while in flight.
//   * Each warp owns a ring of `stages` tile buffers.  The first `stages`
//     tiles are requested before the kernel waits for the previous grid
//     (programmatic dependent launch), so a GEMV's first weight bytes are on
//     their way while the kernel before it drains; afterwards the warp refills
//     a buffer as soon as it has decoded it.  Completion is the hardware's
//     cp.async.wait_group: the kernel has no spin-waits and cannot hang on a
//     copy.
//   * Tile rows are padded in shared memory so that the 8 lanes of a 128-bit
//     read phase (RW rows of 8/RW units) hit distinct bank quads; lane (u, r)
//     decodes unit u of row r.  The RW lanes of one unit read the same
//     activation addresses, which shared memory serves by broadcast.
//   * One CTA per SM by default, of up to 12 warps and at most half of the
//     SM's shared memory (and, for one column, registers), so that the next
//     GEMV's CTAs fit beside it and have their first tiles in flight before
//     this one ends.  Every warp owns a balanced contiguous range of RW-row
//     groups; a row's partial sums meet in a warp-shuffle reduction (no
//     cross-warp traffic).
#pragma once

#include "gemv_mma.cuh"
#include "gemv_units.cuh"
#include "q8_1.cuh"

#include <utility>

namespace qmv {

constexpr int TILE_MAX_THREADS = 384;
constexpr int TILE_MAX_STAGES = 4;
constexpr int STAGE_BATCH = 4;  // q8_1 staging: 16-byte loads in flight per thread
constexpr int TRACE_WORDS = 6;  // timeline stamps per CTA (qmv_debug_trace)
constexpr int MOE_MAX_SLOTS = 256;  // n_tokens * top_k <= 8 * 32
constexpr int MOE_COL_WEIGHT = 6;   // MoE grid split: an expert's work ~ 6 + the tokens (columns) it serves

// Tile geometry for format F and RW rows per tile: UW = 32/RW units per tile
// row (one per lane), the row segment SEG 16-byte pieces long, copied
// row-wise (LPR = 32/RW lanes per row, NJ instructions each, copy_row_pieces).  Rows are padded in shared memory (stride SS):
//   Q4_0 / Q4_K (144-byte units): SS/16 = 8/RW mod 8, so the 8 lanes of a
//     128-bit read phase (RW rows of 8/RW units) hit distinct bank quads;
//   Q6_K (210-byte units, RW = 4): SS = 1,696 bytes = 32 mod 128, which spreads
//     the 32 lanes' 32-bit word reads of 2-byte aligned super-blocks over the
//     banks (at most 2-way, 1.5 on average) and leaves room for the
//     over-read of the last super-block of a row;
//   TC (the tensor-core decode, gemv_mma.cuh; Q4_K, RW = 8): SS = 608 = 96
//     mod 128, so the 16 lanes of a 64-bit read phase (4 rows x 32 bytes) hit
//     distinct banks.
template <int F, int RW, bool TC = false>
struct TileGeom {
    static constexpr int UW = 32 / RW;
    static constexpr int UNIT = unit_bytes<F>();
    static_assert((UW * UNIT) % 16 == 0, "a tile row segment must be whole 16-byte pieces");
    static_assert(F != FMT_Q6_K || RW == 4, "Q6_K tiles are 4 rows x 8 super-blocks");
    static constexpr int SEG = UW * UNIT / 16;
    static constexpr int LPR = 32 / RW;                // row-wise copy: lanes per tile row
    static constexpr int NJ = (SEG + LPR - 1) / LPR;   // row-wise copy: instructions per lane
    static constexpr int SS = F == FMT_Q6_K ? UW * UNIT + 16
                              : TC ? UW * UNIT + 32
                                   : (RW == 1 ? UW * UNIT : UW * UNIT + ((8 / RW - UW % 8 + 8) % 8) * 16);
    static_assert(!TC || (F == FMT_Q4_K && RW == MMA_RW && SS % 128 == 96), "tensor-core tiles: Q4_K, 8 rows");
    static constexpr int TB = RW * SS;
};

// Host-visible geometry: bytes of one tile buffer (0: no such tile); tc: the
// tensor-core tiles.
inline int tile_bytes_rt(int type, int rw, bool tc = false)
{
    if (tc) return (type == FMT_Q4_K && rw == MMA_RW) ? TileGeom<FMT_Q4_K, MMA_RW, true>::TB : 0;
    if (type == FMT_Q6_K) return rw == 4 ? TileGeom<FMT_Q6_K, 4>::TB : 0;
    switch (rw) {
    case 2: return TileGeom<FMT_Q4_K, 2>::TB;
    case 4: return TileGeom<FMT_Q4_K, 4>::TB;
    case 8: return TileGeom<FMT_Q4_K, 8>::TB;
    default: return 0;
    }
}

// Activation staging of the tile kernel.  Every CTA reads the same few KB of
// q8_1 blocks right after the dependency wait, while its weight copies keep
// L2 busy, so the reads go out as whole 128-bit pieces (one request per 16
// bytes instead of one per 4) into a raw shared copy, which is then repacked
// like stage_units_activations (natural-order codes, per-block scalars).
// Falls back to stage_units_activations when xq is not 16-byte aligned or no
// raw area was planned.
//
// With fp32 input (p.xf) the activations are quantized here, straight into the
// repacked layout, with the q8_1 block arithmetic of the standalone quantizer
// (q8_1.cuh): the staged values, and so y, are bit-identical to quantizing
// first and passing the q8_1 blocks.  In a cluster of ncta CTAs, CTA crank
// quantizes only its share of the blocks (a contiguous 1/ncta of them) and
// stores each result into the shared memory of every CTA of the cluster
// (distributed shared memory), so the work is not repeated in every CTA; the
// caller has made sure every CTA of the cluster is running, and completes the
// exchange with a cluster barrier.  Instrumented kernels only: WITHHOLD (when
// p.withhold is set, the CTA of rank 1 keeps its share to itself) and tr, the
// CTA's timeline (thread 0 stamps [2] when its first activation loads have
// returned and [3] when its own part of the staging is done).
template <int F, int NC, bool WITHHOLD, typename ColFn>
__device__ __forceinline__ void stage_tile_activations(const GemvParams &p, uint8_t *smem, int n_active, ColFn src_col,
                                                       uint32_t crank, uint32_t ncta, uint32_t xbar,
                                                       unsigned long long *tr)
{
    if (p.xf != nullptr) {
        const int U = p.units_per_row;
        const int nblk = U * 8;                 // q8_1 blocks per column (K = 256 U)
        const int n_all = n_active * nblk;      // blocks of all columns
        const int blk0 = static_cast<int>(static_cast<int64_t>(crank) * n_all / ncta);
        const int blk1 = static_cast<int>(static_cast<int64_t>(crank + 1) * n_all / ncta);
        const int tasks = (blk1 - blk0) * 4;    // 4 lanes per block
        const bool vec = ((reinterpret_cast<uintptr_t>(p.xf) | static_cast<uintptr_t>(p.ldx * 4)) & 15u) == 0;
        const uint32_t act_qs = smem_u32(smem);
        const uint32_t act_sc = act_qs + static_cast<uint32_t>(NC * U * ACT_QS_STRIDE);
        const int rounds = (tasks + blockDim.x - 1) / blockDim.x;  // the same for every thread
        // One round (blockDim.x tasks) at a time, the next round's loads issued
        // before this round's arithmetic: the load latency overlaps the
        // quantization while the code holds a single copy of it (the staging
        // runs once per CTA, from a cold instruction cache when kernels of
        // another instance share the SM).
        auto load = [&](int r, float (&v)[8]) {
            const int t = r * blockDim.x + threadIdx.x;
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
            if (t < tasks) {
                const int g = blk0 * 4 + t;
                const int c = NC == 1 ? 0 : g / (nblk * 4);
                const int rem = g - c * nblk * 4;
                q8_1_load8(p.xf + (size_t)src_col(c) * p.ldx, (int64_t)(rem >> 2) * QK8_1 + 8 * (rem & 3), p.K, vec, v);
            }
        };
        float v[8];
        if (rounds > 0) load(0, v);
        for (int r = 0; r < rounds; ++r) {
            float vn[8];
            load(r + 1, vn);  // zeros past the last round
            const int t = r * blockDim.x + threadIdx.x;
            uint32_t w0, w1, ds;
            int S, part;
            q8_1_block_group4(v, w0, w1, ds, S, part);
            if (tr && r == 0 && threadIdx.x == 0) tr[2] = global_timer_ns();
            // half sums: codes 0..15 (lanes 0, 1 of the group), 16..31 (lanes 2, 3)
            const int half = part + __shfl_xor_sync(0xffffffffu, part, 1);
            const int other = __shfl_xor_sync(0xffffffffu, half, 2);
            if (t < tasks) {
                const int g = blk0 * 4 + t;
                const int c = NC == 1 ? 0 : g / (nblk * 4);
                const int rem = g - c * nblk * 4;
                const int n = rem >> 2, j = rem & 3;
                const int u = n >> 3, sub = n & 7;
                const uint32_t dq = act_qs + static_cast<uint32_t>((c * U + u) * ACT_QS_STRIDE + 32 * sub + 8 * j);
                const uint32_t sc = act_sc + static_cast<uint32_t>((c * U + u) * act_sc_stride<F>());
                uint32_t off[3], val[3];
                const int nw = act_scalar_words<F>(sub, ds, S, half, other, off, val);
                if (ncta == 1) {
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dq), "r"(w0), "r"(w1) : "memory");
                    if (j == 0) {
#pragma unroll
                        for (int i = 0; i < 3; ++i)
                            if (i < nw) asm volatile("st.shared.u32 [%0], %1;" ::"r"(sc + off[i]), "r"(val[i]) : "memory");
                    }
                } else {
                    // this CTA's copy directly; the others' through st.async,
                    // counted on their mbarrier (cluster_share_bytes per block)
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dq), "r"(w0), "r"(w1) : "memory");
                    if (j == 0) {
#pragma unroll
                        for (int i = 0; i < 3; ++i)
                            if (i < nw) asm volatile("st.shared.u32 [%0], %1;" ::"r"(sc + off[i]), "r"(val[i]) : "memory");
                    }
                    for (uint32_t q = 0; q < ncta; ++q) {
                        if (q == crank || (WITHHOLD && p.withhold && crank == 1)) continue;
                        const uint32_t bq = mapa_shared(xbar, q);
                        st_async_v2(mapa_shared(dq, q), w0, w1, bq);
                        if (j == 0) {
                            const uint32_t scq = mapa_shared(sc, q);
#pragma unroll
                            for (int i = 0; i < 3; ++i)
                                if (i < nw) st_async_u32(scq + off[i], val[i], bq);
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = vn[i];
        }
        if (tr && threadIdx.x == 0) tr[3] = global_timer_ns();
        return;
    }
    if (p.raw_off == 0 || (reinterpret_cast<uintptr_t>(p.xq) & 15u) != 0) {
        stage_units_activations<F, NC>(p, smem, n_active, src_col);
        return;
    }
    const int U = p.units_per_row;
    const int nblk = U * 8;   // q8_1 blocks per column
    const int n16 = U * 18;   // 16-byte pieces per column (8 blocks x 36 bytes per unit)
    uint8_t *raw = smem + p.raw_off;
    const int total16 = n_active * n16;
    for (int base = 0; base < total16; base += STAGE_BATCH * blockDim.x) {  // STAGE_BATCH loads in flight
        uint4 v[STAGE_BATCH];
#pragma unroll
        for (int r = 0; r < STAGE_BATCH; ++r) {
            const int idx = base + r * blockDim.x + threadIdx.x;
            if (idx < total16) {
                const int c = idx / n16;
                const int k = idx - c * n16;
                v[r] = ld_cg_u4(p.xq + (size_t)src_col(c) * p.xq_col_bytes + (size_t)k * 16);
            }
        }
#pragma unroll
        for (int r = 0; r < STAGE_BATCH; ++r) {
            const int idx = base + r * blockDim.x + threadIdx.x;
            if (idx < total16) *reinterpret_cast<uint4 *>(raw + (size_t)idx * 16) = v[r];
        }
        if (tr && base == 0 && threadIdx.x == 0) tr[2] = global_timer_ns();
    }
    __syncthreads();
    uint8_t *act_qs = smem;
    uint8_t *act_sc = smem + (size_t)NC * U * ACT_QS_STRIDE;
    for (int idx = threadIdx.x; idx < NC * nblk; idx += blockDim.x) {
        const int c = idx / nblk;
        const int n = idx - c * nblk;
        uint32_t w[9] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (c < n_active) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(raw + (size_t)idx * Q8_1_BYTES);
#pragma unroll
            for (int i = 0; i < 9; ++i) w[i] = src[i];
        }
        int S_lo = 0, S_hi = 0;
#pragma unroll
        for (int i = 1; i < 5; ++i) S_lo = dp4a_ss(w[i], 0x01010101u, S_lo);
#pragma unroll
        for (int i = 5; i < 9; ++i) S_hi = dp4a_ss(w[i], 0x01010101u, S_hi);
        const int u = n >> 3, sub = n & 7;
        uint4 *dq = reinterpret_cast<uint4 *>(act_qs + ((size_t)c * U + u) * ACT_QS_STRIDE + 32 * sub);
        dq[0] = make_uint4(w[1], w[2], w[3], w[4]);
        dq[1] = make_uint4(w[5], w[6], w[7], w[8]);
        store_act_scalars<F>(act_sc + ((size_t)c * U + u) * act_sc_stride<F>(), sub, w[0], S_lo + S_hi, S_lo, S_hi);
    }
    if (tr && threadIdx.x == 0) tr[3] = global_timer_ns();
}

// Bytes the other CTAs of a cluster store into this CTA's shared memory while
// staging fp32 input (stage_tile_activations): every block of their shares of
// the n_all blocks, as 4 lanes x 8 bytes of codes plus the block's scalar
// words (act_scalar_words: 2, or 3 for Q6_K).
template <int F>
__device__ __forceinline__ uint32_t cluster_share_bytes(int n_all, uint32_t crank, uint32_t ncta)
{
    const int blk0 = static_cast<int>(static_cast<int64_t>(crank) * n_all / ncta);
    const int blk1 = static_cast<int>(static_cast<int64_t>(crank + 1) * n_all / ncta);
    constexpr int per_block = 4 * 8 + 4 * (F == FMT_Q6_K ? 3 : 2);
    return static_cast<uint32_t>((n_all - (blk1 - blk0)) * per_block);
}

// A warp whose activations never arrived: code 2 in the fault word, and NaN in
// every output of its rows r0 .. r_end-1 (y if given, and the CTA's buffer of
// rows for the q8_1 output, whose blocks then carry a NaN scale:
// mark_nan_block_group4), so a bad result cannot pass for a good one.  Out of line, so that the code the warp
// runs when the activations do arrive stays as short as without it (inline,
// it made the step's launches about 0.5 % slower on GB300).
static __device__ __noinline__ void give_up_rows(float *y, int64_t ldy, int ncols, int64_t r0, int64_t r_end, int lane,
                                                 unsigned int *fault, float *ybuf, int ybuf_rows, int64_t yrow0)
{
    if (lane == 0 && fault) atomicOr(fault, FAULT_CLUSTER_STAGING);
    for (int64_t r = r0 + lane; r < r_end; r += 32)
        for (int c = 0; c < ncols; ++c) {
            if (y) y[(size_t)c * ldy + r] = __int_as_float(0x7fc00000);
            if (ybuf) ybuf[c * ybuf_rows + (r - yrow0)] = __int_as_float(0x7fc00000);
        }
}

// A block holding a NaN (the rows of a warp that gave up, see give_up_rows)
// gets a NaN scale, so that no consumer can take it for a good block: the
// quantizer's amax would pass over the NaN (fmaxf returns the other operand)
// and its code would not show it either.  Called like q8_1_block_group4, by
// every lane of the warp, lanes 4g..4g+3 holding one block.
__device__ __forceinline__ void mark_nan_block_group4(const float (&v)[8], uint32_t &ds)
{
    int bad = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) bad |= v[i] != v[i] ? 1 : 0;
    bad |= __shfl_xor_sync(0xffffffffu, bad, 1);
    bad |= __shfl_xor_sync(0xffffffffu, bad, 2);
    if (bad) ds = (ds & 0xffff0000u) | 0x7e00u;
}

// The q8_1 output (p.yq): after the CTA barrier, the CTA's fp32 rows in ybuf
// (whole 32-row blocks from row yrow0, column c at ybuf + c*ybuf_rows) are
// quantized with the arithmetic of the standalone quantizer (q8_1.cuh), 4
// lanes per block, rows at and past M as zeros; the CTA holding the last block
// also writes the padding blocks (all zero bytes, the quantization of zeros).
// Every thread of the CTA takes part (the group reductions shuffle over whole
// warps).
__device__ __forceinline__ void store_rows_q8_1(const GemvParams &p, const float *ybuf, int64_t b0, int64_t b1,
                                                int64_t n_blk)
{
    const int nb_cta = static_cast<int>(b1 - b0);
    const int n_out = nb_cta + (b1 == n_blk && b1 > b0 ? p.yq_nb_pad - static_cast<int>(n_blk) : 0);
    const int tasks = n_out * p.ncols * 4;
    const int rounds = (tasks + blockDim.x - 1) / blockDim.x;
    for (int rd = 0; rd < rounds; ++rd) {
        const int t = rd * blockDim.x + threadIdx.x;
        const bool ok = t < tasks;
        const int tt = ok ? t : 0;
        const int c = tt / (n_out * 4);
        const int rem = tt - c * n_out * 4;
        const int b = rem >> 2, j = rem & 3;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = (b0 + b) * 32 + 8 * j + i;
            v[i] = (ok && b < nb_cta && row < p.M) ? ybuf[c * p.ybuf_rows + static_cast<int>(row - b0 * 32)] : 0.f;
        }
        uint32_t w0, w1, ds;
        int sum, part;
        q8_1_block_group4(v, w0, w1, ds, sum, part);
        mark_nan_block_group4(v, ds);
        if (ok) {
            uint32_t *o = reinterpret_cast<uint32_t *>(p.yq + (size_t)c * p.yq_col_bytes + (size_t)(b0 + b) * Q8_1_BYTES);
            o[1 + 2 * j] = w0;
            o[2 + 2 * j] = w1;
            if (j == 0) o[0] = ds;
        }
    }
}

// One tile row's copy: lane kq of the row's LPR lanes copies its 16-byte
// pieces kq, kq + LPR, kq + 2 LPR, ... (the J-th at byte 16 (kq + LPR J) of
// both the row segment and its shared copy), so a lane's addresses are one
// base plus constant offsets and the copy costs one instruction per piece.
// Only pieces below lim are copied (a partial last k-tile).  Each instruction
// moves 16 LPR contiguous bytes of every row of the tile.  On GB300, against a
// per-piece division of one run of pieces over the warp: Q4_0 / Q4_K (144-byte
// units) the step 1.020 -> 1.002 ms and the MoE calls 5 % faster; Q6_K (with
// each lane's first piece rotated to a line boundary) 4096x14336 11.40 -> 10.96
// us and 5-8 columns 4-5 % faster, its 32000x4096 launch 2.6 % slower -- that
// one, two tiles per row group, takes the ROWRUN variant (whole warp on one
// row, 512 bytes per instruction): 21.75 -> 20.94 us.
template <int LPR, int SEG, int... J>
__device__ __forceinline__ void copy_row_pieces(uint32_t dst, const uint8_t *src, int kq, int lim,
                                                std::integer_sequence<int, J...>)
{
    if (lim >= SEG)
        ((((J + 1) * LPR <= SEG || kq + LPR * J < SEG) ? cp_async16_at<16 * LPR * J>(dst, src) : void()), ...);
    else
        ((kq + LPR * J < lim ? cp_async16_at<16 * LPR * J>(dst, src) : void()), ...);
}

// PROBE: the instrumented twin of a kernel (qmv_debug.h): the same code plus
// the timeline stores (p.trace) and the withheld share (p.withhold).  The
// ordinary kernels carry neither: the instructions would sit on the path from
// the dependency wait to the first decode, which every launch pays.
template <int F, int NC, int MODE, int RW, bool TC = false, bool PROBE = false, bool YQ = false, bool ROWRUN = false>
__global__ void __launch_bounds__(TILE_MAX_THREADS, (NC == 1 && MODE != MODE_DEBUG) ? 2 : 1)
    gemv_tiles_kernel(const GemvParams p)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    __shared__ int s_tok[8];
    __shared__ uint32_t s_slots[8];
    __shared__ int s_cnt;

    using G = TileGeom<F, RW, TC>;
    constexpr int UW = G::UW;                        // units per tile row
    constexpr int SEG = G::SEG;                      // 16-byte pieces per tile row
    constexpr int SS = G::SS;                        // shared bytes per tile row
    constexpr int TB = G::TB;                        // shared bytes per tile
    constexpr int UNIT = G::UNIT;                    // bytes per unit
    constexpr bool IS_MOE = MODE == MODE_MOE || MODE == MODE_MOE_GATE;
    constexpr int NM = (MODE == MODE_GATE || MODE == MODE_MOE_GATE) ? 2 : 1;  // matrices (up, gate)
    constexpr bool MMA = TC;  // tensor-core decode (gemv_mma.cuh): Q4_K, plain, up to 8 columns
    static_assert(!MMA || (F == FMT_Q4_K && MODE == MODE_PLAIN && NC == MMA_COLS), "tensor-core tiles: Q4_K plain");
    static_assert(!YQ || (!MMA && (MODE == MODE_PLAIN || MODE == MODE_GATE)), "q8_1 output: plain or gate/up, dp4a");
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = p.dec_warps;  // warps that stream and decode; the others only help staging
    const int U = p.units_per_row;
    const int r_l = lane % RW;  // this lane's row inside a tile
    const int u_l = lane / RW;  // this lane's unit inside a tile
    const int n_kt = (U + UW - 1) / UW;
    const int64_t rb = p.row_bytes;
    const int stages = p.stages;

    pdl_launch_dependents();
    // optional timeline (qmv_debug_trace, TRACE_WORDS stamps per CTA): entry,
    // after the dependency wait, first activation loads returned, own staging
    // done, activations complete in shared memory, last warp done
    unsigned long long *const trace = (PROBE && p.trace) ? p.trace + TRACE_WORDS * blockIdx.x : nullptr;
    if (trace && threadIdx.x == 0) trace[0] = global_timer_ns();
    // fp32 input in a cluster: the CTAs share the quantization (see
    // stage_tile_activations); this arrive lets the others know this CTA runs
    uint32_t crank = 0, ncta = 1;
    // fp32 staging in a cluster: the partners' shares complete on this
    // mbarrier.  It sits right after the used dynamic area (activations, then
    // every decoding warp's ring and scratch), inside the 128 bytes of
    // alignment slack the host adds: the slack before `smem` is a multiple of
    // 16 below 128, so at least 16 bytes of it remain after the used area.
    // (Static shared memory would cost the whole CTA 128 bytes of budget.)
    constexpr int WARP_EXTRA = MMA ? MMA_FAC_BYTES : 0;
    const uint32_t xbar =
        smem_u32(smem) + p.act_bytes + static_cast<uint32_t>(p.dec_warps * (p.stages * TB + WARP_EXTRA));
    if constexpr (MODE == MODE_PLAIN || MODE == MODE_GATE) {
        ncta = cluster_nctarank();
        if (ncta > 1) {
            crank = cluster_ctarank();
            if (!MMA && threadIdx.x == 0) {
                mbar_init(xbar, 1);
                fence_mbar_init();  // visible to the partners before they pass the cluster wait below
            }
            // Every CTA of the cluster runs (its shared memory may be written)
            // once this wait returns.  The CTAs of a cluster start together, so
            // it returns at once here, where the CTA has no copies in flight;
            // after the dependency wait it sat on the path to the staging (the
            // step 0.3 % slower on GB300).
            cluster_arrive_relaxed();
            cluster_wait();
        }
    }
    // This CTA's share of x's 32-value blocks (fp32 input: the blocks it will
    // quantize), fetched into L2 before the dependency wait, so that the
    // staging loads after it hit L2 instead of queueing for HBM.  Safe even
    // when the previous kernel writes x: L2 is where this GPU's global memory
    // is coherent, so its stores update the lines (only L1 could go stale,
    // and the staging loads bypass L1).  Issued at entry where the early
    // weight requests are held back (p.early_delay), else right after those
    // requests.  Measured on GB300 with activations not in L2: the step 1.030
    // -> 1.004 ms with the prefetch at entry; without the hold-back, qkv,
    // gate+up and down a further 1 % faster with it after their early
    // requests (o 7 % slower); with it, the step 0.6 % slower that way.
    auto prefetch_x = [&]() {
        if constexpr ((MODE == MODE_PLAIN || MODE == MODE_GATE) && !MMA) {
            if (p.xf != nullptr) {
                const int nblk = U * 8;
                const int n_all = p.ncols * nblk;
                const int b0 = static_cast<int>(static_cast<int64_t>(crank) * n_all / ncta);
                const int b1 = static_cast<int>(static_cast<int64_t>(crank + 1) * n_all / ncta);
                for (int b = b0 + static_cast<int>(threadIdx.x); b < b1; b += blockDim.x) {
                    const int c = b / nblk;
                    const float *a = p.xf + (size_t)c * p.ldx + (size_t)(b - c * nblk) * 32;
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
                }
            }
        }
    };
    if (p.early_delay > 0) prefetch_x();

    int n_active = p.ncols;
    int64_t row_base = 0;    // MoE: first row of this CTA's expert
    const uint8_t *W0 = p.W;  // first matrix (MoE: the experts, or the shared expert)
    const uint8_t *W1 = MODE == MODE_MOE_GATE ? p.W3 : p.W2;  // gate matrix (GATE, MOE_GATE)
    bool moe_shared = false;  // MoE: this CTA serves the shared expert
    int64_t cta_index = blockIdx.x, cta_count = gridDim.x;
    if constexpr (IS_MOE) {
        // Routing is known only here (ids come from the previous grid).  The
        // ids are read once into shared memory; the experts some token picks
        // are listed in ascending order (then the shared expert, if any) and
        // the grid is shared among them in proportion to their work, one CTA
        // each plus a share of the rest weighted by MOE_COL_WEIGHT + the
        // number of tokens they serve, so every SM works whatever the routing.
        // CTA 0 also zero-fills the outputs of invalid ids and counts them.
        __shared__ int s_ids[MOE_MAX_SLOTS];
        __shared__ int s_exp[MOE_MAX_SLOTS + 1];   // the picked experts ascending, then the shared one
        __shared__ int s_ntok[MOE_MAX_SLOTS + 1];  // tokens each listed expert serves
        __shared__ int s_eidx;
        __shared__ int64_t s_first, s_next;
        pdl_wait();
        const int n_slots = p.n_tokens * p.top_k;
        for (int s = threadIdx.x; s < n_slots; s += blockDim.x) s_ids[s] = ld_cg_s32(p.ids + s);
        __syncthreads();
        // slot s represents its id if the id is valid and no earlier slot holds it;
        // a representative's place in the list is the number of smaller represented ids
        __shared__ unsigned char s_isrep[MOE_MAX_SLOTS];
        __shared__ int s_nrouted;
        if (threadIdx.x == 0) s_nrouted = 0;
        for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
            const int e = s_ids[s];
            bool rep = e >= 0 && e < p.n_expert;
            for (int j = 0; j < s && rep; ++j) rep = s_ids[j] != e;
            s_isrep[s] = rep ? 1 : 0;
        }
        __syncthreads();
        for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
            if (!s_isrep[s]) continue;
            const int e = s_ids[s];
            int rank = 0;
            for (int j = 0; j < n_slots; ++j) rank += (s_isrep[j] && s_ids[j] < e) ? 1 : 0;
            s_exp[rank] = e;
            atomicAdd(&s_nrouted, 1);
        }
        __syncthreads();
        const int n_routed = s_nrouted;
        const int ne = n_routed + (p.W2 != nullptr ? 1 : 0);
        if (p.W2 != nullptr && threadIdx.x == 0) s_exp[n_routed] = p.n_expert;  // every token, its own output
        __syncthreads();
        for (int i = threadIdx.x; i < ne; i += blockDim.x) {
            const int e = s_exp[i];
            int n = 0;
            for (int t = 0; t < p.n_tokens; ++t) {
                bool hit = e == p.n_expert;
                for (int k = 0; k < p.top_k && !hit; ++k) hit = s_ids[t * p.top_k + k] == e;
                n += hit ? 1 : 0;
            }
            s_ntok[i] = n;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int64_t wsum = 0;
            for (int i = 0; i < ne; ++i) wsum += MOE_COL_WEIGHT + s_ntok[i];
            const int64_t G = gridDim.x, spare = G - ne;  // the planner gives every listable expert a CTA
            int64_t pre = 0, start = 0;
            s_eidx = ne - 1;
            s_first = 0;
            s_next = G;
            for (int i = 0; i < ne; ++i) {
                pre += MOE_COL_WEIGHT + s_ntok[i];
                const int64_t end = (i + 1) + pre * spare / wsum;
                if (static_cast<int64_t>(blockIdx.x) < end) {
                    s_eidx = i;
                    s_first = start;
                    s_next = end;
                    break;
                }
                start = end;
            }
        }
        __syncthreads();
        if (blockIdx.x == 0) {
            int bad = 0;
            for (int s = 0; s < n_slots; ++s) {
                const int e = s_ids[s];
                if (e < 0 || e >= p.n_expert) {
                    ++bad;
                    float *ys = p.y + (size_t)s * p.M;
                    for (int64_t r = threadIdx.x; r < p.M; r += blockDim.x) ys[r] = 0.f;
                }
            }
            if (threadIdx.x == 0 && p.status) *p.status = bad;
        }
        if (ne == 0) return;
        const int expert = s_exp[s_eidx];
        moe_shared = expert == p.n_expert;
        cta_index = blockIdx.x - s_first;
        cta_count = s_next - s_first;
        if (threadIdx.x == 0) {
            int cnt = 0;
            for (int t = 0; t < p.n_tokens; ++t) {
                uint32_t mask = 0;
                if (moe_shared) {
                    mask = 1u;
                } else {
                    for (int k = 0; k < p.top_k; ++k)
                        if (s_ids[t * p.top_k + k] == expert) mask |= 1u << k;
                }
                if (mask) { s_tok[cnt] = t; s_slots[cnt] = mask; ++cnt; }
            }
            s_cnt = cnt;
        }
        __syncthreads();
        n_active = s_cnt;
        if (moe_shared) {
            W0 = p.W2;
            W1 = p.W4;
        }
        else row_base = static_cast<int64_t>(expert) * p.M;
    }

    // every warp (of the grid; MoE: of the expert's CTAs) owns a contiguous,
    // balanced range of row groups (whole groups: a row's partial sums never
    // leave the warp).  With the q8_1 output (PLAIN/GATE), every CTA owns whole
    // 32-row blocks of y (blocks yb0 .. yb1-1 from row yrow0), its warps a
    // balanced share of their row groups.
    int64_t g_begin, my_groups, yb0 = 0, yb1 = 0, yrow0 = 0;
    const int64_t n_yblk = (p.M + 31) / 32;
    if constexpr (YQ) {
        yb0 = cta_index * n_yblk / cta_count;
        yb1 = (cta_index + 1) * n_yblk / cta_count;
        yrow0 = yb0 * 32;
        const int64_t cg0 = yb0 * (32 / RW);
        const int64_t ng = min64(yb1 * (32 / RW), p.n_groups) - cg0;
        g_begin = warp < nwarps ? cg0 + (warp * ng) / nwarps : 0;
        my_groups = warp < nwarps ? cg0 + ((warp + 1) * ng) / nwarps - g_begin : 0;
    } else {
        const int64_t gwarp = cta_index * nwarps + warp;
        const int64_t wtot = cta_count * nwarps;
        g_begin = warp < nwarps ? (gwarp * p.n_groups) / wtot : 0;
        my_groups = warp < nwarps ? ((gwarp + 1) * p.n_groups) / wtot - g_begin : 0;
    }
    float *const ybuf = reinterpret_cast<float *>(smem + p.ybuf_off);  // YQ only
    const int64_t total = my_groups * n_kt * NM;

    // this warp's ring of tile buffers (tensor-core decode: then its row-factor scratch)
    const uint32_t ring =
        smem_u32(smem + p.act_bytes) + static_cast<uint32_t>(min(warp, nwarps - 1) * (stages * TB + WARP_EXTRA));

    // ---- copies: tile (group, k-tile, matrix) -> ring buffer, one group per tile ----
    // Q4_0 / Q4_K: the loader walks its tiles incrementally: ld_row is this
    // lane's row of the current group (matrix 0), advanced by one group's rows
    // at the end of each group; the gate matrix sits a fixed distance dW from
    // it (the step's launches 0.9-1.6 % faster than with the tile's address
    // computed from its indices).  Q6_K keeps that computation: incrementally
    // its 4096x14336 launch was 7 % slower.
    const int cr = lane / G::LPR, ck = lane % G::LPR;  // row-wise copy: this lane's tile row and first piece
    const uint8_t *ld_row = W0 + (row_base + g_begin * RW + cr) * rb;
    const int64_t dW = NM == 2 ? static_cast<int64_t>(W1 - W0) : 0;
    int64_t ld_rows_left = p.M - g_begin * RW - cr;  // > 0: this lane's row exists
    const int lim_last = (U - (n_kt - 1) * UW) * UNIT / 16;  // valid pieces per row of the last k-tile
    int64_t ld_g = g_begin;
    int ld_kt = 0, ld_m = 0, ld_buf = 0;
    int64_t issued = 0;
    auto issue_tile = [&]() {
        if constexpr (F == FMT_Q6_K) {
            // each lane's first piece rotated so that every instruction covers
            // one aligned 128-byte line of each row (1,680-byte row segments)
            const uint8_t *W = (NM == 2 && ld_m) ? W1 : W0;
            const int64_t grow = ld_g * RW;  // first row of the group inside the matrix
            const uint8_t *base = W + (row_base + grow) * rb + static_cast<int64_t>(ld_kt) * (UW * UNIT);
            const int lim = min(UW, U - ld_kt * UW) * UNIT / 16;  // valid pieces per tile row
            if constexpr (ROWRUN) {
                // the whole warp on one row at a time: 512 contiguous bytes per
                // instruction, each lane's first piece rotated to a 512-byte block
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    if (r < p.M - grow) {
                        const uint8_t *rowp = base + r * rb;
                        const int k0 = (lane - static_cast<int>(reinterpret_cast<uintptr_t>(rowp) >> 4)) & 31;
                        copy_row_pieces<32, SEG>(ring + static_cast<uint32_t>(ld_buf * TB + r * SS + k0 * 16),
                                                 rowp + k0 * 16, k0, lim,
                                                 std::make_integer_sequence<int, (SEG + 31) / 32>{});
                    }
                }
            } else if (cr < p.M - grow) {
                const uint8_t *rowp = base + cr * rb;
                const int k0 = (ck - static_cast<int>(reinterpret_cast<uintptr_t>(rowp) >> 4)) & (G::LPR - 1);
                copy_row_pieces<G::LPR, SEG>(ring + static_cast<uint32_t>(ld_buf * TB + cr * SS + k0 * 16),
                                             rowp + k0 * 16, k0, lim, std::make_integer_sequence<int, G::NJ>{});
            }
        } else {
            const uint8_t *rowp = ld_row + static_cast<int64_t>(ld_kt) * (UW * UNIT) + ((NM == 2 && ld_m) ? dW : 0);
            const int lim = ld_kt == n_kt - 1 ? lim_last : SEG;
            if (ld_rows_left > 0)
                copy_row_pieces<G::LPR, SEG>(ring + static_cast<uint32_t>(ld_buf * TB + cr * SS + ck * 16),
                                             rowp + ck * 16, ck, lim, std::make_integer_sequence<int, G::NJ>{});
        }
        cp_async_commit();
        if (++ld_m == NM) {
            ld_m = 0;
            if (++ld_kt == n_kt) {
                ld_kt = 0;
                if constexpr (F == FMT_Q6_K) {
                    ++ld_g;
                } else {
                    ld_row += RW * rb;
                    ld_rows_left -= RW;
                }
            }
        }
        if (++ld_buf == stages) ld_buf = 0;
        ++issued;
    };

    if constexpr (!IS_MOE) {
        // A CTA usually starts as the kernel beside it on the SM passes its
        // own dependency wait and loads its activations.  Where this launch
        // requests its whole matrix early, the planner holds those requests
        // back briefly (p.early_delay), so that the neighbour's activation
        // loads reach the memory system first; the tiles still land long
        // before this launch needs them.  Bounded by the clock alone.
        // That neighbour exists only while the kernel before this one on the
        // stream still runs (a GEMV of this library, which lets this launch
        // start early).  So the CTA's last warp, where it neither decodes nor
        // requests tiles early, waits for that kernel at once and raises a
        // flag in shared memory (in the slack after the mbarrier) when the
        // wait returns: after a kernel that was already done when this CTA
        // started, the hold-back ends at once instead of only postponing the
        // first tiles.
        if (p.early_delay > 0) {
            const uint32_t flag = xbar + 8;
            const int last = static_cast<int>(blockDim.x >> 5) - 1;
            const bool sentinel = last >= nwarps && last >= p.early_warps;
            if (sentinel) {
                if (threadIdx.x == 0) asm volatile("st.volatile.shared.u32 [%0], 0;" ::"r"(flag) : "memory");
                __syncthreads();
                if (warp == last) {
                    pdl_wait();
                    if (lane == 0) asm volatile("st.volatile.shared.u32 [%0], 1;" ::"r"(flag) : "memory");
                }
            }
            const long long c0 = clock64();
            while (clock64() - c0 < p.early_delay) {
                if (sentinel) {
                    uint32_t done;
                    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(done) : "r"(flag) : "memory");
                    if (done) break;
                }
                __nanosleep(64);
            }
        }
    }
    if (warp < p.early_warps)
        while (issued < total && issued < p.pre_tiles) issue_tile();  // weights first
    if (p.early_delay == 0) prefetch_x();
    if constexpr (!IS_MOE) pdl_wait();
    if (trace && threadIdx.x == 0) trace[1] = global_timer_ns();
    if (!MMA && ncta > 1 && threadIdx.x == 0)
        mbar_arrive_expect_tx(xbar, cluster_share_bytes<F>(p.ncols * p.units_per_row * 8, crank, ncta));
    if constexpr (IS_MOE)
        stage_tile_activations<F, NC, PROBE>(p, smem, n_active, [&](int c) { return s_tok[c]; }, 0u, 1u, 0u, nullptr);
    else if constexpr (MMA)
        stage_mma_activations(p, smem, n_active, [](int c) { return c; }, crank, ncta);
    else
        stage_tile_activations<F, NC, PROBE>(p, smem, n_active, [](int c) { return c; }, crank, ncta, xbar, trace);
    if (ncta > 1 && MMA) {
        cluster_arrive();  // this CTA's share is stored everywhere ...
        cluster_wait();    // ... and every share is here; no remote access after this point
    } else if (ncta > 1) {
        // this CTA's own share is here after the CTA barrier; the partners'
        // shares once their bytes have completed on the mbarrier (every byte
        // a partner stores here is counted, so none is still in flight after
        // the wait and no CTA can exit while a partner writes to it)
        __syncthreads();
        const unsigned long long lim = (PROBE && p.withhold && crank == 0) ? p.withhold_wait_ns : WAIT_LIMIT_NS;
        if (__builtin_expect(__any_sync(0xffffffffu, !mbar_wait_bounded(xbar, 0, lim)), 0)) {
            // A partner's share never arrived: this warp computes nothing
            // (give_up_rows), and leaves once its own weight copies have
            // landed.  Each warp decides for itself, so a share that lands
            // just at the limit leaves every row either right or NaN.  With
            // the q8_1 output the warp stays for the CTA's final quantization.
            give_up_rows(p.y, p.ldy, p.ncols, g_begin * RW, min64(p.M, (g_begin + my_groups) * RW), lane, p.fault,
                         YQ ? ybuf : nullptr, p.ybuf_rows, yrow0);
            cp_async_wait(0);
            if constexpr (YQ) {
                __syncthreads();  // the other warps' rows (they meet the barrier after their loop)
                store_rows_q8_1(p, ybuf, yb0, yb1, n_yblk);
            }
            return;
        }
    } else {
        __syncthreads();
    }

    if (trace && threadIdx.x == 0) trace[4] = global_timer_ns();
    while (issued < total && issued < stages) issue_tile();  // the rest of the ring

    const uint32_t act_qs = smem_u32(smem);
    const uint32_t act_sc = act_qs + NC * U * ACT_QS_STRIDE;

    float acc[NM][NC];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[m][c] = 0.f;

    float b_up = 0.f, b_gate = 0.f;  // this lane's row biases (lanes of unit 0)
    // tensor-core decode: lane 4*mg + mt owns y[column mg][rows 2mt, 2mt + 1 of the group]
    const int mg = lane >> 2, mt = lane & 3;
    const uint32_t m_cs = MMA ? static_cast<uint32_t>(mma_col_stride(U * 8)) : 0u;
    const uint32_t m_ss = MMA ? static_cast<uint32_t>(mma_sc_stride(U * 8)) : 0u;
    const uint32_t m_act = act_qs + static_cast<uint32_t>(mg) * m_cs + 16u * mt;  // column mg, lane part mt
    const uint32_t m_scl = act_qs + static_cast<uint32_t>(p.ncols) * m_cs + static_cast<uint32_t>(mg) * m_ss;
    const uint32_t m_fac = ring + static_cast<uint32_t>(stages * TB);  // this warp's row-factor scratch
    float mv[2] = {0.f, 0.f};
    float mb[2] = {0.f, 0.f};  // biases of rows 2mt, 2mt + 1
    int64_t cg = g_begin;  // compute position
    int ckt = 0, cm = 0, cbuf = 0;
    for (int64_t t = 0; t < total; ++t) {
        cp_async_wait(static_cast<int>(issued - t - 1));  // tile t has landed (this lane's pieces)
        __syncwarp();                                     // ... and every lane's

        const int64_t row = cg * RW + r_l;
        const int u = ckt * UW + u_l;
        if constexpr (MMA) {
            // every lane takes part in the mma (rows past M compute on stale
            // tile bytes and are not written); units past the row are skipped
            // by the whole warp
            const int64_t r0 = cg * RW + 2 * mt;
            if (ckt == 0 && p.bias) {
                mb[0] = r0 < p.M ? ld_nc_f32(p.bias + r0) : 0.f;
                mb[1] = r0 + 1 < p.M ? ld_nc_f32(p.bias + r0 + 1) : 0.f;
            }
            const uint32_t tb = ring + static_cast<uint32_t>(cbuf * TB);
            mma_row_factors_q4_K<G::SS, UNIT>(tb, m_fac, lane);
            __syncwarp();  // the factors are in the scratch
            const uint32_t wrow = tb + static_cast<uint32_t>(mg * G::SS + 16 + 8 * mt);
#pragma unroll
            for (int i = 0; i < UW; ++i) {
                const int um = ckt * UW + i;
                const uint32_t fu = m_fac + static_cast<uint32_t>(i * (RW * MMA_FAC_ROW) + 2 * mt * MMA_FAC_ROW);
                if (um < U)
                    mma_unit_q4_K(wrow + i * UNIT, m_act + static_cast<uint32_t>(um * 8 * MMA_BLK_BYTES),
                                  m_scl + static_cast<uint32_t>(um * 8 * 8), mg < n_active, fu, fu + MMA_FAC_ROW, mv);
            }
        } else {
        if constexpr (MODE == MODE_PLAIN || MODE == MODE_GATE) {
            // the row's biases (after the dependency wait; nothing writes them while
            // this kernel runs), requested at the group's first tile so that its
            // decode hides the latency
            if (ckt == 0 && cm == 0 && u_l == 0 && row < p.M) {
                if (p.bias) b_up = ld_nc_f32(p.bias + row);
                if (MODE == MODE_GATE && p.gate_bias) b_gate = ld_nc_f32(p.gate_bias + row);
            }
        }
        if (u < U && row < p.M) {
            uint32_t ub[1] = {ring + static_cast<uint32_t>(cbuf * TB) + r_l * SS + u_l * UNIT};
            const bool live[1] = {true};
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                if (MODE != MODE_PLAIN && c >= n_active) break;
                const uint32_t aq = act_qs + (c * U + u) * ACT_QS_STRIDE;
                const uint32_t as = act_sc + (c * U + u) * act_sc_stride<F>();
                float vv[1] = {0.f};
                int32_t *dbg[1] = {nullptr};
                if constexpr (MODE == MODE_DEBUG) {
                    dbg[0] = p.dbg + ((size_t)c * p.M + row) * (size_t)(F == FMT_Q4_0 ? p.K / 32 : p.K / 16) +
                             (size_t)u * (F == FMT_Q4_0 ? 8 : 16);
                    unit_dot<F, 1, true>(ub, live, aq, as, vv, dbg);
                } else {
                    unit_dot<F, 1, false>(ub, live, aq, as, vv, dbg);
                    if (NM == 2 && cm) acc[NM - 1][c] += vv[0];
                    else acc[0][c] += vv[0];
                }
            }
        }
        }  // dp4a decode
        __syncwarp();  // every lane is done with the buffer
        if (issued < total) issue_tile();

        const bool group_done = (ckt == n_kt - 1) && (cm == NM - 1);
        if constexpr (MMA) {
            if (group_done) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int64_t r = cg * RW + 2 * mt + k;
                    if (r < p.M && mg < n_active) p.y[(size_t)mg * p.ldy + r] = p.bias ? mv[k] + mb[k] : mv[k];
                    mv[k] = 0.f;
                }
            }
        } else if constexpr (MODE != MODE_DEBUG) {
            if (group_done) {
                // the lanes of one row are those with the same r_l (xor over the unit bits)
#pragma unroll
                for (int m = 0; m < NM; ++m)
#pragma unroll
                    for (int c = 0; c < NC; ++c)
#pragma unroll
                        for (int o = 16; o >= RW; o >>= 1) acc[m][c] += __shfl_xor_sync(0xffffffffu, acc[m][c], o);
                if (u_l == 0 && row < p.M) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        if (c >= n_active) break;
                        if constexpr (MODE == MODE_PLAIN || MODE == MODE_GATE) {
                            float out;
                            if constexpr (MODE == MODE_PLAIN) {
                                out = p.bias ? acc[0][c] + b_up : acc[0][c];
                            } else {
                                const float up = p.bias ? acc[0][c] + b_up : acc[0][c];
                                const float gate = p.gate_bias ? acc[NM - 1][c] + b_gate : acc[NM - 1][c];
                                out = up * silu_f32(gate);
                            }
                            if (!YQ || p.y) p.y[(size_t)c * p.ldy + row] = out;
                            if constexpr (YQ) ybuf[c * p.ybuf_rows + static_cast<int>(row - yrow0)] = out;
                        } else {
                            const int tok = s_tok[c];
                            const float v = MODE == MODE_MOE_GATE ? acc[0][c] * silu_f32(acc[NM - 1][c]) : acc[0][c];
                            if (moe_shared) {
                                p.y_shared[(size_t)tok * p.M + row] = v;
                                continue;
                            }
                            uint32_t mask = s_slots[c];
                            while (mask) {
                                const int k = __ffs(mask) - 1;
                                mask &= mask - 1;
                                p.y[((size_t)tok * p.top_k + k) * p.M + row] = v;
                            }
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < NM; ++m)
#pragma unroll
                    for (int c = 0; c < NC; ++c) acc[m][c] = 0.f;
            }
        }
        if (++cm == NM) {
            cm = 0;
            if (++ckt == n_kt) { ckt = 0; ++cg; }
        }
        if (++cbuf == stages) cbuf = 0;
    }
    if (trace && lane == 0) atomicMax(trace + 5, global_timer_ns());
    if constexpr (YQ) {
        __syncthreads();  // every row of the CTA's blocks is in ybuf
        store_rows_q8_1(p, ybuf, yb0, yb1, n_yblk);
    }
}

// Kernel table of the tile path for one format (instantiated only in that
// format's translation unit).  RW = 4 serves every mode and column count;
// for Q4_0 / Q4_K, RW = 2 and 8 exist for one plain column, for geometry sweeps;
// the tensor-core decode (TC) of the plain Q4_K GEMV takes 1..8 columns.
template <int F>
const void *tiles_mma_kernel_fn(int mode)
{
    if constexpr (F == FMT_Q4_K)
        if (mode == MODE_PLAIN)
            return reinterpret_cast<const void *>(&gemv_tiles_kernel<F, MMA_COLS, MODE_PLAIN, MMA_RW, true>);
    return nullptr;
}

// The instrumented twins (PROBE) exist for the plain GEMV of one or two
// columns and the fused gate/up GEMV of one column, 4-row tiles, dp4a decode.
template <int F>
const void *tiles_probe_kernel_fn(int mode, int nc)
{
    if (mode == MODE_PLAIN && nc == 1) return reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 1, MODE_PLAIN, 4, false, true>);
    if (mode == MODE_PLAIN && nc == 2) return reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 2, MODE_PLAIN, 4, false, true>);
    if (mode == MODE_GATE && nc == 1) return reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 1, MODE_GATE, 4, false, true>);
    return nullptr;
}

// The row-run variant (ROWRUN) of the plain Q6_K GEMV of one column: tiles
// copied one row at a time by the whole warp (the planner's choice for short
// rows, where the stream rather than the decode bounds the launch).
template <int F>
const void *tiles_rowrun_kernel_fn(int mode, int nc)
{
    if constexpr (F == FMT_Q6_K)
        if (mode == MODE_PLAIN && nc == 1)
            return reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 1, MODE_PLAIN, 4, false, false, false, true>);
    return nullptr;
}

// The q8_1-output variants (YQ): plain and gate/up GEMV of one column, 4-row
// tiles, dp4a decode; probe: their instrumented twins.
template <int F>
const void *tiles_yq_kernel_fn(int mode, bool probe)
{
    if (mode == MODE_PLAIN)
        return probe ? reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 1, MODE_PLAIN, 4, false, true, true>)
                     : reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 1, MODE_PLAIN, 4, false, false, true>);
    if (mode == MODE_GATE)
        return probe ? reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 1, MODE_GATE, 4, false, true, true>)
                     : reinterpret_cast<const void *>(&gemv_tiles_kernel<F, 1, MODE_GATE, 4, false, false, true>);
    return nullptr;
}

template <int F>
const void *tiles_kernel_fn(int mode, int nc, int rw)
{
#define QMV_TK(NC_, MODE_, RW_) reinterpret_cast<const void *>(&gemv_tiles_kernel<F, NC_, MODE_, RW_>)
    if constexpr (F != FMT_Q6_K) {
        if (rw == 2) return (mode == MODE_PLAIN && nc == 1) ? QMV_TK(1, MODE_PLAIN, 2) : nullptr;
        if (rw == 8) return (mode == MODE_PLAIN && nc == 1) ? QMV_TK(1, MODE_PLAIN, 8) : nullptr;
    }
    if (rw != 4) return nullptr;
    if (mode == MODE_PLAIN) {
        switch (nc) {
        case 1: return QMV_TK(1, MODE_PLAIN, 4);
        case 2: return QMV_TK(2, MODE_PLAIN, 4);
        case 3: return QMV_TK(3, MODE_PLAIN, 4);
        case 4: return QMV_TK(4, MODE_PLAIN, 4);
        case 5: return QMV_TK(5, MODE_PLAIN, 4);
        case 6: return QMV_TK(6, MODE_PLAIN, 4);
        case 7: return QMV_TK(7, MODE_PLAIN, 4);
        case 8: return QMV_TK(8, MODE_PLAIN, 4);
        default: return nullptr;
        }
    }
#define QMV_TK_MODE(MODE_)                    \
    switch (nc) {                             \
    case 1: return QMV_TK(1, MODE_, 4);       \
    case 2: return QMV_TK(2, MODE_, 4);       \
    case 4: return QMV_TK(4, MODE_, 4);       \
    case 8: return QMV_TK(8, MODE_, 4);       \
    default: return nullptr;                  \
    }
    if (mode == MODE_GATE) { QMV_TK_MODE(MODE_GATE) }
    if (mode == MODE_MOE) { QMV_TK_MODE(MODE_MOE) }
    if (mode == MODE_MOE_GATE) { QMV_TK_MODE(MODE_MOE_GATE) }
    if (mode == MODE_DEBUG) { QMV_TK_MODE(MODE_DEBUG) }
#undef QMV_TK_MODE
#undef QMV_TK
    return nullptr;
}

}  // namespace qmv
