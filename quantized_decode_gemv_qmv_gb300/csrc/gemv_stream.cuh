// Streaming quantized GEMV for sm_103a.
//
// What it computes is the method of "llama.cpp 源码完全拆解(十四)：
// mul_mat_vec_q": every weight row is an int8 dot product per block with the
// q8_1 activations (dp4a), scaled by the block scales; the "sign moved into
// constants" corrections of the page are kept (Q4_0 subtracts 8*s, Q4_K
// subtracts dmin*m*d8*sum(qy), Q6_K subtracts 32*sum(qy) per sub-block).
//
// How it computes it is a GB300 design, not the page's:
//   * A light persistent grid (a few CTAs per SM) in which each CTA owns a
//     contiguous, balanced range of row groups.  The kernel signals
//     programmatic completion at entry and issues its first weight copies
//     before waiting on the previous grid (griddepcontrol), so consecutive
//     GEMVs co-reside and keep HBM busy across kernel boundaries.
//   * Weights stream into a per-warp ring of shared-memory slots with
//     per-lane 16-byte cp.async copies (no register cost, no per-copy engine
//     overhead), several slots in flight per warp.
//   * The CTA's warps split K: warp w owns a contiguous run of weight units of
//     every row of the group; each slot holds one K-slice of R rows.  Lanes
//     split the slice into 32-weight items (format-specific) so a warp's
//     shared-memory reads hit 32 distinct banks.
//   * Activations are repacked once per CTA into shared memory in the order
//     the items read them; each item loads its activations once and reuses
//     them for all R rows, and decodes each weight item once and reuses it for
//     all ncols columns (the page re-decodes per column).
//   * Lane partials are reduced with warp shuffles, the warps' partials once
//     per row group through shared memory.
#pragma once

#include "common.cuh"

namespace qmv {

enum Mode { MODE_PLAIN = 0, MODE_GATE = 1, MODE_MOE = 2, MODE_DEBUG = 3 };

constexpr int NR = 4;           // row-slices held by one ring slot
constexpr int MAX_THREADS = 256;

// Streaming unit: the smallest run of whole blocks whose byte size is a
// multiple of 16 (so every slice of a 16-byte-aligned row can be a bulk copy).
// Items: 32-weight pieces, 8 per 256 weights for every format.
template <int F> struct FmtTraits;
template <> struct FmtTraits<FMT_Q4_0> {
    static constexpr int UNIT_BYTES = 8 * Q4_0_BYTES;  // 8 blocks = 144 B
    static constexpr int UNIT_ELEMS = 256;
    static constexpr int ITEMS_PER_UNIT = 8;  // one item per block
    static constexpr int BLOCK_ELEMS = QK4_0;
};
template <> struct FmtTraits<FMT_Q4_K> {
    static constexpr int UNIT_BYTES = Q4_K_BYTES;  // 1 super-block = 144 B
    static constexpr int UNIT_ELEMS = 256;
    static constexpr int ITEMS_PER_UNIT = 8;  // one item per 16 bytes of qs
    static constexpr int BLOCK_ELEMS = QK_K;
};
template <> struct FmtTraits<FMT_Q6_K> {
    static constexpr int UNIT_BYTES = 8 * Q6_K_BYTES;  // 8 super-blocks = 1680 B
    static constexpr int UNIT_ELEMS = 2048;
    static constexpr int ITEMS_PER_UNIT = 64;  // 8 per super-block
    static constexpr int BLOCK_ELEMS = QK_K;
};

struct GemvParams {
    const uint8_t *W;    // weights (MoE: expert 0); GATE: the up matrix
    const uint8_t *W2;   // GATE: the gate matrix
    const uint8_t *xq;   // q8_1 activations, column c at xq + c*xq_col_bytes
    const float *xf;     // fp32 activations quantized in place (tile kernel), column c at xf + c*ldx; or null
    int64_t ldx;
    float *y;            // PLAIN/GATE: y[c*ldy + r]; MOE: y[(t*top_k + k)*M + r]
    int32_t *dbg;        // DEBUG: per-sub-block int sums
    const int32_t *ids;  // MOE: [n_tokens][top_k]
    int32_t *status;     // MOE: number of invalid ids (nullable)
    int64_t M;
    int64_t ldy;
    int64_t row_bytes;
    int64_t xq_col_bytes;
    int64_t expert_bytes;
    int64_t n_groups;    // ceil(M / rows per group)
    int K;
    int ncols;           // active columns (PLAIN/GATE/DEBUG)
    int n_tokens, top_k, n_expert;
    int units_per_row;
    int slice_units;
    int n_slices;
    int stages;
    uint32_t act_bytes;     // shared bytes of the activation area
    uint32_t raw_off;       // tile kernel: offset of the raw q8_1 copy inside the activation area (0: none)
    uint32_t slot_bytes;    // shared bytes of one ring slot
    uint32_t slice_stride;  // shared bytes of one row-slice inside a slot
};

// ---- activation staging ----------------------------------------------------
//
// Per column, for every 256 activations (a "group"), the 16-value runs are
// stored item-major: [low run of item 0..7][high run of item 0..7], 16 B each.
// Item t's low/high runs are the activations its weight nibbles multiply:
//   Q4_0  item t = block t:      low = elems 32t+0..15,        high = 32t+16..31
//   Q4_K  item t = qs bytes 16t: low = 64(t/2)+16(t%2)+0..15,  high = low + 32
//   Q6_K  item t = ql bytes 16t: low = 128(t/4)+16(t%4)+0..15, high = low + 64
// and per item 16 B of scalars:
//   Q4_0 {d8, s8, -, -}   Q4_K {d8_lo, d8_hi, d8_lo*S_lo, d8_hi*S_hi}
//   Q6_K {d8_lo, d8_hi, S_lo (int), S_hi (int)}   with S = sum of the run's qy.

template <int F>
__device__ __forceinline__ void run_position(int rho, int &t, int &half)
{
    if (F == FMT_Q4_0) { t = rho >> 1; half = rho & 1; }
    else if (F == FMT_Q4_K) { t = 2 * (rho >> 2) + (rho & 1); half = (rho >> 1) & 1; }
    else { t = 4 * (rho >> 3) + (rho & 3); half = (rho >> 2) & 1; }
}

// Stages NC columns; column c < n_active reads q8_1 row src_col(c), the rest
// are zero.  Called by all threads of the CTA.
template <int F, int NC, typename ColFn>
__device__ __forceinline__ void stage_activations(const GemvParams &p, uint8_t *smem, int n_active,
                                                  ColFn src_col)
{
    const int K = p.K;
    const int runs = K >> 4;
    const int items_row = K >> 5;
    uint8_t *act_qs = smem;
    uint8_t *act_sc = smem + (size_t)NC * K;
    for (int idx = threadIdx.x; idx < NC * runs; idx += blockDim.x) {
        const int c = idx / runs;
        const int rr = idx - c * runs;
        uint32_t q[4] = {0u, 0u, 0u, 0u};
        uint32_t ds = 0u;
        if (c < n_active) {
            const uint8_t *blk = p.xq + (size_t)src_col(c) * p.xq_col_bytes + (size_t)(rr >> 1) * Q8_1_BYTES;
            const uint32_t *w = reinterpret_cast<const uint32_t *>(blk);
            ds = w[0];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = w[1 + 4 * (rr & 1) + i];
        }
        int S = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) S = dp4a(static_cast<int>(q[i]), 0x01010101, S);
        const float d8 = half_bits_to_float(ds);
        const int G = rr >> 4;
        int t, half;
        run_position<F>(rr & 15, t, half);
        *reinterpret_cast<uint4 *>(act_qs + (size_t)c * K + 256 * G + 128 * half + 16 * t) =
            make_uint4(q[0], q[1], q[2], q[3]);
        float *sc = reinterpret_cast<float *>(act_sc + ((size_t)c * items_row + 8 * G + t) * 16);
        if (F == FMT_Q4_0) {
            if (half == 0) { sc[0] = d8; sc[1] = half_bits_to_float(ds >> 16); }
        } else if (F == FMT_Q4_K) {
            sc[half] = d8;
            sc[2 + half] = d8 * static_cast<float>(S);
        } else {
            sc[half] = d8;
            reinterpret_cast<int *>(sc)[2 + half] = S;
        }
    }
}

// ---- weight items ------------------------------------------------------------

struct WItem {
    uint32_t lo[4], hi[4];  // 16 codes multiplying the low run, 16 the high run
    float a, b, c, e;       // format scalars (see decode_item)
};

// Decodes item `it` of a row-slice at shared address rs.
//   Q4_0: it = block in slice.           a = d4
//   Q4_K: it = 8*unit + j.               a = d*sc_lo, b = d*sc_hi, c = dmin*m_lo, e = dmin*m_hi
//   Q6_K: it = 64*unit + 8*b + k.        a = d*sc_lo, b = d*sc_hi
template <int F>
__device__ __forceinline__ WItem decode_item(uint32_t rs, int it)
{
    WItem o;
    if (F == FMT_Q4_0) {
        const uint32_t blk = rs + Q4_0_BYTES * it;
        uint32_t q[4];
        lds16_unaligned2(blk + 2, q);
        o.a = half_bits_to_float(lds_u16(blk));
        o.b = o.c = o.e = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o.lo[i] = q[i] & 0x0F0F0F0Fu;
            o.hi[i] = (q[i] >> 4) & 0x0F0F0F0Fu;
        }
    } else if (F == FMT_Q4_K) {
        const int j = it & 7;
        const uint32_t blk = rs + Q4_K_BYTES * (it >> 3);
        const uint4 hdr = lds128(blk);
        const uint4 q = lds128(blk + 16 + 16 * j);
        const float d = half_bits_to_float(hdr.x);
        const float dmin = half_bits_to_float(hdr.x >> 16);
        // 6-bit scale/min of sub-blocks 2*(j/2) and 2*(j/2)+1, branch free:
        // sub-blocks 0-3 keep the low 6 bits of bytes 0-3 (scales) and 4-7
        // (mins); sub-blocks 4-7 join a nibble of bytes 8-11 with the top two
        // bits of bytes 0-3 (scales) or 4-7 (mins).
        const int cp = j >> 1;
        const int sh = (cp & 1) * 16;
        const uint32_t s0 = (hdr.y >> sh) & 0xffffu;
        const uint32_t s1 = (hdr.z >> sh) & 0xffffu;
        const uint32_t s2 = (hdr.w >> sh) & 0xffffu;
        const bool upper = cp >= 2;
        const uint32_t sc2 = upper ? ((s2 & 0x0f0fu) | ((s0 & 0xc0c0u) >> 2)) : (s0 & 0x3f3fu);
        const uint32_t m2 = upper ? (((s2 >> 4) & 0x0f0fu) | ((s1 & 0xc0c0u) >> 2)) : (s1 & 0x3f3fu);
        o.a = d * static_cast<float>(sc2 & 0xffu);
        o.b = d * static_cast<float>(sc2 >> 8);
        o.c = dmin * static_cast<float>(m2 & 0xffu);
        o.e = dmin * static_cast<float>(m2 >> 8);
        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o.lo[i] = qq[i] & 0x0F0F0F0Fu;
            o.hi[i] = (qq[i] >> 4) & 0x0F0F0F0Fu;
        }
    } else {
        const int k = it & 7;
        const int bb = (it >> 3) & 7;
        const uint32_t blk = rs + Q6_K_BYTES * (8 * (it >> 6) + bb);
        const int h = k >> 2;
        uint32_t ql[4], qh[4];
        lds16_unaligned2(blk + 16 * k, ql);
        lds16_unaligned2(blk + 128 + 32 * h + 16 * (k & 1), qh);
        const int shl = 2 * ((k >> 1) & 1);
        const float d = half_bits_to_float(lds_u16(blk + 208));
        o.a = d * static_cast<float>(lds_s8(blk + 192 + 8 * h + (k & 3)));
        o.b = d * static_cast<float>(lds_s8(blk + 192 + 8 * h + 4 + (k & 3)));
        o.c = o.e = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o.lo[i] = (ql[i] & 0x0F0F0F0Fu) | (((qh[i] >> shl) & 0x03030303u) << 4);
            o.hi[i] = ((ql[i] >> 4) & 0x0F0F0F0Fu) | (((qh[i] >> (shl + 4)) & 0x03030303u) << 4);
        }
    }
    return o;
}

struct AItem {
    uint4 lo, hi;
    float4 s;
};

__device__ __forceinline__ AItem load_act(uint32_t act_qs_c, uint32_t act_sc_c, int g)
{
    AItem a;
    const uint32_t qa = act_qs_c + 256u * (g >> 3) + 16u * (g & 7);
    a.lo = lds128(qa);
    a.hi = lds128(qa + 128u);
    const uint4 s = lds128(act_sc_c + 16u * g);
    a.s = make_float4(__uint_as_float(s.x), __uint_as_float(s.y), __uint_as_float(s.z), __uint_as_float(s.w));
    return a;
}

__device__ __forceinline__ void dots(const WItem &w, const AItem &a, int &dlo, int &dhi)
{
    dlo = dp4a(static_cast<int>(w.lo[0]), static_cast<int>(a.lo.x), 0);
    dlo = dp4a(static_cast<int>(w.lo[1]), static_cast<int>(a.lo.y), dlo);
    dlo = dp4a(static_cast<int>(w.lo[2]), static_cast<int>(a.lo.z), dlo);
    dlo = dp4a(static_cast<int>(w.lo[3]), static_cast<int>(a.lo.w), dlo);
    dhi = dp4a(static_cast<int>(w.hi[0]), static_cast<int>(a.hi.x), 0);
    dhi = dp4a(static_cast<int>(w.hi[1]), static_cast<int>(a.hi.y), dhi);
    dhi = dp4a(static_cast<int>(w.hi[2]), static_cast<int>(a.hi.z), dhi);
    dhi = dp4a(static_cast<int>(w.hi[3]), static_cast<int>(a.hi.w), dhi);
}

// Contribution of one item to one (row, column) accumulator: the block
// formula of the format restricted to the item's 32 weights.
template <int F>
__device__ __forceinline__ float item_value(const WItem &w, const AItem &a, int dlo, int dhi)
{
    if (F == FMT_Q4_0) {
        // d4 * (d8*sumi - 8*s): the whole block is one item
        return w.a * (a.s.x * static_cast<float>(dlo + dhi) - 8.0f * a.s.y);
    } else if (F == FMT_Q4_K) {
        // d*sc*d8*dot1 - dmin*m*d8*dot2 over the item's two 16-value halves
        return w.a * (a.s.x * static_cast<float>(dlo)) + w.b * (a.s.y * static_cast<float>(dhi)) -
               (w.c * a.s.z + w.e * a.s.w);
    } else {
        // d*sc*d8*(sum v*qy - 32*sum qy) per 16-value sub-block
        const int slo = dlo - 32 * __float_as_int(a.s.z);
        const int shi = dhi - 32 * __float_as_int(a.s.w);
        return w.a * (a.s.x * static_cast<float>(slo)) + w.b * (a.s.y * static_cast<float>(shi));
    }
}

// Per-sub-block integer sums of one item, written to the debug buffer
// (layout of qmv_debug_subblock_sums).  g is the item index along the row.
template <int F>
__device__ __forceinline__ void debug_item(int32_t *out_row, int g, const AItem &a, int dlo, int dhi)
{
    if (F == FMT_Q4_0) {
        out_row[g] = dlo + dhi;
    } else if (F == FMT_Q4_K) {
        const int sb_lo = 8 * (g >> 3) + 2 * ((g & 7) >> 1);
        int s_lo = 0, s_hi = 0;  // sum of qy, as the page computes it: dp4a with 0x01010101
        s_lo = dp4a(0x01010101, static_cast<int>(a.lo.x), s_lo);
        s_lo = dp4a(0x01010101, static_cast<int>(a.lo.y), s_lo);
        s_lo = dp4a(0x01010101, static_cast<int>(a.lo.z), s_lo);
        s_lo = dp4a(0x01010101, static_cast<int>(a.lo.w), s_lo);
        s_hi = dp4a(0x01010101, static_cast<int>(a.hi.x), s_hi);
        s_hi = dp4a(0x01010101, static_cast<int>(a.hi.y), s_hi);
        s_hi = dp4a(0x01010101, static_cast<int>(a.hi.z), s_hi);
        s_hi = dp4a(0x01010101, static_cast<int>(a.hi.w), s_hi);
        atomicAdd(out_row + 2 * sb_lo, dlo);
        atomicAdd(out_row + 2 * sb_lo + 1, s_lo);
        atomicAdd(out_row + 2 * (sb_lo + 1), dhi);
        atomicAdd(out_row + 2 * (sb_lo + 1) + 1, s_hi);
    } else {
        const int k = g & 7;
        const int sb_lo = 16 * (g >> 3) + 8 * (k >> 2) + (k & 3);
        out_row[sb_lo] = dlo - 32 * __float_as_int(a.s.z);
        out_row[sb_lo + 4] = dhi - 32 * __float_as_int(a.s.w);
    }
}

__device__ __forceinline__ float silu_f32(float g)
{
    return g / (1.0f + expf(-g));
}

// ---- the kernel ------------------------------------------------------------
//
// CTA b owns row groups [b*G/grid, (b+1)*G/grid) (G = ceil(M/R)).  Warp w
// streams weight units [w*U/S, (w+1)*U/S) of each of those groups' rows
// through its own ring of `stages` slots; every lane commits exactly one
// cp.async group per slot, so "slot n has landed" is wait_group(issued-n-1)
// followed by __syncwarp.  Ring cursors are 32-bit counters advanced
// incrementally.  Once per group the warps' partial sums meet in shared memory
// (double-buffered by group parity, one __syncthreads per group) and warp 0
// writes the outputs.

template <int F, int NC, int MODE>
__global__ void __launch_bounds__(MAX_THREADS) gemv_stream_kernel(const GemvParams p)
{
    using T = FmtTraits<F>;
    constexpr int R = (MODE == MODE_GATE) ? NR / 2 : NR;  // output rows per group
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // 128-byte aligned base (the host reserves 128 extra bytes)
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    __shared__ int s_tok[8];
    __shared__ uint32_t s_slots[8];
    __shared__ int s_cnt;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = blockDim.x >> 5;
    const int K = p.K;
    const int items_row = K >> 5;

    const uint8_t *W = p.W;
    const uint8_t *W2 = p.W2;
    int n_active = p.ncols;

    if constexpr (MODE == MODE_MOE) {
        pdl_launch_dependents();
        pdl_wait();  // ids and activations come from earlier kernels
        if (blockIdx.y == static_cast<unsigned>(p.n_expert)) {
            // invalid-id slice: zero the outputs of slots whose id is out of range
            int bad = 0;
            for (int s = 0; s < p.n_tokens * p.top_k; ++s) {
                const int e = p.ids[s];
                if (e < 0 || e >= p.n_expert) {
                    ++bad;
                    float *ys = p.y + (size_t)s * p.M;
                    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < p.M;
                         r += (int64_t)gridDim.x * blockDim.x)
                        ys[r] = 0.f;
                }
            }
            if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) *p.status = bad;
            return;
        }
        if (threadIdx.x == 0) {
            int cnt = 0;
            for (int t = 0; t < p.n_tokens; ++t) {
                uint32_t mask = 0;
                for (int k = 0; k < p.top_k; ++k)
                    if (p.ids[t * p.top_k + k] == static_cast<int>(blockIdx.y)) mask |= 1u << k;
                if (mask) { s_tok[cnt] = t; s_slots[cnt] = mask; ++cnt; }
            }
            s_cnt = cnt;
        }
        __syncthreads();
        n_active = s_cnt;
        if (n_active == 0) return;  // expert not selected: its weights are never read
        W = p.W + (size_t)blockIdx.y * p.expert_bytes;
    }

    // shared layout: [activations][rings S x stages x slot][16 B over-read pad][partials 2 x S x NR x NC]
    uint8_t *ring = smem + p.act_bytes + (size_t)warp * p.stages * p.slot_bytes;
    float *partials = reinterpret_cast<float *>(smem + p.act_bytes + (size_t)S * p.stages * p.slot_bytes + 16);

    const int U = p.units_per_row;
    const int ub = (warp * U) / S;            // this warp's units [ub, ue)
    const int ue = ((warp + 1) * U) / S;
    const int KS = p.slice_units;
    const int n_sl = (ue - ub + KS - 1) / KS;  // slices per group (0 if the warp has no units)
    const int64_t g_begin = (static_cast<int64_t>(blockIdx.x) * p.n_groups) / gridDim.x;
    const int64_t g_end = (static_cast<int64_t>(blockIdx.x + 1) * p.n_groups) / gridDim.x;
    const int64_t my_groups = g_end - g_begin;
    const int64_t total = my_groups * n_sl;   // slices this warp streams in the whole call
    const int stages = p.stages;

    // issue cursor (all lanes advance it identically)
    int64_t is_grp = g_begin;
    int is_s = 0, is_slot = 0;
    int64_t issued = 0;
    auto issue_next = [&]() {
        if (issued < total) {
            const int64_t r0 = is_grp * R;
            const int nvalid = static_cast<int>(min64(R, p.M - r0));
            const int u0 = ub + is_s * KS;
            const int nu = min(KS, ue - u0);
            const int bytes = nu * T::UNIT_BYTES;
            const uint32_t dst = smem_u32(ring + (size_t)is_slot * p.slot_bytes);
            const uint8_t *src = W + (size_t)r0 * p.row_bytes + (size_t)u0 * T::UNIT_BYTES;
            for (int i = 0; i < nvalid; ++i)
                for (int o = 16 * lane; o < bytes; o += 512)
                    cp_async16(dst + i * p.slice_stride + o, src + (size_t)i * p.row_bytes + o);
            if constexpr (MODE == MODE_GATE) {
                const uint8_t *src2 = W2 + (size_t)r0 * p.row_bytes + (size_t)u0 * T::UNIT_BYTES;
                for (int i = 0; i < nvalid; ++i)
                    for (int o = 16 * lane; o < bytes; o += 512)
                        cp_async16(dst + (R + i) * p.slice_stride + o, src2 + (size_t)i * p.row_bytes + o);
            }
            if (++is_s == n_sl) { is_s = 0; ++is_grp; }
            if (++is_slot == stages) is_slot = 0;
        }
        cp_async_commit();  // one group per slot per lane, possibly empty
        ++issued;
    };

    // weights do not depend on the previous kernel: start streaming them first
    for (int s = 0; s < stages; ++s) issue_next();

    if constexpr (MODE != MODE_MOE) {
        pdl_launch_dependents();
        pdl_wait();  // activations come from the previous kernel
    }
    if constexpr (MODE == MODE_MOE)
        stage_activations<F, NC>(p, smem, n_active, [&](int c) { return s_tok[c]; });
    else
        stage_activations<F, NC>(p, smem, n_active, [](int c) { return c; });
    __syncthreads();

    const uint32_t act_qs = smem_u32(smem);
    const uint32_t act_sc = act_qs + NC * K;

    float acc[NR][NC];
#pragma unroll
    for (int i = 0; i < NR; ++i)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[i][c] = 0.f;

    int64_t consumed = 0;
    int c_slot = 0;
    for (int64_t gi = 0; gi < my_groups; ++gi) {
        const int64_t r0 = (g_begin + gi) * R;
        const int nvalid = static_cast<int>(min64(R, p.M - r0));
        for (int s = 0; s < n_sl; ++s) {
            cp_async_wait(static_cast<int>(issued - consumed - 1));
            __syncwarp();
            const int u0 = ub + s * KS;
            const int nu = min(KS, ue - u0);
            const uint32_t slotp = smem_u32(ring + (size_t)c_slot * p.slot_bytes);
            const int item0 = u0 * T::ITEMS_PER_UNIT;  // first item of the slice along the row
            const int n_iter = (F == FMT_Q6_K) ? 2 * nu : (nu * T::ITEMS_PER_UNIT + 31) / 32;

            for (int iter = 0; iter < n_iter; ++iter) {
                int it;
                if (F == FMT_Q6_K) {
                    // lanes 8p..8p+7 take items k = 0..7 of super-block 2p + (iter & 1)
                    // of unit iter/2: the four super-blocks of one instruction start
                    // at distinct word offsets mod 4, so the warp's shared reads
                    // fall in 32 distinct banks.
                    it = 64 * (iter >> 1) + 8 * (2 * (lane >> 3) + (iter & 1)) + (lane & 7);
                } else {
                    it = lane + 32 * iter;
                    if (it >= nu * T::ITEMS_PER_UNIT) break;
                }
                const int g = item0 + it;
                WItem w[NR];
#pragma unroll
                for (int i = 0; i < NR; ++i) {
                    const int row_ok = (MODE == MODE_GATE) ? ((i % R) < nvalid) : (i < nvalid);
                    if (row_ok) w[i] = decode_item<F>(slotp + i * p.slice_stride, it);
                }
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    if (MODE != MODE_PLAIN && c >= n_active) break;
                    const AItem a = load_act(act_qs + c * K, act_sc + c * items_row * 16, g);
#pragma unroll
                    for (int i = 0; i < NR; ++i) {
                        const int row_ok = (MODE == MODE_GATE) ? ((i % R) < nvalid) : (i < nvalid);
                        if (!row_ok) continue;
                        int dlo, dhi;
                        dots(w[i], a, dlo, dhi);
                        if constexpr (MODE == MODE_DEBUG)
                            debug_item<F>(p.dbg + ((size_t)c * p.M + r0 + i) * (size_t)(F == FMT_Q4_0 ? K / 32 : K / 16),
                                          g, a, dlo, dhi);
                        else
                            acc[i][c] += item_value<F>(w[i], a, dlo, dhi);
                    }
                }
            }
            __syncwarp();  // every lane is done with the slot before it is refilled
            ++consumed;
            issue_next();
            if (++c_slot == stages) c_slot = 0;
        }

        // ---- group epilogue: lanes -> warp -> CTA, then outputs ----
        if constexpr (MODE != MODE_DEBUG) {
            float *part = partials + (size_t)(gi & 1) * S * NR * NC;
#pragma unroll
            for (int i = 0; i < NR; ++i)
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const float v = warp_sum(acc[i][c]);
                    if (lane == 0) part[(warp * NR + i) * NC + c] = v;
                    acc[i][c] = 0.f;
                }
            __syncthreads();
            if (warp == 0) {
                for (int idx = lane; idx < R * NC; idx += 32) {
                    const int i = idx / NC, c = idx - (idx / NC) * NC;
                    if (i >= nvalid || c >= n_active) continue;
                    float v = 0.f;
                    for (int w2 = 0; w2 < S; ++w2) v += part[(w2 * NR + i) * NC + c];
                    const int64_t row = r0 + i;
                    if constexpr (MODE == MODE_PLAIN) {
                        p.y[(size_t)c * p.ldy + row] = v;
                    } else if constexpr (MODE == MODE_GATE) {
                        float gsum = 0.f;
                        for (int w2 = 0; w2 < S; ++w2) gsum += part[(w2 * NR + R + i) * NC + c];
                        p.y[(size_t)c * p.ldy + row] = v * silu_f32(gsum);
                    } else {
                        const int tok = s_tok[c];
                        uint32_t mask = s_slots[c];
                        while (mask) {
                            const int k = __ffs(mask) - 1;
                            mask &= mask - 1;
                            p.y[((size_t)tok * p.top_k + k) * p.M + row] = v;
                        }
                    }
                }
            }
        }
    }
    cp_async_wait(0);  // no copy may still target shared memory at exit
}

}  // namespace qmv
