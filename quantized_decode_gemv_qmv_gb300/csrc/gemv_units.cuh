// Streaming GEMV for the 144-byte-unit formats (Q4_K super-blocks; Q4_0 in
// runs of 8 blocks), sm_103a.
//
// Method: "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q" (vec_dot_q4_0_q8_1_impl,
// vec_dot_q4_K_q8_1_impl_vmmq): int8 dot products per block scaled by the
// block scales, with the page's constant corrections (Q4_0: -8*s; Q4_K:
// -dmin*m*d8*sum(qy)).
//
// Design (GB300-specific):
//   * Weight tiles move by TMA: a tensor map views W as [rows][units][144 B],
//     and one cp.async.bulk.tensor.3d per ring slot brings RT rows x KW units
//     (a few KB) into shared memory, completing on an mbarrier.  No
//     thread spends instructions on copies; rows or units past the matrix read
//     as zeros.  Each warp owns a ring of `stages` slots and issues the first
//     ones before waiting on the previous grid (programmatic dependent launch).
//   * Lane <-> (rows, unit).  A warp works on RT = RPL*32/KW rows at a time;
//     lane (rw, kw) decodes unit kw of rows rw, rw + 32/KW, ... (RPL rows):
//     one header decode per 256 weights, the 6-bit scales/mins of all 8
//     sub-blocks unpacked word-parallel, the high nibbles used in place
//     (dp4a.u32.s32 on q & 0xF0F0F0F0 is 16x the dot; the 1/16 folds into the
//     scale exactly), and each activation load is shared by the lane's RPL
//     rows (two independent dp4a chains).
//   * Units sit 144 bytes apart in a slot and activations 272 / 80 bytes apart
//     per unit, so the 8 lanes of every 128-bit shared read phase hit distinct
//     bank quads.
//   * Warps are independent (no cross-warp reduction): each warp owns whole
//     row groups; a row's KW lane partials are combined with xor shuffles.
#pragma once

#include <cuda.h>

#include "gemv_stream.cuh"

namespace qmv {

constexpr int UNIT_B = 144;         // bytes of a unit (both formats)
constexpr int ACT_QS_STRIDE = 272;  // shared bytes per unit of staged activation codes (256 + pad)
constexpr int ACT_SC_STRIDE = 80;   // shared bytes per unit of staged activation scalars (64 + pad)
constexpr int UNITS_RPL = 2;        // rows per lane

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// 3D tensor tile global -> shared, completing on an mbarrier.  The tensor
// map views W as [rows][units][144 bytes] (18 eight-byte elements per unit).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int unit, int row, uint32_t bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(unit), "r"(row), "r"(bar), "l"(policy)
        : "memory");
}

// Activation staging for the units path.  Per column and unit u (256 values):
// the 256 codes in natural order at c*U*272 + u*272, and 16 scalars at
// sc + (c*U + u)*80:
//   Q4_K: per sub-block pair j (= 32-byte qs chunk j): {d8[2j], d8[2j+1], D[2j], D[2j+1]}
//         with D = d8 * sum(qy over the 32-value sub-block);
//   Q4_0: per block t: {d8[t], s8[t]}.
template <int F, int NC, typename ColFn>
__device__ __forceinline__ void stage_units_activations(const GemvParams &p, uint8_t *smem, int n_active,
                                                        ColFn src_col)
{
    const int U = p.units_per_row;
    const int nblk = U * 8;  // q8_1 blocks per column
    uint8_t *act_qs = smem;
    uint8_t *act_sc = smem + (size_t)NC * U * ACT_QS_STRIDE;
    for (int idx = threadIdx.x; idx < NC * nblk; idx += blockDim.x) {
        const int c = idx / nblk;
        const int n = idx - c * nblk;
        uint32_t w[9] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (c < n_active) {
            const uint32_t *src =
                reinterpret_cast<const uint32_t *>(p.xq + (size_t)src_col(c) * p.xq_col_bytes + (size_t)n * Q8_1_BYTES);
#pragma unroll
            for (int i = 0; i < 9; ++i) w[i] = src[i];
        }
        int S = 0;
#pragma unroll
        for (int i = 1; i < 9; ++i) S = dp4a_ss(w[i], 0x01010101u, S);
        const int u = n >> 3, sub = n & 7;
        uint4 *dq = reinterpret_cast<uint4 *>(act_qs + ((size_t)c * U + u) * ACT_QS_STRIDE + 32 * sub);
        dq[0] = make_uint4(w[1], w[2], w[3], w[4]);
        dq[1] = make_uint4(w[5], w[6], w[7], w[8]);
        float *sc = reinterpret_cast<float *>(act_sc + ((size_t)c * U + u) * ACT_SC_STRIDE);
        const float d8 = half_bits_to_float(w[0]);
        if (F == FMT_Q4_K) {
            sc[4 * (sub >> 1) + (sub & 1)] = d8;
            sc[4 * (sub >> 1) + 2 + (sub & 1)] = d8 * static_cast<float>(S);
        } else {
            sc[2 * sub] = d8;
            sc[2 * sub + 1] = half_bits_to_float(w[0] >> 16);
        }
    }
}

// One unit of NRL rows (shared addresses ub[r], rows with live[r] false are
// skipped) against one activation column (codes at aq, scalars at as):
// v[r] += the unit's contribution.  With DEBUG, writes the unit's integer
// sums (layout of qmv_debug_subblock_sums) to dbg[r].
template <int F, int NRL, bool DEBUG>
__device__ __forceinline__ void unit_dot(const uint32_t (&ub)[NRL], const bool (&live)[NRL], uint32_t aq, uint32_t as,
                                         float (&v)[NRL], int32_t *const (&dbg)[NRL])
{
    if (F == FMT_Q4_K) {
        float d[NRL], dmin[NRL];
        uint32_t sc_lo[NRL], m_lo[NRL], sc_hi[NRL], m_hi[NRL];
#pragma unroll
        for (int r = 0; r < NRL; ++r) {
            if (!live[r]) continue;
            const uint4 hdr = lds128(ub[r]);
            d[r] = half_bits_to_float(hdr.x);
            dmin[r] = half_bits_to_float(hdr.x >> 16);
            // byte k of these words: scale / min of sub-block k (lo) and 4+k (hi)
            sc_lo[r] = hdr.y & 0x3F3F3F3Fu;
            m_lo[r] = hdr.z & 0x3F3F3F3Fu;
            sc_hi[r] = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
            m_hi[r] = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 a0 = lds128(aq + 64 * j);
            const uint4 a1 = lds128(aq + 64 * j + 16);
            const uint4 a2 = lds128(aq + 64 * j + 32);
            const uint4 a3 = lds128(aq + 64 * j + 48);
            const uint4 sv = lds128(as + 16 * j);
            const uint32_t alo[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t ahi[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
            const float d8lo = __uint_as_float(sv.x), d8hi = __uint_as_float(sv.y);
            const float Dlo = __uint_as_float(sv.z), Dhi = __uint_as_float(sv.w);
            const int sh = 16 * (j & 1);
#pragma unroll
            for (int r = 0; r < NRL; ++r) {
                if (!live[r]) continue;
                const uint4 q0 = lds128(ub[r] + 16 + 32 * j);
                const uint4 q1 = lds128(ub[r] + 32 + 32 * j);
                const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                int l0 = 0, l1 = 0, h0 = 0, h1 = 0;  // four short chains for ILP
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    l0 = dp4a_ss(q[i] & 0x0F0F0F0Fu, alo[i], l0);
                    l1 = dp4a_ss(q[i + 1] & 0x0F0F0F0Fu, alo[i + 1], l1);
                    h0 = dp4a_us(q[i] & 0xF0F0F0F0u, ahi[i], h0);
                    h1 = dp4a_us(q[i + 1] & 0xF0F0F0F0u, ahi[i + 1], h1);
                }
                const int dlo = l0 + l1, dhi16 = h0 + h1;
                const uint32_t scw = (j < 2) ? sc_lo[r] : sc_hi[r];
                const uint32_t mw = (j < 2) ? m_lo[r] : m_hi[r];
                const float sc0 = static_cast<float>((scw >> sh) & 0xffu);
                const float sc1 = static_cast<float>((scw >> (sh + 8)) & 0xffu);
                const float m0 = static_cast<float>((mw >> sh) & 0xffu);
                const float m1 = static_cast<float>((mw >> (sh + 8)) & 0xffu);
                v[r] += (d[r] * sc0) * (d8lo * static_cast<float>(dlo)) +
                        (d[r] * sc1 * 0.0625f) * (d8hi * static_cast<float>(dhi16)) - dmin[r] * (m0 * Dlo + m1 * Dhi);
                if constexpr (DEBUG) {
                    int s0 = 0, s1 = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        s0 = dp4a_ss(0x01010101u, alo[i], s0);
                        s1 = dp4a_ss(0x01010101u, ahi[i], s1);
                    }
                    dbg[r][4 * j + 0] = dlo;
                    dbg[r][4 * j + 1] = s0;
                    dbg[r][4 * j + 2] = dhi16 >> 4;
                    dbg[r][4 * j + 3] = s1;
                }
            }
        }
    } else {
        // 8 Q4_0 blocks: block t occupies bytes [18t, 18t+18) of the unit, i.e.
        // bytes [2t, 2t+18) of the 16-byte chunks t and t+1: a sliding window.
        uint32_t win[NRL][8];
#pragma unroll
        for (int r = 0; r < NRL; ++r) {
            if (!live[r]) continue;
            const uint4 c0 = lds128(ub[r]);
            win[r][4] = c0.x; win[r][5] = c0.y; win[r][6] = c0.z; win[r][7] = c0.w;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint4 alo = lds128(aq + 32 * t);
            const uint4 ahi = lds128(aq + 32 * t + 16);
            uint32_t s0, s1;
            asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(s0), "=r"(s1) : "r"(as + 8 * t));
            const uint32_t al[4] = {alo.x, alo.y, alo.z, alo.w};
            const uint32_t ah[4] = {ahi.x, ahi.y, ahi.z, ahi.w};
#pragma unroll
            for (int r = 0; r < NRL; ++r) {
                if (!live[r]) continue;
                const uint4 cn = lds128(ub[r] + 16 * (t + 1));
                win[r][0] = win[r][4]; win[r][1] = win[r][5]; win[r][2] = win[r][6]; win[r][3] = win[r][7];
                win[r][4] = cn.x; win[r][5] = cn.y; win[r][6] = cn.z; win[r][7] = cn.w;
                const int db = 2 * t;      // byte of d in the window
                const int qb = 2 * t + 2;  // first byte of qs in the window
                const float d4 = half_bits_to_float(win[r][db >> 2] >> (8 * (db & 3)));
                uint32_t q[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    q[i] = (qb & 3) ? __funnelshift_r(win[r][(qb >> 2) + i], win[r][(qb >> 2) + i + 1], 8 * (qb & 3))
                                    : win[r][(qb >> 2) + i];
                int dlo = 0, dhi16 = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    dlo = dp4a_ss(q[i] & 0x0F0F0F0Fu, al[i], dlo);
                    dhi16 = dp4a_us(q[i] & 0xF0F0F0F0u, ah[i], dhi16);
                }
                const int sumi = dlo + (dhi16 >> 4);
                v[r] += d4 * (__uint_as_float(s0) * static_cast<float>(sumi) - 8.0f * __uint_as_float(s1));
                if constexpr (DEBUG) dbg[r][t] = sumi;
            }
        }
    }
}

// tm0: tensor map of W (MoE: of all experts' rows stacked); tm1: of the gate
// matrix (GATE mode; otherwise unused).  Box = [18 eight-byte elements] x
// [KW units] x [RT rows], RT = rows-per-lane * 32/KW.
template <int F, int NC, int MODE>
__global__ void __launch_bounds__(MAX_THREADS) gemv_units_kernel(const __grid_constant__ CUtensorMap tm0,
                                                                 const __grid_constant__ CUtensorMap tm1,
                                                                 const GemvParams p, unsigned int *fault)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    __shared__ int s_tok[8];
    __shared__ uint32_t s_slots[8];
    __shared__ int s_cnt;

    constexpr int NM = (MODE == MODE_GATE) ? 2 : 1;  // matrices streamed per group
    constexpr int NRL = NM * UNITS_RPL;              // row-slices per lane
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int U = p.units_per_row;
    const int KW = p.slice_units;  // lanes per row (power of two)
    const int RW = 32 / KW;
    const int RPL = p.rpl;          // rows per lane, 1..UNITS_RPL
    const int RT = RW * RPL;        // rows per group
    const int rw = lane / KW, kw = lane & (KW - 1);
    int n_active = p.ncols;
    int row_base = 0;  // row offset of the streamed matrix inside the tensor map

    if constexpr (MODE == MODE_MOE) {
        pdl_launch_dependents();
        pdl_wait();
        if (blockIdx.y == static_cast<unsigned>(p.n_expert)) {
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
        if (n_active == 0) return;
        row_base = static_cast<int>(blockIdx.y) * static_cast<int>(p.M);
    }

    // shared layout: [activations][rings nwarps x stages x slot][mbarriers nwarps x stages]
    uint8_t *ring = smem + p.act_bytes + (size_t)warp * p.stages * p.slot_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.act_bytes + (size_t)nwarps * p.stages * p.slot_bytes) +
                     (size_t)warp * p.stages;
    const int n_sl = (U + KW - 1) / KW;
    // every warp of the grid owns a contiguous, balanced range of row groups
    const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
    const int64_t wtot = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t g_begin = (gwarp * p.n_groups) / wtot;
    const int64_t my_groups = ((gwarp + 1) * p.n_groups) / wtot - g_begin;
    const int64_t total = my_groups * n_sl;
    const int stages = p.stages;
    const uint32_t box_bytes = static_cast<uint32_t>(RT) * KW * UNIT_B;
    const uint64_t policy = policy_evict_first();

    int64_t is_grp = g_begin;
    int is_s = 0, is_slot = 0;
    int64_t issued = 0;
    auto issue_next = [&]() {  // lane 0 only
        const uint32_t bar = smem_u32(bars + is_slot);
        const uint32_t dst = smem_u32(ring + (size_t)is_slot * p.slot_bytes);
        const int u0 = is_s * KW;
        const int y = row_base + static_cast<int>(is_grp * RT);
        mbar_arrive_expect_tx(bar, box_bytes * NM);
        tma_load_3d(dst, &tm0, u0, y, bar, policy);
        if constexpr (MODE == MODE_GATE) tma_load_3d(dst + box_bytes, &tm1, u0, y, bar, policy);
        if (++is_s == n_sl) { is_s = 0; ++is_grp; }
        if (++is_slot == stages) is_slot = 0;
        ++issued;
    };

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_u32(bars + s), 1);
        fence_mbar_init();
        fence_proxy_async_shared();
        while (issued < total && issued < stages) issue_next();  // weights first
    }
    __syncwarp();

    if constexpr (MODE != MODE_MOE) {
        pdl_launch_dependents();
        pdl_wait();
    }
    if constexpr (MODE == MODE_MOE)
        stage_units_activations<F, NC>(p, smem, n_active, [&](int c) { return s_tok[c]; });
    else
        stage_units_activations<F, NC>(p, smem, n_active, [](int c) { return c; });
    __syncthreads();

    const uint32_t act_qs = smem_u32(smem);
    const uint32_t act_sc = act_qs + NC * U * ACT_QS_STRIDE;

    float acc[NRL][NC];
#pragma unroll
    for (int r = 0; r < NRL; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;

    bool ok = true;
    int64_t waited = 0;
    int c_slot = 0;
    uint32_t c_par = 0;
    for (int64_t gi = 0; gi < my_groups && ok; ++gi) {
        const int64_t r0 = (g_begin + gi) * RT;
        for (int s = 0; s < n_sl; ++s) {
            const bool got = mbar_wait_bounded(smem_u32(bars + c_slot), c_par);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            ++waited;
            const int u = s * KW + kw;  // this lane's unit
            if (u < U) {
                const uint32_t slotp = smem_u32(ring + (size_t)c_slot * p.slot_bytes);
                uint32_t ub[NRL];
                bool live[NRL];
                int32_t *dbg[NRL];
#pragma unroll
                for (int m = 0; m < NM; ++m)
#pragma unroll
                    for (int q = 0; q < UNITS_RPL; ++q) {
                        const int rr = rw + RW * q;  // row inside the group
                        ub[m * UNITS_RPL + q] = slotp + m * box_bytes + (rr * KW + kw) * UNIT_B;
                        live[m * UNITS_RPL + q] = q < RPL && r0 + rr < p.M;
                        dbg[m * UNITS_RPL + q] = nullptr;
                    }
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    if (MODE != MODE_PLAIN && c >= n_active) break;
                    const uint32_t aq = act_qs + (c * U + u) * ACT_QS_STRIDE;
                    const uint32_t as = act_sc + (c * U + u) * ACT_SC_STRIDE;
                    if constexpr (MODE == MODE_DEBUG) {
#pragma unroll
                        for (int q = 0; q < UNITS_RPL; ++q)
                            if (live[q])
                                dbg[q] = p.dbg + ((size_t)c * p.M + r0 + rw + RW * q) * (size_t)(F == FMT_Q4_0 ? p.K / 32 : p.K / 16) +
                                         (size_t)u * (F == FMT_Q4_0 ? 8 : 16);
                        float scratch[NRL];
#pragma unroll
                        for (int r = 0; r < NRL; ++r) scratch[r] = 0.f;
                        unit_dot<F, NRL, true>(ub, live, aq, as, scratch, dbg);
                    } else {
                        float vv[NRL];
#pragma unroll
                        for (int r = 0; r < NRL; ++r) vv[r] = 0.f;
                        unit_dot<F, NRL, false>(ub, live, aq, as, vv, dbg);
#pragma unroll
                        for (int r = 0; r < NRL; ++r) acc[r][c] += vv[r];
                    }
                }
            }
            __syncwarp();  // the slot is free before it is refilled
            if (lane == 0 && issued < total) {
                fence_proxy_async_shared();
                issue_next();
            }
            if (++c_slot == stages) { c_slot = 0; c_par ^= 1u; }
        }
        if (!ok) break;
        if constexpr (MODE != MODE_DEBUG) {
#pragma unroll
            for (int r = 0; r < NRL; ++r)
#pragma unroll
                for (int c = 0; c < NC; ++c)
                    for (int o = KW >> 1; o > 0; o >>= 1) acc[r][c] += __shfl_xor_sync(0xffffffffu, acc[r][c], o);
            if (kw == 0) {
#pragma unroll
                for (int q = 0; q < UNITS_RPL; ++q) {
                    const int64_t row = r0 + rw + RW * q;
                    if (q >= RPL || row >= p.M) continue;
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        if (c >= n_active) break;
                        if constexpr (MODE == MODE_PLAIN) {
                            p.y[(size_t)c * p.ldy + row] = acc[q][c];
                        } else if constexpr (MODE == MODE_GATE) {
                            p.y[(size_t)c * p.ldy + row] = acc[q][c] * silu_f32(acc[UNITS_RPL + q][c]);
                        } else {
                            const int tok = s_tok[c];
                            uint32_t mask = s_slots[c];
                            while (mask) {
                                const int k = __ffs(mask) - 1;
                                mask &= mask - 1;
                                p.y[((size_t)tok * p.top_k + k) * p.M + row] = acc[q][c];
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NRL; ++r)
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;
        }
    }

    if (!ok) {
        if (lane == 0) atomicExch(fault, FAULT_WAIT_TIMEOUT);
        // let every copy this warp still has in flight land before exiting
        const int64_t n_issued = __shfl_sync(0xffffffffu, issued, 0);
        for (int64_t m = waited; m < n_issued; ++m)
            (void)mbar_wait_bounded(smem_u32(bars + (m % stages)), static_cast<uint32_t>((m / stages) & 1));
    }
}

}  // namespace qmv
