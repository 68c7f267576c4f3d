// Per-unit arithmetic of the 144-byte-unit formats (Q4_K super-blocks; Q4_0
// in runs of 8 blocks), shared by the tile kernel (gemv_tiles.cuh).
//
// Method: "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q" (vec_dot_q4_0_q8_1_impl,
// vec_dot_q4_K_q8_1_impl_vmmq): int8 dot products per block scaled by the
// block scales, with the page's constant corrections (Q4_0: -8*s; Q4_K:
// -dmin*m*d8*sum(qy)).
//
// GB300 choices: one lane decodes a whole unit (one header decode per 256
// weights, the 6-bit scales/mins of all 8 sub-blocks unpacked word-parallel),
// the high nibbles are used in place (dp4a.u32.s32 on q & 0xF0F0F0F0 is 16x
// the dot; the 1/16 folds into the scale exactly), and activations are
// restaged once per CTA so that every 128-bit shared read is aligned and the
// 8 lanes of a read phase hit distinct bank quads (units 272 / 80 bytes apart).
#pragma once

#include "gemv_stream.cuh"

namespace qmv {

constexpr int UNIT_B = 144;         // bytes of a unit (both formats)
constexpr int ACT_QS_STRIDE = 272;  // shared bytes per unit of staged activation codes (256 + pad)
constexpr int ACT_SC_STRIDE = 80;   // shared bytes per unit of staged activation scalars (64 + pad)

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

// Activation staging (4-byte loads; any 4-byte aligned xq).  Per column and unit u (256 values):
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

}  // namespace qmv
