// Per-unit arithmetic of the tile kernel (gemv_tiles.cuh): a unit is 256
// weights -- a Q4_K super-block (144 bytes), 8 Q4_0 blocks (144 bytes) or a
// Q6_K super-block (210 bytes).
//
// Method: "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q" (vec_dot_q4_0_q8_1_impl,
// vec_dot_q4_K_q8_1_impl_vmmq and the Q6_K snippet): int8 dot products per
// block scaled by the block scales, with the page's constant corrections
// (Q4_0: -8*s; Q4_K: -dmin*m*d8*sum(qy); Q6_K: -32*sum(qy) per sub-block).
//
// GB300 choices: one lane decodes a whole unit (one header decode per 256
// weights, the 6-bit scales/mins of all 8 sub-blocks unpacked word-parallel),
// the high nibbles are used in place (dp4a.u32.s32 on q & 0xF0F0F0F0 is 16x
// the dot; the 1/16 folds into the scale exactly), and activations are
// restaged once per CTA so that every 128-bit shared read is aligned and the
// 8 lanes of a read phase hit distinct bank quads (units 272 / 80 bytes apart).
#pragma once

#include "gemv_params.cuh"

namespace qmv {

constexpr int UNIT_B = 144;         // bytes of a Q4_0 / Q4_K unit
constexpr int ACT_QS_STRIDE = 272;  // shared bytes per unit of staged activation codes (256 + pad)
constexpr int ACT_SC_STRIDE = 80;   // Q4_0 / Q4_K: shared bytes per unit of staged activation scalars (64 + pad)

template <int F>
__host__ __device__ constexpr int unit_bytes()
{
    return F == FMT_Q6_K ? Q6_K_BYTES : UNIT_B;
}

// Staged scalars per unit: Q4_K {d8[2j], d8[2j+1], D[2j], D[2j+1]} per qs chunk j
// with D = d8 * sum(qy over the 32-value block); Q4_0 {d8[t], s8[t]} per block;
// Q6_K d8[0..7] then the 16-value half sums S16[0..15] (int).
template <int F>
__host__ __device__ constexpr int act_sc_stride()
{
    return F == FMT_Q6_K ? 96 : ACT_SC_STRIDE;
}

// The scalars of q8_1 block `sub` (0..7) of a unit as 32-bit words of the
// unit's scalar area: n words, word i at byte offset off[i] holding val[i].
// ds = (half d | half s << 16) as stored, S = the block's code sum, S_lo / S_hi
// = the sums of its codes 0..15 / 16..31.
template <int F>
__device__ __forceinline__ int act_scalar_words(int sub, uint32_t ds, int S, int S_lo, int S_hi, uint32_t (&off)[3],
                                                uint32_t (&val)[3])
{
    const float d8 = half_bits_to_float(ds);
    if constexpr (F == FMT_Q4_K) {
        off[0] = 4u * (4 * (sub >> 1) + (sub & 1));
        val[0] = __float_as_uint(d8);
        off[1] = 4u * (4 * (sub >> 1) + 2 + (sub & 1));
        val[1] = __float_as_uint(d8 * static_cast<float>(S));
        return 2;
    } else if constexpr (F == FMT_Q4_0) {
        off[0] = 8u * sub;
        val[0] = __float_as_uint(d8);
        off[1] = 8u * sub + 4u;
        val[1] = __float_as_uint(half_bits_to_float(ds >> 16));
        return 2;
    } else {
        off[0] = 4u * sub;
        val[0] = __float_as_uint(d8);
        off[1] = 32u + 8u * sub;
        val[1] = static_cast<uint32_t>(S_lo);
        off[2] = 36u + 8u * sub;
        val[2] = static_cast<uint32_t>(S_hi);
        return 3;
    }
}

// Writes the scalars of q8_1 block `sub` of a unit (act_scalar_words) into this
// CTA's shared memory at sc_unit.
template <int F>
__device__ __forceinline__ void store_act_scalars(uint8_t *sc_unit, int sub, uint32_t ds, int S, int S_lo, int S_hi)
{
    uint32_t off[3], val[3];
    const int n = act_scalar_words<F>(sub, ds, S, S_lo, S_hi, off, val);
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (i < n) *reinterpret_cast<uint32_t *>(sc_unit + off[i]) = val[i];
}

// NW consecutive 32-bit words starting at a 2-byte aligned shared address: the
// covering aligned words are read once each and funnel-shifted pairwise (Q6_K
// super-blocks are 210 bytes, so they start on 2-byte boundaries).  Reads the
// aligned words [a & ~3, (a & ~3) + 4*(NW+1)).
template <int NW>
__device__ __forceinline__ void lds_run_u2(uint32_t a, uint32_t (&out)[NW])
{
    const uint32_t base = a & ~3u;
    const uint32_t sh = (a & 2u) << 3;  // 0 or 16 bits
    uint32_t prev = lds32(base);
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        const uint32_t nxt = lds32(base + 4u * (k + 1));
        out[k] = __funnelshift_r(prev, nxt, sh);
        prev = nxt;
    }
}

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

// Activation staging (4-byte loads; any 4-byte aligned xq): per column and unit
// u the 256 codes in natural order at c*U*272 + u*272, then the unit's scalars
// (store_act_scalars) at sc + (c*U + u)*act_sc_stride, sc = NC*U*272.
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
    } else if (F == FMT_Q6_K) {
        // One super-block (210 bytes, 2-byte aligned): ql[128] at 0, qh[64] at
        // 128, int8 scales[16] at 192, half d at 208.  Element e = 128h + 32g + l
        // (h < 2, g < 4, l < 32) has low 4 bits in ql[64h + 32(g&1) + l]
        // (nibble g>>1) and high 2 bits in qh[32h + l] (bits 2g, 2g+1); its
        // 16-value sub-block is e/16.  Per (h, word w of l), the words of ql_a =
        // ql[64h..], ql_b = ql[64h+32..] and qh hold 4 elements of each g.
#pragma unroll
        for (int r = 0; r < NRL; ++r) {
            if (!live[r]) continue;
            uint32_t dw[1], scw[4];
            lds_run_u2<1>(ub[r] + 208, dw);
            lds_run_u2<4>(ub[r] + 192, scw);
            const float d = half_bits_to_float(dw[0]);
            float acc = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t qa[8], qb[8], qh[8];
                lds_run_u2<8>(ub[r] + 64 * h, qa);
                lds_run_u2<8>(ub[r] + 64 * h + 32, qb);
                lds_run_u2<8>(ub[r] + 128 + 32 * h, qh);
                const uint4 d8v = lds128(as + 16 * h);          // d8 of q8_1 blocks 4h..4h+3
                const uint4 s16a = lds128(as + 32 + 32 * h);    // S16 of sub-blocks 8h..8h+3
                const uint4 s16b = lds128(as + 48 + 32 * h);    // S16 of sub-blocks 8h+4..8h+7
                const float d8s[4] = {__uint_as_float(d8v.x), __uint_as_float(d8v.y), __uint_as_float(d8v.z),
                                      __uint_as_float(d8v.w)};
                const int s16[8] = {static_cast<int>(s16a.x), static_cast<int>(s16a.y), static_cast<int>(s16a.z),
                                    static_cast<int>(s16a.w), static_cast<int>(s16b.x), static_cast<int>(s16b.y),
                                    static_cast<int>(s16b.z), static_cast<int>(s16b.w)};
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint4 a0 = lds128(aq + 128 * h + 32 * g);
                    const uint4 a1 = lds128(aq + 128 * h + 32 * g + 16);
                    const uint32_t act[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    int dlo = 0, dhi = 0;
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint32_t ql = (g & 1) ? qb[w] : qa[w];
                        const uint32_t lo4 = (g & 2) ? ((ql >> 4) & 0x0F0F0F0Fu) : (ql & 0x0F0F0F0Fu);
                        const uint32_t hi2 = g == 0 ? (qh[w] << 4) : g == 1 ? (qh[w] << 2) : g == 2 ? qh[w] : (qh[w] >> 2);
                        const uint32_t q = lo4 | (hi2 & 0x30303030u);  // 6-bit codes 0..63
                        if (w < 4) dlo = dp4a_us(q, act[w], dlo);
                        else dhi = dp4a_us(q, act[w], dhi);
                    }
                    const int sb0 = 8 * h + 2 * g;
                    const int t0 = dlo - 32 * s16[2 * g];      // sum (v - 32) * qy, sub-block sb0
                    const int t1 = dhi - 32 * s16[2 * g + 1];  // sub-block sb0 + 1
                    const float sc0 = static_cast<float>(static_cast<int8_t>((scw[sb0 >> 2] >> (8 * (sb0 & 3))) & 0xffu));
                    const float sc1 =
                        static_cast<float>(static_cast<int8_t>((scw[(sb0 + 1) >> 2] >> (8 * ((sb0 + 1) & 3))) & 0xffu));
                    acc += d8s[g] * (sc0 * static_cast<float>(t0) + sc1 * static_cast<float>(t1));
                    if constexpr (DEBUG) {
                        dbg[r][sb0] = t0;
                        dbg[r][sb0 + 1] = t1;
                    }
                }
            }
            v[r] += d * acc;
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
