// Tensor-core decode of the tile kernel (gemv_tiles.cuh) for several
// activation columns: Q4_K.
//
// Method: the block products of "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q"
// (vec_dot_q4_K_q8_1_impl_vmmq), as in unit_dot: per 32-weight sub-block the
// integer dot sum(q * qy), scaled by d*sc*d8, minus dmin*m*d8*sum(qy).
//
// Why it exists.  From about three columns on, the per-column dp4a decode is
// bound by instruction issue, not by HBM: every column repeats 64 dp4a, the
// activation loads and the scaling per 256 weights.  This decode is the
// decode-once alternative for that regime.  On GB300 it measured slower than
// the dp4a decode at every column count up to 8 (14336x4096: 16.1 vs 7.6 us at
// one column, 20.3 vs 16.7 us at eight), with one HMMA per mma.sync and the
// time spent in the integer and fp32 work around it, so it is off by default
// and selected with qmv_set_mma_min_cols.  Here a warp multiplies
// its tile's 8 weight rows by all 8 columns at once with mma.sync m16n8k16
// (fp16 operands, fp32 accumulators; A = the activation columns, rows 8..15
// zero, B = the weight rows), two instructions per 32-weight sub-block:
//   * the weights enter as fp16 1024 + q (low nibbles) or 1024 + 16q (high
//     nibbles used in place), the bit patterns 0x6400 | code, one logic op per
//     two codes; the activations as their exact int8 codes, staged once per
//     CTA as fp16;
//   * every product and every partial sum of a sub-block is an integer below
//     2^23 (|sum| <= 32 * 1264 * 127), so the fp32 accumulators hold exact
//     integers, and the bias is removed exactly: 16^h * sum(q*qy) = C -
//     1024*sum(qy);
//   * the block scaling that follows is plain fp32: per output and sub-block
//     two products and four fused multiply-adds.  The per-row factors d*sc and
//     dmin*m are computed once per tile (one lane per row and unit) into a
//     small per-warp scratch, not by every lane that needs them.
// The operands' k order inside a sub-block is a permutation shared by A and B
// (lane t of a row holds the 8 codes 8t..8t+7 of the sub-block), so each lane
// reads its weights as one 8-byte piece and converts them without shuffles.
// tcgen05 does not fit this contraction: each 32-term block dot must be
// rescaled by its own per-column d8 before it is summed, i.e. read back from
// the accumulator every two k-steps, which mma.sync's register accumulators do
// for free and tensor memory does not.
#pragma once

#include "gemv_units.cuh"
#include "q8_1.cuh"

namespace qmv {

constexpr int MMA_RW = 8;              // weight rows per tile (the mma's N)
constexpr int MMA_COLS = 8;            // activation columns of one mma (its M rows 0..7)
constexpr int MMA_BLK_BYTES = 64;      // staged fp16 codes of one q8_1 block
constexpr int MMA_FAC_ROW = 80;        // scratch bytes per row and unit: 16 factors + 16 of padding
constexpr int MMA_MIN_COLS = 9;        // default: never (measured slower than dp4a at 1..8 columns on GB300)

// Per-warp scratch of a tile's row factors: 4 units x 8 rows x 80 bytes.  The
// 80-byte row stride puts the rows 2t and 2t+1 read by the lanes of one read
// phase on distinct banks.
constexpr int MMA_FAC_BYTES = 4 * MMA_RW * MMA_FAC_ROW;

// Shared bytes per staged column of nblk q8_1 blocks: 64 bytes of fp16 codes
// per block plus 64, so that consecutive columns start 64 bytes apart modulo
// 128 (a 128-bit read phase of 8 lanes covers two columns' 64-byte pieces, on
// distinct banks).
__host__ __device__ constexpr int64_t mma_col_stride(int64_t nblk) { return nblk * MMA_BLK_BYTES + 64; }

// Shared bytes per staged column of (d8, S) float pairs: 8 per block plus 16,
// for the same reason.
__host__ __device__ constexpr int64_t mma_sc_stride(int64_t nblk) { return nblk * 8 + 16; }

// Shared bytes of the activation area: nc columns of codes, then nc columns
// of block scalars.
__host__ __device__ constexpr int64_t mma_act_bytes(int64_t nc, int64_t nblk)
{
    return nc * (mma_col_stride(nblk) + mma_sc_stride(nblk));
}

__device__ __forceinline__ uint2 lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t a, float x, float y, float z, float w)
{
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t a, uint4 v)
{
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulators.  Fragments (lane =
// 4g + t): a0 = A[g][2t..2t+1], a1 = A[g+8][2t..2t+1], a2 = A[g][2t+8..2t+9],
// a3 = A[g+8][2t+8..2t+9]; b0 = B[2t..2t+1][g], b1 = B[2t+8..2t+9][g];
// d = {D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1]}.  Here A's rows 8..15
// are zero (a1 = a3 = 0), so d[2] and d[3] stay zero.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Four int8 codes b0..b3 (bytes of w) as exact fp16 pairs: even = (b0, b2),
// odd = (b1, b3), the lower-indexed code in the low half.  0x6400 | u is the
// half 1024 + u for u < 1024; u = byte ^ 0x80 = code + 128, so the value is
// 1152 + code, and subtracting 1152 (0x6480) is exact.
__device__ __forceinline__ void i8x4_to_h2(uint32_t w, uint32_t &even, uint32_t &odd)
{
    const uint32_t e = (w & 0x00FF00FFu) ^ 0x64806480u;
    const uint32_t o = ((w >> 8) & 0x00FF00FFu) ^ 0x64806480u;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(even) : "r"(e), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(odd) : "r"(o), "r"(0x64806480u));
}

// 4-bit codes of bytes (0, 2) of w as the fp16 pair 1024 + code: MASK
// 0x000F000F takes the low nibbles (1024 + q), 0x00F000F0 the high nibbles in
// place (1024 + 16q).  For bytes (1, 3) pass w >> 8.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t nib_h2(uint32_t w)
{
    return (w & MASK) | 0x64006400u;
}

// Activation staging for this decode (fp32 input quantized here, or q8_1
// blocks copied): column c's block n at a16 + c*cs + 64n, lane part t (codes
// 8t..8t+7) as the 16 bytes (even, odd) of codes 8t..8t+3 then of 8t+4..8t+7
// at +16t; the block's d8 and code sum S as floats at sc + c*ss + 8n, sc =
// a16 + ncols*cs.  The q8_1 arithmetic is that of the standalone quantizer
// (q8_1_block_group4), so the codes are bit-identical to quantizing first.  In
// a cluster of ncta CTAs, CTA crank converts a contiguous 1/ncta of the blocks
// and stores them into every CTA's shared memory; the caller completes the
// exchange with a cluster barrier.
template <typename ColFn>
__device__ __forceinline__ void stage_mma_activations(const GemvParams &p, uint8_t *smem, int n_active, ColFn src_col,
                                                      uint32_t crank, uint32_t ncta)
{
    const int U = p.units_per_row;
    const int nblk = U * 8;
    const uint32_t cs = static_cast<uint32_t>(mma_col_stride(nblk));
    const uint32_t ss = static_cast<uint32_t>(mma_sc_stride(nblk));
    const uint32_t a16 = smem_u32(smem);
    const uint32_t scal = a16 + static_cast<uint32_t>(p.ncols) * cs;
    const int n_all = n_active * nblk;
    const int blk0 = static_cast<int>(static_cast<int64_t>(crank) * n_all / ncta);
    const int blk1 = static_cast<int>(static_cast<int64_t>(crank + 1) * n_all / ncta);
    const int tasks = (blk1 - blk0) * 4;  // 4 lanes per block
    const bool vec = ((reinterpret_cast<uintptr_t>(p.xf) | static_cast<uintptr_t>(p.ldx * 4)) & 15u) == 0;
    const int rounds = (tasks + blockDim.x - 1) / blockDim.x;  // the same for every thread
    for (int r = 0; r < rounds; ++r) {
        const int ti = r * blockDim.x + threadIdx.x;
        const bool active = ti < tasks;  // whole groups of 4 lanes
        const int g = blk0 * 4 + ti;
        const int c = active ? g / (nblk * 4) : 0;
        const int rem = g - c * nblk * 4;
        const int n = rem >> 2, j = rem & 3;
        uint32_t w0 = 0u, w1 = 0u, ds = 0u;
        int S = 0;
        if (p.xf != nullptr) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
            if (active)
                q8_1_load8(p.xf + (size_t)src_col(c) * p.ldx, (int64_t)n * QK8_1 + 8 * j, p.K, vec, v);
            int part;
            q8_1_block_group4(v, w0, w1, ds, S, part);  // every lane of the warp takes part
        } else {
            if (active) {
                const uint8_t *blk = p.xq + (size_t)src_col(c) * p.xq_col_bytes + (size_t)n * Q8_1_BYTES;
                ds = __ldcg(reinterpret_cast<const unsigned int *>(blk));
                w0 = __ldcg(reinterpret_cast<const unsigned int *>(blk + 4 + 8 * j));
                w1 = __ldcg(reinterpret_cast<const unsigned int *>(blk + 8 + 8 * j));
            }
            S = dp4a_ss(w1, 0x01010101u, dp4a_ss(w0, 0x01010101u, 0));
            S += __shfl_xor_sync(0xffffffffu, S, 1);
            S += __shfl_xor_sync(0xffffffffu, S, 2);
        }
        if (active) {
            uint4 h;
            i8x4_to_h2(w0, h.x, h.y);
            i8x4_to_h2(w1, h.z, h.w);
            const uint32_t dq = a16 + static_cast<uint32_t>(c) * cs + static_cast<uint32_t>(n * MMA_BLK_BYTES + 16 * j);
            const uint32_t dsc = scal + static_cast<uint32_t>(c) * ss + static_cast<uint32_t>(n * 8);
            const uint32_t d8 = __float_as_uint(half_bits_to_float(ds));
            const uint32_t sf = __float_as_uint(static_cast<float>(S));
            if (ncta == 1) {
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dq), "r"(h.x), "r"(h.y), "r"(h.z),
                             "r"(h.w)
                             : "memory");
                if (j == 0) asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dsc), "r"(d8), "r"(sf) : "memory");
            } else {
                for (uint32_t q = 0; q < ncta; ++q) {
                    st_cluster_v4(mapa_shared(dq, q), h);
                    if (j == 0) st_cluster_v2(mapa_shared(dsc, q), d8, sf);
                }
            }
        }
    }
}

// Row factors of a Q4_K tile (8 rows x 4 units at tb, row stride SS) into the
// warp's scratch fac: lane (row fr = lane & 7, unit fu = lane >> 3) decodes its
// unit's header and stores, per qs chunk j (sub-blocks 2j, 2j+1), the floats
// (d*sc[2j], d*sc[2j+1]/16, dmin*m[2j], dmin*m[2j+1]) at fac + fu*640 + fr*80
// + 16j.  The high-nibble factor carries the 1/16 of the in-place nibbles
// (exact: a power of two).
template <int SS, int UNIT>
__device__ __forceinline__ void mma_row_factors_q4_K(uint32_t tb, uint32_t fac, int lane)
{
    const int fr = lane & 7, fu = lane >> 3;
    const uint4 hdr = lds128(tb + static_cast<uint32_t>(fr * SS + fu * UNIT));
    const float d = half_bits_to_float(hdr.x);
    const float d16 = d * 0.0625f;
    const float dmin = half_bits_to_float(hdr.x >> 16);
    // byte k of these words: scale / min of sub-block k (lo) and 4+k (hi)
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu;
    const uint32_t m_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    const uint32_t dst = fac + static_cast<uint32_t>(fu * (MMA_RW * MMA_FAC_ROW) + fr * MMA_FAC_ROW);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t scw = (j < 2) ? sc_lo : sc_hi;
        const uint32_t mw = (j < 2) ? m_lo : m_hi;
        const int sft = 16 * (j & 1);
        sts128(dst + 16u * j, d * static_cast<float>((scw >> sft) & 0xffu),
               d16 * static_cast<float>((scw >> (sft + 8)) & 0xffu), dmin * static_cast<float>((mw >> sft) & 0xffu),
               dmin * static_cast<float>((mw >> (sft + 8)) & 0xffu));
    }
}

// One Q4_K super-block of the tile's 8 rows against the staged columns
// (lane = 4g + t): w = the unit in row g plus 16 + 8t (its qs bytes 8t..8t+7
// of each 32-byte chunk); act = column g's first block of the unit plus 16t
// and scl = its first (d8, S) pair (both skipped when act_live is false:
// column g multiplies as zero); fr0 / fr1 = the scratch factors of rows 2t and
// 2t+1 for this unit.  v = {y[g][row 2t], y[g][row 2t+1]} += the unit's
// contribution.
__device__ __forceinline__ void mma_unit_q4_K(uint32_t w, uint32_t act, uint32_t scl, bool act_live, uint32_t fr0,
                                              uint32_t fr1, float (&v)[2])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // low nibbles = sub-block 2j, high nibbles = sub-block 2j + 1
        const uint2 q = lds64(w + 32 * j);
        uint4 xl = make_uint4(0u, 0u, 0u, 0u), xh = make_uint4(0u, 0u, 0u, 0u), sc = make_uint4(0u, 0u, 0u, 0u);
        if (act_live) {
            xl = lds128(act + (2 * j) * MMA_BLK_BYTES);
            xh = lds128(act + (2 * j + 1) * MMA_BLK_BYTES);
            sc = lds128(scl + 16 * j);  // (d8, S) of sub-blocks 2j, 2j + 1
        }
        const uint4 f0 = lds128(fr0 + 16 * j);  // (d*sc_lo, d*sc_hi/16, dmin*m_lo, dmin*m_hi) of row 2t
        const uint4 f1 = lds128(fr1 + 16 * j);  // ... of row 2t + 1
        const uint32_t qx8 = q.x >> 8, qy8 = q.y >> 8;
        float cl[4] = {0.f, 0.f, 0.f, 0.f}, ch[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(cl, xl.x, xl.y, nib_h2<0x000F000Fu>(q.x), nib_h2<0x000F000Fu>(qx8));
        mma_16816(cl, xl.z, xl.w, nib_h2<0x000F000Fu>(q.y), nib_h2<0x000F000Fu>(qy8));
        mma_16816(ch, xh.x, xh.y, nib_h2<0x00F000F0u>(q.x), nib_h2<0x00F000F0u>(qx8));
        mma_16816(ch, xh.z, xh.w, nib_h2<0x00F000F0u>(q.y), nib_h2<0x00F000F0u>(qy8));
        const float d8l = __uint_as_float(sc.x), Sl = __uint_as_float(sc.y);
        const float d8h = __uint_as_float(sc.z), Sh = __uint_as_float(sc.w);
        const float Dl = d8l * Sl, Dh = d8h * Sh;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint4 f = k ? f1 : f0;
            const float dl = fmaf(-1024.0f, Sl, cl[k]);  // sum(q*qy), exact
            const float dh = fmaf(-1024.0f, Sh, ch[k]);  // 16 * sum(q*qy), exact
            float a = v[k];
            a = fmaf(__uint_as_float(f.x), d8l * dl, a);
            a = fmaf(__uint_as_float(f.y), d8h * dh, a);
            a = fmaf(-__uint_as_float(f.z), Dl, a);
            a = fmaf(-__uint_as_float(f.w), Dh, a);
            v[k] = a;
        }
    }
}

}  // namespace qmv
