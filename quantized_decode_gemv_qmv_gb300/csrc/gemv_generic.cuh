// Generic quantized GEMV: any K that is a multiple of the block size, any
// 2-byte aligned W, activations read straight from global memory.  Used for
// shapes the tile kernel cannot take (rows whose byte size is not a multiple
// of 16, e.g. Q4_0 with K % 256 != 0 or Q6_K with K % 2048 != 0; misaligned
// W; activations larger than the shared-memory budget).  One warp per output
// row, lanes over blocks, byte-granular loads; the arithmetic is the same
// block formula as the streaming kernel, integer sums by dp4a.
#pragma once

#include "gemv_params.cuh"

namespace qmv {

__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p)
{
    return static_cast<uint32_t>(__ldg(p)) | (static_cast<uint32_t>(__ldg(p + 1)) << 8);
}

// four bytes as a packed int, any alignment
__device__ __forceinline__ int ld_i8x4(const uint8_t *p)
{
    return static_cast<int>(static_cast<uint32_t>(__ldg(p)) | (static_cast<uint32_t>(__ldg(p + 1)) << 8) |
                            (static_cast<uint32_t>(__ldg(p + 2)) << 16) |
                            (static_cast<uint32_t>(__ldg(p + 3)) << 24));
}

// q8_1 block n of column xc: 4 packed ints per 16-value half h
__device__ __forceinline__ int q8_word(const uint8_t *xc, int n, int w)
{
    return *reinterpret_cast<const int *>(xc + (size_t)n * Q8_1_BYTES + 4 + 4 * w);
}

__device__ __forceinline__ float q8_d(const uint8_t *xc, int n)
{
    return half_bits_to_float(*reinterpret_cast<const uint16_t *>(xc + (size_t)n * Q8_1_BYTES));
}

__device__ __forceinline__ float q8_s(const uint8_t *xc, int n)
{
    return half_bits_to_float(*reinterpret_cast<const uint16_t *>(xc + (size_t)n * Q8_1_BYTES + 2));
}

// Value of block b of a row for one activation column; also writes the
// block's integer sums to dbg_row when it is not null.
template <int F>
__device__ float generic_block(const uint8_t *row, int b, const uint8_t *xc, int32_t *dbg_row)
{
    if (F == FMT_Q4_0) {
        const uint8_t *blk = row + (size_t)b * Q4_0_BYTES;
        int sumi = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int v = ld_i8x4(blk + 2 + 4 * w);
            sumi = dp4a(v & 0x0F0F0F0F, q8_word(xc, b, w), sumi);
            sumi = dp4a((v >> 4) & 0x0F0F0F0F, q8_word(xc, b, 4 + w), sumi);
        }
        if (dbg_row) dbg_row[b] = sumi;
        return half_bits_to_float(ld_u16(blk)) * (q8_d(xc, b) * static_cast<float>(sumi) - 8.0f * q8_s(xc, b));
    } else if (F == FMT_Q4_K) {
        const uint8_t *blk = row + (size_t)b * Q4_K_BYTES;
        const float d = half_bits_to_float(ld_u16(blk));
        const float dmin = half_bits_to_float(ld_u16(blk + 2));
        const uint8_t *s = blk + 4;
        float v = 0.f;
        for (int sb = 0; sb < 8; ++sb) {
            int sc, m;
            if (sb < 4) {
                sc = __ldg(s + sb) & 63;
                m = __ldg(s + sb + 4) & 63;
            } else {
                sc = (__ldg(s + sb + 4) & 15) | ((__ldg(s + sb - 4) >> 6) << 4);
                m = (__ldg(s + sb + 4) >> 4) | ((__ldg(s + sb) >> 6) << 4);
            }
            const uint8_t *q = blk + 16 + 32 * (sb >> 1);
            const int shift = 4 * (sb & 1);
            const int n8 = 8 * b + sb;
            int dot1 = 0, dot2 = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int u = q8_word(xc, n8, w);
                dot1 = dp4a((ld_i8x4(q + 4 * w) >> shift) & 0x0F0F0F0F, u, dot1);
                dot2 = dp4a(0x01010101, u, dot2);
            }
            if (dbg_row) { dbg_row[2 * n8] = dot1; dbg_row[2 * n8 + 1] = dot2; }
            const float d8 = q8_d(xc, n8);
            v += d * static_cast<float>(sc) * (d8 * static_cast<float>(dot1)) -
                 dmin * static_cast<float>(m) * (d8 * static_cast<float>(dot2));
        }
        return v;
    } else {
        const uint8_t *blk = row + (size_t)b * Q6_K_BYTES;
        const float d = half_bits_to_float(ld_u16(blk + 208));
        float v = 0.f;
        for (int sb = 0; sb < 16; ++sb) {
            // elements 16sb..16sb+15: half h, group g, positions l0..l0+15
            const int e0 = 16 * sb;
            const int h = e0 >> 7, r = e0 & 127, g = r >> 5, l0 = r & 31;
            const uint8_t *ql = blk + 64 * h + 32 * (g & 1) + l0;
            const uint8_t *qh = blk + 128 + 32 * h + l0;
            const int n8 = 8 * b + (sb >> 1);
            int sumi = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int lo = (ld_i8x4(ql + 4 * w) >> (4 * (g >> 1))) & 0x0F0F0F0F;
                const int hi = ((ld_i8x4(qh + 4 * w) >> (2 * g)) & 0x03030303) << 4;
                const int u = q8_word(xc, n8, 4 * (sb & 1) + w);
                sumi = dp4a(lo | hi, u, sumi);
                sumi = dp4a(static_cast<int>(0xE0E0E0E0u), u, sumi);  // -32 per value
            }
            if (dbg_row) dbg_row[16 * b + sb] = sumi;
            v += d * static_cast<float>(static_cast<int8_t>(__ldg(blk + 192 + sb))) *
                 (q8_d(xc, n8) * static_cast<float>(sumi));
        }
        return v;
    }
}

template <int F, int MODE>
__global__ void __launch_bounds__(256) gemv_generic_kernel(const GemvParams p)
{
    constexpr int BE = (F == FMT_Q4_0) ? QK4_0 : QK_K;
    __shared__ int s_tok[8];
    __shared__ uint32_t s_slots[8];
    __shared__ int s_cnt;
    pdl_launch_dependents();
    pdl_wait();

    const uint8_t *W = p.W;
    int n_active = p.ncols;
    if constexpr (MODE == MODE_MOE) {
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
        W = p.W + (size_t)blockIdx.y * p.expert_bytes;
    }

    const int lane = threadIdx.x & 31;
    const int nb = p.K / BE;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < p.M; row += warps) {
        float acc[8], accg[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = accg[c] = 0.f;
        for (int b = lane; b < nb; b += 32) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                if (c >= n_active) break;
                const int col = (MODE == MODE_MOE) ? s_tok[c] : c;
                const uint8_t *xc = p.xq + (size_t)col * p.xq_col_bytes;
                int32_t *dbg = nullptr;
                if constexpr (MODE == MODE_DEBUG)
                    dbg = p.dbg + ((size_t)c * p.M + row) * (size_t)(F == FMT_Q4_0 ? p.K / 32 : p.K / 16);
                acc[c] += generic_block<F>(W + (size_t)row * p.row_bytes, b, xc, dbg);
                if constexpr (MODE == MODE_GATE)
                    accg[c] += generic_block<F>(p.W2 + (size_t)row * p.row_bytes, b, xc, nullptr);
            }
        }
        if constexpr (MODE == MODE_DEBUG) continue;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (c >= n_active) break;
            const float v = warp_sum(acc[c]);
            const float vg = (MODE == MODE_GATE) ? warp_sum(accg[c]) : 0.f;
            if (lane != 0) continue;
            if constexpr (MODE == MODE_PLAIN) p.y[(size_t)c * p.ldy + row] = v;
            else if constexpr (MODE == MODE_GATE) p.y[(size_t)c * p.ldy + row] = v * silu_f32(vg);
            else {
                uint32_t mask = s_slots[c];
                while (mask) {
                    const int k = __ffs(mask) - 1;
                    mask &= mask - 1;
                    p.y[((size_t)s_tok[c] * p.top_k + k) * p.M + row] = v;
                }
            }
        }
    }
}

}  // namespace qmv
