// q8_1 block quantization shared by the standalone quantizer and the GEMV
// kernels that quantize their fp32 input while staging it.
//
// "llama.cpp 源码完全拆解(十四)：mul_mat_vec_q", section "激活的量化:为什么是
// q8_1,而不是 q8_0": per 32 values amax = max|x|, d = amax/127, q = round(x/d),
// block = (half d, half s, 32 int8).  s = half(d * sum(q)) with sum(q) the exact
// integer sum (the page's struct comment; its kernel stores the float sum of
// x instead).  The zero test is taken on d == 0 and q is clamped to +-127:
// for normal inputs this is the page's amax == 0 test; it only differs for
// subnormal blocks whose d underflows.
//
// Every code is decided with explicitly rounded fp32 operations (__fdiv_rn,
// __fmul_rn), C roundf (halfway away from zero) and round-to-nearest-even half
// conversion, so the bytes are a fixed function of the input floats no matter
// which kernel or lane mapping computes them.
#pragma once

#include "common.cuh"

namespace qmv {

__device__ __forceinline__ int clamp_round(float z, float lo, float hi)
{
    float r = roundf(z);
    if (r < lo) r = lo;
    if (r > hi) r = hi;
    return static_cast<int>(r);
}

__device__ __forceinline__ uint32_t f2h_bits(float f)
{
    return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(f)));
}

__device__ __forceinline__ float h2f(uint32_t bits)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// One q8_1 block quantized by 4 consecutive lanes (lanes 4g..4g+3 of the warp),
// lane j holding values 8j..8j+7 of the block in v.  Every lane of the warp must
// call it (the reductions shuffle across the group with the full mask).
// Returns in w0 / w1 the lane's two code words (codes 8j..8j+3, 8j+4..8j+7,
// byte i = code i), in ds the block's (half d | half s << 16) word, in sum the
// exact integer code sum of the block and in part the sum of the lane's own 8
// codes.
__device__ __forceinline__ void q8_1_block_group4(const float (&v)[8], uint32_t &w0, uint32_t &w1, uint32_t &ds,
                                                  int &sum, int &part)
{
    float amax = fabsf(v[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    int s = 0;
    uint32_t b[8];
    // x/d is needed correctly rounded (the integer code is rounded from the
    // fp32 quotient).  With y = RN(1/d), Markstein's correction (Markstein,
    // "Computation of elementary functions on the IBM RISC System/6000
    // processor", IBM J. Res. Dev. 34(1), 1990) q' = RN(q + y*(x - d*q)), the
    // residual x - d*q formed exactly by one FMA, returns RN(x/d) when q is
    // within one ulp of x/d.  q0 = RN(x*y) can be up to 1.5 ulp off, so the
    // correction is applied twice: q0 + y*(x - d*q0) = x/d + (q0 - x/d)(1 - d*y)
    // with |1 - d*y| <= 2^-24, so even with the residual rounded the first step
    // leaves q1 within 1/2 ulp + 3*2^-24 ulp < 1 ulp of x/d, and the second
    // step is the theorem's case.  No intermediate over- or underflows for d in
    // [2^-40, 2^40] and |x/d| >= 2^-30; smaller quotients give code 0 from
    // either quotient.  Since d = RN(amax/127), |x/d| <= 127 (1 + 2^-23) and the
    // codes need no clamp.  Other scales use the IEEE division itself.
    const bool fast = d >= 0x1p-40f && d <= 0x1p40f;  // the same for all 4 lanes of the block
    const float y = fast ? __frcp_rn(d) : 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q;
        if (fast) {
            const float q0 = __fmul_rn(v[i], y);
            const float q1 = __fmaf_rn(__fmaf_rn(-d, q0, v[i]), y, q0);
            const float q2 = __fmaf_rn(__fmaf_rn(-d, q1, v[i]), y, q1);
            q = static_cast<int>(roundf(q2));
        } else {
            q = clamp_round((d == 0.0f) ? 0.0f : __fdiv_rn(v[i], d), -127.0f, 127.0f);
        }
        s += q;
        b[i] = static_cast<uint32_t>(q) & 0xffu;
    }
    part = s;
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    w0 = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    w1 = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    ds = f2h_bits(d) | (f2h_bits(__fmul_rn(d, static_cast<float>(s))) << 16);
    sum = s;
}

// The 8 values of lane j of a block: x[k0 + 8j .. k0 + 8j + 7], reading zero at
// and past K.  vec: x and the column stride allow 16-byte loads.
__device__ __forceinline__ void q8_1_load8(const float *__restrict__ col, int64_t k, int64_t K, bool vec,
                                           float (&v)[8])
{
    if (vec && k + 8 <= K) {
        const float4 a = ld_cg_f4(col + k);
        const float4 b = ld_cg_f4(col + k + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (k + i < K) ? ld_cg_f32(col + k + i) : 0.0f;
    }
}

}  // namespace qmv
