/*
 * IEEE-754 binary16 <-> binary32 conversion, written from the format's
 * definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits;
 * exponent 0 encodes zero and subnormals of weight 2^-24, exponent 31 encodes
 * infinities and NaNs).  Test infrastructure for the oracle only.
 *
 * float -> half rounds to nearest, ties to even, and overflows to infinity,
 * which is the conversion the GGUF block fields (ggml_half) are stored with.
 */
#include <math.h>
#include <string.h>

#include "qmv_oracle.h"

/* Shift m right by s bits, rounding to nearest with ties to even. */
static uint32_t shift_rne(uint32_t m, int s)
{
    if (s <= 0) return m << (-s);
    if (s >= 32) return 0; /* m < 2^24, so m < half of 2^s: rounds to zero */
    uint32_t q = m >> s;
    uint32_t rem = m & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return q;
}

uint16_t oracle_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ef = (x >> 23) & 0xffu;
    uint32_t mf = x & 0x7fffffu;

    if (ef == 0xffu) {                       /* inf or NaN */
        if (mf == 0) return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | 0x7e00u | (mf >> 13)); /* quiet NaN */
    }
    if (ef == 0 && mf == 0) return sign;    /* signed zero */

    /* value = m * 2^E exactly, with m an integer < 2^24 */
    uint32_t m;
    int E;
    int p; /* floor(log2 |value|) for normal floats */
    if (ef == 0) { m = mf; E = -149; p = -127; /* below every half exponent */ }
    else { m = mf | 0x800000u; E = (int)ef - 150; p = (int)ef - 127; }

    /* half value = q * 2^Eh with q < 2048: Eh = p - 10 for normal halves,
     * Eh = -24 (the subnormal grid) below 2^-14. */
    int Eh = (p >= -14) ? p - 10 : -24;
    uint32_t q = shift_rne(m, Eh - E);
    if (q == 2048u) { q = 1024u; Eh += 1; }  /* rounding carried into the next binade */
    if (Eh + 25 >= 31) return (uint16_t)(sign | 0x7c00u); /* >= 2^16 after rounding: overflow */
    if (q >= 1024u) return (uint16_t)(sign | ((uint32_t)(Eh + 25) << 10) | (q - 1024u));
    return (uint16_t)(sign | q);             /* subnormal half (Eh == -24) */
}

float oracle_f16_to_f32(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(1024 + f), e - 25);
    return (float)(s ? -v : v);
}

void oracle_f32_to_f16_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}

void oracle_f16_to_f32_array(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(in[i]);
}
