// Device-side NVFP4 encoders shared by the weight quantiser and the prefill
// activation quantiser.  Both round to nearest, ties to even, and saturate.
#pragma once
#include "ft_internal.cuh"

namespace ft {

struct RecordOffsets {
    size_t gu_codes, gu_scales, d_codes, d_scales, s_gu, s_d;
};

// Unsigned E4M3 (bias 7, max 448, no infinities) of a finite v >= 0.
__device__ __forceinline__ uint8_t e4m3_encode_rne(float v) {
    if (!(v > 0.f)) return 0;
    if (v >= 448.f) return 0x7E;
    const uint32_t b = __float_as_uint(v);
    const int e = (int)(b >> 23) - 127;
    if (e < -6) {
        // subnormal grid m * 2^-9, m = 0..8 (m = 8 is the smallest normal, code 0x08)
        return (uint8_t)(int)rintf(v * 512.0f);
    }
    const uint32_t mant = b & 0x7FFFFFu;
    uint32_t code = ((uint32_t)(e + 7) << 3) | (mant >> 20);
    const uint32_t rem = mant & 0xFFFFFu;
    if (rem > 0x80000u || (rem == 0x80000u && (code & 1u))) ++code;   // carries into the exponent
    return (uint8_t)(code > 0x7Eu ? 0x7Eu : code);
}

// Value of an unsigned E4M3 byte (exact in fp32).
__device__ __forceinline__ float e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 0) return (float)m * (1.0f / 512.0f);
    return __uint_as_float((uint32_t)(e - 7 + 127) << 23 | (uint32_t)m << 20);
}

// E2M1 code of an fp32 value, RNE, saturating at +-6; zero magnitudes are +0.
// Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; the ties .25, 1.25, 2.5, 5 fall to the
// even code below them and .75, 1.75, 3.5 rise to the even code above.
__device__ __forceinline__ uint8_t e2m1_encode_rne(float v) {
    const float a = fabsf(v);
    const uint32_t mag = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) +
                         (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
    return (uint8_t)(mag | ((v < 0.f && mag) ? 8u : 0u));
}

// Activation quantiser of one 16-element block (unit tensor scale), fp32 IEEE
// steps: s = E4M3_RNE(amax / 6), code = E2M1_RNE_sat(v / s); s = 0 gives zeros.
// Codes of elements 0..7 go to lo (element j at bits 4j), 8..15 to hi.
__device__ __forceinline__ uint8_t quant_block16(const float (&v)[16], uint32_t& lo, uint32_t& hi) {
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
    const uint8_t sc = e4m3_encode_rne(__fdiv_rn(amax, 6.0f));
    const float s = e4m3_value(sc);
    lo = 0;
    hi = 0;
    if (s != 0.f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            lo |= (uint32_t)e2m1_encode_rne(__fdiv_rn(v[j], s)) << (4 * j);
            hi |= (uint32_t)e2m1_encode_rne(__fdiv_rn(v[8 + j], s)) << (4 * j);
        }
    }
    return sc;
}

}  // namespace ft
