// decode.cuh -- register-level unpacking of packed quant words into fp32.
//
// Integers become floats without a conversion instruction: an integer u
// placed in the mantissa of a float whose exponent makes bit p worth 1 reads
// as 2^(23-p) + u, and one subtraction of a constant removes the bias and the
// format's offset exactly (both operands lie in one binade, so the difference
// is exact).  One AND+OR (a single LOP3) per weight and one paired fp32 add
// per two weights give the exact integer value (q - offset) as fp32.
//
// Every function returns exact values: q - 8 for Q4_0, q for the int8
// formats, q - 32 for Q6_K.  The scales are applied by the caller per block.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace lean {

// magic exponents: bit p of the mantissa worth 1.0
__device__ __forceinline__ float mant_u(uint32_t bits_at_p, uint32_t magic) {
    return __uint_as_float(bits_at_p | magic);
}

constexpr uint32_t kMagic0 = 0x4B000000u;   // 2^23 : bit 0 worth 1
constexpr uint32_t kMagic4 = 0x49000000u;   // 2^19 : bit 4 worth 1
constexpr uint32_t kMagic6 = 0x48000000u;   // 2^17 : bit 6 worth 1
constexpr uint32_t kMagic8 = 0x47000000u;   // 2^15 : bit 8 worth 1
constexpr uint32_t kMagic12 = 0x45000000u;  // 2^11 : bit 12 worth 1
constexpr uint32_t kMagic14 = 0x44000000u;  // 2^9  : bit 14 worth 1
constexpr uint32_t kMagic16 = 0x43000000u;  // 2^7  : bit 16 worth 1

// ---- Q4_0: one word = 8 nibbles, element i in bits 4i..4i+3 -------------------
// out[j] = (q_{2j} - 8, q_{2j+1} - 8)
__device__ __forceinline__ void dec_q4_word(uint32_t w, float2 out[4]) {
    const uint32_t h = w >> 12;  // nibbles 5, 6, 7 -> bits 8, 12, 16
    const float f0 = mant_u(w & 0x0000000Fu, kMagic0);
    const float f1 = mant_u(w & 0x000000F0u, kMagic4);
    const float f2 = mant_u(w & 0x00000F00u, kMagic8);
    const float f3 = mant_u(w & 0x0000F000u, kMagic12);
    const float f4 = mant_u(w & 0x000F0000u, kMagic16);
    const float f5 = mant_u(h & 0x00000F00u, kMagic8);
    const float f6 = mant_u(h & 0x0000F000u, kMagic12);
    const float f7 = mant_u(h & 0x000F0000u, kMagic16);
    out[0] = __fadd2_rn(make_float2(f0, f1), make_float2(-8388616.0f, -524296.0f));
    out[1] = __fadd2_rn(make_float2(f2, f3), make_float2(-32776.0f, -2056.0f));
    out[2] = __fadd2_rn(make_float2(f4, f5), make_float2(-136.0f, -32776.0f));
    out[3] = __fadd2_rn(make_float2(f6, f7), make_float2(-2056.0f, -136.0f));
}

// ---- int8 (stored biased by 128): one word = 4 elements, byte i = element i ----
// out[0] = (q0, q1), out[1] = (q2, q3)
__device__ __forceinline__ void dec_i8_word(uint32_t w, float2 out[2]) {
    const uint32_t h = w >> 16;
    const float f0 = mant_u(w & 0x000000FFu, kMagic0);
    const float f1 = mant_u(w & 0x0000FF00u, kMagic8);
    const float f2 = mant_u(h & 0x000000FFu, kMagic0);
    const float f3 = mant_u(h & 0x0000FF00u, kMagic8);
    out[0] = __fadd2_rn(make_float2(f0, f1), make_float2(-8388736.0f, -32896.0f));
    out[1] = __fadd2_rn(make_float2(f2, f3), make_float2(-8388736.0f, -32896.0f));
}

// ---- Q6_K sub-block: 3 words = 16 six-bit values -------------------------------
// Element i < 15 sits in word i/5 at bit 6*(i%5); element 15 is split into the
// top two bits of the three words.  out[j] = (q_{2j} - 32, q_{2j+1} - 32).
__device__ __forceinline__ void dec_q6_group(uint32_t w0, uint32_t w1, uint32_t w2,
                                             float2 out[8]) {
    const uint32_t s0 = w0 >> 12, s1 = w1 >> 12, s2 = w2 >> 12;
    float f[16];
    f[0] = mant_u(w0 & 0x0000003Fu, kMagic0);
    f[1] = mant_u(w0 & 0x00000FC0u, kMagic6);
    f[2] = mant_u(w0 & 0x0003F000u, kMagic12);
    f[3] = mant_u(s0 & 0x00000FC0u, kMagic6);
    f[4] = mant_u(s0 & 0x0003F000u, kMagic12);
    f[5] = mant_u(w1 & 0x0000003Fu, kMagic0);
    f[6] = mant_u(w1 & 0x00000FC0u, kMagic6);
    f[7] = mant_u(w1 & 0x0003F000u, kMagic12);
    f[8] = mant_u(s1 & 0x00000FC0u, kMagic6);
    f[9] = mant_u(s1 & 0x0003F000u, kMagic12);
    f[10] = mant_u(w2 & 0x0000003Fu, kMagic0);
    f[11] = mant_u(w2 & 0x00000FC0u, kMagic6);
    f[12] = mant_u(w2 & 0x0003F000u, kMagic12);
    f[13] = mant_u(s2 & 0x00000FC0u, kMagic6);
    f[14] = mant_u(s2 & 0x0003F000u, kMagic12);
    // element 15 at bit 14: bits 14-15 <- w2[30:31], 16-17 <- w1[30:31], 18-19 <- w0[30:31]
    f[15] = __uint_as_float((s0 & 0x000C0000u) | ((w1 >> 14) & 0x00030000u) |
                            ((w2 >> 16) & 0x0000C000u) | kMagic14);
    const float c0 = -8388640.0f;  // 2^23 + 32
    const float c6 = -131104.0f;   // 2^17 + 32
    const float c12 = -2080.0f;    // 2^11 + 32
    const float c14 = -544.0f;     // 2^9 + 32
    out[0] = __fadd2_rn(make_float2(f[0], f[1]), make_float2(c0, c6));
    out[1] = __fadd2_rn(make_float2(f[2], f[3]), make_float2(c12, c6));
    out[2] = __fadd2_rn(make_float2(f[4], f[5]), make_float2(c12, c0));
    out[3] = __fadd2_rn(make_float2(f[6], f[7]), make_float2(c6, c12));
    out[4] = __fadd2_rn(make_float2(f[8], f[9]), make_float2(c6, c12));
    out[5] = __fadd2_rn(make_float2(f[10], f[11]), make_float2(c0, c6));
    out[6] = __fadd2_rn(make_float2(f[12], f[13]), make_float2(c12, c6));
    out[7] = __fadd2_rn(make_float2(f[14], f[15]), make_float2(c12, c14));
}

__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
}

}  // namespace lean
