// decode.cuh -- register-level unpacking of packed quant words into fp32.
//
// Integers become floats without a conversion instruction: an integer u
// placed in the mantissa of a float whose exponent makes bit p worth 1 reads
// as 2^(23-p) + u, and one subtraction of a constant removes that bias and the
// format's offset exactly (both operands lie in one binade, so the difference
// is exact).  One LOP3 ((word & mask) | magic) per weight and one paired fp32
// add per two weights give the exact integer (q - offset) as fp32, which a
// paired fp32 FMA multiplies into the running sum.  The magic exponents come
// from kernel parameters so that each LOP3 keeps its mask as the immediate.
//
// Values: q - 8 for Q4_0, q for the int8 formats, q - 32 for Q6_K.  Scales are
// applied by the callers once per block (sub-block for Q6_K).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "layout.h"
#include "ptx.cuh"

namespace lean {

struct Magic {
    uint32_t m0, m4, m6, m8, m12, m14, m16;  // bit p of the mantissa worth 1.0
    uint32_t pad;
    // (bias + offset) pairs subtracted after the LOP3, as f32x2 bit patterns
    unsigned long long q4[4];  // Q4_0 element pairs (0,1) (2,3) (4,5) (6,7) of a word
    unsigned long long i8;     // int8 byte pairs (0,1) / (2,3)
    unsigned long long q6[8];  // Q6_K element pairs of a sub-block
};
inline unsigned long long f2_bits(float lo, float hi) {
    uint32_t a, b;
    memcpy(&a, &lo, 4);
    memcpy(&b, &hi, 4);
    return ((unsigned long long)b << 32) | a;
}
inline Magic make_magic() {
    // exponent field 150 - p: the float 2^(23-p) has mantissa bit p worth 1
    Magic m;
    m.m0 = 0x4B000000u; m.m4 = 0x49000000u; m.m6 = 0x48000000u; m.m8 = 0x47000000u;
    m.m12 = 0x45000000u; m.m14 = 0x44000000u; m.m16 = 0x43000000u; m.pad = 0;
    // Q4_0: bias 2^(23-p) plus the offset 8
    m.q4[0] = f2_bits(-8388616.0f, -524296.0f);  // p = 0, 4
    m.q4[1] = f2_bits(-32776.0f, -2056.0f);      // p = 8, 12
    m.q4[2] = f2_bits(-136.0f, -32776.0f);       // p = 16, 8
    m.q4[3] = f2_bits(-2056.0f, -136.0f);        // p = 12, 16
    m.i8 = f2_bits(-8388736.0f, -32896.0f);      // bias 2^23 / 2^15 plus 128
    const float c0 = -8388640.0f, c6 = -131104.0f, c12 = -2080.0f, c14 = -544.0f;  // + 32
    m.q6[0] = f2_bits(c0, c6);
    m.q6[1] = f2_bits(c12, c6);
    m.q6[2] = f2_bits(c12, c0);
    m.q6[3] = f2_bits(c6, c12);
    m.q6[4] = f2_bits(c6, c12);
    m.q6[5] = f2_bits(c0, c6);
    m.q6[6] = f2_bits(c12, c6);
    m.q6[7] = f2_bits(c12, c14);
    return m;
}

// Copy the constants into registers once per thread: the opaque moves keep
// the compiler from re-materialising them inside the streaming loops.
__device__ __forceinline__ uint32_t pin32(uint32_t v) {
    asm volatile("mov.b32 %0, %0;" : "+r"(v));
    return v;
}
__device__ __forceinline__ unsigned long long pin64(unsigned long long v) {
    asm volatile("mov.b64 %0, %0;" : "+l"(v));
    return v;
}
__device__ __forceinline__ Magic pin(const Magic &g) {
    Magic m;
    m.m0 = pin32(g.m0); m.m4 = pin32(g.m4); m.m6 = pin32(g.m6); m.m8 = pin32(g.m8);
    m.m12 = pin32(g.m12); m.m14 = pin32(g.m14); m.m16 = pin32(g.m16); m.pad = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m.q4[i] = pin64(g.q4[i]);
    m.i8 = pin64(g.i8);
#pragma unroll
    for (int i = 0; i < 8; ++i) m.q6[i] = pin64(g.q6[i]);
    return m;
}

// The same, for one format: only the constants its decoder uses are copied
// (the others stay zero and are never read), which saves about twenty
// registers in the Q4_0 and int8 kernels.
template <int FMT>
__device__ __forceinline__ Magic pin_fmt(const Magic &g) {
    Magic m = {};
    m.m0 = pin32(g.m0);  // every format (int8 sub-scales use it too)
    if (FMT == Q4_0) {
        m.m4 = pin32(g.m4); m.m8 = pin32(g.m8); m.m12 = pin32(g.m12); m.m16 = pin32(g.m16);
#pragma unroll
        for (int i = 0; i < 4; ++i) m.q4[i] = pin64(g.q4[i]);
    } else if (FMT == Q6_K) {
        m.m6 = pin32(g.m6); m.m12 = pin32(g.m12); m.m14 = pin32(g.m14);
#pragma unroll
        for (int i = 0; i < 8; ++i) m.q6[i] = pin64(g.q6[i]);
    } else {  // Q8_0, I8_B64
        m.m8 = pin32(g.m8);
        m.i8 = pin64(g.i8);
    }
    return m;
}

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// ---- Q4_0: one word = 8 nibbles, element i in bits 4i..4i+3 -------------------
// p[j] = (q_{2j} - 8, q_{2j+1} - 8)
__device__ __forceinline__ void q4_word(uint32_t w, const Magic &mg, f32x2 p[4]) {
    const uint32_t h = w >> 12;  // nibbles 5, 6, 7 -> bits 8, 12, 16
    p[0] = add2(pack2(as_f(and_or(w, 0x0000000Fu, mg.m0)), as_f(and_or(w, 0x000000F0u, mg.m4))),
                mg.q4[0]);
    p[1] = add2(pack2(as_f(and_or(w, 0x00000F00u, mg.m8)), as_f(and_or(w, 0x0000F000u, mg.m12))),
                mg.q4[1]);
    p[2] = add2(pack2(as_f(and_or(w, 0x000F0000u, mg.m16)), as_f(and_or(h, 0x00000F00u, mg.m8))),
                mg.q4[2]);
    p[3] = add2(pack2(as_f(and_or(h, 0x0000F000u, mg.m12)), as_f(and_or(h, 0x000F0000u, mg.m16))),
                mg.q4[3]);
}

// ---- int8 stored + 128: one word = 4 elements, byte i = element i ------------
// p[0] = (q0, q1), p[1] = (q2, q3)
__device__ __forceinline__ void i8_word(uint32_t w, const Magic &mg, f32x2 p[2]) {
    const uint32_t h = w >> 16;
    p[0] = add2(pack2(as_f(and_or(w, 0x000000FFu, mg.m0)), as_f(and_or(w, 0x0000FF00u, mg.m8))),
                mg.i8);
    p[1] = add2(pack2(as_f(and_or(h, 0x000000FFu, mg.m0)), as_f(and_or(h, 0x0000FF00u, mg.m8))),
                mg.i8);
}

// ---- Q6_K sub-block: 3 words = 16 six-bit values --------------------------------
// Element i < 15 sits in word i/5 at bit 6*(i%5); element 15 is split into the
// top two bits of the three words.  p[j] = (q_{2j} - 32, q_{2j+1} - 32).
__device__ __forceinline__ void q6_group(uint32_t w0, uint32_t w1, uint32_t w2, const Magic &mg,
                                         f32x2 p[8]) {
    const uint32_t s0 = w0 >> 12, s1 = w1 >> 12, s2 = w2 >> 12;
    // element 15 at bit 14: bits 14-15 <- w2[30:31], 16-17 <- w1[30:31], 18-19 <- w0[30:31]
    uint32_t e15 = and_or(s0, 0x000C0000u, mg.m14);
    e15 = and_or(w1 >> 14, 0x00030000u, e15);
    e15 = and_or(w2 >> 16, 0x0000C000u, e15);
    p[0] = add2(pack2(as_f(and_or(w0, 0x0000003Fu, mg.m0)), as_f(and_or(w0, 0x00000FC0u, mg.m6))),
                mg.q6[0]);
    p[1] = add2(pack2(as_f(and_or(w0, 0x0003F000u, mg.m12)), as_f(and_or(s0, 0x00000FC0u, mg.m6))),
                mg.q6[1]);
    p[2] = add2(pack2(as_f(and_or(s0, 0x0003F000u, mg.m12)), as_f(and_or(w1, 0x0000003Fu, mg.m0))),
                mg.q6[2]);
    p[3] = add2(pack2(as_f(and_or(w1, 0x00000FC0u, mg.m6)), as_f(and_or(w1, 0x0003F000u, mg.m12))),
                mg.q6[3]);
    p[4] = add2(pack2(as_f(and_or(s1, 0x00000FC0u, mg.m6)), as_f(and_or(s1, 0x0003F000u, mg.m12))),
                mg.q6[4]);
    p[5] = add2(pack2(as_f(and_or(w2, 0x0000003Fu, mg.m0)), as_f(and_or(w2, 0x00000FC0u, mg.m6))),
                mg.q6[5]);
    p[6] = add2(pack2(as_f(and_or(w2, 0x0003F000u, mg.m12)), as_f(and_or(s2, 0x00000FC0u, mg.m6))),
                mg.q6[6]);
    p[7] = add2(pack2(as_f(and_or(s2, 0x0003F000u, mg.m12)), as_f(e15)), mg.q6[7]);
}

// int8 sub-scale stored + 128, byte i of word w
__device__ __forceinline__ float i8_byte(uint32_t w, int i, const Magic &mg) {
    return as_f(and_or(w >> (8 * i), 0xFFu, mg.m0)) - 8388736.0f;
}

__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int t) {
    return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w;
}

// fp16 scale of block b (0..7) of a scale vector
__device__ __forceinline__ float scale_of(const uint4 &s, int b) {
    const uint32_t w = word_of(s, b >> 1);
    return h2f((b & 1) ? (w >> 16) : w);
}

}  // namespace lean
