// pack.cpp -- host repacking between the canonical block layout and the
// packed device layout (layout.h).  Bits are moved, never rounded: every
// canonical byte is recoverable with lean_unpack_canonical.
//
// Formats (canonical side): "oxinfer" crate page, How it works (Q4_0: two
// nibbles per byte + f16 scale per 32; Q8: 32 weights per scale);
// "wgpu-llm" README, INT8 mode (block 64); "lean" README model table (Q6_K).
//
// Packed side, per format (one row n; vector = 16 bytes):
//   Q4_0   vector c = block c; word t bits 4i..4i+3 = q of block element 8t+i.
//   Q8_0   vectors 2c, 2c+1 = block c; byte i = (q of element 16*(j%2)+i) + 128.
//   I8_B64 vectors 4c..4c+3 = block c; byte i of vector 4c+j = element 16j+i,
//          biased by 128.
//   Q6_K   vectors 13s..13s+11 hold the 256 6-bit q of super-block s as 16
//          sub-blocks of 3 words (48 words); vector 13s+12 holds the 16
//          sub-scales, biased by 128.  Sub-block b (elements 16b..16b+15)
//          occupies words 3b, 3b+1, 3b+2 =: W0, W1, W2, with local element
//          i = 0..14 in word i/5 at bit 6*(i%5) and element 15 split into
//          2-bit pieces: bits 0-1 in W2[30:31], bits 2-3 in W1[30:31],
//          bits 4-5 in W0[30:31].
//   Scales: fp16 bits copied as they are; Q4_0/Q8_0/I8_B64 one per block,
//   Q6_K one d per super-block, 8 per scale vector.
#include <cstring>

#include "../../include/lean_qmatmul.h"
#include "layout.h"

using namespace lean;

namespace {

inline uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
inline void wr16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }
inline uint32_t rd32(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
inline void wr32(uint8_t *p, uint32_t v) {
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}

// Q6_K: 6-bit q of canonical element e of a super-block
inline int q6k_get(const uint8_t *blk, int e) {
    int h = e / 128, g = (e % 128) / 32, l = e % 32;
    int lo = (blk[64 * h + 32 * (g % 2) + l] >> (4 * (g / 2))) & 0xf;
    int hi = (blk[128 + 32 * h + l] >> (2 * g)) & 0x3;
    return lo | (hi << 4);
}
inline void q6k_put(uint8_t *blk, int e, int q) {
    int h = e / 128, g = (e % 128) / 32, l = e % 32;
    blk[64 * h + 32 * (g % 2) + l] |= (uint8_t)((q & 0xf) << (4 * (g / 2)));
    blk[128 + 32 * h + l] |= (uint8_t)(((q >> 4) & 0x3) << (2 * g));
}

// packed Q6_K sub-block: 16 six-bit values <-> 3 words
inline void q6_words_from(const int *q, uint32_t *w) {
    w[0] = w[1] = w[2] = 0;
    for (int i = 0; i < 15; ++i) w[i / 5] |= (uint32_t)q[i] << (6 * (i % 5));
    w[2] |= (uint32_t)(q[15] & 0x3) << 30;
    w[1] |= (uint32_t)((q[15] >> 2) & 0x3) << 30;
    w[0] |= (uint32_t)((q[15] >> 4) & 0x3) << 30;
}
inline void q6_words_to(const uint32_t *w, int *q) {
    for (int i = 0; i < 15; ++i) q[i] = (int)((w[i / 5] >> (6 * (i % 5))) & 0x3f);
    q[15] = (int)((w[2] >> 30) | (((w[1] >> 30) & 3) << 2) | (((w[0] >> 30) & 3) << 4));
}

template <bool TO_PACKED>
lean_status convert(int fmt, const uint8_t *canon, uint8_t *packed, int64_t N, int64_t K) {
    Geom g;
    if (!make_geom(fmt, N, K, &g)) return LEAN_ERR_SHAPE;
    const int be = block_elems(fmt);
    const int64_t bb = block_bytes(fmt);
    const int64_t nblk = K / be;
    if (TO_PACKED) std::memset(packed, 0, (size_t)g.total);
    uint8_t *qp = packed;
    uint8_t *sp = packed + g.s_off;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < nblk; ++c) {
            const int64_t coff = (n * nblk + c) * bb;
            // scale slot: blocks (Q4_0/Q8_0/I8) or super-blocks (Q6_K), 8 per vector
            uint8_t *sv = sp + vec_offset(n, c / 8, g.svec) + 2 * (c % 8);
            if (fmt == Q4_0) {
                uint8_t *v = qp + vec_offset(n, c, g.qvec);
                if (TO_PACKED) {
                    const uint8_t *b = canon + coff;
                    wr16(sv, rd16(b));
                    for (int t = 0; t < 4; ++t) {
                        uint32_t w = 0;
                        for (int i = 0; i < 8; ++i) {
                            int e = 8 * t + i;
                            int q = e < 16 ? (b[2 + e] & 0xf) : (b[2 + e - 16] >> 4);
                            w |= (uint32_t)q << (4 * i);
                        }
                        wr32(v + 4 * t, w);
                    }
                } else {
                    uint8_t *b = const_cast<uint8_t *>(canon) + coff;
                    wr16(b, rd16(sv));
                    std::memset(b + 2, 0, 16);
                    for (int t = 0; t < 4; ++t) {
                        uint32_t w = rd32(v + 4 * t);
                        for (int i = 0; i < 8; ++i) {
                            int e = 8 * t + i, q = (w >> (4 * i)) & 0xf;
                            if (e < 16) b[2 + e] |= (uint8_t)q;
                            else b[2 + e - 16] |= (uint8_t)(q << 4);
                        }
                    }
                }
            } else if (fmt == Q8_0 || fmt == I8_B64) {
                const int nv = be / 16;  // vectors per block
                if (TO_PACKED) {
                    const uint8_t *b = canon + coff;
                    wr16(sv, rd16(b));
                    for (int j = 0; j < nv; ++j) {
                        uint8_t *v = qp + vec_offset(n, c * nv + j, g.qvec);
                        for (int i = 0; i < 16; ++i) v[i] = (uint8_t)(b[2 + 16 * j + i] ^ 0x80);
                    }
                } else {
                    uint8_t *b = const_cast<uint8_t *>(canon) + coff;
                    wr16(b, rd16(sv));
                    for (int j = 0; j < nv; ++j) {
                        const uint8_t *v = qp + vec_offset(n, c * nv + j, g.qvec);
                        for (int i = 0; i < 16; ++i) b[2 + 16 * j + i] = (uint8_t)(v[i] ^ 0x80);
                    }
                }
            } else {  // Q6_K
                uint8_t words[13 * 16];
                if (TO_PACKED) {
                    const uint8_t *b = canon + coff;
                    wr16(sv, rd16(b + 208));
                    for (int s = 0; s < 16; ++s) {
                        int q[16];
                        uint32_t w[3];
                        for (int i = 0; i < 16; ++i) q[i] = q6k_get(b, 16 * s + i);
                        q6_words_from(q, w);
                        for (int k = 0; k < 3; ++k) wr32(words + 4 * (3 * s + k), w[k]);
                        words[192 + s] = (uint8_t)(b[192 + s] ^ 0x80);
                    }
                    for (int j = 0; j < 13; ++j)
                        std::memcpy(qp + vec_offset(n, c * 13 + j, g.qvec), words + 16 * j, 16);
                } else {
                    uint8_t *b = const_cast<uint8_t *>(canon) + coff;
                    std::memset(b, 0, 210);
                    wr16(b + 208, rd16(sv));
                    for (int j = 0; j < 13; ++j)
                        std::memcpy(words + 16 * j, qp + vec_offset(n, c * 13 + j, g.qvec), 16);
                    for (int s = 0; s < 16; ++s) {
                        int q[16];
                        uint32_t w[3];
                        for (int k = 0; k < 3; ++k) w[k] = rd32(words + 4 * (3 * s + k));
                        q6_words_to(w, q);
                        for (int i = 0; i < 16; ++i) q6k_put(b, 16 * s + i, q[i]);
                        b[192 + s] = (uint8_t)(words[192 + s] ^ 0x80);
                    }
                }
            }
        }
    }
    return LEAN_OK;
}

}  // namespace

extern "C" {

int lean_block_elems(int fmt) { return block_elems(fmt); }

int64_t lean_block_bytes(int fmt) { return block_bytes(fmt); }

int64_t lean_canonical_bytes(int fmt, int64_t N, int64_t K) {
    Geom g;
    if (!make_geom(fmt, N, K, &g)) return -1;
    return N * (K / block_elems(fmt)) * block_bytes(fmt);
}

int64_t lean_packed_bytes(int fmt, int64_t N, int64_t K) {
    Geom g;
    if (!make_geom(fmt, N, K, &g)) return -1;
    return g.total;
}

lean_status lean_pack(int fmt, const void *canon_host, void *packed_host, int64_t N, int64_t K) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    if (!canon_host || !packed_host) return LEAN_ERR_NULL;
    return convert<true>(fmt, (const uint8_t *)canon_host, (uint8_t *)packed_host, N, K);
}

lean_status lean_unpack_canonical(int fmt, const void *packed_host, void *canon_host, int64_t N,
                                  int64_t K) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    if (!canon_host || !packed_host) return LEAN_ERR_NULL;
    return convert<false>(fmt, (const uint8_t *)canon_host, (uint8_t *)packed_host, N, K);
}

const char *lean_status_str(int status) {
    switch (status) {
    case LEAN_OK: return "ok";
    case LEAN_ERR_FORMAT: return "unknown weight format";
    case LEAN_ERR_SHAPE: return "bad shape (N, K, M <= 0, K not a multiple of the block, or too large)";
    case LEAN_ERR_NULL: return "null pointer";
    case LEAN_ERR_ALIGN: return "misaligned pointer";
    case LEAN_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

}  // extern "C"
