// pack.cpp -- host repacking between the canonical block layout and the
// packed device layout (layout.h).  Bits are moved, never rounded: every
// canonical byte is recoverable with lean_unpack_canonical.
//
// Formats (canonical side): "oxinfer" crate page, How it works (Q4_0: two
// nibbles per byte + f16 scale per 32; Q8: 32 weights per scale);
// "wgpu-llm" README, INT8 mode (block 64); "lean" README model table (Q6_K).
//
// Packed side: see layout.h (row groups of 32, steps of 8 blocks, quant
// vectors then one scale vector per step).  Scales are fp16 bits copied as
// they are; int8 values and Q6_K sub-scales are stored biased by 128.
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
    const int64_t bb = block_bytes(fmt);
    const int64_t nblk = g.blocks;
    const int vpb = g.vpb;
    if (TO_PACKED) std::memset(packed, 0, (size_t)g.total);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < nblk; ++c) {
            const int64_t coff = (n * nblk + c) * bb;
            const int64_t s = c / kBlocksPerStep;
            const int i = (int)(c % kBlocksPerStep);
            // the step's scale vector follows its quant vectors; halfword i is block i's d
            uint8_t *sv = packed + vec_offset(g, n, s, (int64_t)step_blocks(g, s) * vpb) + 2 * i;
            auto qv = [&](int j) { return packed + vec_offset(g, n, s, (int64_t)i * vpb + j); };
            if (fmt == Q4_0) {
                uint8_t *v = qv(0);
                if (TO_PACKED) {
                    const uint8_t *b = canon + coff;
                    wr16(sv, rd16(b));
                    for (int t = 0; t < 4; ++t) {
                        uint32_t w = 0;
                        for (int k = 0; k < 8; ++k) {
                            int e = 8 * t + k;
                            int q = e < 16 ? (b[2 + e] & 0xf) : (b[2 + e - 16] >> 4);
                            w |= (uint32_t)q << (4 * k);
                        }
                        wr32(v + 4 * t, w);
                    }
                } else {
                    uint8_t *b = const_cast<uint8_t *>(canon) + coff;
                    wr16(b, rd16(sv));
                    std::memset(b + 2, 0, 16);
                    for (int t = 0; t < 4; ++t) {
                        uint32_t w = rd32(v + 4 * t);
                        for (int k = 0; k < 8; ++k) {
                            int e = 8 * t + k, q = (w >> (4 * k)) & 0xf;
                            if (e < 16) b[2 + e] |= (uint8_t)q;
                            else b[2 + e - 16] |= (uint8_t)(q << 4);
                        }
                    }
                }
            } else if (fmt == Q8_0 || fmt == I8_B64) {
                if (TO_PACKED) {
                    const uint8_t *b = canon + coff;
                    wr16(sv, rd16(b));
                    for (int j = 0; j < vpb; ++j) {
                        uint8_t *v = qv(j);
                        for (int k = 0; k < 16; ++k) v[k] = (uint8_t)(b[2 + 16 * j + k] ^ 0x80);
                    }
                } else {
                    uint8_t *b = const_cast<uint8_t *>(canon) + coff;
                    wr16(b, rd16(sv));
                    for (int j = 0; j < vpb; ++j) {
                        const uint8_t *v = qv(j);
                        for (int k = 0; k < 16; ++k) b[2 + 16 * j + k] = (uint8_t)(v[k] ^ 0x80);
                    }
                }
            } else {  // Q6_K
                uint8_t words[13 * 16];
                if (TO_PACKED) {
                    const uint8_t *b = canon + coff;
                    wr16(sv, rd16(b + 208));
                    for (int sb = 0; sb < 16; ++sb) {
                        int q[16];
                        uint32_t w[3];
                        for (int k = 0; k < 16; ++k) q[k] = q6k_get(b, 16 * sb + k);
                        q6_words_from(q, w);
                        for (int k = 0; k < 3; ++k) wr32(words + 4 * (3 * sb + k), w[k]);
                        words[192 + sb] = (uint8_t)(b[192 + sb] ^ 0x80);
                    }
                    for (int j = 0; j < 13; ++j) std::memcpy(qv(j), words + 16 * j, 16);
                } else {
                    uint8_t *b = const_cast<uint8_t *>(canon) + coff;
                    std::memset(b, 0, 210);
                    wr16(b + 208, rd16(sv));
                    for (int j = 0; j < 13; ++j) std::memcpy(words + 16 * j, qv(j), 16);
                    for (int sb = 0; sb < 16; ++sb) {
                        int q[16];
                        uint32_t w[3];
                        for (int k = 0; k < 3; ++k) w[k] = rd32(words + 4 * (3 * sb + k));
                        q6_words_to(w, q);
                        for (int k = 0; k < 16; ++k) q6k_put(b, 16 * sb + k, q[k]);
                        b[192 + sb] = (uint8_t)(words[192 + sb] ^ 0x80);
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
    case LEAN_ERR_KERNEL_BOUNDS: return "a kernel met an index outside its buffers (LEAN_DEBUG build)";
    case LEAN_ERR_DEVICE: return "a kernel reported an error in the device error word";
    }
    return "unknown status";
}

}  // extern "C"
