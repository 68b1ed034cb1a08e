// layout.h -- geometry of the packed (device) layout, shared by the host
// packer and the kernels.  Internal to the library.
//
// Every format is stored as planes of 16-byte vectors.  Rows are taken in
// groups of 32 ("row groups", one row per lane of a warp); inside a plane the
// 16-byte vector j of all 32 rows of group g is stored contiguously:
//
//     plane offset of (row n, vector j) = ((g * per_row + j) * 32 + n % 32) * 16
//     with g = n / 32
//
// so a warp whose lane r reads row g*32+r touches 512 contiguous bytes.  This
// is the "oxinfer" crate page's quant plane + scale plane idea (Pre-quantized
// checkpoints) laid out for 32-wide warps.
//
//   quant plane  Q4_0   : K/32 vectors per row, one per block, 32 nibbles.
//                         Word t of a vector holds block elements 8t..8t+7,
//                         element 8t+i in bits 4i..4i+3.
//                Q8_0   : K/16 vectors per row, two per block, 16 int8 each,
//                         stored biased (q + 128 as an unsigned byte);
//                         byte i of vector j is element 16*(j%2) + i of block j/2.
//                I8_B64 : K/16 vectors per row, four per block, as Q8_0.
//                Q6_K   : 13 vectors per super-block (see q6k layout below).
//   scale plane  Q4_0, Q8_0, I8_B64: one fp16 per block, 8 per vector:
//                         vector v holds the scales of blocks 8v..8v+7.
//                Q6_K   : one fp16 d per super-block, 8 per vector.
// Padding rows (n >= N in the last group) and padding scale slots are zero.
// The scale plane starts at a 256-byte aligned offset after the quant plane.
#pragma once
#include <stdint.h>

namespace lean {

constexpr int kRowsPerGroup = 32;
constexpr int kVec = 16;  // bytes per vector

enum Fmt { Q4_0 = 0, Q8_0 = 1, I8_B64 = 2, Q6_K = 3 };

struct Geom {
    int64_t N, K;
    int64_t groups;      // ceil(N / 32)
    int64_t qvec;        // quant vectors per row
    int64_t svec;        // scale vectors per row
    int64_t q_bytes;     // size of the quant plane
    int64_t s_off;       // byte offset of the scale plane
    int64_t total;       // packed bytes
};

inline int block_elems(int fmt) {
    switch (fmt) {
    case Q4_0: return 32;
    case Q8_0: return 32;
    case I8_B64: return 64;
    case Q6_K: return 256;
    }
    return 0;
}

inline int64_t block_bytes(int fmt) {
    switch (fmt) {
    case Q4_0: return 18;
    case Q8_0: return 34;
    case I8_B64: return 66;
    case Q6_K: return 210;
    }
    return 0;
}

// quant vectors per block
inline int qvec_per_block(int fmt) {
    switch (fmt) {
    case Q4_0: return 1;
    case Q8_0: return 2;
    case I8_B64: return 4;
    case Q6_K: return 13;
    }
    return 0;
}

inline bool make_geom(int fmt, int64_t N, int64_t K, Geom *g) {
    int be = block_elems(fmt);
    if (be == 0 || N <= 0 || K <= 0 || K % be) return false;
    // keep every index of the kernels inside int32 per row and int64 overall
    if (K > (int64_t)1 << 24 || N > (int64_t)1 << 31) return false;
    int64_t blocks = K / be;
    g->N = N;
    g->K = K;
    g->groups = (N + kRowsPerGroup - 1) / kRowsPerGroup;
    g->qvec = blocks * qvec_per_block(fmt);
    g->svec = (blocks + 7) / 8;
    g->q_bytes = g->groups * g->qvec * kRowsPerGroup * kVec;
    g->s_off = (g->q_bytes + 255) / 256 * 256;
    g->total = g->s_off + g->groups * g->svec * kRowsPerGroup * kVec;
    return true;
}

// byte offset of vector j of row n inside a plane with per_row vectors per row
inline int64_t vec_offset(int64_t n, int64_t j, int64_t per_row) {
    return (((n / kRowsPerGroup) * per_row + j) * kRowsPerGroup + n % kRowsPerGroup) * kVec;
}

}  // namespace lean
