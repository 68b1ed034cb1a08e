// layout.h -- geometry of the packed (device) layout, shared by the host
// packer and the kernels.  Internal to the library.
//
// Rows are taken in groups of 32 ("row groups", one row per lane of a warp).
// The unit of storage is a "vector": 16 bytes for each of the 32 rows of a
// group, 512 contiguous bytes in all, so that a warp whose lane r handles row
// g*32+r reads one vector with a single coalesced 512-byte access.
//
// Each row group is one contiguous stream of "steps".  A step covers 8 blocks
// along K (Q6_K: 8 super-blocks) and holds first their quant vectors, then one
// scale vector with the 8 fp16 scales of those blocks -- the "oxinfer" crate
// page's quant plane + scale plane (Pre-quantized checkpoints), interleaved
// per step so that a single contiguous copy brings a step's quants together
// with its scales.  The last step of a row may hold fewer than 8 blocks.
//
//   quant vectors per block (VPB) and their contents, per format:
//     Q4_0   1: word t holds block elements 8t..8t+7, element 8t+i in bits 4i..4i+3
//     Q8_0   2: vector j holds elements 16j..16j+15, one byte each, q + 128
//     I8_B64 4: as Q8_0
//     Q6_K  13: vectors 0..11 hold the 256 six-bit q as 16 sub-blocks of 3 words
//               (sub-block b: words 3b..3b+2 =: W0,W1,W2; local element i < 15
//               in word i/5 at bit 6*(i%5); element 15 split into W2[30:31]
//               (bits 0-1), W1[30:31] (bits 2-3), W0[30:31] (bits 4-5));
//               vector 12 holds the 16 int8 sub-scales, each + 128.
//   scale vector: fp16 scale d of block i of the step in halfword i (Q6_K: the
//               super-block's d); unused slots are zero.
// Padding rows (n >= N in the last group) are zero.
#pragma once
#include <stdint.h>

namespace lean {

constexpr int kRowsPerGroup = 32;
constexpr int kVec = 16;                       // bytes per row per vector
constexpr int kVecBytes = kVec * kRowsPerGroup;  // 512 bytes per vector
constexpr int kBlocksPerStep = 8;
// x of the M = 1 product as integer planes: bytes per 32-element block
// (a 32-byte header, then four 32-byte planes)
constexpr int kXqBlockBytes = 160;

enum Fmt { Q4_0 = 0, Q8_0 = 1, I8_B64 = 2, Q6_K = 3 };

// Device error word bit of a LEAN_DEBUG build's index check (debug.cuh).
constexpr unsigned kErrBounds = 32u;

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
inline int vecs_per_block(int fmt) {
    switch (fmt) {
    case Q4_0: return 1;
    case Q8_0: return 2;
    case I8_B64: return 4;
    case Q6_K: return 13;
    }
    return 0;
}

struct Geom {
    int64_t N, K;
    int64_t groups;      // ceil(N / 32)
    int64_t blocks;      // blocks per row
    int steps;           // steps per row group
    int last_blocks;     // blocks in the last step (1..8)
    int vpb;             // quant vectors per block
    int step_vecs;       // vectors of a full step (8 * vpb + 1)
    int64_t group_vecs;  // vectors per row group
    int64_t total;       // packed bytes
};

inline bool make_geom(int fmt, int64_t N, int64_t K, Geom *g) {
    const int be = block_elems(fmt);
    if (be == 0 || N <= 0 || K <= 0 || K % be) return false;
    // keep per-row indices inside int32 and the total inside int64
    if (K > ((int64_t)1 << 24) || N > ((int64_t)1 << 31)) return false;
    g->N = N;
    g->K = K;
    g->groups = (N + kRowsPerGroup - 1) / kRowsPerGroup;
    g->blocks = K / be;
    g->steps = (int)((g->blocks + kBlocksPerStep - 1) / kBlocksPerStep);
    g->last_blocks = (int)(g->blocks - (int64_t)(g->steps - 1) * kBlocksPerStep);
    g->vpb = vecs_per_block(fmt);
    g->step_vecs = kBlocksPerStep * g->vpb + 1;
    g->group_vecs = (int64_t)(g->steps - 1) * g->step_vecs + g->last_blocks * g->vpb + 1;
    g->total = g->groups * g->group_vecs * kVecBytes;
    return true;
}

// byte offset of vector v of step s of row n's group, for row n's 16 bytes
inline int64_t vec_offset(const Geom &g, int64_t n, int64_t s, int64_t v) {
    return ((n / kRowsPerGroup) * g.group_vecs + s * g.step_vecs + v) * kVecBytes +
           (n % kRowsPerGroup) * kVec;
}

// blocks held by step s
inline int step_blocks(const Geom &g, int64_t s) {
    return s == g.steps - 1 ? g.last_blocks : kBlocksPerStep;
}

}  // namespace lean
