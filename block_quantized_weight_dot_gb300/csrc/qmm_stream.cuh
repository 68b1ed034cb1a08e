// qmm_stream.cuh -- the decode GEMV (M = 1) as a TMA-fed streaming kernel.
//
// Decode streams every weight once ("oxinfer" crate page, Performance: decode
// is memory-bandwidth bound, each generated token streams all dense weights
// once), so this kernel is a pipeline whose only job is to keep HBM busy:
//
//  - work is cut into units: one chunk of K (BPC blocks of one step) for each
//    of 8 consecutive 32-row groups of one matrix.  A producer lane copies a
//    unit -- the 8 groups' quant vectors of the chunk with their scale vector,
//    and the chunk's x once for all 8 -- into a shared-memory slot with bulk
//    asynchronous copies (cp.async.bulk), counting the bytes on the slot's
//    mbarrier;
//  - with a workspace, the integer formats (Q4_0, Q8_0, I8_B64) take x as
//    integer planes written once per call by xprep_kernel, so that the dot
//    products run on dp4a: each 32-element block of x is scaled by a power of
//    two 2^sf chosen from its largest magnitude, rounded to integers X with
//    |X| < 2^31 and cut into four byte planes (X = X3*2^24 + X2*2^16 +
//    X1*2^8 + X0, X3 signed).  Every plane's dp4a sum starts at -128 * (sum of
//    the plane) and so ends as the exact integer sum of (q - offset) * plane
//    (the raw weight bytes carry offset 128: int8 stored + 128, and Q4_0
//    nibbles read as 16 * q with offset 16 * 8); the four sums combine exactly
//    in integers, round once to fp32 and scale by d * 2^-sf.
//    xprep_kernel checks every element: X is rounded on a grid 256 times
//    coarser (lowest plane all zero) when that moves no element by more than
//    2^-14 of itself, as for about 98 blocks in 100 of N(0,1) activations;
//    else on the fine grid; and a block that even the fine grid cannot hold to
//    2^-14 (a small value next to an outlier channel), or that holds an Inf or
//    NaN, is marked, and the consumers take the exact fp32 dot for it from x
//    itself.  The grid is decided per chunk (the x blocks of one unit), so the
//    consumers branch once per chunk: three planes when all blocks are coarse,
//    four otherwise, block by block only where a block is marked.  Each
//    product w*x therefore errs by at most 2^-14 of |w*x| plus fp32 rounding,
//    whatever x is.  Without a workspace, and for Q6_K (whose 6-bit fields do
//    not come out as bytes cheaply), x stays fp32 and the decode is the exact
//    mantissa-bias conversion with paired fp32 FMAs;
//  - consumer warp w owns group w of every unit: lane r decodes row r from
//    shared memory (conflict-free 16-byte reads, x as a broadcast read) and
//    keeps the group's running sum in a register across units, so no warp
//    ever waits for another; the slot is released on a second mbarrier;
//  - a CTA works on a contiguous range of the flattened (problem, group
//    block, chunk) list.  Without a workspace the ranges hold whole group
//    blocks; with one they hold equal numbers of units (stream-K) and a group
//    split between CTAs is completed by the last CTA to arrive, which adds the
//    parts in CTA order: results are deterministic either way;
//  - a batch with many more group blocks than CTAs (a whole decode step) is
//    instead handed out at run time, one whole group block at a time, largest
//    blocks first, from a counter in the workspace: CTAs that run faster
//    take more blocks, so they all finish within about one block of each
//    other (static ranges left the slowest SM several microseconds behind).
//    A group block never splits, so each row is still summed in one fixed
//    order;
//  - weights are requested before griddepcontrol.wait and x after it, so with
//    programmatic dependent launch the weight stream of one product overlaps
//    the tail of the previous kernel on the stream;
//  - every wait is bounded (globaltimer); on timeout the kernel records an
//    error code, lets its own copies land and returns.
//
// Several independent products (same format, M = 1) can share one launch: the
// list of problems is a kernel parameter and their units are concatenated.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "debug.cuh"
#include "decode.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace lean {

constexpr int kStreamWarps = 8;                          // consumer warps per CTA
constexpr int kMaxGroupsPerUnit = 16;                    // workspace slots per CTA side
constexpr int kStreamThreads = 32 * (kStreamWarps + 1);  // + one producer warp
constexpr uint64_t kWaitLimitNs = 2000000000ull;        // 2 s

enum StreamError : unsigned {
    kErrFullTimeout = 1u,   // a consumer waited too long for a slot
    kErrEmptyTimeout = 2u,  // the producer waited too long for a free slot
};

struct StreamProb {
    const uint8_t *W;
    const float *x;
    float *y;
    int N, K;
    int steps, last_blocks;  // steps per group, blocks in a group's last step
    int chunks;              // chunks per group
    int pad;
    int64_t group_vecs;      // vectors per row group
    int64_t groups;          // row groups
    int64_t gblocks;         // group blocks (8 groups each)
    int64_t unit0, gblock0;  // first global unit / group block of this problem
    int64_t group0;          // first global group
    int64_t xq0;             // byte offset of this problem's x planes in xq
};

template <int NP>
struct StreamArgs {
    int nprob;
    int ctas;
    int balanced;  // 1: equal units per CTA (needs part/cnt); 0: whole group blocks;
                   // 3: whole group blocks taken at run time (needs dyn)
    int pad;
    int64_t total_units, total_gblocks;
    float *part;    // [ctas][2][8][32] partial sums of groups split between CTAs
    unsigned *cnt;  // [total groups] arrival counters, all zero between calls
    unsigned *err;  // device error word (bits of StreamError)
    const uint8_t *xq;  // x as planes (xprep_kernel), or null: fp32 x
    unsigned *dyn;      // balanced == 3: [0] blocks taken after the first one of
                        // each CTA, [1] CTAs done taking; both zero between calls
    int nruns;          // balanced == 3: runs of group blocks, largest blocks first
    int pad2;
    Magic mg;
    StreamProb p[NP];
    // run r: problem run_prob[r] & 0xFFFF, its full group blocks (bit 16 clear)
    // or its last, partial one (set); its blocks are items run_item0[r] ..
    // run_item0[r + 1] - 1 of the hand-out order
    int32_t run_prob[2 * NP];
    int32_t run_item0[2 * NP + 1];
};
static_assert(sizeof(StreamArgs<256>) <= 32764, "kernel parameters fit the launch limit");

template <int FMT> struct StreamCfg;
// VPB: quant vectors per block; BPC: blocks per chunk; E: weights per block;
// S: slots in the ring; CPS: CTAs per SM.  A unit is 8 x BPC blocks of 32
// rows plus x: about 37 KB (Q6_K 58 KB).
// GPW: row groups per consumer warp (the warps share the unit's x reads).
#ifndef LEAN_Q4_BPC
#define LEAN_Q4_BPC 8
#endif
#ifndef LEAN_Q4_GPW
#define LEAN_Q4_GPW 1
#endif
#ifndef LEAN_Q4_S
#define LEAN_Q4_S 3
#endif
#ifndef LEAN_Q4_CPS
#define LEAN_Q4_CPS 2
#endif
template <> struct StreamCfg<Q4_0> {
    static constexpr int VPB = 1, BPC = LEAN_Q4_BPC, E = 32, S = LEAN_Q4_S, CPS = LEAN_Q4_CPS,
                         GPW = LEAN_Q4_GPW;
};
template <> struct StreamCfg<Q8_0> { static constexpr int VPB = 2, BPC = 4, E = 32, S = 2, CPS = 2, GPW = 1; };
template <> struct StreamCfg<I8_B64> { static constexpr int VPB = 4, BPC = 2, E = 64, S = 2, CPS = 2, GPW = 1; };
template <> struct StreamCfg<Q6_K> { static constexpr int VPB = 13, BPC = 1, E = 256, S = 3, CPS = 1, GPW = 1; };

// Ring depth and CTAs per SM of a kernel variant (PL: x as planes, dp4a; that
// variant needs no decode constants in registers, so more CTAs may fit).
#ifndef LEAN_Q4P_S
#define LEAN_Q4P_S 3
#endif
#ifndef LEAN_Q4P_CPS
#define LEAN_Q4P_CPS 2
#endif
template <int FMT, bool PL>
struct StreamRing {
    static constexpr int S = StreamCfg<FMT>::S, CPS = StreamCfg<FMT>::CPS;
};
template <>
struct StreamRing<Q4_0, true> {
    static constexpr int S = LEAN_Q4P_S, CPS = LEAN_Q4P_CPS;
};

// x as integer planes (dp4a) for the integer formats
template <int FMT> struct XPlanes { static constexpr bool on = FMT != Q6_K; };
// One 32-element block of x in plane form: a 32-byte header {init3, init2,
// init1, init0 (the scale in chunks of tier 0 or 3), scale, tier of the
// chunk, 0, 0} (scale = 2^-sf, 1/16 more for Q4_0; -1 marks a block that takes
// the exact fp32 dot), then planes 3 (the top digits), 2, 1 and 0, 32 bytes
// each.
constexpr int kXqBytes = kXqBlockBytes;
constexpr int kXqHeader = 32;
static_assert(kXqBytes == kXqHeader + 4 * 32, "header + four planes");

template <int FMT, bool PL = false>
struct StreamLayout {
    using C = StreamCfg<FMT>;
    static constexpr int S = StreamRing<FMT, PL>::S;
    static constexpr int CPSTEP = 8 / C::BPC;                          // chunks of a full step
    static constexpr int CHUNK_BYTES = (C::BPC * C::VPB + 1) * kVecBytes;  // one group's chunk
    static constexpr int XE = C::BPC * C::E;                           // x elements of a unit
    static constexpr int GPU = kStreamWarps * C::GPW;                  // row groups of a unit
    // x of a unit: fp32, or its planes (5 bytes per element)
    static constexpr int XBYTES = XE * 4 > XE / 32 * kXqBytes ? XE * 4 : XE / 32 * kXqBytes;
    static constexpr int SLOT_BYTES = GPU * CHUNK_BYTES + XBYTES;
    // shared memory: [full S][empty S][abort][info S][ring S*SLOT]; info:
    // which unit a slot holds when units are taken at run time
    static constexpr int OFF_FULL = 0;
    static constexpr int OFF_EMPTY = 8 * S;
    static constexpr int OFF_ABORT = 16 * S;
    static constexpr int OFF_INFO = (OFF_ABORT + 4 + 15) / 16 * 16;
    static constexpr int OFF_RING = (OFF_INFO + 16 * S + 127) / 128 * 128;
    static constexpr int SMEM = OFF_RING + S * SLOT_BYTES;
};

__device__ __forceinline__ int64_t i64min(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t i64max(int64_t a, int64_t b) { return a > b ? a : b; }

template <int NP>
__device__ __forceinline__ int find_prob_by_unit(const StreamArgs<NP> &a, int64_t u) {
    int lo = 0, hi = a.nprob - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.p[mid].unit0 <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}
template <int NP>
__device__ __forceinline__ int find_prob_by_gblock(const StreamArgs<NP> &a, int64_t gb) {
    int lo = 0, hi = a.nprob - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.p[mid].gblock0 <= gb) lo = mid; else hi = mid - 1;
    }
    return lo;
}
// first global unit of global group block gb (gb == total_gblocks gives total_units)
template <int NP>
__device__ __forceinline__ int64_t gblock_first_unit(const StreamArgs<NP> &a, int64_t gb) {
    if (gb >= a.total_gblocks) return a.total_units;
    const StreamProb &p = a.p[find_prob_by_gblock(a, gb)];
    return p.unit0 + (gb - p.gblock0) * p.chunks;
}
template <int NP>
__device__ __forceinline__ int64_t range_begin(const StreamArgs<NP> &a, int64_t i) {
    if (a.balanced) return a.total_units * i / a.ctas;
    return gblock_first_unit(a, a.total_gblocks * i / a.ctas);
}
// the CTA whose balanced range holds unit u
template <int NP>
__device__ __forceinline__ int64_t cta_of_unit(const StreamArgs<NP> &a, int64_t u) {
    int64_t i = u * a.ctas / a.total_units;
    while (i + 1 < a.ctas && a.total_units * (i + 1) / a.ctas <= u) ++i;
    while (i > 0 && a.total_units * i / a.ctas > u) --i;
    return i;
}

// Problem and group block of item k of the run-time hand-out order.
template <int NP>
__device__ __forceinline__ void item_gblock(const StreamArgs<NP> &a, int64_t k, int &pi,
                                            int64_t &gb) {
    int lo = 0, hi = a.nruns - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.run_item0[mid] <= k) lo = mid; else hi = mid - 1;
    }
    const int r = a.run_prob[lo];
    pi = r & 0xFFFF;
    gb = (r >> 16) ? a.p[pi].gblocks - 1 : k - a.run_item0[lo];
}
// the unit a slot holds (run-time hand-out); pi < 0: no more units
struct SlotInfo {
    int pi;
    int c;
    int64_t gb;
};

// Where a unit's chunk sits in its groups' streams.
struct ChunkPos {
    int s;     // step
    int sub;   // chunk inside the step
    int nblk;  // blocks of the step
    int nbc;   // blocks of the chunk
};
template <int FMT>
__device__ __forceinline__ ChunkPos chunk_pos(const StreamProb &p, int c) {
    using C = StreamCfg<FMT>;
    constexpr int CPSTEP = StreamLayout<FMT>::CPSTEP;
    ChunkPos q;
    q.s = c / CPSTEP;
    q.sub = c % CPSTEP;
    q.nblk = q.s == p.steps - 1 ? p.last_blocks : 8;
    q.nbc = min(C::BPC, q.nblk - q.sub * C::BPC);
    return q;
}

// ---- x as integer planes ------------------------------------------------------
// Byte of element l (0..31) of a block in its planes: Q4_0 words hold the
// even elements of a weight word (its low nibbles) then the odd ones (high
// nibbles); the int8 formats keep element order.
template <int FMT>
__device__ __forceinline__ int plane_pos(int l) {
    if (FMT == Q4_0) return 4 * (2 * (l >> 3) + (l & 1)) + ((l & 7) >> 1);
    return l;
}
// x blocks (of 32 elements) in one chunk of the stream kernel: xprep_kernel
// gives all x blocks of a chunk one grid tier, so that a consumer branches
// once per chunk.
template <int FMT>
constexpr int xq_chunk_blocks() { return StreamCfg<FMT>::BPC * StreamCfg<FMT>::E / 32; }

// One 32-element block of x rounded to integers (the warp works on one block;
// lane l holds element l in v).
//   The fine grid: t = v * 2^sf, sf = 30 - floor(log2(max |v|)), so the
//   block's largest |t| lies in [2^30, 2^31) and X = round(t) fits int32 (sf is
//   capped at 122 for blocks of tiny values: 2^-(sf+4) stays a normal float).
//   The coarse grid is 256 times wider (t / 256, |.| < 2^23).  t, t / 256 and
//   their rounding residues are exact in fp32.  An element is held precisely
//   enough when its residue is at most 2^-14 of itself.
//   tier 0: every element is, on the coarse grid: X = 256 * round(t / 256)
//           (clamped to 2^23 - 1 before the product), lowest byte zero;
//   tier 1: every element is on the fine grid: X = round(t);
//   tier 2: not even that (a small value next to an outlier channel), or an
//           Inf or NaN in the block: the consumers take the exact fp32 dot.
struct XBlock {
    int X;     // this lane's integer
    int sf;    // fine-grid exponent
    int tier;  // 0, 1, 2 (warp-uniform)
};
__device__ __forceinline__ XBlock x_block_quantize(float v) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7fffffffu);
    const int e = (int)(mx >> 23) - 127;  // floor(log2 max|v|); -127 for zero / subnormal
    XBlock r;
    r.sf = min(30 - e, 122);
    const float tf = v * __int_as_float((127 + r.sf) << 23);  // exact
    const float tc = tf * (1.f / 256.f);                      // exact
    const float rc = rintf(tc), rf = rintf(tf);
    // residues within 2^-14 of the element (true for t = 0, whose residue is 0)
    const bool coarse_ok = fabsf(tc - rc) * 16384.f <= fabsf(tc);
    const bool fine_ok = fabsf(tf - rf) * 16384.f <= fabsf(tf);
    if (mx >= 0x7f800000u) r.tier = 2;
    else if (__all_sync(0xffffffffu, coarse_ok)) r.tier = 0;
    else r.tier = __all_sync(0xffffffffu, fine_ok) ? 1 : 2;
    r.X = r.tier == 0 ? __float2int_rn(fminf(rc, 8388607.f)) * 256
          : r.tier == 1 ? __float2int_rn(rf) : 0;
    return r;
}
// x quantized to int8 (LEAN_FLAG_X_INT8), one block: s = max|v| / 127 and
// q = round(v / s), ties away from zero, both fp32 operations as the rule
// states (0 for a block of zeros); the codes go in the top plane (chunk tier
// 3: the consumers read that plane only) with scale s (1/16 more for Q4_0).
// A block holding an Inf or NaN gets a NaN scale.
template <int FMT>
__device__ __forceinline__ void x_block_store_int8(float v, uint8_t *dst, int lane) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7fffffffu);
    const float amax = __uint_as_float(mx);
    const float s = __fdiv_rn(amax, 127.f);
    int q = 0;
    if (mx != 0u && mx < 0x7f800000u)
        q = (int)fminf(fmaxf(roundf(__fdiv_rn(v, s)), -127.f), 127.f);
    dst[kXqHeader + plane_pos<FMT>(lane)] = (uint8_t)q;
    const int sq = __reduce_add_sync(0xffffffffu, q);
    if (lane == 0) {
        const float scale = mx >= 0x7f800000u ? __int_as_float(0x7fc00000)
                                              : (FMT == Q4_0 ? s * (1.f / 16.f) : s);
        reinterpret_cast<int4 *>(dst)[0] = make_int4(-128 * sq, 0, 0, __float_as_int(scale));
        reinterpret_cast<int4 *>(dst)[1] = make_int4(__float_as_int(scale), 3, 0, 0);
    }
}

// Writes the block's planes at dst: the bytes of X, X = X3*2^24 + X2*2^16 +
// X1*2^8 + X0 with X3 signed and the others in 0..255, each plane's header
// init -128 * (its byte sum), the block's scale and the chunk's tier `mode`.
template <int FMT>
__device__ __forceinline__ void x_block_store(const XBlock &xb, int mode, uint8_t *dst, int lane) {
    const int d0 = xb.X & 255, d1 = (xb.X >> 8) & 255, d2 = (xb.X >> 16) & 255, d3 = xb.X >> 24;
    const int pos = kXqHeader + plane_pos<FMT>(lane);
    dst[pos] = (uint8_t)d3;
    dst[pos + 32] = (uint8_t)d2;
    dst[pos + 64] = (uint8_t)d1;
    dst[pos + 96] = (uint8_t)d0;
    const int s3 = __reduce_add_sync(0xffffffffu, d3);
    const int s2 = __reduce_add_sync(0xffffffffu, d2);
    const int s1 = __reduce_add_sync(0xffffffffu, d1);
    const int s0 = __reduce_add_sync(0xffffffffu, d0);
    if (lane == 0) {
        // Q4_0's dp4a sums come out 16 times the integer sum (nibbles read in
        // place as 16 * q): its scale carries the 1/16
        const int sc = xb.sf + (FMT == Q4_0 ? 4 : 0);
        const float scale = xb.tier == 2 ? -1.f : __int_as_float((127 - sc) << 23);
        // chunks of tier 0 need no init of the lowest plane (all zero): its
        // slot carries the scale, times 256 (their sums come out as T / 256),
        // so that one load brings the whole header
        const int w = mode == 0 ? __float_as_int(scale * 256.f) : -128 * s0;
        reinterpret_cast<int4 *>(dst)[0] = make_int4(-128 * s3, -128 * s2, -128 * s1, w);
        reinterpret_cast<int4 *>(dst)[1] = make_int4(__float_as_int(scale), mode, 0, 0);
    }
}

// x of several problems as planes: blockIdx.y = problem; each warp converts
// kXprepBlocks consecutive x blocks (their loads issued first), the CTA's 8
// warps one run of whole chunks of the stream kernel; the blocks' tiers meet
// in shared memory to give each chunk its tier.  xq + p.xq0 receives the
// problem's K/32 plane blocks.
constexpr int kXprepBlocks = 2;
constexpr int kXprepCtaBlocks = 8 * kXprepBlocks;
struct XprepProb {
    const float *x;
    int64_t xq0;
    int nb;  // blocks of 32 elements
    int pad;
};
template <int NP>
struct XprepArgs {
    int nprob;
    int int8;  // 1: quantize x to int8 (LEAN_FLAG_X_INT8) instead of the exact planes
    uint8_t *xq;
    int64_t xq_bytes;  // bytes of the plane region
    unsigned *err;     // device error word (LEAN_DEBUG index checks)
    XprepProb p[NP];
};
template <int FMT, int NP>
__global__ void __launch_bounds__(256) xprep_kernel(const __grid_constant__ XprepArgs<NP> a) {
    constexpr int G = xq_chunk_blocks<FMT>();
    static_assert(kXprepCtaBlocks % G == 0, "a CTA converts whole chunks");
    __shared__ int tiers[kXprepCtaBlocks];
    pdl_launch_dependents();
    pdl_wait();  // x may come from the previous kernel on the stream
    const XprepProb &p = a.p[blockIdx.y];
    const int lane = (int)(threadIdx.x & 31), warp = (int)(threadIdx.x >> 5);
    const int cta0 = (int)blockIdx.x * kXprepCtaBlocks;
    const int b0 = cta0 + warp * kXprepBlocks;
    float v[kXprepBlocks];
#pragma unroll
    for (int u = 0; u < kXprepBlocks; ++u)
        v[u] = b0 + u < p.nb ? p.x[32 * (int64_t)(b0 + u) + lane] : 0.f;
    if (a.int8) {
#pragma unroll
        for (int u = 0; u < kXprepBlocks; ++u)
            if (b0 + u < p.nb && LEAN_SPAN(p.xq0 + (int64_t)(b0 + u) * kXqBytes, kXqBytes, a.xq_bytes, a.err))
                x_block_store_int8<FMT>(v[u], a.xq + p.xq0 + (int64_t)(b0 + u) * kXqBytes, lane);
        return;
    }
    XBlock xb[kXprepBlocks];
#pragma unroll
    for (int u = 0; u < kXprepBlocks; ++u) {
        xb[u] = x_block_quantize(v[u]);
        if (lane == 0) tiers[warp * kXprepBlocks + u] = b0 + u < p.nb ? xb[u].tier : 0;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kXprepBlocks; ++u) {
        if (b0 + u >= p.nb) break;
        const int c0 = (warp * kXprepBlocks + u) / G * G;  // the chunk's first block in the CTA
        int mode = 0;
#pragma unroll
        for (int j = 0; j < G; ++j) mode = max(mode, tiers[c0 + j]);
        if (LEAN_SPAN(p.xq0 + (int64_t)(b0 + u) * kXqBytes, kXqBytes, a.xq_bytes, a.err))
            x_block_store<FMT>(xb[u], mode, a.xq + p.xq0 + (int64_t)(b0 + u) * kXqBytes, lane);
    }
}

__device__ __forceinline__ uint32_t dp4a_us(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Integer sum over one x block of the weight bytes times x, in the block's
// plane order: w[0..7] hold four raw weight bytes each.  The even words start
// their chains at 0 and the odd ones at the header's -128 * (plane byte sum);
// LO16 scales the even chains by 16 (Q4_0: the even words hold the low
// nibbles, the odd ones the high nibbles in place, i.e. 16 * q).  TIER 1: the
// lowest plane may be nonzero, else (0) it is all zero and skipped; TIER 3:
// x as int8 codes, in the top plane alone.  Returns the block's exact sum of
// (weight byte - offset) * X (times 16 for Q4_0), rounded once to fp32.
template <bool LO16, int TIER>
__device__ __forceinline__ float plane_dot(const uint32_t (&w)[8], const int4 &h, const uint8_t *xq) {
    constexpr bool FINE = TIER == 1;
    constexpr int L = LO16 ? 16 : 1;
    const uint4 *pl = reinterpret_cast<const uint4 *>(xq + kXqHeader);
    const uint4 a3 = pl[0], b3 = pl[1];
    const uint32_t P3[8] = {a3.x, a3.y, a3.z, a3.w, b3.x, b3.y, b3.z, b3.w};
    if (TIER == 3) {  // x as int8 codes: the top plane alone
        uint32_t s3 = 0, t3 = (uint32_t)h.x;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            s3 = dp4a_us(w[i], P3[i], s3);
            t3 = dp4a_us(w[i + 1], P3[i + 1], t3);
        }
        return (float)((int)s3 * L + (int)t3);  // |.| < 2^20: exact
    }
    const uint4 a2 = pl[2], b2 = pl[3], a1 = pl[4], b1 = pl[5];
    const uint32_t P2[8] = {a2.x, a2.y, a2.z, a2.w, b2.x, b2.y, b2.z, b2.w};
    const uint32_t P1[8] = {a1.x, a1.y, a1.z, a1.w, b1.x, b1.y, b1.z, b1.w};
    uint32_t P0[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (FINE) {
        const uint4 a0 = pl[6], b0 = pl[7];
        P0[0] = a0.x; P0[1] = a0.y; P0[2] = a0.z; P0[3] = a0.w;
        P0[4] = b0.x; P0[5] = b0.y; P0[6] = b0.z; P0[7] = b0.w;
    }
    uint32_t s3 = 0, s2 = 0, s1 = 0, s0 = 0;
    uint32_t t3 = (uint32_t)h.x, t2 = (uint32_t)h.y, t1 = (uint32_t)h.z, t0 = (uint32_t)h.w;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        s3 = dp4a_us(w[i], P3[i], s3);
        s2 = dp4a_uu(w[i], P2[i], s2);
        s1 = dp4a_uu(w[i], P1[i], s1);
        t3 = dp4a_us(w[i + 1], P3[i + 1], t3);
        t2 = dp4a_uu(w[i + 1], P2[i + 1], t2);
        t1 = dp4a_uu(w[i + 1], P1[i + 1], t1);
        if (FINE) {
            s0 = dp4a_uu(w[i], P0[i], s0);
            t0 = dp4a_uu(w[i + 1], P0[i + 1], t0);
        }
    }
    const int u3 = (int)s3 * L + (int)t3, u2 = (int)s2 * L + (int)t2, u1 = (int)s1 * L + (int)t1;
    if (!FINE) {
        // the lowest plane is zero: T / 256 = (u3 * 256 + u2) * 256 + u1, with
        // |u1| < 2^21 exact in fp32 and no cancellation against the first
        // term once that one rounds (|u3 * 256 + u2| >= 2^24); one FMA rounds
        // the rest (the tier's scale carries the factor 256)
        return fmaf((float)(u3 * 256 + u2), 256.f, (float)u1);
    }
    const int u0 = (int)s0 * L + (int)t0;
    // |u| < 2^21, so both halves are exact in int32.  T = hi * 2^16 + lo is
    // rewritten as hi' * 2^16 + lo' with lo' = lo mod 2^16 in 0..65535 (the
    // carry moves into hi'): the FMA then rounds once, without cancellation,
    // and needs no 64-bit conversion (which would run on the FP64 pipe).
    const int hi = u3 * 256 + u2, lo = u1 * 256 + u0;
    const int hi2 = hi + (lo >> 16), lo2 = lo & 0xFFFF;
    return fmaf((float)hi2, 65536.f, (float)lo2);
}
// The exact fallback for a marked x block: sum over its 32 elements of the
// weight (d * (q - offset), exact in fp32) times x, in fp32, x read from
// global memory (16-byte aligned).  wa, wb: w[0..3], w[4..7] of plane_dot.
// Not inlined: it is the rare path, kept out of the unrolled block loops.
template <int FMT>
__device__ __noinline__ float exact_block_dot(uint4 wa, uint4 wb, float d, const float *xg) {
    const uint32_t w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    float r = 0.f;
#pragma unroll 1
    for (int l = 0; l < 32; l += 4) {
        const float4 xv = *reinterpret_cast<const float4 *>(xg + l);
        const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = l + j;
            int q;
            if (FMT == Q4_0) {  // element 8t+i: bits 4i..4i+3 of packed word t
                const int t = e >> 3, i = e & 7;
                const uint32_t word = (i & 1) ? (w[2 * t + 1] >> 4) : w[2 * t];
                q = (int)((word >> (8 * (i >> 1))) & 15u) - 8;
            } else {  // byte e, stored + 128
                q = (int)((w[e >> 2] >> (8 * (e & 3))) & 255u) - 128;
            }
            r = fmaf(d * (float)q, xs[j], r);
        }
    }
    return r;
}
// One x block times the weights' scale d: the planes' integer sum times
// d * 2^-sf (the two scales first, so that only a result beyond the fp32
// range can overflow).  MODE is the chunk's tier: 0 all blocks on the coarse
// grid, 1 some on the fine grid, 2 some marked for the exact fp32 dot (this
// block's own scale, -1 when marked, decides), 3 x quantized to int8 codes.
template <int FMT, int MODE>
__device__ __forceinline__ float x_block_dot(const uint32_t (&w)[8], float d, const uint8_t *xq,
                                             const float *xg) {
    const int4 h = *reinterpret_cast<const int4 *>(xq);
    // tiers 0 and 3 carry the scale in the header's last slot
    const float scale = (MODE == 0 || MODE == 3) ? __int_as_float(h.w)
                                                 : *reinterpret_cast<const float *>(xq + 16);
    if (MODE == 2 && scale < 0.f)
        return exact_block_dot<FMT>(make_uint4(w[0], w[1], w[2], w[3]),
                                    make_uint4(w[4], w[5], w[6], w[7]), d, xg);
    return (d * scale) * plane_dot<FMT == Q4_0, MODE == 2 ? 1 : MODE>(w, h, xq);
}
// One block with x as planes: this lane's row, block b of the step at ws, x
// planes of the chunk at xq, fp32 x of the chunk at xg.
template <int FMT, int MODE>
__device__ __forceinline__ float block_dot_q(const uint8_t *ws, const uint8_t *xq, const float *xg,
                                             int b, float d, int lane) {
    using C = StreamCfg<FMT>;
    if (FMT == Q4_0) {
        const uint4 v = *reinterpret_cast<const uint4 *>(ws + b * kVecBytes + lane * 16);
        uint32_t w[8];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t x = word_of(v, t);
            w[2 * t] = x & 0x0F0F0F0Fu;      // low nibbles: q
            w[2 * t + 1] = x & 0xF0F0F0F0u;  // high nibbles in place: 16 * q
        }
        return x_block_dot<FMT, MODE>(w, d, xq + b * kXqBytes, xg + b * 32);
    } else {  // Q8_0 (one x block) or I8_B64 (two): stored bytes q + 128
        float r = 0.f;
#pragma unroll
        for (int h = 0; h < C::E / 32; ++h) {
            const uint4 va = *reinterpret_cast<const uint4 *>(ws + (b * C::VPB + 2 * h) * kVecBytes + lane * 16);
            const uint4 vb = *reinterpret_cast<const uint4 *>(ws + (b * C::VPB + 2 * h + 1) * kVecBytes + lane * 16);
            const uint32_t w[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
            r += x_block_dot<FMT, MODE>(w, d, xq + (b * (C::E / 32) + h) * kXqBytes,
                                        xg + b * C::E + 32 * h);
        }
        return r;
    }
}
// The blocks of one chunk with x as planes, for one chunk tier MODE.
template <int FMT, int MODE>
__device__ __forceinline__ float planes_chunk(const uint8_t *ws, const uint8_t *xq, const float *xg,
                                              const uint4 &sv, int nbc, int sub, int lane) {
    using C = StreamCfg<FMT>;
    // Fully unrolled bodies only where they pay (tier 0, and full chunks of
    // tier 1): more copies of the block body overflow the instruction cache
    float acc = 0.f;
    if (MODE != 2 && nbc == C::BPC) {
#pragma unroll
        for (int i = 0; i < C::BPC; ++i)
            acc += block_dot_q<FMT, MODE>(ws, xq, xg, i, scale_of(sv, sub * C::BPC + i), lane);
    } else if (MODE == 0 || MODE == 3) {
#pragma unroll
        for (int i = 0; i < C::BPC; ++i)
            if (i < nbc)
                acc += block_dot_q<FMT, MODE>(ws, xq, xg, i, scale_of(sv, sub * C::BPC + i), lane);
    } else {
#pragma unroll 1
        for (int i = 0; i < nbc; ++i)
            acc += block_dot_q<FMT, MODE>(ws, xq, xg, i, scale_of(sv, sub * C::BPC + i), lane);
    }
    return acc;
}

// ---- per-format consumer work on one chunk held in shared memory ------------
// One block: this lane's row, block b of the step at ws, x of the block at xb.
template <int FMT>
__device__ __forceinline__ float block_dot(const uint8_t *ws, const float *xb, int b, float d,
                                           int lane, const Magic &mg) {
    using C = StreamCfg<FMT>;
    if (FMT == Q4_0) {
        const uint4 v = *reinterpret_cast<const uint4 *>(ws + b * kVecBytes + lane * 16);
        f32x2 s[4];  // one chain per word: four independent FMA chains
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            f32x2 p[4];
            q4_word(word_of(v, t), mg, p);
            const ulonglong2 xa = *reinterpret_cast<const ulonglong2 *>(xb + 8 * t);
            const ulonglong2 xc = *reinterpret_cast<const ulonglong2 *>(xb + 8 * t + 4);
            s[t] = mul2(p[0], xa.x);
            s[t] = fma2(p[1], xa.y, s[t]);
            s[t] = fma2(p[2], xc.x, s[t]);
            s[t] = fma2(p[3], xc.y, s[t]);
        }
        const float2 r = unpack2(add2(add2(s[0], s[1]), add2(s[2], s[3])));
        return d * (r.x + r.y);
    } else if (FMT == Q8_0 || FMT == I8_B64) {
        f32x2 s[4] = {0ull, 0ull, 0ull, 0ull};  // four independent FMA chains
#pragma unroll
        for (int j = 0; j < C::VPB; ++j) {
            const uint4 v =
                *reinterpret_cast<const uint4 *>(ws + (b * C::VPB + j) * kVecBytes + lane * 16);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                f32x2 p[2];
                i8_word(word_of(v, t), mg, p);
                const ulonglong2 xa = *reinterpret_cast<const ulonglong2 *>(xb + j * 16 + 4 * t);
                s[t] = fma2(p[0], xa.x, s[t]);
                s[t] = fma2(p[1], xa.y, s[t]);
            }
        }
        const float2 r = unpack2(add2(add2(s[0], s[1]), add2(s[2], s[3])));
        return d * (r.x + r.y);
    } else {  // Q6_K super-block: 16 sub-blocks with int8 sub-scales
        const uint8_t *sb = ws + b * C::VPB * kVecBytes + lane * 16;
        const uint4 scv = *reinterpret_cast<const uint4 *>(sb + 12 * kVecBytes);
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 4 sub-blocks per 3 vectors
            const uint4 v0 = *reinterpret_cast<const uint4 *>(sb + (3 * q + 0) * kVecBytes);
            const uint4 v1 = *reinterpret_cast<const uint4 *>(sb + (3 * q + 1) * kVecBytes);
            const uint4 v2 = *reinterpret_cast<const uint4 *>(sb + (3 * q + 2) * kVecBytes);
            const uint32_t w[12] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y,
                                    v1.z, v1.w, v2.x, v2.y, v2.z, v2.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int sub = 4 * q + u;
                f32x2 p[8];
                q6_group(w[3 * u], w[3 * u + 1], w[3 * u + 2], mg, p);
                f32x2 s0 = 0ull, s1 = 0ull;  // two independent FMA chains
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    const ulonglong2 xa =
                        *reinterpret_cast<const ulonglong2 *>(xb + sub * 16 + 4 * j);
                    const ulonglong2 xc =
                        *reinterpret_cast<const ulonglong2 *>(xb + sub * 16 + 4 * j + 4);
                    s0 = fma2(p[2 * j], xa.x, s0);
                    s0 = fma2(p[2 * j + 1], xa.y, s0);
                    s1 = fma2(p[2 * j + 2], xc.x, s1);
                    s1 = fma2(p[2 * j + 3], xc.y, s1);
                }
                const float sc = i8_byte(word_of(scv, sub >> 2), sub & 3, mg);
                const float2 r = unpack2(add2(s0, s1));
                acc = fmaf(d * sc, r.x + r.y, acc);
            }
        }
        return acc;
    }
}

// This lane's row: sum over the chunk's blocks of w * x.  ws: the group's
// chunk (nbc blocks of quant vectors, then the step's scale vector); xs: the
// chunk's x in shared memory (fp32, or its planes); xg: the chunk's fp32 x in
// global memory (read only for x blocks marked for the exact dot); sub: the
// chunk's place in its step (for the scale slots).
template <int FMT>
__device__ __forceinline__ float consume_chunk(const uint8_t *ws, const float *xs, const float *xg,
                                               int nbc, int sub, int lane, const Magic &mg,
                                               bool planes) {
    using C = StreamCfg<FMT>;
    const uint4 sv = *reinterpret_cast<const uint4 *>(ws + nbc * C::VPB * kVecBytes + lane * 16);
    float acc = 0.f;
    if (XPlanes<FMT>::on && planes) {
        const uint8_t *xq = reinterpret_cast<const uint8_t *>(xs);
        const int mode = *reinterpret_cast<const int *>(xq + 20);  // the chunk's tier
        if (mode == 0) return planes_chunk<FMT, 0>(ws, xq, xg, sv, nbc, sub, lane);
        if (mode == 1) return planes_chunk<FMT, 1>(ws, xq, xg, sv, nbc, sub, lane);
        if (mode == 3) return planes_chunk<FMT, 3>(ws, xq, xg, sv, nbc, sub, lane);
        return planes_chunk<FMT, 2>(ws, xq, xg, sv, nbc, sub, lane);
    }
    if (nbc == C::BPC) {
#pragma unroll
        for (int i = 0; i < C::BPC; ++i)
            acc += block_dot<FMT>(ws, xs + i * C::E, i, scale_of(sv, sub * C::BPC + i), lane, mg);
    } else {
#pragma unroll
        for (int i = 0; i < C::BPC; ++i)
            if (i < nbc)
                acc += block_dot<FMT>(ws, xs + i * C::E, i, scale_of(sv, sub * C::BPC + i), lane,
                                      mg);
    }
    return acc;
}

// Q4_0, R row groups sharing each x read: block b of every group's chunk.
template <int R>
__device__ __forceinline__ void q4_block_rows(const uint8_t *ws, int stride, const float *xb, int b,
                                              const float (&d)[R], int lane, const Magic &mg,
                                              float (&acc)[R]) {
    uint4 v[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        v[r] = *reinterpret_cast<const uint4 *>(ws + r * stride + b * kVecBytes + lane * 16);
    f32x2 s[R][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const ulonglong2 xa = *reinterpret_cast<const ulonglong2 *>(xb + 8 * t);
        const ulonglong2 xc = *reinterpret_cast<const ulonglong2 *>(xb + 8 * t + 4);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            f32x2 p[4];
            q4_word(word_of(v[r], t), mg, p);
            s[r][t] = mul2(p[0], xa.x);
            s[r][t] = fma2(p[1], xa.y, s[r][t]);
            s[r][t] = fma2(p[2], xc.x, s[r][t]);
            s[r][t] = fma2(p[3], xc.y, s[r][t]);
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float2 q = unpack2(add2(add2(s[r][0], s[r][1]), add2(s[r][2], s[r][3])));
        acc[r] = fmaf(d[r], q.x + q.y, acc[r]);
    }
}

// All of a warp's live groups (nlive of GPW) on one unit: groups sit
// kStreamWarps chunks apart in the slot.
template <int FMT>
__device__ __forceinline__ void consume_rows(const uint8_t *ws, const float *xs, const float *xg,
                                             int nbc, int sub, int nlive, int lane, const Magic &mg,
                                             bool planes, float (&acc)[StreamCfg<FMT>::GPW]) {
    using C = StreamCfg<FMT>;
    using L = StreamLayout<FMT>;
    constexpr int stride = kStreamWarps * L::CHUNK_BYTES;
    if (FMT == Q4_0 && C::GPW > 1 && nlive == C::GPW && !planes) {
        uint4 sv[C::GPW];
#pragma unroll
        for (int r = 0; r < C::GPW; ++r)
            sv[r] = *reinterpret_cast<const uint4 *>(ws + r * stride + nbc * C::VPB * kVecBytes +
                                                     lane * 16);
        if (nbc == C::BPC) {
#pragma unroll
            for (int i = 0; i < C::BPC; ++i) {
                float d[C::GPW];
#pragma unroll
                for (int r = 0; r < C::GPW; ++r) d[r] = scale_of(sv[r], sub * C::BPC + i);
                q4_block_rows<C::GPW>(ws, stride, xs + i * C::E, i, d, lane, mg, acc);
            }
        } else {
#pragma unroll
            for (int i = 0; i < C::BPC; ++i) {
                if (i < nbc) {
                    float d[C::GPW];
#pragma unroll
                    for (int r = 0; r < C::GPW; ++r) d[r] = scale_of(sv[r], sub * C::BPC + i);
                    q4_block_rows<C::GPW>(ws, stride, xs + i * C::E, i, d, lane, mg, acc);
                }
            }
        }
        return;
    }
#pragma unroll
    for (int r = 0; r < C::GPW; ++r)
        if (r < nlive)
            acc[r] += consume_chunk<FMT>(ws + r * stride, xs, xg, nbc, sub, lane, mg, planes);
}

template <int FMT, int NP, bool PL>
__global__ void __launch_bounds__(kStreamThreads, (StreamRing<FMT, PL>::CPS))
    qmm_stream_kernel(const __grid_constant__ StreamArgs<NP> a) {
    using C = StreamCfg<FMT>;
    using L = StreamLayout<FMT, PL>;
    constexpr int S = L::S;
    constexpr int SV = 8 * C::VPB + 1;  // vectors of a full step
    extern __shared__ __align__(128) uint8_t sbuf[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sbuf + L::OFF_FULL);
    uint64_t *empty = reinterpret_cast<uint64_t *>(sbuf + L::OFF_EMPTY);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbuf + L::OFF_ABORT);
    SlotInfo *info = reinterpret_cast<SlotInfo *>(sbuf + L::OFF_INFO);
    uint8_t *ring = sbuf + L::OFF_RING;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cta = blockIdx.x;
    const bool dyn = a.balanced == 3;  // whole group blocks taken at run time
    const int64_t beg = dyn ? 0 : range_begin(a, cta), end = dyn ? 0 : range_begin(a, cta + 1);
    const int64_t nunits = end - beg;

    // Let the next kernel on the stream start streaming its own weights.
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kStreamWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (!dyn && nunits <= 0) return;

    // cursor over the CTA's units: problem, group block inside it, chunk (with
    // run-time hand-out: the CTA's first group block is item blockIdx.x)
    int pi;
    int64_t gb;
    int c;
    if (dyn) {
        item_gblock(a, cta, pi, gb);
        c = 0;
    } else {
        pi = find_prob_by_unit(a, beg);
        const int64_t o = beg - a.p[pi].unit0;
        gb = o / a.p[pi].chunks;
        c = (int)(o % a.p[pi].chunks);
    }
    auto advance = [&]() {
        if (++c == a.p[pi].chunks) {
            c = 0;
            if (!dyn && ++gb == a.p[pi].gblocks) {
                gb = 0;
                ++pi;
            }
        }
    };

    if (warp == kStreamWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        constexpr bool planes = PL && XPlanes<FMT>::on;
        // Units whose weights go out before griddepcontrol.wait.  With x as
        // planes the kernel before is the plane kernel, whose x reads would
        // queue behind these requests: one unit each (measured on the decode
        // step: 38.9 us against 40.7 us with all S).  Otherwise the whole ring.
        constexpr int PRE = planes ? 1 : S;
        const uint8_t *xsrc[S];
        uint32_t xbytes[S];
        // arm slot j's barrier for the whole unit and copy the weights; returns
        // the x source (fp32 x or its planes) through xs / xb for a later copy
        auto issue_weights = [&](int sl, const uint8_t *&xs, uint32_t &xb) {
            uint8_t *base = ring + sl * L::SLOT_BYTES;
            const StreamProb &p = a.p[pi];
            const ChunkPos q = chunk_pos<FMT>(p, c);
            const int ng = (int)i64min(L::GPU, p.groups - gb * L::GPU);
            const uint32_t qbytes = q.nbc * C::VPB * kVecBytes;
            const int64_t e0 = (int64_t)(q.s * 8 + q.sub * C::BPC) * C::E;  // first x element
            if (planes) {
                xb = q.nbc * (C::E / 32) * kXqBytes;
                xs = a.xq + p.xq0 + (e0 / 32) * kXqBytes;
                if (!LEAN_SPAN((e0 / 32) * kXqBytes, xb, (int64_t)(p.K / 32) * kXqBytes, a.err)) xb = 0;
            } else {
                xb = q.nbc * C::E * 4;
                xs = reinterpret_cast<const uint8_t *>(p.x + e0);
                if (!LEAN_SPAN(e0 * 4, xb, (int64_t)p.K * 4, a.err)) xb = 0;
            }
            const bool merged = q.sub * C::BPC + q.nbc == q.nblk;  // chunk ends at the scale vector
            // (LEAN_DEBUG) only copies inside the packed matrix are made and counted
            const int64_t wbytes = p.groups * p.group_vecs * kVecBytes;
            bool w_in = true;
            for (int w = 0; w < ng; ++w) {
                const int64_t so = ((gb * L::GPU + w) * p.group_vecs + (int64_t)q.s * SV) * kVecBytes;
                w_in = w_in && LEAN_SPAN(so + q.sub * C::BPC * C::VPB * kVecBytes, qbytes, wbytes, a.err) &&
                       LEAN_SPAN(so + q.nblk * C::VPB * kVecBytes, kVecBytes, wbytes, a.err);
            }
            mbar_arrive_expect_tx(&full[sl], (w_in ? ng * (qbytes + kVecBytes) : 0u) + xb);
            for (int w = 0; w < ng && w_in; ++w) {
                const uint8_t *step =
                    p.W + ((gb * L::GPU + w) * p.group_vecs + (int64_t)q.s * SV) * kVecBytes;
                uint8_t *dst = base + w * L::CHUNK_BYTES;
                const uint8_t *qsrc = step + q.sub * C::BPC * C::VPB * kVecBytes;
                if (merged) {
                    bulk_g2s(dst, qsrc, qbytes + kVecBytes, &full[sl]);
                } else {
                    bulk_g2s(dst, qsrc, qbytes, &full[sl]);
                    bulk_g2s(dst + qbytes, step + q.nblk * C::VPB * kVecBytes, kVecBytes, &full[sl]);
                }
            }
            advance();
        };
        auto issue_x = [&](int sl, const uint8_t *xs, uint32_t xb) {
            if (xb) bulk_g2s(ring + sl * L::SLOT_BYTES + L::GPU * L::CHUNK_BYTES, xs, xb, &full[sl]);
        };
        // after a timeout: let the copies already issued (units j - S .. j - 1)
        // land before the CTA can exit
        auto drain = [&](int64_t j) {
            for (int64_t k = i64max(0, j - S); k < j; ++k)
                mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), kWaitLimitNs);
        };
        if (dyn) {
            // Units of the CTA's first group block go out before griddepcontrol.wait
            // (weights only, at most PRE of them); the counter is read after
            // it, once the previous kernel on the stream has finished with it.
            bool waited = false;
            int ndef = 0;  // x copies held back until the wait (slots 0 .. ndef - 1)
            auto wait_prev = [&]() {
                pdl_wait();
                waited = true;
                for (int k = 0; k < ndef; ++k) issue_x(k, xsrc[k], xbytes[k]);
            };
            // unit j >= S waits for the consumers of unit j - S (same slot)
            auto slot_free = [&](int64_t j) {
                return j < S || (!*abort_flag &&
                                 mbar_wait(&empty[j % S], (uint32_t)((j / S - 1) & 1), kWaitLimitNs));
            };
            int64_t j = 0;
            while (pi >= 0) {
                if (!slot_free(j)) {
                    atomicOr(a.err, kErrEmptyTimeout);
                    drain(j);
                    return;
                }
                const int sl = (int)(j % S);
                info[sl] = SlotInfo{pi, c, gb};
                const uint8_t *xs;
                uint32_t xb;
                issue_weights(sl, xs, xb);  // moves c on; c == 0: the block is done
                if (waited) {
                    issue_x(sl, xs, xb);
                } else {
                    xsrc[ndef] = xs;
                    xbytes[ndef] = xb;
                    ++ndef;
                }
                ++j;
                if (!waited && (j == PRE || c == 0)) wait_prev();
                if (c == 0) {  // take the next group block
                    const int64_t k = (int64_t)atomicAdd(&a.dyn[0], 1u) + a.ctas;
                    if (k < a.total_gblocks) item_gblock(a, k, pi, gb); else pi = -1;
                }
            }
            // no more units: the next slot gets an empty unit that stops the consumers
            if (!slot_free(j)) {
                atomicOr(a.err, kErrEmptyTimeout);
                drain(j);
                return;
            }
            info[j % S].pi = -1;
            mbar_arrive(&full[j % S]);
            // the last CTA to finish taking blocks leaves the counters zeroed
            if (atomicAdd(&a.dyn[1], 1u) == (unsigned)a.ctas - 1) {
                atomicExch(&a.dyn[0], 0u);
                atomicExch(&a.dyn[1], 0u);
            }
            return;
        }
        const int64_t nfill = i64min(S, nunits);
#pragma unroll
        for (int j = 0; j < PRE; ++j)
            if (j < nfill) issue_weights(j, xsrc[j], xbytes[j]);
        pdl_wait();  // x (or its planes) may be written by the previous kernel on the stream
#pragma unroll
        for (int j = 0; j < PRE; ++j)
            if (j < nfill) issue_x(j, xsrc[j], xbytes[j]);
#pragma unroll
        for (int j = PRE; j < S; ++j)
            if (j < nfill) {
                issue_weights(j, xsrc[j], xbytes[j]);
                issue_x(j, xsrc[j], xbytes[j]);
            }
        // slot and phase of unit j advance incrementally (no 64-bit division);
        // unit j >= S waits for the consumers of unit j - S (the same slot, the
        // previous phase)
        int sl = (int)(nfill % S);
        uint32_t ph = nfill == S ? 0u : 1u;  // phase parity of unit j - S on `empty`
        for (int64_t j = nfill; j < nunits; ++j) {
            if (*abort_flag || !mbar_wait(&empty[sl], ph, kWaitLimitNs)) {
                atomicOr(a.err, kErrEmptyTimeout);
                drain(j);
                return;
            }
            const uint8_t *xs;
            uint32_t xb;
            issue_weights(sl, xs, xb);
            issue_x(sl, xs, xb);
            if (++sl == S) {
                sl = 0;
                ph ^= 1u;
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Warp w owns groups w, w + 8, ... of each unit and keeps their sums in
    // registers until a group's last chunk in this CTA.  A group complete in
    // the CTA is stored; one shared with other CTAs (workspace mode) is
    // published and finished by the last CTA to arrive.
    constexpr bool planes = PL && XPlanes<FMT>::on;
    Magic mg;  // decode constants, in registers only for the fp32-x variant
    if constexpr (!planes) mg = pin_fmt<FMT>(a.mg);
    float acc[C::GPW];
#pragma unroll
    for (int r = 0; r < C::GPW; ++r) acc[r] = 0.f;
    int sl = 0;
    uint32_t ph = 0;  // phase parity of unit j on `full`
    for (int64_t j = 0; dyn || j < nunits; ++j) {
        if (!mbar_wait(&full[sl], ph, kWaitLimitNs)) {
            if (lane == 0) {
                atomicOr(a.err, kErrFullTimeout);
                *abort_flag = 1;
            }
            return;
        }
        if (dyn) {  // the producer says which unit the slot holds
            const SlotInfo inf = info[sl];
            if (inf.pi < 0) break;
            pi = inf.pi;
            c = inf.c;
            gb = inf.gb;
        }
        const StreamProb &p = a.p[pi];
        const int64_t g0 = gb * L::GPU + warp;  // this warp's first group in the problem
        const int nlive = (int)i64max(0, i64min(C::GPW, (p.groups - g0 + kStreamWarps - 1) / kStreamWarps));
        if (nlive > 0) {
            const ChunkPos q = chunk_pos<FMT>(p, c);
            const uint8_t *ws = ring + sl * L::SLOT_BYTES + warp * L::CHUNK_BYTES;
            const float *xs =
                reinterpret_cast<const float *>(ring + sl * L::SLOT_BYTES + L::GPU * L::CHUNK_BYTES);
            const float *xg = p.x + (int64_t)(q.s * 8 + q.sub * C::BPC) * C::E;
            consume_rows<FMT>(ws, xs, xg, q.nbc, q.sub, nlive, lane, mg, planes, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sl]);  // the slot is free; the sums are in registers
        const bool group_done = c == p.chunks - 1;
        if (group_done || j == nunits - 1) {
            const int64_t u0 = p.unit0 + gb * p.chunks;  // the groups' first and last unit
            const int64_t u1 = u0 + p.chunks - 1;
#pragma unroll
            for (int r = 0; r < C::GPW; ++r) {
                if (r >= nlive) break;
                const int64_t g = g0 + r * kStreamWarps;
                const int slot = warp + r * kStreamWarps;  // the group's place in the unit
                const int64_t n = g * kRowsPerGroup + lane;
                if (dyn || (u0 >= beg && u1 < end)) {  // the whole group is in this CTA
                    if (n < p.N) p.y[n] = acc[r];
                } else {
                    // split between CTAs: publish; the last CTA to arrive adds up
                    const int side = u0 < beg ? 0 : 1;
                    a.part[((cta * 2 + side) * kMaxGroupsPerUnit + slot) * 32 + lane] = acc[r];
                    __threadfence();
                    __syncwarp();
                    const int64_t gg = p.group0 + g;
                    unsigned arrived = 0;
                    if (lane == 0) arrived = atomicAdd(&a.cnt[gg], 1u);
                    arrived = __shfl_sync(0xffffffffu, arrived, 0);
                    const int64_t i0 = cta_of_unit(a, u0), i1 = cta_of_unit(a, u1);
                    if (arrived + 1 == (unsigned)(i1 - i0 + 1)) {
                        __threadfence();
                        float tot = 0.f;
                        for (int64_t i = i0; i <= i1; ++i) {
                            const int sd = (i == i0) ? 1 : 0;
                            tot += __ldcg(&a.part[((i * 2 + sd) * kMaxGroupsPerUnit + slot) * 32 + lane]);
                        }
                        if (n < p.N) p.y[n] = tot;
                        if (lane == 0) a.cnt[gg] = 0;  // ready for the next call
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < C::GPW; ++r) acc[r] = 0.f;
        }
        advance();
        if (++sl == S) {
            sl = 0;
            ph ^= 1u;
        }
    }
}

}  // namespace lean
