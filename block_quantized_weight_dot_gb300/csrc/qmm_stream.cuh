// qmm_stream.cuh -- the decode GEMV (M = 1) as a TMA-fed streaming kernel.
//
// Decode streams every weight once ("oxinfer" crate page, Performance: decode
// is memory-bandwidth bound, each generated token streams all dense weights
// once), so this kernel is a pipeline whose only job is to keep HBM busy:
//
//  - one producer lane per CTA copies whole steps (8 blocks of one 32-row
//    group: their quant vectors and scale vector, contiguous in the packed
//    layout) plus the matching slice of x into a ring of shared-memory slots
//    with bulk asynchronous copies (cp.async.bulk, completion counted in bytes
//    on an mbarrier per slot);
//  - eight consumer warps decode the slot from shared memory (lane r owns row
//    r of the group: conflict-free 16-byte reads; x is a broadcast read) and
//    accumulate in fp32, then release the slot on a second mbarrier;
//  - a CTA works on a contiguous range of the flattened (problem, row group,
//    step) list.  Without a workspace the ranges are whole row groups; with a
//    workspace they are equal numbers of steps (stream-K), and a group split
//    between CTAs is completed by the last CTA to arrive, which adds the
//    parts in CTA order: results are deterministic either way;
//  - weights are requested before griddepcontrol.wait, x after it, so with
//    programmatic dependent launch the weight stream of one product overlaps
//    the tail of the previous kernel on the stream;
//  - every wait is bounded (globaltimer); on timeout the kernel records an
//    error code, lets its own copies land and returns.
//
// Several independent products (same format, M = 1) can share one launch: the
// list of problems is a kernel parameter, and their steps are concatenated.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "decode.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace lean {

constexpr int kStreamWarps = 8;                          // consumer warps per CTA
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
    int64_t group_vecs;      // vectors per row group
    int64_t groups;          // row groups
    int64_t step0, group0;   // first global step / group of this problem
};

template <int NP>
struct StreamArgs {
    int nprob;
    int ctas;
    int balanced;  // 1: equal steps per CTA (needs part/cnt); 0: whole groups per CTA
    int64_t total_steps, total_groups;
    float *part;    // [ctas][2][32] partial sums of groups split between CTAs
    unsigned *cnt;  // [total_groups] arrival counters, all zero between calls
    unsigned *err;  // device error word (bits of StreamError)
    Magic mg;
    StreamProb p[NP];
};

template <int FMT> struct StreamCfg;
// VPB: quant vectors per block; SE: x elements per step; KS: steps per slot;
// S: slots in the ring; CPS: CTAs per SM.  Each consumer warp handles BPW
// blocks of one step per slot (128 or 256 weights per lane); an SM holds
// about 90-190 KB of ring in all.
template <> struct StreamCfg<Q4_0> { static constexpr int VPB = 1, SE = 256, KS = 8, S = 2, CPS = 2; };
template <> struct StreamCfg<Q8_0> { static constexpr int VPB = 2, SE = 256, KS = 4, S = 2, CPS = 2; };
template <> struct StreamCfg<I8_B64> { static constexpr int VPB = 4, SE = 512, KS = 2, S = 2, CPS = 2; };
template <> struct StreamCfg<Q6_K> { static constexpr int VPB = 13, SE = 2048, KS = 1, S = 3, CPS = 1; };

template <int FMT>
struct StreamLayout {
    using C = StreamCfg<FMT>;
    static constexpr int STEP_WBYTES = (8 * C::VPB + 1) * kVecBytes;
    static constexpr int STEP_XBYTES = C::SE * 4;
    static constexpr int STEP_BYTES = STEP_WBYTES + STEP_XBYTES;
    static constexpr int SLOT_BYTES = C::KS * STEP_BYTES;
    static constexpr int WPS = kStreamWarps / C::KS;  // warps per step
    static constexpr int BPW = 8 / WPS;               // blocks per warp
    // shared memory: [full S][empty S][meta S*KS][stage 2*W*32][carry 2*32][abort][ring S*SLOT]
    static constexpr int OFF_FULL = 0;
    static constexpr int OFF_EMPTY = 8 * C::S;
    static constexpr int OFF_META = 16 * C::S;
    static constexpr int OFF_STAGE = OFF_META + 48 * C::S * C::KS;
    static constexpr int OFF_CARRY = OFF_STAGE + 4 * 2 * kStreamWarps * 32;
    static constexpr int OFF_ABORT = OFF_CARRY + 4 * 2 * 32;
    static constexpr int OFF_RING = (OFF_ABORT + 16 + 127) / 128 * 128;
    static constexpr int SMEM = OFF_RING + C::S * SLOT_BYTES;
};

__device__ __forceinline__ int64_t i64min(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t i64max(int64_t a, int64_t b) { return a > b ? a : b; }

template <int NP>
__device__ __forceinline__ int find_prob_by_step(const StreamArgs<NP> &a, int64_t t) {
    int lo = 0, hi = a.nprob - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.p[mid].step0 <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}
template <int NP>
__device__ __forceinline__ int find_prob_by_group(const StreamArgs<NP> &a, int64_t g) {
    int lo = 0, hi = a.nprob - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.p[mid].group0 <= g) lo = mid; else hi = mid - 1;
    }
    return lo;
}
// first global step of global group g (g == total_groups gives total_steps)
template <int NP>
__device__ __forceinline__ int64_t group_first_step(const StreamArgs<NP> &a, int64_t g) {
    if (g >= a.total_groups) return a.total_steps;
    const StreamProb &p = a.p[find_prob_by_group(a, g)];
    return p.step0 + (g - p.group0) * p.steps;
}
template <int NP>
__device__ __forceinline__ int64_t range_begin(const StreamArgs<NP> &a, int64_t i) {
    if (a.balanced) return a.total_steps * i / a.ctas;
    return group_first_step(a, a.total_groups * i / a.ctas);
}
// the CTA whose balanced range holds step t
template <int NP>
__device__ __forceinline__ int64_t cta_of_step(const StreamArgs<NP> &a, int64_t t) {
    int64_t i = t * a.ctas / a.total_steps;
    while (i + 1 < a.ctas && a.total_steps * (i + 1) / a.ctas <= t) ++i;
    while (i > 0 && a.total_steps * i / a.ctas > t) --i;
    return i;
}

// ---- per-format consumer work on one step held in shared memory -------------
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

// This warp's share of sum_k w x for its lane's row: blocks [B0, B0+BPW) of a
// step with nblk blocks.  B0 is a compile-time constant so that every shared
// address below is a constant offset; full steps take the unchecked path.
template <int FMT, int B0>
__device__ __forceinline__ float consume_step(const uint8_t *ws, const float *xs, int nblk,
                                              int lane, const Magic &mg) {
    using C = StreamCfg<FMT>;
    constexpr int BPW = StreamLayout<FMT>::BPW;
    float acc = 0.f;
    if (nblk == 8) {
        const uint4 sv =
            *reinterpret_cast<const uint4 *>(ws + 8 * C::VPB * kVecBytes + lane * 16);
#pragma unroll
        for (int i = 0; i < BPW; ++i)
            acc += block_dot<FMT>(ws, xs + (B0 + i) * (C::SE / 8), B0 + i, scale_of(sv, B0 + i),
                                  lane, mg);
    } else {
        const uint4 sv =
            *reinterpret_cast<const uint4 *>(ws + nblk * C::VPB * kVecBytes + lane * 16);
#pragma unroll
        for (int i = 0; i < BPW; ++i)
            if (B0 + i < nblk)
                acc += block_dot<FMT>(ws, xs + (B0 + i) * (C::SE / 8), B0 + i,
                                      scale_of(sv, B0 + i), lane, mg);
    }
    return acc;
}

// This warp's share with a runtime first block (one code copy for all warps).
template <int FMT>
__device__ __forceinline__ float consume_any(const uint8_t *ws, const float *xs, int nblk, int b0,
                                             int lane, const Magic &mg) {
    using C = StreamCfg<FMT>;
    constexpr int BPW = StreamLayout<FMT>::BPW;
    const uint4 sv = *reinterpret_cast<const uint4 *>(ws + nblk * C::VPB * kVecBytes + lane * 16);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < BPW; ++i) {
        const int b = b0 + i;
        if (b < nblk) acc += block_dot<FMT>(ws, xs + b * (C::SE / 8), b, scale_of(sv, b), lane, mg);
    }
    return acc;
}

// dispatch on the warp's (runtime) first block: compile-time offsets when a
// step is split over at most two warps, a single code copy otherwise
template <int FMT>
__device__ __forceinline__ float consume(const uint8_t *ws, const float *xs, int nblk, int b0,
                                         int lane, const Magic &mg) {
    constexpr int BPW = StreamLayout<FMT>::BPW;
    if (8 / BPW > 2) return consume_any<FMT>(ws, xs, nblk, b0, lane, mg);
    switch (b0 / BPW) {
    case 0: return consume_step<FMT, 0>(ws, xs, nblk, lane, mg);
    case 1: if (BPW * 1 < 8) return consume_step<FMT, (BPW * 1) % 8>(ws, xs, nblk, lane, mg); break;
    case 2: if (BPW * 2 < 8) return consume_step<FMT, (BPW * 2) % 8>(ws, xs, nblk, lane, mg); break;
    case 3: if (BPW * 3 < 8) return consume_step<FMT, (BPW * 3) % 8>(ws, xs, nblk, lane, mg); break;
    case 4: if (BPW * 4 < 8) return consume_step<FMT, (BPW * 4) % 8>(ws, xs, nblk, lane, mg); break;
    case 5: if (BPW * 5 < 8) return consume_step<FMT, (BPW * 5) % 8>(ws, xs, nblk, lane, mg); break;
    case 6: if (BPW * 6 < 8) return consume_step<FMT, (BPW * 6) % 8>(ws, xs, nblk, lane, mg); break;
    case 7: if (BPW * 7 < 8) return consume_step<FMT, (BPW * 7) % 8>(ws, xs, nblk, lane, mg); break;
    }
    return 0.f;
}

// What the producer learned about one step of a slot, for the consumers.
struct StepMeta {
    int64_t g;       // global row group
    int64_t gs, ge;  // global step range of that group
    const float *x;  // x slice copied for the step
    int pi;          // problem index
    int nblk;        // blocks in the step
    int xe;          // x elements copied
    int step;        // step inside the group
};
static_assert(sizeof(StepMeta) == 48, "StepMeta layout");

template <int FMT, int NP>
__global__ void __launch_bounds__(kStreamThreads, StreamCfg<FMT>::CPS)
    qmm_stream_kernel(const __grid_constant__ StreamArgs<NP> a) {
    using C = StreamCfg<FMT>;
    using L = StreamLayout<FMT>;
    constexpr int SV = 8 * C::VPB + 1;  // vectors of a full step
    extern __shared__ __align__(128) uint8_t sbuf[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sbuf + L::OFF_FULL);
    uint64_t *empty = reinterpret_cast<uint64_t *>(sbuf + L::OFF_EMPTY);
    StepMeta *meta = reinterpret_cast<StepMeta *>(sbuf + L::OFF_META);
    float *stage = reinterpret_cast<float *>(sbuf + L::OFF_STAGE);   // [2][W][32]
    float *carry = reinterpret_cast<float *>(sbuf + L::OFF_CARRY);   // [2][32]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbuf + L::OFF_ABORT);
    uint8_t *ring = sbuf + L::OFF_RING;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cta = blockIdx.x;
    const int64_t beg = range_begin(a, cta), end = range_begin(a, cta + 1);
    const int64_t nsteps = end - beg;
    const int64_t nslots = (nsteps + C::KS - 1) / C::KS;

    // Let the next kernel on the stream start streaming its own weights.
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kStreamWarps);
        }
        fence_mbar_init();
        *abort_flag = 0;
    }
    __syncthreads();
    if (nsteps <= 0) return;

    if (warp == kStreamWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        // cursor over the CTA's steps: problem, group inside it, step inside the group
        int pi = find_prob_by_step(a, beg);
        int64_t g, s;
        {
            const int64_t o = beg - a.p[pi].step0;
            g = o / a.p[pi].steps;
            s = o % a.p[pi].steps;
        }
        // fill the metadata of slot j, arm its barrier and copy its weights
        auto issue_weights = [&](int64_t j) {
            const int sl = (int)(j % C::S);
            const int ns = (int)i64min(C::KS, nsteps - j * C::KS);
            uint8_t *base = ring + sl * L::SLOT_BYTES;
            StepMeta *m = meta + sl * C::KS;
            uint32_t bytes = 0;
            for (int i = 0; i < ns; ++i) {
                const StreamProb &p = a.p[pi];
                const int nblk = s == p.steps - 1 ? p.last_blocks : 8;
                const int xe = min(C::SE, p.K - (int)s * C::SE);
                m[i].g = p.group0 + g;
                m[i].gs = p.step0 + g * p.steps;
                m[i].ge = m[i].gs + p.steps;
                m[i].x = p.x + s * C::SE;
                m[i].pi = pi;
                m[i].nblk = nblk;
                m[i].xe = xe;
                m[i].step = (int)s;
                bytes += (nblk * C::VPB + 1) * kVecBytes + xe * 4;
                if (++s == p.steps) {  // advance the cursor
                    s = 0;
                    if (++g == p.groups) {
                        g = 0;
                        ++pi;
                    }
                }
            }
            mbar_arrive_expect_tx(&full[sl], bytes);  // releases the metadata too
            for (int i = 0; i < ns; ++i) {
                const StreamProb &p = a.p[m[i].pi];
                const int64_t lg = m[i].g - p.group0;
                const uint8_t *src =
                    p.W + (lg * p.group_vecs + (int64_t)m[i].step * SV) * kVecBytes;
                bulk_g2s(base + i * L::STEP_BYTES, src, (m[i].nblk * C::VPB + 1) * kVecBytes,
                         &full[sl]);
            }
        };
        auto issue_x = [&](int64_t j) {
            const int sl = (int)(j % C::S);
            const int ns = (int)i64min(C::KS, nsteps - j * C::KS);
            uint8_t *base = ring + sl * L::SLOT_BYTES;
            const StepMeta *m = meta + sl * C::KS;
            for (int i = 0; i < ns; ++i)
                bulk_g2s(base + i * L::STEP_BYTES + L::STEP_WBYTES, m[i].x, m[i].xe * 4, &full[sl]);
        };
        const int64_t nfill = i64min(C::S, nslots);
        for (int64_t j = 0; j < nfill; ++j) issue_weights(j);
        pdl_wait();  // x may be written by the previous kernel on the stream
        for (int64_t j = 0; j < nfill; ++j) issue_x(j);
        for (int64_t j = nfill; j < nslots; ++j) {
            const int sl = (int)(j % C::S);
            if (*abort_flag || !mbar_wait(&empty[sl], (uint32_t)((j / C::S - 1) & 1), kWaitLimitNs)) {
                atomicOr(a.err, kErrEmptyTimeout);
                // let the copies already issued land before the CTA can exit
                for (int64_t k = i64max(0, j - C::S); k < j; ++k)
                    mbar_wait(&full[k % C::S], (uint32_t)((k / C::S) & 1), kWaitLimitNs);
                return;
            }
            issue_weights(j);
            issue_x(j);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Each warp computes its blocks of one step per slot and stages its sum;
    // after a barrier of the consumer warps, warp r adds up run r of the slot
    // (consecutive steps of one row group) in step order, carrying a group
    // that continues into the next slot.  A group complete in this CTA is
    // stored; one shared with other CTAs (workspace mode) is published and
    // finished by the last CTA.  Every sum is taken in a fixed order.
    const int si = warp / L::WPS;             // step of the slot this warp works on
    const int b0 = (warp % L::WPS) * L::BPW;  // its first block in that step
    const Magic mg = pin(a.mg);

    // finish the CTA's part of group g (global steps [gs, ge), problem pi) with value v
    auto finish_group = [&](int64_t g, int64_t gs, int64_t ge, int pi, float v) {
        const StreamProb &p = a.p[pi];
        const int64_t n = (g - p.group0) * kRowsPerGroup + lane;
        if (gs >= beg && ge <= end) {  // the whole group is in this CTA
            if (n < p.N) p.y[n] = v;
            return;
        }
        // group split between CTAs: publish, the last CTA to arrive adds up
        const int side = gs < beg ? 0 : 1;
        a.part[(cta * 2 + side) * 32 + lane] = v;
        __threadfence();
        __syncwarp();
        unsigned arrived = 0;
        if (lane == 0) arrived = atomicAdd(&a.cnt[g], 1u);
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        const int64_t i0 = cta_of_step(a, gs), i1 = cta_of_step(a, ge - 1);
        if (arrived + 1 != (unsigned)(i1 - i0 + 1)) return;
        __threadfence();
        float tot = 0.f;
        for (int64_t i = i0; i <= i1; ++i) {
            const int sd = (i == i0) ? 1 : 0;
            tot += __ldcg(&a.part[(i * 2 + sd) * 32 + lane]);
        }
        if (n < p.N) p.y[n] = tot;
        if (lane == 0) a.cnt[g] = 0;  // ready for the next call
    };

    for (int64_t j = 0; j < nslots; ++j) {
        const int sl = (int)(j % C::S);
        const int ns = (int)i64min(C::KS, nsteps - j * C::KS);
        const bool ok = mbar_wait(&full[sl], (uint32_t)((j / C::S) & 1), kWaitLimitNs);
        if (!ok && lane == 0) {
            atomicOr(a.err, kErrFullTimeout);
            *abort_flag = 1;
        }
        float v = 0.f;
        if (ok && si < ns) {
            const StepMeta &m = meta[sl * C::KS + si];
            const uint8_t *ws = ring + sl * L::SLOT_BYTES + si * L::STEP_BYTES;
            const float *xs = reinterpret_cast<const float *>(ws + L::STEP_WBYTES);
            v = consume<FMT>(ws, xs, m.nblk, b0, lane, mg);
        }
        float *stg = stage + (j & 1) * kStreamWarps * 32;
        stg[warp * 32 + lane] = v;
        named_barrier_sync(1, 32 * kStreamWarps);  // every consumer warp staged its sum
        // all consumer warps read the flag after the same barrier: they stop together
        if (*abort_flag) return;
        {
            // run r of the slot: the r-th maximal run of steps with one group
            const StepMeta *m = meta + sl * C::KS;
            int r = 0, i0 = 0;
            for (int i = 1; i <= ns && r <= warp; ++i) {
                if (i == ns || m[i].g != m[i0].g) {
                    if (r == warp) {
                        const StepMeta &mm = m[i0];
                        float sum = 0.f;
                        const int64_t t0 = beg + j * C::KS + i0;
                        if (t0 != mm.gs && t0 != beg)  // continues a run of the previous slot
                            sum = carry[((j + 1) & 1) * 32 + lane];
                        for (int k = i0 * L::WPS; k < i * L::WPS; ++k) sum += stg[k * 32 + lane];
                        const int64_t t1 = beg + j * C::KS + i;  // one past the run
                        if (t1 == i64min(mm.ge, end)) {
                            finish_group(mm.g, mm.gs, mm.ge, mm.pi, sum);
                        } else {  // the group goes on in the next slot
                            carry[(j & 1) * 32 + lane] = sum;
                        }
                    }
                    ++r;
                    i0 = i;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sl]);
    }
}

}  // namespace lean
