// qmm_simt.cuh -- CUDA-core product for a few activation rows (up to 8 per
// launch), and the dequantisation kernel.
//
// One lane owns one row of a 32-row group and walks its blocks with 16-byte
// loads (512 contiguous bytes per warp); each block is unpacked once into
// exact fp32 integers (decode.cuh) and multiplied into all M rows of x, which
// sit in shared memory (broadcast reads).  The warps of a CTA, and the CTAs
// of a thread-block cluster, split K; partial sums are reduced through shared
// memory and, across the cluster, through distributed shared memory by the
// rank-0 CTA, which alone writes y.  No atomics: the result is deterministic.
#pragma once
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "debug.cuh"
#include "decode.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace lean {

namespace cg = cooperative_groups;

struct SimtArgs {
    const uint8_t *W;  // packed weights
    const float *x;    // x[M][K]
    float *y;          // y[M][N]
    int N, K, M;       // M = rows of x handled by this launch (<= MT)
    int64_t groups;    // row groups
    int64_t blocks;    // blocks per row
    int steps, last_blocks, step_vecs;
    int64_t group_vecs;
    int cl;            // CTAs per cluster (split of K across CTAs)
    int rg;            // row groups per CTA
    int wpr;           // warps per row group inside a CTA
    int xs_stride;     // floats per x row in shared memory
    unsigned *err;     // device error word (LEAN_DEBUG index checks)
    Magic mg;
};

template <int FMT> struct BlockTraits;
template <> struct BlockTraits<Q4_0> { static constexpr int VPB = 1, E = 32; };
template <> struct BlockTraits<Q8_0> { static constexpr int VPB = 2, E = 32; };
template <> struct BlockTraits<I8_B64> { static constexpr int VPB = 4, E = 64; };
template <> struct BlockTraits<Q6_K> { static constexpr int VPB = 13, E = 256; };

template <int FMT>
struct BlockFrag {
    uint4 v[BlockTraits<FMT>::VPB];
    float d;
};

// vectors and scale of block c of this lane's row; grp points at the lane's
// 16 bytes of the row group's first vector
template <int FMT>
__device__ __forceinline__ void load_block(BlockFrag<FMT> &f, const SimtArgs &a, const uint8_t *grp,
                                           int64_t c) {
    constexpr int VPB = BlockTraits<FMT>::VPB;
    const int s = (int)(c >> 3), i = (int)(c & 7);
    const int nblk = s == a.steps - 1 ? a.last_blocks : 8;
    const uint8_t *step = grp + (int64_t)s * a.step_vecs * kVecBytes;
    const int64_t wbytes = a.groups * a.group_vecs * kVecBytes;  // the packed matrix
#pragma unroll
    for (int j = 0; j < VPB; ++j) {
        const uint8_t *vp = step + (i * VPB + j) * kVecBytes;
        f.v[j] = LEAN_SPAN(vp - a.W, 16, wbytes, a.err) ? __ldg(reinterpret_cast<const uint4 *>(vp))
                                                       : make_uint4(0u, 0u, 0u, 0u);
    }
    const unsigned short *sv =
        reinterpret_cast<const unsigned short *>(step + nblk * VPB * kVecBytes);
    f.d = LEAN_SPAN(reinterpret_cast<const uint8_t *>(sv + i) - a.W, 2, wbytes, a.err) ? h2f(__ldg(sv + i))
                                                                                       : 0.f;
}

// tot[m] += sum over the block of w * x[m]; xs = the block's x for row 0
template <int FMT, int MT>
__device__ __forceinline__ void block_fma(const BlockFrag<FMT> &f, const float *xs, int xs_stride,
                                          const Magic &mg, float (&tot)[MT]) {
    if (FMT == Q4_0) {
        f32x2 s[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) s[m] = 0ull;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            f32x2 p[4];
            q4_word(word_of(f.v[0], t), mg, p);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float *xb = xs + m * xs_stride + 8 * t;
                const ulonglong2 xa = *reinterpret_cast<const ulonglong2 *>(xb);
                const ulonglong2 xc = *reinterpret_cast<const ulonglong2 *>(xb + 4);
                s[m] = fma2(p[0], xa.x, s[m]);
                s[m] = fma2(p[1], xa.y, s[m]);
                s[m] = fma2(p[2], xc.x, s[m]);
                s[m] = fma2(p[3], xc.y, s[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float2 r = unpack2(s[m]);
            tot[m] = fmaf(f.d, r.x + r.y, tot[m]);
        }
    } else if (FMT == Q8_0 || FMT == I8_B64) {
        constexpr int VPB = BlockTraits<FMT>::VPB;
        f32x2 s[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) s[m] = 0ull;
#pragma unroll
        for (int j = 0; j < VPB; ++j) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                f32x2 p[2];
                i8_word(word_of(f.v[j], t), mg, p);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const ulonglong2 xa = *reinterpret_cast<const ulonglong2 *>(
                        xs + m * xs_stride + j * 16 + 4 * t);
                    s[m] = fma2(p[0], xa.x, s[m]);
                    s[m] = fma2(p[1], xa.y, s[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float2 r = unpack2(s[m]);
            tot[m] = fmaf(f.d, r.x + r.y, tot[m]);
        }
    } else {  // Q6_K
        const uint4 scv = f.v[12];
#pragma unroll
        for (int sub = 0; sub < 16; ++sub) {
            const int w0 = 3 * sub;
            f32x2 p[8];
            q6_group(word_of(f.v[w0 / 4], w0 % 4), word_of(f.v[(w0 + 1) / 4], (w0 + 1) % 4),
                     word_of(f.v[(w0 + 2) / 4], (w0 + 2) % 4), mg, p);
            const float dsc = f.d * i8_byte(word_of(scv, sub >> 2), sub & 3, mg);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                f32x2 s = 0ull;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const ulonglong2 xa = *reinterpret_cast<const ulonglong2 *>(
                        xs + m * xs_stride + sub * 16 + 4 * j);
                    s = fma2(p[2 * j], xa.x, s);
                    s = fma2(p[2 * j + 1], xa.y, s);
                }
                const float2 r = unpack2(s);
                tot[m] = fmaf(dsc, r.x + r.y, tot[m]);
            }
        }
    }
}

// grid.x = ceil(groups / rg) * cl; cluster = (cl,1,1); blockDim.x = 32 * rg * wpr.
// A CTA owns rg row groups; each row group gets wpr warps that split the
// CTA's blocks.  Dynamic shared memory: MT * xs_stride floats of x, then
// warps * MT * 32 floats of partial sums.
template <int FMT, int MT>
__global__ void __launch_bounds__(512) qmm_simt_kernel(const SimtArgs a) {
    constexpr int E = BlockTraits<FMT>::E;
    extern __shared__ __align__(16) float smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)(blockIdx.x % (unsigned)a.cl);
    const int64_t g0 = (int64_t)(blockIdx.x / (unsigned)a.cl) * a.rg;
    const int gi = warp / a.wpr, sub = warp % a.wpr;
    const int64_t g = g0 + gi;
    const bool live = g < a.groups;

    // this CTA's blocks, then this warp's
    const int64_t c0 = a.blocks * rank / a.cl, c1 = a.blocks * (rank + 1) / a.cl;
    const int64_t w0 = c0 + (c1 - c0) * sub / a.wpr;
    const int64_t w1 = live ? c0 + (c1 - c0) * (sub + 1) / a.wpr : w0;
    const uint8_t *grp = a.W + (g * a.group_vecs) * kVecBytes + lane * kVec;

    pdl_launch_dependents();
    const Magic mg = pin_fmt<FMT>(a.mg);
    BlockFrag<FMT> fa, fb;
    if (w0 < w1) load_block<FMT>(fa, a, grp, w0);
    pdl_wait();  // x may come from the previous kernel on the stream

    // stage x[m][c0*E .. c1*E) into shared memory
    float *xs = smem;
    const int64_t e0 = c0 * E;
    const int elen = (int)((c1 - c0) * E);
    for (int m = 0; m < MT && m < a.M; ++m) {
        const float4 *src = reinterpret_cast<const float4 *>(a.x + (int64_t)m * a.K + e0);
        float4 *dst = reinterpret_cast<float4 *>(xs + m * a.xs_stride);
        for (int i = threadIdx.x; i < (elen >> 2); i += blockDim.x)
            dst[i] = LEAN_SPAN((int64_t)m * a.K + e0 + 4 * i, 4, (int64_t)a.M * a.K, a.err)
                         ? __ldg(src + i)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    float tot[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[m] = 0.f;
    for (int64_t c = w0; c < w1; c += 2) {
        if (c + 1 < w1) load_block<FMT>(fb, a, grp, c + 1);
        block_fma<FMT, MT>(fa, xs + (c - c0) * E, a.xs_stride, mg, tot);
        if (c + 2 < w1) load_block<FMT>(fa, a, grp, c + 2);
        if (c + 1 < w1) block_fma<FMT, MT>(fb, xs + (c + 1 - c0) * E, a.xs_stride, mg, tot);
    }

    // reduce over the wpr warps of each row group: red[warp][m][lane]
    float *red = smem + MT * a.xs_stride;
#pragma unroll
    for (int m = 0; m < MT; ++m) red[(warp * MT + m) * 32 + lane] = tot[m];
    __syncthreads();
    const int nout = a.rg * MT * 32;
    for (int i = threadIdx.x; i < nout; i += blockDim.x) {
        const int gq = i / (MT * 32), rest = i % (MT * 32);
        float s = 0.f;
        for (int w = 0; w < a.wpr; ++w) s += red[((gq * a.wpr + w) * MT) * 32 + rest];
        red[(gq * a.wpr * MT) * 32 + rest] = s;  // the group's warp-0 slot, read by its owner only
    }
    if (a.cl == 1) {
        __syncthreads();
        for (int i = threadIdx.x; i < nout; i += blockDim.x) {
            const int gq = i / (MT * 32), rest = i % (MT * 32);
            const int m = rest >> 5;
            const int64_t n = (g0 + gq) * kRowsPerGroup + (rest & 31);
            if (m < a.M && n < a.N && LEAN_IN((int64_t)m * a.N + n, (int64_t)a.M * a.N, a.err))
                a.y[(int64_t)m * a.N + n] = red[(gq * a.wpr * MT) * 32 + rest];
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (rank == 0) {
        for (int i = threadIdx.x; i < nout; i += blockDim.x) {
            const int gq = i / (MT * 32), rest = i % (MT * 32);
            const int slot = (gq * a.wpr * MT) * 32 + rest;
            float s = red[slot];
            for (int r = 1; r < a.cl; ++r) s += cluster.map_shared_rank(red, r)[slot];
            const int m = rest >> 5;
            const int64_t n = (g0 + gq) * kRowsPerGroup + (rest & 31);
            if (m < a.M && n < a.N && LEAN_IN((int64_t)m * a.N + n, (int64_t)a.M * a.N, a.err))
                a.y[(int64_t)m * a.N + n] = s;
        }
    }
    cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

// ---- dequantisation: w[n][k] fp32; one warp per (row group, block) ----
// The E weights of one block of one row, exact in fp32, to out (16-byte
// aligned): the same decode the products use, then the scale.
template <int FMT>
__device__ __forceinline__ void store_block(const BlockFrag<FMT> &f, const Magic &mg, float *out) {
    constexpr int VPB = BlockTraits<FMT>::VPB;
    if (FMT == Q4_0) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            f32x2 p[4];
            q4_word(word_of(f.v[0], t), mg, p);
            const float2 q0 = unpack2(p[0]), q1 = unpack2(p[1]), q2 = unpack2(p[2]),
                         q3 = unpack2(p[3]);
            float4 *o = reinterpret_cast<float4 *>(out + 8 * t);
            o[0] = make_float4(f.d * q0.x, f.d * q0.y, f.d * q1.x, f.d * q1.y);
            o[1] = make_float4(f.d * q2.x, f.d * q2.y, f.d * q3.x, f.d * q3.y);
        }
    } else if (FMT == Q8_0 || FMT == I8_B64) {
#pragma unroll
        for (int j = 0; j < VPB; ++j) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                f32x2 p[2];
                i8_word(word_of(f.v[j], t), mg, p);
                const float2 q0 = unpack2(p[0]), q1 = unpack2(p[1]);
                *reinterpret_cast<float4 *>(out + 16 * j + 4 * t) =
                    make_float4(f.d * q0.x, f.d * q0.y, f.d * q1.x, f.d * q1.y);
            }
        }
    } else {
        const uint4 scv = f.v[12];
#pragma unroll
        for (int sub = 0; sub < 16; ++sub) {
            const int w0 = 3 * sub;
            f32x2 p[8];
            q6_group(word_of(f.v[w0 / 4], w0 % 4), word_of(f.v[(w0 + 1) / 4], (w0 + 1) % 4),
                     word_of(f.v[(w0 + 2) / 4], (w0 + 2) % 4), mg, p);
            const float dsc = f.d * i8_byte(word_of(scv, sub >> 2), sub & 3, mg);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 q0 = unpack2(p[2 * j]), q1 = unpack2(p[2 * j + 1]);
                *reinterpret_cast<float4 *>(out + 16 * sub + 4 * j) =
                    make_float4(dsc * q0.x, dsc * q0.y, dsc * q1.x, dsc * q1.y);
            }
        }
    }
}

// w[n][k] for the whole matrix: one warp per (row group, block), lane = row.
template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const SimtArgs a, float *w) {
    constexpr int E = BlockTraits<FMT>::E;
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t g = item / a.blocks, c = item % a.blocks;
    if (g >= a.groups) return;
    BlockFrag<FMT> f;
    load_block<FMT>(f, a, a.W + g * a.group_vecs * kVecBytes + lane * kVec, c);
    const int64_t n = g * kRowsPerGroup + lane;
    if (n >= a.N || !LEAN_SPAN(n * a.K + c * E, E, (int64_t)a.N * a.K, a.err)) return;
    store_block<FMT>(f, a.mg, w + n * a.K + c * E);
}

// Error bit of an embedding id outside 0..N-1.
constexpr unsigned kErrEmbedId = 16u;

// Selected rows of the matrix (an embedding lookup): out[i][k] = w[ids[i]][k],
// one thread per (id, block), consecutive threads on consecutive blocks of
// one id.  An id outside 0..N-1 gives a row of NaN and sets kErrEmbedId in
// the device error word.
template <int FMT>
__global__ void __launch_bounds__(256) embed_kernel(const SimtArgs a, const int32_t *ids,
                                                    int64_t n_ids, float *out, unsigned *err) {
    constexpr int E = BlockTraits<FMT>::E;
    const int64_t item = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (item >= n_ids * a.blocks) return;
    const int64_t i = item / a.blocks, c = item % a.blocks;
    const int64_t n = ids[i];
    float *o = out + i * a.K + c * E;
    if (!LEAN_SPAN(i * a.K + c * E, E, n_ids * a.K, a.err)) return;
    if (n < 0 || n >= a.N) {
        const float4 nan4 = make_float4(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                        __int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
#pragma unroll
        for (int j = 0; j < E; j += 4) *reinterpret_cast<float4 *>(o + j) = nan4;
        if (c == 0) atomicOr(err, kErrEmbedId);
        return;
    }
    BlockFrag<FMT> f;
    load_block<FMT>(f, a, a.W + (n / kRowsPerGroup) * a.group_vecs * kVecBytes + (n % kRowsPerGroup) * kVec,
                    c);
    store_block<FMT>(f, a.mg, o);
}

}  // namespace lean
