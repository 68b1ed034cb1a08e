// qmm_simt.cuh -- the CUDA-core product kernel: y[m][n] = sum_k w[n][k] x[m][k]
// for M <= 16 activation rows (M = 1 is the decode GEMV).
//
// Decode streams every weight once ("oxinfer" crate page, Performance: decode
// is memory-bandwidth bound, every token streams all dense weights once), so
// the kernel is built around the packed stream:
//
//  - one lane owns one weight row of a 32-row group and walks along K with
//    16-byte loads; a warp's load is 512 contiguous bytes (layout.h);
//  - the CTA's slice of x[M][K] sits in shared memory; every lane of a warp
//    reads the same x element, so the shared loads are broadcasts;
//  - quant words are unpacked to exact fp32 integers in registers (decode.cuh)
//    and accumulated with paired fp32 FMAs per block; the block's scale is
//    applied once per block;
//  - the warps of a CTA, and the CTAs of a thread-block cluster, split K; the
//    per-lane sums are reduced through shared memory and then, across the
//    cluster, through distributed shared memory by the cluster's rank-0 CTA,
//    which alone writes y.  No global scratch and no atomics: the result is
//    deterministic.
//
// A "step" is the unit of work along K: 8 quant vectors (Q4_0: 8 blocks,
// Q8_0: 4 blocks, I8_B64: 2 blocks) or one Q6_K super-block (12 quant vectors
// + 1 sub-scale vector).  Warps take contiguous runs of steps and prefetch the
// next step's vectors while they compute the current one.
#pragma once
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "decode.cuh"
#include "layout.h"

namespace lean {

namespace cg = cooperative_groups;

struct SimtArgs {
    const uint8_t *W;      // packed weights
    const float *x;        // x[M][K]
    float *y;              // y[M][N]
    int64_t s_off;         // scale plane offset (bytes)
    int N, K, M;           // M = rows of x handled by this launch (<= MT)
    int qvec, svec;        // vectors per row in the quant / scale planes
    int steps;             // steps per row
    int64_t groups;        // row groups (ceil(N / 32))
    int cl;                // CTAs per cluster (split of K across CTAs)
    int rg;                // row groups per CTA
    int wpr;               // warps per row group inside a CTA
    int xs_stride;         // floats per x row in shared memory
};

template <int FMT> struct StepTraits;
template <> struct StepTraits<Q4_0> { static constexpr int VECS = 8, ELEMS = 256; };
template <> struct StepTraits<Q8_0> { static constexpr int VECS = 8, ELEMS = 128; };
template <> struct StepTraits<I8_B64> { static constexpr int VECS = 8, ELEMS = 128; };
template <> struct StepTraits<Q6_K> { static constexpr int VECS = 13, ELEMS = 256; };

template <int FMT>
struct StepFrag {
    uint4 v[StepTraits<FMT>::VECS];
    uint32_t s0, s1, s2, s3;  // raw scale bits for the step
};

// Load the quant vectors and scales of step `st` of this lane's row.
template <int FMT>
__device__ __forceinline__ void load_step(StepFrag<FMT> &f, const SimtArgs &a, int64_t qrow,
                                          int64_t srow_vec0, int st) {
    constexpr int V = StepTraits<FMT>::VECS;
    const uint4 *q = reinterpret_cast<const uint4 *>(a.W) + qrow;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int vi = st * V + j;
        if (FMT == Q6_K || vi < a.qvec)
            f.v[j] = __ldg(q + (int64_t)vi * kRowsPerGroup);
        else
            f.v[j] = make_uint4(0u, 0u, 0u, 0u);
    }
    // scale plane: vector index v covers 8 blocks / super-blocks
    const uint8_t *sbase = a.W + a.s_off;
    if (FMT == Q4_0) {
        uint4 s = __ldg(reinterpret_cast<const uint4 *>(sbase) + srow_vec0 +
                        (int64_t)st * kRowsPerGroup);
        f.s0 = s.x; f.s1 = s.y; f.s2 = s.z; f.s3 = s.w;
    } else if (FMT == Q8_0) {  // 4 blocks per step: half a scale vector
        const uint2 *p = reinterpret_cast<const uint2 *>(
            reinterpret_cast<const uint4 *>(sbase) + srow_vec0 + (int64_t)(st >> 1) * kRowsPerGroup);
        uint2 s = __ldg(p + (st & 1));
        f.s0 = s.x; f.s1 = s.y; f.s2 = 0; f.s3 = 0;
    } else if (FMT == I8_B64) {  // 2 blocks per step: a quarter vector
        const uint32_t *p = reinterpret_cast<const uint32_t *>(
            reinterpret_cast<const uint4 *>(sbase) + srow_vec0 + (int64_t)(st >> 2) * kRowsPerGroup);
        f.s0 = __ldg(p + (st & 3)); f.s1 = f.s2 = f.s3 = 0;
    } else {  // Q6_K: one fp16 d per super-block
        const unsigned short *p = reinterpret_cast<const unsigned short *>(
            reinterpret_cast<const uint4 *>(sbase) + srow_vec0 + (int64_t)(st >> 3) * kRowsPerGroup);
        f.s0 = __ldg(p + (st & 7)); f.s1 = f.s2 = f.s3 = 0;
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int t) {
    return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t scale_half(const uint32_t s0, const uint32_t s1,
                                               const uint32_t s2, const uint32_t s3, int b) {
    const uint32_t w = (b >> 1) == 0 ? s0 : (b >> 1) == 1 ? s1 : (b >> 1) == 2 ? s2 : s3;
    return (b & 1) ? (w >> 16) : (w & 0xffffu);
}

// x pairs for elements e, e+1 .. e+3 of row m from shared memory (broadcast)
__device__ __forceinline__ void lds_x4(const float *xs, float2 &a, float2 &b) {
    const float4 v = *reinterpret_cast<const float4 *>(xs);
    a = make_float2(v.x, v.y);
    b = make_float2(v.z, v.w);
}

// Accumulate one step into tot[m].  xs points at the step's first element of
// row 0 in shared memory; rows are xs_stride floats apart.
template <int FMT, int MT>
__device__ __forceinline__ void compute_step(const StepFrag<FMT> &f, const float *xs, int xs_stride,
                                             int qvec_left, float (&tot)[MT]) {
    if (FMT == Q4_0) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {           // vector b = block b of the step
            if (b < qvec_left) {
                const float d = h2f(scale_half(f.s0, f.s1, f.s2, f.s3, b));
                float2 acc[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = make_float2(0.f, 0.f);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float2 w[4];
                    dec_q4_word(word_of(f.v[b], t), w);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float2 x0, x1, x2, x3;
                        const float *xp = xs + m * xs_stride + b * 32 + t * 8;
                        lds_x4(xp, x0, x1);
                        lds_x4(xp + 4, x2, x3);
                        acc[m] = __ffma2_rn(w[0], x0, acc[m]);
                        acc[m] = __ffma2_rn(w[1], x1, acc[m]);
                        acc[m] = __ffma2_rn(w[2], x2, acc[m]);
                        acc[m] = __ffma2_rn(w[3], x3, acc[m]);
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) tot[m] = fmaf(d, acc[m].x + acc[m].y, tot[m]);
            }
        }
    } else if (FMT == Q8_0 || FMT == I8_B64) {
        constexpr int VPB = (FMT == Q8_0) ? 2 : 4;  // vectors per block
#pragma unroll
        for (int b = 0; b < 8 / VPB; ++b) {
            if (b * VPB < qvec_left) {
                const float d = h2f(scale_half(f.s0, f.s1, f.s2, f.s3, b));
                float2 acc[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < VPB; ++j) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        float2 w[2];
                        dec_i8_word(word_of(f.v[b * VPB + j], t), w);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            float2 x0, x1;
                            lds_x4(xs + m * xs_stride + (b * VPB + j) * 16 + t * 4, x0, x1);
                            acc[m] = __ffma2_rn(w[0], x0, acc[m]);
                            acc[m] = __ffma2_rn(w[1], x1, acc[m]);
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) tot[m] = fmaf(d, acc[m].x + acc[m].y, tot[m]);
            }
        }
    } else {  // Q6_K: 16 sub-blocks of 16 elements, one int8 sub-scale each
        const float d = h2f(f.s0);
        const uint4 scv = f.v[12];
#pragma unroll
        for (int sb = 0; sb < 16; ++sb) {
            const int wi = 3 * sb;  // word index inside the 12 quant vectors
            const uint32_t w0 = word_of(f.v[wi / 4], wi % 4);
            const uint32_t w1 = word_of(f.v[(wi + 1) / 4], (wi + 1) % 4);
            const uint32_t w2 = word_of(f.v[(wi + 2) / 4], (wi + 2) % 4);
            float2 w[8];
            dec_q6_group(w0, w1, w2, w);
            // sub-scale sb: byte sb%4 of word sb/4 of the scale vector, biased by 128
            const uint32_t scw = word_of(scv, sb / 4);
            const float sc = __uint_as_float(((scw >> (8 * (sb % 4))) & 0xffu) | kMagic0) - 8388736.0f;
            const float dsc = d * sc;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float2 x0, x1;
                    lds_x4(xs + m * xs_stride + sb * 16 + j * 4, x0, x1);
                    acc = __ffma2_rn(w[2 * j], x0, acc);
                    acc = __ffma2_rn(w[2 * j + 1], x1, acc);
                }
                tot[m] = fmaf(dsc, acc.x + acc.y, tot[m]);
            }
        }
    }
}

// grid.x = ceil(groups / rg) * cl; cluster = (cl,1,1); blockDim.x = 32 * rg * wpr.
// A CTA owns rg row groups; each row group gets wpr warps that split the
// CTA's steps.  Dynamic shared memory: MT * xs_stride floats of x, then
// warps * MT * 32 floats of partial sums.
template <int FMT, int MT, bool DB>
__global__ void __launch_bounds__(512) qmm_simt_kernel(const SimtArgs a) {
    constexpr int SE = StepTraits<FMT>::ELEMS;
    constexpr int V = StepTraits<FMT>::VECS;
    extern __shared__ __align__(16) float smem[];
    const int warps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)(blockIdx.x % (unsigned)a.cl);
    const int64_t g0 = (int64_t)(blockIdx.x / (unsigned)a.cl) * a.rg;
    const int gi = warp / a.wpr, sub = warp % a.wpr;
    const int64_t g = g0 + gi;
    const bool live = g < a.groups;

    // this CTA's steps, then this warp's
    const int c0 = (int)((int64_t)a.steps * rank / a.cl);
    const int c1 = (int)((int64_t)a.steps * (rank + 1) / a.cl);
    const int w0 = c0 + (int)((int64_t)(c1 - c0) * sub / a.wpr);
    const int w1 = live ? c0 + (int)((int64_t)(c1 - c0) * (sub + 1) / a.wpr) : w0;

    // lane's row inside the planes (uint4 units)
    const int64_t qrow = g * a.qvec * kRowsPerGroup + lane;
    const int64_t srow = g * a.svec * kRowsPerGroup + lane;

    // Programmatic dependent launch: let the next kernel on the stream start
    // its own weight loads now; weights are never written by these kernels.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    StepFrag<FMT> fa, fb;
    if (w0 < w1) load_step<FMT>(fa, a, qrow, srow, w0);

    // x may be produced by the preceding kernel: wait for it to complete
    // (a no-op when the launch has no programmatic dependency).
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // stage x[m][c0*SE .. min(c1*SE, K)) into shared memory
    float *xs = smem;
    const int e0 = c0 * SE;
    const int elen = min(c1 * SE, a.K) - e0;
    for (int m = 0; m < MT; ++m) {
        if (m >= a.M) break;
        const float4 *src = reinterpret_cast<const float4 *>(a.x + (int64_t)m * a.K + e0);
        float4 *dst = reinterpret_cast<float4 *>(xs + m * a.xs_stride);
        for (int i = threadIdx.x; i < (elen >> 2); i += blockDim.x) dst[i] = __ldg(src + i);
    }
    __syncthreads();

    float tot[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[m] = 0.f;

    if (DB) {  // prefetch the next step while computing this one
        for (int st = w0; st < w1; st += 2) {
            if (st + 1 < w1) load_step<FMT>(fb, a, qrow, srow, st + 1);
            compute_step<FMT, MT>(fa, xs + (st - c0) * SE, a.xs_stride, a.qvec - st * V, tot);
            if (st + 2 < w1) load_step<FMT>(fa, a, qrow, srow, st + 2);
            if (st + 1 < w1)
                compute_step<FMT, MT>(fb, xs + (st + 1 - c0) * SE, a.xs_stride,
                                      a.qvec - (st + 1) * V, tot);
        }
    } else {
        for (int st = w0; st < w1; ++st) {
            if (st > w0) load_step<FMT>(fa, a, qrow, srow, st);
            compute_step<FMT, MT>(fa, xs + (st - c0) * SE, a.xs_stride, a.qvec - st * V, tot);
        }
    }

    // reduce over the wpr warps of each row group: red[warp][m][lane]
    float *red = smem + MT * a.xs_stride;
#pragma unroll
    for (int m = 0; m < MT; ++m) red[(warp * MT + m) * 32 + lane] = tot[m];
    __syncthreads();
    // out slot i = (gi * MT + m) * 32 + row, stored over the first warp of each group
    const int nout = a.rg * MT * 32;
    for (int i = threadIdx.x; i < nout; i += blockDim.x) {
        const int gq = i / (MT * 32), rest = i % (MT * 32);
        float s = 0.f;
        for (int w = 0; w < a.wpr; ++w) s += red[((gq * a.wpr + w) * MT) * 32 + rest];
        red[(gq * a.wpr * MT) * 32 + rest] = s;  // overwrites the group's warp-0 slot only
    }
    if (a.cl == 1) {
        __syncthreads();
        for (int i = threadIdx.x; i < nout; i += blockDim.x) {
            const int gq = i / (MT * 32), rest = i % (MT * 32);
            const int m = rest >> 5;
            const int64_t n = (g0 + gq) * kRowsPerGroup + (rest & 31);
            if (m < a.M && n < a.N) a.y[(int64_t)m * a.N + n] = red[(gq * a.wpr * MT) * 32 + rest];
        }
        return;
    }
    // reduce over the CTAs of the cluster through distributed shared memory
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
            if (m < a.M && n < a.N) a.y[(int64_t)m * a.N + n] = s;
        }
    }
    cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

// ---- dequantisation: w[n][k] fp32, one lane per row, one step per warp ----
template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const SimtArgs a, float *w) {
    constexpr int SE = StepTraits<FMT>::ELEMS;
    constexpr int V = StepTraits<FMT>::VECS;
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t g = item / a.steps;
    const int st = (int)(item % a.steps);
    if (g * kRowsPerGroup >= a.N) return;
    const int64_t n = g * kRowsPerGroup + lane;
    StepFrag<FMT> f;
    load_step<FMT>(f, a, g * a.qvec * kRowsPerGroup + lane, g * a.svec * kRowsPerGroup + lane, st);
    if (n >= a.N) return;
    float *out = w + n * a.K + (int64_t)st * SE;
    const int left = a.qvec - st * V;
    if (FMT == Q4_0) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (b < left) {
                const float d = h2f(scale_half(f.s0, f.s1, f.s2, f.s3, b));
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float2 q[4];
                    dec_q4_word(word_of(f.v[b], t), q);
                    float4 *o = reinterpret_cast<float4 *>(out + b * 32 + t * 8);
                    o[0] = make_float4(d * q[0].x, d * q[0].y, d * q[1].x, d * q[1].y);
                    o[1] = make_float4(d * q[2].x, d * q[2].y, d * q[3].x, d * q[3].y);
                }
            }
        }
    } else if (FMT == Q8_0 || FMT == I8_B64) {
        constexpr int VPB = (FMT == Q8_0) ? 2 : 4;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < left) {
                const float d = h2f(scale_half(f.s0, f.s1, f.s2, f.s3, j / VPB));
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float2 q[2];
                    dec_i8_word(word_of(f.v[j], t), q);
                    *reinterpret_cast<float4 *>(out + j * 16 + t * 4) =
                        make_float4(d * q[0].x, d * q[0].y, d * q[1].x, d * q[1].y);
                }
            }
        }
    } else {
        const float d = h2f(f.s0);
#pragma unroll
        for (int sb = 0; sb < 16; ++sb) {
            const int wi = 3 * sb;
            float2 q[8];
            dec_q6_group(word_of(f.v[wi / 4], wi % 4), word_of(f.v[(wi + 1) / 4], (wi + 1) % 4),
                         word_of(f.v[(wi + 2) / 4], (wi + 2) % 4), q);
            const uint32_t scw = word_of(f.v[12], sb / 4);
            const float sc = __uint_as_float(((scw >> (8 * (sb % 4))) & 0xffu) | kMagic0) - 8388736.0f;
            const float dsc = d * sc;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4 *>(out + sb * 16 + 4 * j) =
                    make_float4(dsc * q[2 * j].x, dsc * q[2 * j].y, dsc * q[2 * j + 1].x,
                                dsc * q[2 * j + 1].y);
        }
    }
}

}  // namespace lean
