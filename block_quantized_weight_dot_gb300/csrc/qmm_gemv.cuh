// qmm_gemv.cuh -- the M = 1 product for problems that fit the GPU in one
// wave: latency first.
//
// A decode step is a chain of GEMVs in which each one's x is the previous
// one's output ("wgpu-llm" README, Architecture at a Glance: N x (Attn + FFN)),
// so what a single product costs after its input exists is what the step
// pays.  This kernel takes every weight it needs off the critical path:
//
//  - a CTA of 8 warps owns one 32-row group (lane = row) and a range of its
//    blocks along K; each warp takes at most NB consecutive blocks, and a
//    cluster of up to 8 CTAs splits longer rows;
//  - every lane loads all of its blocks (16-byte loads, 512 contiguous bytes
//    per warp) before griddepcontrol.wait, so with programmatic dependent
//    launch the weights stream while the previous kernel is still running;
//  - after the wait the CTA stages its slice of x in shared memory (coalesced
//    16-byte loads), each lane decodes its blocks exactly (decode.cuh) and
//    sums w * x with paired fp32 FMAs, the warps' partial sums meet in shared
//    memory and the cluster's in distributed shared memory, in a fixed order:
//    no atomics, no workspace, deterministic.
//
// Several problems of one format can share a launch (a list of problems, each
// owning a run of clusters), like the q, k and v projections of one layer.
#pragma once
#include <cooperative_groups.h>
#include <stdint.h>

#include "debug.cuh"
#include "decode.cuh"
#include "layout.h"
#include "ptx.cuh"
#include "qmm_simt.cuh"

namespace lean {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = 32 * kGemvWarps;
constexpr int kGemvMaxCluster = 8;

// Blocks a lane holds in registers at most (four 16-byte vectors per block of
// the int8 formats: Q8_0 2, I8_B64 4; Q6_K 13 vectors), for MT rows of x: with
// 8 rows fewer, so that the CTA's x slice stays within 32 KB.
template <int FMT> struct GemvCfg;
template <> struct GemvCfg<Q4_0> { static constexpr int NB = 8; };
template <> struct GemvCfg<Q8_0> { static constexpr int NB = 4; };
template <> struct GemvCfg<I8_B64> { static constexpr int NB = 2; };
template <> struct GemvCfg<Q6_K> { static constexpr int NB = 1; };
template <int FMT, int MT>
constexpr int gemv_nb() {
    return MT <= 4 ? GemvCfg<FMT>::NB
                   : (GemvCfg<FMT>::NB * 4 / MT > 0 ? GemvCfg<FMT>::NB * 4 / MT : 1);
}
// floats of x one CTA stages per row of x
template <int FMT, int MT>
constexpr int gemv_xstride() { return kGemvWarps * gemv_nb<FMT, MT>() * BlockTraits<FMT>::E; }
template <int FMT, int MT>
constexpr int gemv_smem_bytes() {
    return (MT * gemv_xstride<FMT, MT>() + kGemvWarps * MT * 32) * 4;
}

struct GemvProb {
    const uint8_t *W;
    const float *x;
    float *y;
    int N, K;
    int blocks;      // blocks per row
    int steps, last_blocks, step_vecs;
    int nbw;         // blocks per warp (<= NB)
    int cta0;        // first CTA of this problem (a multiple of the cluster size)
    int64_t group_vecs;
};

template <int NP>
struct GemvArgs {
    int nprob;
    int cl;  // CTAs per cluster (K split), the same for every problem
    int M;   // rows of x (<= MT of the kernel); x[M][K], y[M][N]
    int pad;
    unsigned *err;  // device error word (LEAN_DEBUG index checks)
    Magic mg;
    GemvProb p[NP];
};

// vectors and scale of block c of this lane's row (as load_block, for a
// GemvProb)
template <int FMT>
__device__ __forceinline__ void gemv_load(BlockFrag<FMT> &f, const GemvProb &p, const uint8_t *grp,
                                          int c, unsigned *err) {
    constexpr int VPB = BlockTraits<FMT>::VPB;
    const int s = c >> 3, i = c & 7;
    const int nblk = s == p.steps - 1 ? p.last_blocks : 8;
    const uint8_t *step = grp + (int64_t)s * p.step_vecs * kVecBytes;
    const int64_t wbytes = (int64_t)((p.N + kRowsPerGroup - 1) / kRowsPerGroup) * p.group_vecs * kVecBytes;
#pragma unroll
    for (int j = 0; j < VPB; ++j) {
        const uint8_t *vp = step + (i * VPB + j) * kVecBytes;
        f.v[j] = LEAN_SPAN(vp - p.W, 16, wbytes, err) ? __ldg(reinterpret_cast<const uint4 *>(vp))
                                                     : make_uint4(0u, 0u, 0u, 0u);
    }
    const unsigned short *sv = reinterpret_cast<const unsigned short *>(step + nblk * VPB * kVecBytes);
    f.d = LEAN_SPAN(reinterpret_cast<const uint8_t *>(sv + i) - p.W, 2, wbytes, err) ? h2f(__ldg(sv + i))
                                                                                    : 0.f;
}

// grid.x = sum over problems of groups * cl; cluster = (cl, 1, 1);
// blockDim.x = 256; dynamic shared memory gemv_smem_bytes<FMT, MT>(): the
// CTA's slice of each of the MT rows of x, then 8 x MT x 32 partial sums.
// MT > 1: the same for up to MT rows of x, each decoded weight multiplied into
// all of them (x rows past M read as zero).
// SWIGLU (MT = 1): the problems come in pairs (gate, up) of one shape, x and
// output; each row group gets a cluster of cl = 2 * (K split) CTAs, the first
// half on the gate rows, the second on the up rows, and rank 0 writes
// h = silu(gate . x) * (up . x) (the input of the FFN's down projection).
// A pair's two entries carry the same cta0.
template <int FMT, int NP, bool SWIGLU, int MT>
__global__ void __launch_bounds__(kGemvThreads, MT == 1 ? 3 : 2)
    qmm_gemv_kernel(const __grid_constant__ GemvArgs<NP> a) {
    namespace cg = cooperative_groups;
    constexpr int E = BlockTraits<FMT>::E;
    constexpr int NB = gemv_nb<FMT, MT>();
    constexpr int XS = gemv_xstride<FMT, MT>();
    extern __shared__ __align__(16) float gsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's problem: the last one whose first CTA is at or before it
    int lo = 0, hi = a.nprob - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.p[mid].cta0 <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const int base = SWIGLU ? (lo & ~1) : lo;
    const int local = (int)blockIdx.x - a.p[base].cta0;
    const int rank = local % a.cl;              // rank in the cluster
    const int64_t g = local / a.cl;
    const int ks = SWIGLU ? a.cl >> 1 : a.cl;   // CTAs splitting one row's K
    const int role = SWIGLU ? rank / ks : 0;    // SWIGLU: 0 gate, 1 up
    const int krank = rank % ks;
    const GemvProb &p = a.p[base + role];
    // blocks of this CTA and of this warp
    const int span = kGemvWarps * p.nbw;
    const int c0 = min(p.blocks, krank * span), c1 = min(p.blocks, c0 + span);
    const int w0 = min(c1, c0 + warp * p.nbw), w1 = min(c1, w0 + p.nbw);
    const uint8_t *grp = p.W + g * p.group_vecs * kVecBytes + lane * kVec;

    pdl_launch_dependents();
    BlockFrag<FMT> f[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i)
        if (w0 + i < w1) gemv_load<FMT>(f[i], p, grp, w0 + i, a.err);
    const Magic mg = pin_fmt<FMT>(a.mg);
    pdl_wait();  // x may come from the previous kernel on the stream

    float *xs = gsm;
    const int nv = (c1 - c0) * (E / 4);  // float4 per row of the slice
    for (int i = threadIdx.x; i < MT * nv; i += kGemvThreads) {
        const int m = i / nv, v = i % nv;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < a.M && LEAN_SPAN((int64_t)m * p.K + (int64_t)c0 * E + 4 * v, 4, (int64_t)a.M * p.K, a.err))
            val = reinterpret_cast<const float4 *>(p.x + (int64_t)m * p.K + (int64_t)c0 * E)[v];
        reinterpret_cast<float4 *>(xs + m * XS)[v] = val;
    }
    __syncthreads();

    float tot[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[m] = 0.f;
#pragma unroll
    for (int i = 0; i < NB; ++i)
        if (w0 + i < w1) block_fma<FMT, MT>(f[i], xs + (w0 + i - c0) * E, XS, mg, tot);

    // the 8 warps' sums, then (cluster) the CTAs' sums, each in a fixed order
    float *red = gsm + MT * XS;
#pragma unroll
    for (int m = 0; m < MT; ++m) red[(warp * MT + m) * 32 + lane] = tot[m];
    __syncthreads();
    for (int i = threadIdx.x; i < MT * 32; i += kGemvThreads) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kGemvWarps; ++w) s += red[w * MT * 32 + i];
        red[i] = s;  // warp 0's slots: row m = i / 32, lane i % 32
        const int m = i >> 5;
        const int64_t n = g * kRowsPerGroup + (i & 31);
        if (!SWIGLU && a.cl == 1 && m < a.M && n < p.N &&
            LEAN_IN((int64_t)m * p.N + n, (int64_t)a.M * p.N, a.err))
            p.y[(int64_t)m * p.N + n] = s;
    }
    if (!SWIGLU && a.cl == 1) return;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (rank == 0) {
        for (int i = threadIdx.x; i < MT * 32; i += kGemvThreads) {
            const int m = i >> 5;
            const int64_t n = g * kRowsPerGroup + (i & 31);
            if (!SWIGLU) {
                float s = red[i];
                for (int r = 1; r < a.cl; ++r) s += cluster.map_shared_rank(red, r)[i];
                if (m < a.M && n < p.N && LEAN_IN((int64_t)m * p.N + n, (int64_t)a.M * p.N, a.err))
                    p.y[(int64_t)m * p.N + n] = s;
            } else {
                float gs = red[i], us = 0.f;
                for (int r = 1; r < ks; ++r) gs += cluster.map_shared_rank(red, r)[i];
                for (int r = ks; r < a.cl; ++r) us += cluster.map_shared_rank(red, r)[i];
                if (n < p.N && LEAN_IN(n, p.N, a.err)) p.y[n] = gs / (1.f + expf(-gs)) * us;  // silu(g) * u
            }
        }
    }
    cluster.sync();  // no CTA leaves while rank 0 reads its shared memory
}

}  // namespace lean
