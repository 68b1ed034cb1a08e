// simt_launch.cuh -- launch planning for the CUDA-core kernels.  Included by
// one translation unit per weight format (qmm_<fmt>.cu), each of which
// instantiates qmm_fmt<FMT> and dequant_fmt<FMT>.
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "../../include/lean_qmatmul.h"
#include "layout.h"
#include "qmm_simt.cuh"

namespace lean {


constexpr int kMaxDevices = 64;
constexpr int kMaxWarpsPerCta = 16;
constexpr int kMaxCluster = 8;
constexpr size_t kMaxSmem = 200 * 1024;

// Per-device SM count, read once.
inline int sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

template <int FMT> constexpr int step_elems() { return StepTraits<FMT>::ELEMS; }
template <int FMT> constexpr int step_vecs() { return StepTraits<FMT>::VECS; }

struct Plan {
    int cl, rg, wpr, mt, per_warp;
    int64_t ctas;
    size_t smem;
    int xs_stride;
};

// Launch shape for the CUDA-core kernel.  Aim for about 16 resident warps per
// SM with every warp doing a whole number of steps; split K over the warps of
// a CTA first and over the CTAs of a cluster when one CTA is not enough.
template <int FMT>
bool plan_simt(const Geom &g, int mt, Plan *p) {
    const int V = step_vecs<FMT>(), SE = step_elems<FMT>();
    const int steps = (int)((g.qvec + V - 1) / V);
    const int64_t target = (int64_t)sm_count() * 16;
    int64_t want = (target + g.groups - 1) / g.groups;          // warps per row group
    want = std::max<int64_t>(1, std::min<int64_t>(want, steps));
    const int per_warp = (int)((steps + want - 1) / want);       // steps per warp
    int wtot = (steps + per_warp - 1) / per_warp;                // warps per row group
    int cl = (wtot + kMaxWarpsPerCta - 1) / kMaxWarpsPerCta;
    cl = std::min(cl, kMaxCluster);
    // shared memory for x: grow the cluster until the slice fits
    auto slice_floats = [&](int c) { return (int)(((steps + c - 1) / c) * (int64_t)SE); };
    while (cl < kMaxCluster && (size_t)mt * slice_floats(cl) * 4 > kMaxSmem / 2) ++cl;
    const int wpr = std::max(1, std::min(kMaxWarpsPerCta, (wtot + cl - 1) / cl));
    // several row groups per CTA when a group needs few warps
    int rg = 1;
    while (rg * 2 * wpr <= 8 && rg * 2 <= g.groups) rg *= 2;
    const int xs_stride = slice_floats(cl);
    const size_t smem = (size_t)mt * xs_stride * 4 + (size_t)rg * wpr * mt * 32 * 4;
    if (smem > kMaxSmem) return false;
    p->cl = cl;
    p->rg = rg;
    p->wpr = wpr;
    p->mt = mt;
    p->per_warp = per_warp;
    p->ctas = (g.groups + rg - 1) / rg * cl;
    p->smem = smem;
    p->xs_stride = xs_stride;
    return true;
}

template <int FMT, int MT>
lean_status launch_simt(const Geom &g, const uint8_t *W, const float *x, float *y, int M,
                        unsigned flags, cudaStream_t stream) {
    Plan p;
    if (!plan_simt<FMT>(g, MT, &p)) return LEAN_ERR_SHAPE;
    SimtArgs a;
    a.W = W;
    a.x = x;
    a.y = y;
    a.s_off = g.s_off;
    a.N = (int)g.N;
    a.K = (int)g.K;
    a.M = M;
    a.qvec = (int)g.qvec;
    a.svec = (int)g.svec;
    a.steps = (int)((g.qvec + step_vecs<FMT>() - 1) / step_vecs<FMT>());
    a.groups = g.groups;
    a.cl = p.cl;
    a.rg = p.rg;
    a.wpr = p.wpr;
    a.xs_stride = p.xs_stride;
    // double-buffer the steps only when a warp has several and registers allow
    auto kern = (p.per_warp >= 2 && MT <= 2) ? qmm_simt_kernel<FMT, MT, true>
                                              : qmm_simt_kernel<FMT, MT, false>;
    if (p.smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) !=
            cudaSuccess)
            return LEAN_ERR_CUDA;
    }
    if (p.ctas > INT32_MAX) return LEAN_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)(32 * p.rg * p.wpr), 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.cl > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = p.cl;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (flags & LEAN_FLAG_EARLY_WEIGHTS) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return LEAN_ERR_CUDA;
    return LEAN_OK;
}

template <int FMT>
lean_status qmm_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                    unsigned flags, cudaStream_t stream) {
    // M rows of x in tiles of at most 16; each tile re-streams the weights.
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        const int mt = (int)std::min<int64_t>(16, M - m0);
        const float *xt = x + m0 * g.K;
        float *yt = y + m0 * g.N;
        lean_status s;
        if (mt == 1) s = launch_simt<FMT, 1>(g, W, xt, yt, mt, flags, stream);
        else if (mt == 2) s = launch_simt<FMT, 2>(g, W, xt, yt, mt, flags, stream);
        else if (mt <= 4) s = launch_simt<FMT, 4>(g, W, xt, yt, mt, flags, stream);
        else if (mt <= 8) s = launch_simt<FMT, 8>(g, W, xt, yt, mt, flags, stream);
        else s = launch_simt<FMT, 16>(g, W, xt, yt, mt, flags, stream);
        if (s != LEAN_OK) return s;
    }
    return LEAN_OK;
}


template <int FMT>
lean_status dequant_fmt(const Geom &g, const uint8_t *W, float *w, cudaStream_t stream) {
    SimtArgs a = {};
    a.W = W;
    a.s_off = g.s_off;
    a.N = (int)g.N;
    a.K = (int)g.K;
    a.qvec = (int)g.qvec;
    a.svec = (int)g.svec;
    a.steps = (int)((g.qvec + step_vecs<FMT>() - 1) / step_vecs<FMT>());
    a.groups = g.groups;
    const int64_t items = g.groups * a.steps;  // one warp each
    const int64_t blocks = (items + 7) / 8;
    if (blocks > INT32_MAX) return LEAN_ERR_SHAPE;
    dequant_kernel<FMT><<<(unsigned)blocks, 256, 0, stream>>>(a, w);
    return cudaGetLastError() == cudaSuccess ? LEAN_OK : LEAN_ERR_CUDA;
}


}  // namespace lean
