// launch.cuh -- launch planning for the product kernels.  Included by one
// translation unit per weight format (qmm_<fmt>.cu), each of which
// instantiates the entry templates declared in dispatch.h.
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "../../include/lean_qmatmul.h"
#include "dispatch.h"
#include "layout.h"
#include "qmm_gemv.cuh"
#include "qmm_mma.cuh"
#include "qmm_mma_wide.cuh"
#include "qmm_simt.cuh"
#include "qmm_stream.cuh"

namespace lean {

constexpr int kMaxDevices = 64;
constexpr int kMaxWarpsPerCta = 16;
constexpr int kMaxCluster = 8;
constexpr size_t kMaxSimtSmem = 200 * 1024;

inline int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Per-device SM count, read once.
inline int sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Raise a kernel's dynamic shared memory limit once per device.
template <typename Kern>
inline bool ensure_smem(Kern kern, size_t bytes, std::atomic<uint64_t> &done) {
    if (bytes <= 48 * 1024) return true;
    const int dev = current_device();
    if (dev < 0) return false;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_relaxed) & bit) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
        return false;
    done.fetch_or(bit, std::memory_order_relaxed);
    return true;
}

inline void fill_launch(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int cluster,
                        unsigned flags) {
    int na = 0;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
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
}

// ------------------------------------------------------------ CUDA-core path ---

struct SimtPlan {
    int cl, rg, wpr;
    int64_t ctas;
    size_t smem;
    int xs_stride;
};

// Aim for about 16 resident warps per SM with every warp owning a run of
// blocks; split K over the warps of a CTA first, then over a cluster when x
// does not fit one CTA's shared memory or one CTA has too few warps.
template <int FMT>
bool plan_simt(const Geom &g, int mt, SimtPlan *p) {
    constexpr int E = BlockTraits<FMT>::E;
    const int64_t target = (int64_t)sm_count() * 16;
    int64_t want = (target + g.groups - 1) / g.groups;  // warps per row group
    want = std::max<int64_t>(1, std::min<int64_t>(want, g.blocks));
    const int64_t per_warp = (g.blocks + want - 1) / want;  // blocks per warp
    const int wtot = (int)((g.blocks + per_warp - 1) / per_warp);
    int cl = std::min(kMaxCluster, (wtot + kMaxWarpsPerCta - 1) / kMaxWarpsPerCta);
    auto slice_floats = [&](int c) { return (int)(((g.blocks + c - 1) / c) * E); };
    while (cl < kMaxCluster && (size_t)mt * slice_floats(cl) * 4 > kMaxSimtSmem / 2) ++cl;
    const int wpr = std::max(1, std::min(kMaxWarpsPerCta, (wtot + cl - 1) / cl));
    int rg = 1;
    while (rg * 2 * wpr <= 8 && rg * 2 <= g.groups) rg *= 2;
    const int xs_stride = slice_floats(cl);
    const size_t smem = (size_t)mt * xs_stride * 4 + (size_t)rg * wpr * mt * 32 * 4;
    if (smem > kMaxSimtSmem) return false;
    p->cl = cl;
    p->rg = rg;
    p->wpr = wpr;
    p->ctas = (g.groups + rg - 1) / rg * cl;
    p->smem = smem;
    p->xs_stride = xs_stride;
    return true;
}

inline SimtArgs simt_args(const Geom &g, const uint8_t *W, const float *x, float *y, int M) {
    SimtArgs a = {};
    a.W = W;
    a.x = x;
    a.y = y;
    a.N = (int)g.N;
    a.K = (int)g.K;
    a.M = M;
    a.groups = g.groups;
    a.blocks = g.blocks;
    a.steps = g.steps;
    a.last_blocks = g.last_blocks;
    a.step_vecs = g.step_vecs;
    a.group_vecs = g.group_vecs;
    a.mg = make_magic();
#ifdef LEAN_DEBUG
    a.err = error_word();
#endif
    return a;
}

template <int FMT, int MT>
lean_status launch_simt(const Geom &g, const uint8_t *W, const float *x, float *y, int M,
                        unsigned flags, cudaStream_t stream) {
    static std::atomic<uint64_t> smem_done{0};
    SimtPlan p;
    if (!plan_simt<FMT>(g, MT, &p)) return LEAN_ERR_SHAPE;
    if (p.ctas > INT32_MAX) return LEAN_ERR_SHAPE;
    SimtArgs a = simt_args(g, W, x, y, M);
    a.cl = p.cl;
    a.rg = p.rg;
    a.wpr = p.wpr;
    a.xs_stride = p.xs_stride;
    auto kern = qmm_simt_kernel<FMT, MT>;
    // the attribute is set once per device, to the most any plan asks for
    if (!ensure_smem(kern, kMaxSimtSmem, smem_done)) return LEAN_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)(32 * p.rg * p.wpr), 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    fill_launch(cfg, attr, p.cl, flags);
    return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? LEAN_OK : LEAN_ERR_CUDA;
}

template <int FMT>
lean_status simt_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                     unsigned flags, cudaStream_t stream) {
    // M rows of x in tiles of at most 8 (the library sends fewer rows than
    // the tensor-core switch, at most 8); each tile re-streams the weights
    for (int64_t m0 = 0; m0 < M; m0 += 8) {
        const int mt = (int)std::min<int64_t>(8, M - m0);
        const float *xt = x + m0 * g.K;
        float *yt = y + m0 * g.N;
        lean_status s;
        if (mt <= 2) s = launch_simt<FMT, 2>(g, W, xt, yt, mt, flags, stream);
        else if (mt <= 4) s = launch_simt<FMT, 4>(g, W, xt, yt, mt, flags, stream);
        else s = launch_simt<FMT, 8>(g, W, xt, yt, mt, flags, stream);
        if (s != LEAN_OK) return s;
    }
    return LEAN_OK;
}

template <int FMT>
lean_status dequant_fmt(const Geom &g, const uint8_t *W, float *w, cudaStream_t stream) {
    SimtArgs a = simt_args(g, W, nullptr, nullptr, 0);
    const int64_t items = g.groups * g.blocks;  // one warp each
    const int64_t blocks = (items + 7) / 8;
    if (blocks > INT32_MAX) return LEAN_ERR_SHAPE;
    dequant_kernel<FMT><<<(unsigned)blocks, 256, 0, stream>>>(a, w);
    return cudaGetLastError() == cudaSuccess ? LEAN_OK : LEAN_ERR_CUDA;
}

template <int FMT>
lean_status embed_fmt(const Geom &g, const uint8_t *W, const int32_t *ids, int64_t n_ids,
                      float *out, unsigned *err, cudaStream_t stream) {
    SimtArgs a = simt_args(g, W, nullptr, nullptr, 0);
    const int64_t items = n_ids * g.blocks;  // one thread each
    const int64_t blocks = (items + 255) / 256;
    if (blocks > INT32_MAX) return LEAN_ERR_SHAPE;
    embed_kernel<FMT><<<(unsigned)blocks, 256, 0, stream>>>(a, ids, n_ids, out, err);
    return cudaGetLastError() == cudaSuccess ? LEAN_OK : LEAN_ERR_CUDA;
}

// --------------------------------------------------------- tensor-core path ---


// Clusters of c CTAs of `kern` (one CTA per SM) that fit the GPU at once:
// cudaOccupancyMaxActiveClusters, which knows how the SMs are grouped (16
// row tiles in clusters of 8 did not all fit in one wave).  Read once per
// device and c; 0 when the query fails.
template <typename Kern>
inline int mma_active_clusters(Kern kern, int c, size_t smem, int threads) {
    static std::atomic<int> cache[kMaxDevices][kMmaMaxSplit + 1];
    const int dev = current_device();
    if (dev < 0 || c < 1 || c > kMmaMaxSplit) return 0;
    int v = cache[dev][c].load(std::memory_order_relaxed);
    if (v == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)c, 1, 1);
        cfg.blockDim = dim3((unsigned)threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess || v <= 0) {
            (void)cudaGetLastError();
            return 0;
        }
        cache[dev][c].store(v, std::memory_order_relaxed);
    }
    return v;
}

// K split of a tensor-core product: the cluster size c that minimises
// waves x (256-wide K slots per CTA + fixed + reduce when c > 1), in units of
// one slot's time, the waves counted from the clusters that fit at once.
// Constants from timing the Qwen2.5-3B FFN shapes (11008 x 2048 and 2048 x
// 11008) at every c: for the integer-code kernel (M = 16, 64) a CTA's fixed
// cost (start, epilogue) is about two slots and the cluster reduction 0.7;
// the split-weight kernel's slots cost about three times as much, so its
// fixed costs are smaller in slots (1 and 0.3).
template <typename ClusterFn>
inline int mma_split_clusters(int64_t tiles, int nsl, double fixed, double reduce, ClusterFn clusters) {
    int ks = 1;
    double best = 1e300;
    for (int c = 1; c <= kMmaMaxSplit && c <= nsl; ++c) {
        const int n = clusters(c);
        if (n <= 0) continue;
        const int64_t waves = (tiles + n - 1) / n;
        const double cost = (double)waves * ((nsl + c - 1) / c + fixed + (c > 1 ? reduce : 0.0));
        if (cost < best - 1e-9) {
            best = cost;
            ks = c;
        }
    }
    return ks;
}

// The tensor-core product for more than 64 rows of x (qmm_mma_wide.cuh):
// weights split on the CUDA cores, 256-row tiles of x.
template <int FMT>
lean_status mma_wide_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                    unsigned flags, void *ws, int64_t ws_bytes, unsigned *err,
                    cudaStream_t stream) {
    static std::atomic<uint64_t> smem_done{0}, smem_done_x{0};
    const int64_t tiles = (g.N + wide::kMmaRows - 1) / wide::kMmaRows;
    const int nkb = (int)((g.K + wide::kMmaKB - 1) / wide::kMmaKB);
    const int nsl = (nkb + wide::kMmaSub - 1) / wide::kMmaSub;
    const int64_t mtiles = (M + wide::kMmaMaxN - 1) / wide::kMmaMaxN;
    const int mpad = ((int)std::min<int64_t>(M, wide::kMmaMaxN) + 15) & ~15;
    const int RS = wide::mma_raw_slots<FMT>(mpad);
    const size_t smem = (size_t)wide::mma_smem_bytes<FMT>(mpad, RS);
    // one CTA per SM: the rings take most of the shared memory and all 512
    // tensor-memory columns are allocated
    if (RS < 1) return LEAN_ERR_SHAPE;
    const int64_t xs_bytes = wide::mma_xs_bytes(M, g.K);
    if (ws && ws_bytes < xs_bytes) return LEAN_ERR_SHAPE;
    uint8_t *xs = static_cast<uint8_t *>(ws);
    wide::MmaArgs a = {};
    a.W = W;
    a.x = x;
    a.xs = xs;
    a.y = y;
    a.N = (int)g.N;
    a.K = (int)g.K;
    a.M = (int)M;
    a.nkb = nkb;
    a.nsl = nsl;
    a.RS = RS;
    a.BS = wide::mma_b_stages(mpad);
    a.raw_off = wide::mma_raw_off(mpad);
    a.groups = g.groups;
    a.steps = g.steps;
    a.last_blocks = g.last_blocks;
    a.step_vecs = g.step_vecs;
    a.group_vecs = g.group_vecs;
    a.err = err;
    a.xs_bytes = xs ? xs_bytes : 0;
    a.mg = make_magic();
    if (xs) {
        // x -> bf16 hi / lo operand tiles, once
        wide::XsplitArgs xa;
        xa.x = x;
        xa.xs = xs;
        xa.M = (int)M;
        xa.K = (int)g.K;
        xa.nkb = nkb;
        xa.mtiles = (int)mtiles;
        xa.xs_bytes = xs_bytes;
        xa.err = err;
        xa.rows = (mtiles - 1) * wide::kMmaMaxN + (((M - (mtiles - 1) * wide::kMmaMaxN) + 15) & ~15);
        const int64_t blocks = (xa.rows * nkb * 8 + 255) / 256;
        if (blocks > INT32_MAX) return LEAN_ERR_SHAPE;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        fill_launch(cfg, attr, 1, flags);
        if (cudaLaunchKernelEx(&cfg, wide::xsplit_kernel, xa) != cudaSuccess) return LEAN_ERR_CUDA;
    }
    auto kern = xs ? wide::qmm_mma_kernel<FMT, true> : wide::qmm_mma_kernel<FMT, false>;
    std::atomic<uint64_t> &sd = xs ? smem_done : smem_done_x;
    if (!ensure_smem(kern, (size_t)wide::kMmaSmemLimit, sd)) return LEAN_ERR_CUDA;
    const int ks = mma_split_clusters(tiles * mtiles, nsl, 1.0, 0.3, [&](int c) {
        return mma_active_clusters(kern, c, smem, wide::kMmaThreads);
    });
    if (tiles * ks > INT32_MAX) return LEAN_ERR_SHAPE;
    a.ks = ks;
    for (int64_t t0 = 0; t0 < mtiles; t0 += 65535) {
        a.m_base = (int)(t0 * wide::kMmaMaxN);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim =
            dim3((unsigned)(tiles * ks), (unsigned)std::min<int64_t>(65535, mtiles - t0), 1);
        cfg.blockDim = dim3(wide::kMmaThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        // after the split kernel (which itself starts only when the caller's
        // flags allow) the launch is always programmatic
        fill_launch(cfg, attr, ks, xs ? (unsigned)LEAN_FLAG_EARLY_WEIGHTS : flags);
        if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return LEAN_ERR_CUDA;
    }
    return LEAN_OK;
}

template <int FMT>
lean_status mma_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                    unsigned flags, void *ws, int64_t ws_bytes, unsigned *err,
                    cudaStream_t stream) {
    // more than one 64-row tile of x: one weight conversion per 256 rows.
    // Q6_K and Q8_0 take it from 33 rows already: there the full epilogue of
    // the integer-code kernel (32 columns per warp and group) costs more than
    // the split weights' third MMA (measured: Q6_K 18992 x 2048, 48 rows,
    // 32.0 -> 29.7 us; Q4_0 and INT8-B64 at 11008 x 2048 and 2048 x 5632 lose).
    constexpr int64_t wide_from = (FMT == Q6_K || FMT == Q8_0) ? 32 : kMmaMaxN;
    if (M > wide_from) return mma_wide_fmt<FMT>(g, W, x, y, M, flags, ws, ws_bytes, err, stream);
    static std::atomic<uint64_t> smem_done{0}, smem_done_x{0};
    const int64_t tiles = (g.N + kMmaRows - 1) / kMmaRows;
    const int nkb = (int)((g.K + kMmaKB - 1) / kMmaKB);
    const int nsl = (nkb + kMmaSub - 1) / kMmaSub;
    const int64_t mtiles = (M + kMmaMaxN - 1) / kMmaMaxN;
    const int mpad = ((int)std::min<int64_t>(M, kMmaMaxN) + 15) & ~15;
    const int RS = mma_raw_slots<FMT>(mpad);
    const size_t smem = (size_t)mma_smem_bytes<FMT>(mpad, RS);
    if (RS < 1) return LEAN_ERR_SHAPE;
    const int64_t xs_bytes = mma_xs_bytes(M, g.K);
    if (ws && ws_bytes < xs_bytes) return LEAN_ERR_SHAPE;
    uint8_t *xs = static_cast<uint8_t *>(ws);
    MmaArgs a = {};
    a.W = W;
    a.x = x;
    a.xs = xs;
    a.y = y;
    a.N = (int)g.N;
    a.K = (int)g.K;
    a.M = (int)M;
    a.nkb = nkb;
    a.nsl = nsl;
    a.RS = RS;
    a.raw_off = mma_raw_off(mpad);
    a.groups = g.groups;
    a.steps = g.steps;
    a.last_blocks = g.last_blocks;
    a.step_vecs = g.step_vecs;
    a.group_vecs = g.group_vecs;
    a.err = err;
    a.xs_bytes = xs ? xs_bytes : 0;
    a.mg = make_magic();
    if (xs) {
        // x -> bf16 hi / lo operand tiles, once
        XsplitArgs xa;
        xa.x = x;
        xa.xs = xs;
        xa.M = (int)M;
        xa.K = (int)g.K;
        xa.nkb = nkb;
        xa.mtiles = (int)mtiles;
        xa.xs_bytes = xs_bytes;
        xa.err = err;
        xa.rows = (mtiles - 1) * kMmaMaxN + (((M - (mtiles - 1) * kMmaMaxN) + 15) & ~15);
        const int64_t blocks = (xa.rows * nkb * 8 + 255) / 256;
        if (blocks > INT32_MAX) return LEAN_ERR_SHAPE;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        fill_launch(cfg, attr, 1, flags);
        if (cudaLaunchKernelEx(&cfg, xsplit_kernel, xa) != cudaSuccess) return LEAN_ERR_CUDA;
    }
    auto kern = xs ? qmm_mma_kernel<FMT, true> : qmm_mma_kernel<FMT, false>;
    std::atomic<uint64_t> &sd = xs ? smem_done : smem_done_x;
    if (!ensure_smem(kern, (size_t)kMmaSmemLimit, sd)) return LEAN_ERR_CUDA;
    // one CTA per SM: the rings take most of the shared memory and all 512
    // tensor-memory columns are allocated
    const int ks = mma_split_clusters(tiles * mtiles, nsl, 2.0, 0.7, [&](int c) {
        return mma_active_clusters(kern, c, smem, kMmaThreads);
    });
    if (tiles * ks > INT32_MAX) return LEAN_ERR_SHAPE;
    a.ks = ks;
    for (int64_t t0 = 0; t0 < mtiles; t0 += 65535) {
        a.m_base = (int)(t0 * kMmaMaxN);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim =
            dim3((unsigned)(tiles * ks), (unsigned)std::min<int64_t>(65535, mtiles - t0), 1);
        cfg.blockDim = dim3(kMmaThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        // after the split kernel (which itself starts only when the caller's
        // flags allow) the launch is always programmatic
        fill_launch(cfg, attr, ks, xs ? (unsigned)LEAN_FLAG_EARLY_WEIGHTS : flags);
        if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return LEAN_ERR_CUDA;
    }
    return LEAN_OK;
}

// ------------------------------------------------------- one-wave M = 1 path ---

// CTAs of qmm_gemv_kernel<FMT, NP, false, 1> resident per SM (read once per device).
template <int FMT, int NP>
inline int gemv_ctas_per_sm() {
    static std::atomic<int> cache[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, qmm_gemv_kernel<FMT, NP, false, 1>,
                                                          kGemvThreads,
                                                          gemv_smem_bytes<FMT, 1>()) != cudaSuccess ||
            v <= 0)
            v = -1;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// The product on qmm_gemv_kernel for MT rows of x (M <= MT) when every
// problem's row fits a cluster of 8 CTAs; with one_wave, only when the whole
// grid also fits the GPU at once.  *done = false leaves the call to the other
// kernels.  SWIGLU: ph[0] gate, ph[1] up (n = 2), h = silu(g) * u.
template <int FMT, int NP, int MT, bool SWIGLU>
lean_status launch_gemv(const HostProb *ph, int n, int M, unsigned flags, bool one_wave,
                        cudaStream_t stream, bool *done) {
    constexpr int NB = gemv_nb<FMT, MT>();
    static std::atomic<uint64_t> smem_done{0};
    *done = false;
    int64_t maxb = 0, groups = 0;
    for (int i = 0; i < n; ++i) {
        maxb = std::max<int64_t>(maxb, ph[i].g.blocks);
        groups += ph[i].g.groups;
    }
    if (SWIGLU) groups = ph[0].g.groups;
    // the smallest K split for which every row's blocks fit 8 warps x NB
    const int ks = (int)((maxb + kGemvWarps * NB - 1) / (kGemvWarps * NB));
    const int cl = SWIGLU ? 2 * ks : ks;
    if (cl > kGemvMaxCluster) return SWIGLU ? LEAN_ERR_SHAPE : LEAN_OK;
    if (groups * cl > INT32_MAX) return LEAN_ERR_SHAPE;
    if (one_wave) {
        const int per_sm = gemv_ctas_per_sm<FMT, NP>();
        if (per_sm <= 0 || groups * cl > (int64_t)per_sm * sm_count()) return LEAN_OK;
    }
    auto kern = qmm_gemv_kernel<FMT, NP, SWIGLU, MT>;
    if (!ensure_smem(kern, (size_t)gemv_smem_bytes<FMT, MT>(), smem_done)) return LEAN_ERR_CUDA;
    GemvArgs<NP> a;
    a.nprob = n;
    a.cl = cl;
    a.M = M;
    a.pad = 0;
    a.err = nullptr;
#ifdef LEAN_DEBUG
    a.err = error_word();
#endif
    a.mg = make_magic();
    int cta = 0;
    for (int i = 0; i < n; ++i) {
        const Geom &g = ph[i].g;
        GemvProb &p = a.p[i];
        p.W = ph[i].W;
        p.x = SWIGLU ? ph[0].x : ph[i].x;
        p.y = SWIGLU ? ph[0].y : ph[i].y;
        p.N = (int)g.N;
        p.K = (int)g.K;
        p.blocks = (int)g.blocks;
        p.steps = g.steps;
        p.last_blocks = g.last_blocks;
        p.step_vecs = g.step_vecs;
        p.nbw = (int)((g.blocks + kGemvWarps * ks - 1) / (kGemvWarps * ks));
        p.cta0 = cta;
        p.group_vecs = g.group_vecs;
        if (!SWIGLU) cta += (int)g.groups * cl;
    }
    if (SWIGLU) cta = (int)groups * cl;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cta, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = gemv_smem_bytes<FMT, MT>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    fill_launch(cfg, attr, cl, flags);
    *done = true;
    return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? LEAN_OK : LEAN_ERR_CUDA;
}

// h = silu(W_gate x) * (W_up x) on the one-wave kernel (any number of waves):
// a cluster of 2 x (K split) CTAs per row group.  ph[0] gate, ph[1] up.
template <int FMT>
lean_status swiglu_fmt(const HostProb *ph, unsigned flags, cudaStream_t stream) {
    bool done = false;
    return launch_gemv<FMT, 2, 1, true>(ph, 2, 1, flags, false, stream, &done);
}

// M = 1: the one-wave kernel when the grid fits the GPU at once.
template <int FMT>
lean_status gemv_fmt(const HostProb *ph, int n, unsigned flags, cudaStream_t stream, bool *done) {
    if (n == 1) return launch_gemv<FMT, 1, 1, false>(ph, n, 1, flags, true, stream, done);
    if (n <= 8) return launch_gemv<FMT, 8, 1, false>(ph, n, 1, flags, true, stream, done);
    return launch_gemv<FMT, kMaxBatch, 1, false>(ph, n, 1, flags, true, stream, done);
}

// M = 2..8 rows of x on the same kernel (several waves allowed; the library
// sends it fewer rows than the tensor-core switch) when a row fits a cluster;
// *done = false leaves the call to the row-tiled CUDA-core kernel.
template <int FMT>
lean_status gemv_small_m_fmt(const HostProb &hp, int M, unsigned flags, cudaStream_t stream,
                             bool *done) {
    if (M <= 2) return launch_gemv<FMT, 1, 2, false>(&hp, 1, M, flags, false, stream, done);
    if (M <= 4) return launch_gemv<FMT, 1, 4, false>(&hp, 1, M, flags, false, stream, done);
    if (FMT == Q6_K) {  // its x slice would not fit for 8 rows or more
        *done = false;
        return LEAN_OK;
    }
    if (M <= 8) return launch_gemv<FMT, 1, 8, false>(&hp, 1, M, flags, false, stream, done);
    *done = false;
    return LEAN_OK;
}

// -------------------------------------------------------------- stream path ---

// Total row groups of a problem list; false when the list is too long.
inline bool stream_totals(const HostProb *ph, int n, int64_t *groups) {
    if (n < 1 || n > kMaxBatch) return false;
    int64_t gg = 0;
    for (int i = 0; i < n; ++i) gg += ph[i].g.groups;
    *groups = gg;
    return true;
}

// Set the variant's shared-memory limit once per device and launch it.
template <int FMT, int NP, bool PL>
lean_status launch_stream_kernel(const StreamArgs<NP> &a, unsigned kflags, cudaStream_t stream) {
    using L = StreamLayout<FMT, PL>;
    static std::atomic<uint64_t> smem_done{0};
    auto kern = qmm_stream_kernel<FMT, NP, PL>;
    if (!ensure_smem(kern, L::SMEM, smem_done)) return LEAN_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.ctas, 1, 1);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    fill_launch(cfg, attr, 1, kflags);
    return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? LEAN_OK : LEAN_ERR_CUDA;
}

// Run-time hand-out of whole group blocks: worth it when a batch has many more
// group blocks than CTAs, so that the last blocks taken are short.
constexpr int64_t kDynMinBlocksPerCta = 3;
// On the decode step one unit costs its consumer warps about as long as
// streaming this many bytes, on top of its own bytes (measured: the finish
// time of a CTA grew by ~0.7 us per unit and ~0.026 us per KB).
constexpr int64_t kUnitFixedBytes = 27 * 1024;

// Runs of group blocks in hand-out order, largest blocks first: for each
// problem its full group blocks (one run) and its last, partial block (a run of
// one), sorted by the cost of one block (bytes copied plus a fixed cost per
// unit); ties keep problem order.
template <int FMT, bool PL, int NP>
void dyn_runs(StreamArgs<NP> &a) {
    using C = StreamCfg<FMT>;
    using L = StreamLayout<FMT, PL>;
    auto unit_bytes = [](int64_t ng, int nbc) -> int64_t {
        const int64_t xb = (PL && XPlanes<FMT>::on) ? (int64_t)nbc * (C::E / 32) * kXqBytes
                                                    : (int64_t)nbc * C::E * 4;
        return ng * ((int64_t)nbc * C::VPB + 1) * kVecBytes + xb;
    };
    struct Run {
        int32_t code;
        int64_t count, cost;
    };
    Run runs[2 * NP];
    int nr = 0;
    for (int i = 0; i < a.nprob; ++i) {
        const StreamProb &p = a.p[i];
        const int last_nbc = p.last_blocks - ((p.last_blocks + C::BPC - 1) / C::BPC - 1) * C::BPC;
        auto block_cost = [&](int64_t ng) {
            return (p.chunks - 1) * unit_bytes(ng, C::BPC) + unit_bytes(ng, last_nbc) +
                   p.chunks * kUnitFixedBytes;
        };
        const int64_t full = p.groups / L::GPU, part = p.groups % L::GPU;
        if (full > 0) runs[nr++] = Run{i, full, block_cost(L::GPU)};
        if (part > 0) runs[nr++] = Run{i | (1 << 16), 1, block_cost(part)};
    }
    std::stable_sort(runs, runs + nr, [](const Run &x, const Run &y) { return x.cost > y.cost; });
    int64_t item = 0;
    for (int r = 0; r < nr; ++r) {
        a.run_prob[r] = runs[r].code;
        a.run_item0[r] = (int32_t)item;
        item += runs[r].count;
    }
    a.run_item0[nr] = (int32_t)item;
    a.nruns = nr;
}

template <int FMT, int NP>
lean_status launch_stream(const HostProb *ph, int n, unsigned flags, void *ws, int64_t ws_bytes,
                          bool planes, unsigned *err, cudaStream_t stream) {
    using C = StreamCfg<FMT>;
    using L = StreamLayout<FMT>;  // the ring geometry that both variants share
    StreamArgs<NP> a;
    a.nprob = n;
    a.pad = 0;
    int64_t units = 0, gblocks = 0, groups = 0;
    for (int i = 0; i < n; ++i) {
        const Geom &g = ph[i].g;
        StreamProb &p = a.p[i];
        p.W = ph[i].W;
        p.x = ph[i].x;
        p.y = ph[i].y;
        p.N = (int)g.N;
        p.K = (int)g.K;
        p.steps = g.steps;
        p.last_blocks = g.last_blocks;
        p.chunks = (g.steps - 1) * L::CPSTEP + (g.last_blocks + C::BPC - 1) / C::BPC;
        p.pad = 0;
        p.group_vecs = g.group_vecs;
        p.groups = g.groups;
        p.gblocks = (g.groups + L::GPU - 1) / L::GPU;
        p.unit0 = units;
        p.gblock0 = gblocks;
        p.group0 = groups;
        p.xq0 = 0;
        units += p.gblocks * p.chunks;
        gblocks += p.gblocks;
        groups += g.groups;
    }
    a.total_units = units;
    a.total_gblocks = gblocks;
    a.mg = make_magic();
    a.err = err;
    a.xq = nullptr;
    a.dyn = nullptr;
    a.nruns = 0;
    a.pad2 = 0;
    unsigned kflags = flags;
    bool use_planes = false;
    if (ws != nullptr) {
        // room for the x planes of every problem, back to back (the layout is
        // the one lean_*_workspace_bytes describe, planes used or not)
        int64_t xqb = 0, wbytes = 0;
        int max_nb = 0;
        if (planes && XPlanes<FMT>::on) {
            for (int i = 0; i < n; ++i) {
                a.p[i].xq0 = xqb;
                xqb += xq_bytes(FMT, ph[i].g.K);
                wbytes += ph[i].g.total;
                max_nb = std::max<int>(max_nb, (int)(ph[i].g.K / 32));
            }
        }
        use_planes = xqb > 0 && (wbytes >= kPlanesMinWeightBytes ||
                                 (flags & (LEAN_FLAG_X_PLANES | LEAN_FLAG_X_INT8)));
        const WorkspaceLayout wl = workspace_layout(groups, xqb, n > 1);
        if (ws_bytes < wl.total) return LEAN_ERR_SHAPE;
        const int cps = use_planes ? StreamRing<FMT, true>::CPS : StreamRing<FMT, false>::CPS;
        const int64_t slots = std::min<int64_t>((int64_t)sm_count() * cps, kMaxStreamCtas);
        a.balanced = 1;
        a.ctas = (int)std::max<int64_t>(1, std::min<int64_t>(slots, units));
        a.part = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + wl.part_off);
        a.cnt = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(ws) + wl.cnt_off);
        if (n > 1 && gblocks >= kDynMinBlocksPerCta * slots && gblocks <= INT32_MAX &&
            a.nprob <= 0xFFFF) {
            a.balanced = 3;
            a.ctas = (int)slots;
            a.dyn = a.cnt + groups;
            if (use_planes) dyn_runs<FMT, true>(a); else dyn_runs<FMT, false>(a);
        }
        if (use_planes) {
            XprepArgs<NP> xa;
            xa.nprob = n;
            xa.int8 = (flags & LEAN_FLAG_X_INT8) ? 1 : 0;
            xa.xq = static_cast<uint8_t *>(ws) + wl.xq_off;
            xa.xq_bytes = wl.cnt_off - wl.xq_off;
            xa.err = err;
            for (int i = 0; i < n; ++i) {
                xa.p[i].x = ph[i].x;
                xa.p[i].xq0 = a.p[i].xq0;
                xa.p[i].nb = (int)(ph[i].g.K / 32);
                xa.p[i].pad = 0;
            }
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)((max_nb + kXprepCtaBlocks - 1) / kXprepCtaBlocks),
                               (unsigned)n, 1);
            cfg.blockDim = dim3(256, 1, 1);
            cfg.stream = stream;
            cudaLaunchAttribute attr[2];
            fill_launch(cfg, attr, 1, flags & LEAN_FLAG_EARLY_WEIGHTS);
            if (cudaLaunchKernelEx(&cfg, xprep_kernel<FMT, NP>, xa) != cudaSuccess)
                return LEAN_ERR_CUDA;
            a.xq = xa.xq;
            // after the plane kernel (which itself starts only when the caller's
            // flags allow) the product is always launched programmatically
            kflags = LEAN_FLAG_EARLY_WEIGHTS;
        }
    } else {
        const int64_t slots =
            std::min<int64_t>((int64_t)sm_count() * StreamRing<FMT, false>::CPS, kMaxStreamCtas);
        a.balanced = 0;
        a.ctas = (int)std::max<int64_t>(1, std::min<int64_t>(slots, gblocks));
        a.part = nullptr;
        a.cnt = nullptr;
    }
    if (use_planes) return launch_stream_kernel<FMT, NP, true>(a, kflags, stream);
    return launch_stream_kernel<FMT, NP, false>(a, kflags, stream);
}

template <int FMT>
lean_status stream_fmt(const HostProb *ph, int n, unsigned flags, void *ws, int64_t ws_bytes,
                       bool planes, unsigned *err, cudaStream_t stream) {
    int64_t groups;
    if (!stream_totals(ph, n, &groups)) return LEAN_ERR_SHAPE;
    if (n == 1) return launch_stream<FMT, 1>(ph, n, flags, ws, ws_bytes, planes, err, stream);
    return launch_stream<FMT, kMaxBatch>(ph, n, flags, ws, ws_bytes, planes, err, stream);
}

}  // namespace lean

// explicit instantiation of a format's entry templates (use inside namespace lean)
#define LEAN_INSTANTIATE(FMT)                                                                  \
    template lean_status simt_fmt<FMT>(const Geom &, const uint8_t *, const float *, float *,  \
                                       int64_t, unsigned, cudaStream_t);                       \
    template lean_status dequant_fmt<FMT>(const Geom &, const uint8_t *, float *, cudaStream_t); \
    template lean_status embed_fmt<FMT>(const Geom &, const uint8_t *, const int32_t *, int64_t, \
                                        float *, unsigned *, cudaStream_t);                    \
    template lean_status stream_fmt<FMT>(const HostProb *, int, unsigned, void *, int64_t,     \
                                         bool, unsigned *, cudaStream_t);                      \
    template lean_status gemv_fmt<FMT>(const HostProb *, int, unsigned, cudaStream_t, bool *); \
    template lean_status swiglu_fmt<FMT>(const HostProb *, unsigned, cudaStream_t);              \
    template lean_status gemv_small_m_fmt<FMT>(const HostProb &, int, unsigned, cudaStream_t,    \
                                               bool *);                                           \
    template lean_status mma_fmt<FMT>(const Geom &, const uint8_t *, const float *, float *,   \
                                      int64_t, unsigned, void *, int64_t, unsigned *,          \
                                      cudaStream_t);
