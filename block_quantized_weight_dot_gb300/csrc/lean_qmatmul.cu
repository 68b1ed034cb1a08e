// lean_qmatmul.cu -- C ABI entry points for the device calls: argument
// checks and dispatch by format and M.  The kernels and their launch
// planning live in one translation unit per format (qmm_<fmt>.cu).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "../../include/lean_qmatmul.h"
#include "dispatch.h"
#include "layout.h"
#include "qmm_mma.cuh"

using namespace lean;

// Device error word written by kernels whose bounded waits time out.
__device__ unsigned lean_error_word;

namespace {
constexpr unsigned kErrSelftest = 8u;

// One block waits on an mbarrier that nothing completes, for limit_ns.
__global__ void wait_selftest_kernel(unsigned *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const bool done = mbar_wait(&bar, 0u, limit_ns);
    if (__syncthreads_or(!done) && threadIdx.x == 0) atomicOr(err, kErrSelftest);
}
}  // namespace

namespace lean {

// Device address of the error word on the current device (looked up once).
unsigned *error_word() {
    static std::atomic<unsigned *> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    unsigned *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, lean_error_word) != cudaSuccess) return nullptr;
        p = static_cast<unsigned *>(a);
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace lean

namespace {

bool aligned(const void *p, size_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

template <int FMT>
lean_status run_stream(const HostProb *ph, int n, unsigned flags, void *ws, int64_t wsb,
                       bool planes, cudaStream_t s) {
    unsigned *err = error_word();
    if (!err) return LEAN_ERR_CUDA;
    return stream_fmt<FMT>(ph, n, flags, ws, wsb, planes, err, s);
}

lean_status dispatch_stream(int fmt, const HostProb *ph, int n, unsigned flags, void *ws,
                            int64_t wsb, bool planes, cudaStream_t s) {
    switch (fmt) {
    case LEAN_Q4_0: return run_stream<Q4_0>(ph, n, flags, ws, wsb, planes, s);
    case LEAN_Q8_0: return run_stream<Q8_0>(ph, n, flags, ws, wsb, planes, s);
    case LEAN_I8_B64: return run_stream<I8_B64>(ph, n, flags, ws, wsb, planes, s);
    case LEAN_Q6_K: return run_stream<Q6_K>(ph, n, flags, ws, wsb, planes, s);
    }
    return LEAN_ERR_FORMAT;
}

// M = 1: the one-wave kernel when the problems fit it, unless the caller asks
// for the streaming kernel or the call takes x as integer planes (with a
// workspace, Q4_0 / Q8_0 / I8_B64, LEAN_FLAG_X_PLANES or >= 32 MiB of weights);
// otherwise the streaming kernel.
lean_status dispatch_m1(int fmt, const HostProb *ph, int n, unsigned flags, void *ws,
                        int64_t wsb, cudaStream_t s) {
    int64_t wbytes = 0, groups = 0, xqb = 0;
    for (int i = 0; i < n; ++i) {
        wbytes += ph[i].g.total;
        groups += ph[i].g.groups;
        xqb += xq_bytes(fmt, ph[i].g.K);
    }
    // a workspace smaller than the size query gives is refused whichever
    // kernel runs
    if (ws && wsb < workspace_layout(groups, xqb, n > 1).total) return LEAN_ERR_SHAPE;
    if (flags & LEAN_FLAG_X_INT8) {  // x quantized to int8: needs the planes' workspace
        if (fmt == LEAN_Q6_K) return LEAN_ERR_FORMAT;
        if (!ws) return LEAN_ERR_NULL;
    }
    const bool planes = ws && fmt != LEAN_Q6_K &&
                        ((flags & (LEAN_FLAG_X_PLANES | LEAN_FLAG_X_INT8)) ||
                         wbytes >= kPlanesMinWeightBytes);
    if (!(flags & LEAN_FLAG_STREAM) && !planes) {
        bool done = false;
        lean_status st = LEAN_OK;
        switch (fmt) {
        case LEAN_Q4_0: st = gemv_fmt<Q4_0>(ph, n, flags, s, &done); break;
        case LEAN_Q8_0: st = gemv_fmt<Q8_0>(ph, n, flags, s, &done); break;
        case LEAN_I8_B64: st = gemv_fmt<I8_B64>(ph, n, flags, s, &done); break;
        case LEAN_Q6_K: st = gemv_fmt<Q6_K>(ph, n, flags, s, &done); break;
        }
        if (done || st != LEAN_OK) return st;
    }
    return dispatch_stream(fmt, ph, n, flags, ws, wsb, true, s);
}

lean_status check_product(int fmt, const void *W, const float *x, const float *y, int64_t N,
                          int64_t K, int64_t M, unsigned flags, Geom *g) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    if (M <= 0 || !make_geom(fmt, N, K, g)) return LEAN_ERR_SHAPE;
    if (M > ((int64_t)1 << 31) / std::max<int64_t>(K, N)) return LEAN_ERR_SHAPE;
    if (!W || !x || !y) return LEAN_ERR_NULL;
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4)) return LEAN_ERR_ALIGN;
    if (flags & ~(unsigned)(LEAN_FLAG_EARLY_WEIGHTS | LEAN_FLAG_X_PLANES | LEAN_FLAG_STREAM |
                            LEAN_FLAG_X_INT8))
        return LEAN_ERR_FORMAT;
    if ((flags & LEAN_FLAG_X_INT8) && M != 1) return LEAN_ERR_FORMAT;
    return LEAN_OK;
}

}  // namespace

namespace lean {
lean_status qmatmul_m1_ws(int fmt, const void *W, const float *x, float *y, int64_t N,
                          int64_t K, unsigned flags, void *ws, int64_t ws_bytes, bool planes,
                          bool clear_counters, cudaStream_t stream) {
    Geom g;
    lean_status st = check_product(fmt, W, x, y, N, K, 1, flags, &g);
    if (st != LEAN_OK) return st;
    if (!ws || !aligned(ws, 256)) return ws ? LEAN_ERR_ALIGN : LEAN_ERR_NULL;
    const WorkspaceLayout wl = workspace_layout(g.groups, planes ? xq_bytes(fmt, K) : 0);
    if (ws_bytes < wl.total) return LEAN_ERR_SHAPE;
    cudaGetLastError();
    // every argument is valid: only now may anything be queued on the stream
    if (clear_counters &&
        cudaMemsetAsync(static_cast<uint8_t *>(ws) + wl.cnt_off, 0, (size_t)(g.groups * 4),
                        stream) != cudaSuccess)
        return LEAN_ERR_CUDA;
    HostProb hp = {(const uint8_t *)W, x, y, g};
    return dispatch_stream(fmt, &hp, 1, flags, ws, ws_bytes, planes, stream);
}
}  // namespace lean

extern "C" {

lean_status lean_qmatmul_ws(int fmt, const void *W_packed_dev, const float *x_dev, float *y_dev,
                            int64_t N, int64_t K, int64_t M, unsigned flags, void *workspace,
                            int64_t workspace_bytes, void *stream) {
    Geom g;
    lean_status st = check_product(fmt, W_packed_dev, x_dev, y_dev, N, K, M, flags, &g);
    if (st != LEAN_OK) return st;
    if (workspace && !aligned(workspace, 256)) return LEAN_ERR_ALIGN;
    cudaGetLastError();  // start from a clean error state
    const uint8_t *W = (const uint8_t *)W_packed_dev;
    cudaStream_t s = (cudaStream_t)stream;
    if (M == 1) {
        HostProb hp = {W, x_dev, y_dev, g};
        return dispatch_m1(fmt, &hp, 1, flags, workspace, workspace_bytes, s);
    }
    if (M >= mma_min_m(fmt)) {
        unsigned *err = error_word();
        if (!err) return LEAN_ERR_CUDA;
        void *ws = workspace;
        const int64_t wsb = workspace_bytes;
        switch (fmt) {
        case LEAN_Q4_0: return mma_fmt<Q4_0>(g, W, x_dev, y_dev, M, flags, ws, wsb, err, s);
        case LEAN_Q8_0: return mma_fmt<Q8_0>(g, W, x_dev, y_dev, M, flags, ws, wsb, err, s);
        case LEAN_I8_B64: return mma_fmt<I8_B64>(g, W, x_dev, y_dev, M, flags, ws, wsb, err, s);
        case LEAN_Q6_K: return mma_fmt<Q6_K>(g, W, x_dev, y_dev, M, flags, ws, wsb, err, s);
        }
        return LEAN_ERR_FORMAT;
    }
    {  // fewer rows: the one-wave kernel when a row fits a cluster of it
        HostProb hp = {W, x_dev, y_dev, g};
        bool done = false;
        lean_status st2 = LEAN_OK;
        if (!(flags & LEAN_FLAG_STREAM)) {
            switch (fmt) {
            case LEAN_Q4_0: st2 = gemv_small_m_fmt<Q4_0>(hp, (int)M, flags, s, &done); break;
            case LEAN_Q8_0: st2 = gemv_small_m_fmt<Q8_0>(hp, (int)M, flags, s, &done); break;
            case LEAN_I8_B64: st2 = gemv_small_m_fmt<I8_B64>(hp, (int)M, flags, s, &done); break;
            case LEAN_Q6_K: st2 = gemv_small_m_fmt<Q6_K>(hp, (int)M, flags, s, &done); break;
            }
        }
        if (done || st2 != LEAN_OK) return st2;
    }
    switch (fmt) {
    case LEAN_Q4_0: return simt_fmt<Q4_0>(g, W, x_dev, y_dev, M, flags, s);
    case LEAN_Q8_0: return simt_fmt<Q8_0>(g, W, x_dev, y_dev, M, flags, s);
    case LEAN_I8_B64: return simt_fmt<I8_B64>(g, W, x_dev, y_dev, M, flags, s);
    case LEAN_Q6_K: return simt_fmt<Q6_K>(g, W, x_dev, y_dev, M, flags, s);
    }
    return LEAN_ERR_FORMAT;
}

lean_status lean_qmatmul_ex(int fmt, const void *W_packed_dev, const float *x_dev, float *y_dev,
                            int64_t N, int64_t K, int64_t M, unsigned flags, void *stream) {
    return lean_qmatmul_ws(fmt, W_packed_dev, x_dev, y_dev, N, K, M, flags, nullptr, 0, stream);
}

lean_status lean_qmatmul(int fmt, const void *W_packed_dev, const float *x_dev, float *y_dev,
                         int64_t N, int64_t K, int64_t M, void *stream) {
    return lean_qmatmul_ws(fmt, W_packed_dev, x_dev, y_dev, N, K, M, 0u, nullptr, 0, stream);
}

int lean_tensor_core_min_m(int fmt) { return lean_block_elems(fmt) > 0 ? (int)mma_min_m(fmt) : -1; }

int64_t lean_qmatmul_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t M) {
    Geom g;
    if (M <= 0 || !make_geom(fmt, N, K, &g)) return -1;
    if (M >= mma_min_m(fmt)) return mma_xs_bytes(M, K);
    if (M > 1) return 0;
    return workspace_layout(g.groups, xq_bytes(fmt, K)).total;
}

int64_t lean_batch_workspace_bytes(int fmt, int count, const lean_problem *problems) {
    if (count < 1 || count > LEAN_MAX_BATCH || !problems) return -1;
    int64_t groups = 0, xqb = 0;
    for (int i = 0; i < count; ++i) {
        Geom g;
        if (!make_geom(fmt, problems[i].N, problems[i].K, &g)) return -1;
        groups += g.groups;
        xqb += xq_bytes(fmt, problems[i].K);
    }
    return workspace_layout(groups, xqb, count > 1).total;
}

lean_status lean_qmatmul_batch(int fmt, int count, const lean_problem *problems, unsigned flags,
                               void *workspace, int64_t workspace_bytes, void *stream) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    if (count < 1 || count > LEAN_MAX_BATCH) return LEAN_ERR_SHAPE;
    if (!problems) return LEAN_ERR_NULL;
    if (workspace && !aligned(workspace, 256)) return LEAN_ERR_ALIGN;
    HostProb hp[LEAN_MAX_BATCH];
    for (int i = 0; i < count; ++i) {
        const lean_problem &p = problems[i];
        lean_status st = check_product(fmt, p.W, p.x, p.y, p.N, p.K, 1, flags, &hp[i].g);
        if (st != LEAN_OK) return st;
        hp[i].W = (const uint8_t *)p.W;
        hp[i].x = p.x;
        hp[i].y = p.y;
    }
    cudaGetLastError();
    return dispatch_m1(fmt, hp, count, flags, workspace, workspace_bytes, (cudaStream_t)stream);
}

lean_status lean_dequant(int fmt, const void *W_packed_dev, float *w_dev, int64_t N, int64_t K,
                         void *stream) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    Geom g;
    if (!make_geom(fmt, N, K, &g)) return LEAN_ERR_SHAPE;
    if (!W_packed_dev || !w_dev) return LEAN_ERR_NULL;
    if (!aligned(W_packed_dev, 16) || !aligned(w_dev, 16)) return LEAN_ERR_ALIGN;
    cudaGetLastError();
    const uint8_t *W = (const uint8_t *)W_packed_dev;
    cudaStream_t s = (cudaStream_t)stream;
    switch (fmt) {
    case LEAN_Q4_0: return dequant_fmt<Q4_0>(g, W, w_dev, s);
    case LEAN_Q8_0: return dequant_fmt<Q8_0>(g, W, w_dev, s);
    case LEAN_I8_B64: return dequant_fmt<I8_B64>(g, W, w_dev, s);
    case LEAN_Q6_K: return dequant_fmt<Q6_K>(g, W, w_dev, s);
    }
    return LEAN_ERR_FORMAT;
}

lean_status lean_embed_rows(int fmt, const void *W_packed_dev, const int32_t *ids_dev,
                            float *out_dev, int64_t n_ids, int64_t N, int64_t K, void *stream) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    Geom g;
    if (n_ids <= 0 || !make_geom(fmt, N, K, &g)) return LEAN_ERR_SHAPE;
    if (n_ids > ((int64_t)1 << 40) / K) return LEAN_ERR_SHAPE;
    if (!W_packed_dev || !ids_dev || !out_dev) return LEAN_ERR_NULL;
    if (!aligned(W_packed_dev, 16) || !aligned(ids_dev, 4) || !aligned(out_dev, 16))
        return LEAN_ERR_ALIGN;
    unsigned *err = error_word();
    if (!err) return LEAN_ERR_CUDA;
    cudaGetLastError();
    const uint8_t *W = (const uint8_t *)W_packed_dev;
    cudaStream_t s = (cudaStream_t)stream;
    switch (fmt) {
    case LEAN_Q4_0: return embed_fmt<Q4_0>(g, W, ids_dev, n_ids, out_dev, err, s);
    case LEAN_Q8_0: return embed_fmt<Q8_0>(g, W, ids_dev, n_ids, out_dev, err, s);
    case LEAN_I8_B64: return embed_fmt<I8_B64>(g, W, ids_dev, n_ids, out_dev, err, s);
    case LEAN_Q6_K: return embed_fmt<Q6_K>(g, W, ids_dev, n_ids, out_dev, err, s);
    }
    return LEAN_ERR_FORMAT;
}

lean_status lean_qmatmul_swiglu(int fmt, const void *W_gate_dev, const void *W_up_dev,
                                const float *x_dev, float *h_dev, int64_t N, int64_t K,
                                unsigned flags, void *stream) {
    HostProb hp[2];
    lean_status st = check_product(fmt, W_gate_dev, x_dev, h_dev, N, K, 1, flags, &hp[0].g);
    if (st != LEAN_OK) return st;
    st = check_product(fmt, W_up_dev, x_dev, h_dev, N, K, 1, flags, &hp[1].g);
    if (st != LEAN_OK) return st;
    if (flags & ~(unsigned)LEAN_FLAG_EARLY_WEIGHTS) return LEAN_ERR_FORMAT;
    hp[0].W = (const uint8_t *)W_gate_dev;
    hp[1].W = (const uint8_t *)W_up_dev;
    hp[0].x = hp[1].x = x_dev;
    hp[0].y = hp[1].y = h_dev;
    cudaGetLastError();
    cudaStream_t s = (cudaStream_t)stream;
    switch (fmt) {
    case LEAN_Q4_0: return swiglu_fmt<Q4_0>(hp, flags, s);
    case LEAN_Q8_0: return swiglu_fmt<Q8_0>(hp, flags, s);
    case LEAN_I8_B64: return swiglu_fmt<I8_B64>(hp, flags, s);
    case LEAN_Q6_K: return swiglu_fmt<Q6_K>(hp, flags, s);
    }
    return LEAN_ERR_FORMAT;
}

lean_status lean_wait_selftest(unsigned limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 1000000) return LEAN_ERR_SHAPE;
    unsigned *err = error_word();
    if (!err) return LEAN_ERR_CUDA;
    cudaGetLastError();
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, (uint64_t)limit_us * 1000u);
    return cudaGetLastError() == cudaSuccess ? LEAN_OK : LEAN_ERR_CUDA;
}

lean_status lean_device_status(int clear) {
    const unsigned v = lean_device_error(clear);
    if (v == 0xFFFFFFFFu) return LEAN_ERR_CUDA;
    if (v & kErrBounds) return LEAN_ERR_KERNEL_BOUNDS;
    return v ? LEAN_ERR_DEVICE : LEAN_OK;
}

int lean_debug_build(void) {
#ifdef LEAN_DEBUG
    return 1;
#else
    return 0;
#endif
}

unsigned lean_device_error(int clear) {
    unsigned v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return 0xFFFFFFFFu;
    if (cudaMemcpyFromSymbol(&v, lean_error_word, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    if (clear && v) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(lean_error_word, &zero, sizeof(zero)) != cudaSuccess)
            return 0xFFFFFFFFu;
    }
    return v;
}

}  // extern "C"
