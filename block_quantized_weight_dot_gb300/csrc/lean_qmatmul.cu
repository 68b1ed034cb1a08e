// lean_qmatmul.cu -- C ABI entry points for the device calls: argument
// checks and dispatch by format.  The kernels and their launch planning live
// in one translation unit per format (qmm_<fmt>.cu).
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/lean_qmatmul.h"
#include "layout.h"

namespace lean {
template <int FMT>
lean_status qmm_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                    unsigned flags, cudaStream_t stream);
template <int FMT>
lean_status dequant_fmt(const Geom &g, const uint8_t *W, float *w, cudaStream_t stream);
}  // namespace lean

using namespace lean;

namespace {
bool aligned(const void *p, size_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
}  // namespace

extern "C" {

lean_status lean_qmatmul_ex(int fmt, const void *W_packed_dev, const float *x_dev, float *y_dev,
                            int64_t N, int64_t K, int64_t M, unsigned flags, void *stream) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    Geom g;
    if (M <= 0 || !make_geom(fmt, N, K, &g)) return LEAN_ERR_SHAPE;
    if (M > ((int64_t)1 << 31) / std::max<int64_t>(K, N)) return LEAN_ERR_SHAPE;
    if (!W_packed_dev || !x_dev || !y_dev) return LEAN_ERR_NULL;
    if (!aligned(W_packed_dev, 16) || !aligned(x_dev, 16) || !aligned(y_dev, 4)) return LEAN_ERR_ALIGN;
    if (flags & ~(unsigned)LEAN_FLAG_EARLY_WEIGHTS) return LEAN_ERR_FORMAT;
    cudaGetLastError();  // start from a clean error state
    const uint8_t *W = (const uint8_t *)W_packed_dev;
    cudaStream_t s = (cudaStream_t)stream;
    switch (fmt) {
    case LEAN_Q4_0: return qmm_fmt<Q4_0>(g, W, x_dev, y_dev, M, flags, s);
    case LEAN_Q8_0: return qmm_fmt<Q8_0>(g, W, x_dev, y_dev, M, flags, s);
    case LEAN_I8_B64: return qmm_fmt<I8_B64>(g, W, x_dev, y_dev, M, flags, s);
    case LEAN_Q6_K: return qmm_fmt<Q6_K>(g, W, x_dev, y_dev, M, flags, s);
    }
    return LEAN_ERR_FORMAT;
}

lean_status lean_qmatmul(int fmt, const void *W_packed_dev, const float *x_dev, float *y_dev,
                         int64_t N, int64_t K, int64_t M, void *stream) {
    return lean_qmatmul_ex(fmt, W_packed_dev, x_dev, y_dev, N, K, M, 0u, stream);
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

}  // extern "C"
