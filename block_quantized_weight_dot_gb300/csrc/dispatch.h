// dispatch.h -- what the C-ABI translation unit needs from the per-format
// kernel translation units (qmm_<fmt>.cu): problem descriptors, the workspace
// layout and the per-format entry templates.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lean_qmatmul.h"
#include "layout.h"

namespace lean {

constexpr int kMaxBatch = LEAN_MAX_BATCH;  // problems per batched launch
constexpr int kMaxStreamCtas = 512;        // CTAs of one streaming launch, at most
#ifndef LEAN_MMA_MIN_M
#define LEAN_MMA_MIN_M 16
#endif
constexpr int64_t kMmaMinM = LEAN_MMA_MIN_M;  // rows of x from which the tensor cores take over

struct HostProb {
    const uint8_t *W;
    const float *x;
    float *y;
    Geom g;
};

// Workspace of the balanced (stream-K) GEMV: per-CTA partial sums of the row
// groups split between CTAs (two sides x 16 groups x 32 rows), then one
// arrival counter per row group.
struct WorkspaceLayout {
    int64_t part_off, cnt_off, total;
};
inline WorkspaceLayout workspace_layout(int64_t groups) {
    WorkspaceLayout w;
    w.part_off = 0;
    w.cnt_off = (int64_t)kMaxStreamCtas * 2 * 16 * 32 * 4;
    w.total = (w.cnt_off + groups * 4 + 255) / 256 * 256;
    return w;
}

template <int FMT>
lean_status simt_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                     unsigned flags, cudaStream_t stream);
template <int FMT>
lean_status dequant_fmt(const Geom &g, const uint8_t *W, float *w, cudaStream_t stream);
template <int FMT>
lean_status mma_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                    unsigned flags, void *ws, int64_t ws_bytes, unsigned *err,
                    cudaStream_t stream);
template <int FMT>
lean_status stream_fmt(const HostProb *ph, int n, unsigned flags, void *ws, int64_t ws_bytes,
                       unsigned *err, cudaStream_t stream);

}  // namespace lean
