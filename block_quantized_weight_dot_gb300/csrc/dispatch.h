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
// Rows of x from which the tensor cores take over, measured: the CUDA-core
// kernels cost about M times their one-row work (their M = 9..15 variant twice
// the M = 5..8 one), the tensor-core kernel is flat up to 64 rows (x rows are
// padded to 16).  At 9 rows it is ahead for every format and shape measured
// (1.2-2.5x); Q6_K, whose 6-bit fields are dear to decode on the CUDA cores,
// already from 5.
inline int64_t mma_min_m(int fmt) { return fmt == LEAN_Q6_K ? 5 : 9; }

struct HostProb {
    const uint8_t *W;
    const float *x;
    float *y;
    Geom g;
};

// Workspace of the balanced (stream-K) GEMV: per-CTA partial sums of the row
// groups split between CTAs (two sides x 16 groups x 32 rows), then x as
// integer planes (xq_bytes, may be 0), then one arrival counter per row group
// and, for a batch (handout), the two counters of the run-time hand-out of
// group blocks.
struct WorkspaceLayout {
    int64_t part_off, xq_off, cnt_off, total;
};
inline WorkspaceLayout workspace_layout(int64_t groups, int64_t xq_bytes = 0,
                                        bool handout = false) {
    WorkspaceLayout w;
    w.part_off = 0;
    w.xq_off = (int64_t)kMaxStreamCtas * 2 * 16 * 32 * 4;
    w.cnt_off = w.xq_off + (xq_bytes + 255) / 256 * 256;
    w.total = w.cnt_off + ((groups + (handout ? 2 : 0)) * 4 + 255) / 256 * 256;
    return w;
}
// x planes pay for their extra launch only when the call streams this many
// weight bytes or more (a single mid-size GEMV is bound by launch latency)
constexpr int64_t kPlanesMinWeightBytes = (int64_t)32 << 20;
// bytes of the x planes of one M = 1 product (0 for Q6_K, which takes fp32 x)
inline int64_t xq_bytes(int fmt, int64_t K) { return fmt == Q6_K ? 0 : K / 32 * kXqBlockBytes; }

template <int FMT>
lean_status simt_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                     unsigned flags, cudaStream_t stream);
template <int FMT>
lean_status dequant_fmt(const Geom &g, const uint8_t *W, float *w, cudaStream_t stream);
template <int FMT>
lean_status embed_fmt(const Geom &g, const uint8_t *W, const int32_t *ids, int64_t n_ids,
                      float *out, unsigned *err, cudaStream_t stream);
template <int FMT>
lean_status mma_fmt(const Geom &g, const uint8_t *W, const float *x, float *y, int64_t M,
                    unsigned flags, void *ws, int64_t ws_bytes, unsigned *err,
                    cudaStream_t stream);
// M = 1 on the one-wave kernel; *done = false when the problems do not fit it
template <int FMT>
lean_status gemv_fmt(const HostProb *ph, int n, unsigned flags, cudaStream_t stream, bool *done);
// M = 2..8 on the one-wave kernel; *done = false when a row does not fit it
template <int FMT>
lean_status gemv_small_m_fmt(const HostProb &hp, int M, unsigned flags, cudaStream_t stream,
                             bool *done);
// h = silu(W_gate x) * (W_up x); ph[0] gate (its x and y are the call's), ph[1] up
template <int FMT>
lean_status swiglu_fmt(const HostProb *ph, unsigned flags, cudaStream_t stream);
// planes: with a workspace, hand x to the integer formats as planes (dp4a)
template <int FMT>
lean_status stream_fmt(const HostProb *ph, int n, unsigned flags, void *ws, int64_t ws_bytes,
                       bool planes, unsigned *err, cudaStream_t stream);

// Device address of the library's error word on the current device (looked up
// once per device), or null.
unsigned *error_word();

// The M = 1 product with a workspace; planes = false keeps x in fp32 (the
// layout without a plane region, as the fixed array of lean_qmatmul_fixed_ws).
// clear_counters: once every argument has been checked, zero the arrival
// counters on the stream before the product (a rejected call queues nothing).
lean_status qmatmul_m1_ws(int fmt, const void *W, const float *x, float *y, int64_t N,
                          int64_t K, unsigned flags, void *ws, int64_t ws_bytes, bool planes,
                          bool clear_counters, cudaStream_t stream);

}  // namespace lean
