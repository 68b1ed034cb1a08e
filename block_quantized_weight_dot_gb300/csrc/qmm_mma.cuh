// qmm_mma.cuh -- the product for larger M on the fifth-generation tensor cores
// (tcgen05.mma with accumulators in tensor memory).
//
// With many rows of x the product is a dense contraction.  The pages' GPU
// path dequantizes weight tiles and multiplies them in f32 ("oxinfer" crate
// page, Platforms and accelerators: Browser (WebGPU)).  Here the tensor cores
// multiply the integer codes themselves and the block scales are applied
// afterwards, once per block and row of x:
//
//   y[m, n] = sum over scale groups g of  d[n, g] * D_g[n, m],
//   D_g[n, m] = sum over k in g of  c[n, k] * x[m, k],
//
// c the integer code (Q4_0 q - 8, the int8 formats q; Q6_K sc * (q - 32) with
// the super-block's d as the group scale).  Every code of Q4_0, Q8_0 and
// INT8-B64 is exact in bf16; Q6_K's sc * (q - 32) has up to 13 significant
// bits and is split exactly into two bf16 parts c_hi + c_lo.  x is split into
// bf16 x_hi + x_lo (x_lo rounded: below 2^-17 of |x|), so D_g takes two MMAs
// per 16-wide K step (c * x_hi, c * x_lo) -- three for Q6_K (c_hi * x_hi,
// c_hi * x_lo, c_lo * x_hi; the dropped c_lo * x_lo is below 2^-16 of |c x|).
// bf16 operands alone would miss the 1e-4 tolerance (one bf16 rounding of x
// is 2^-9 relative).
//
// Two kernels.  xsplit_kernel writes x once as bf16 hi / lo tiles already in
// the shared-memory operand layout, one contiguous piece per (64-row tile of
// x, 64-wide K block), into a caller workspace; without one, the converter
// warps split each CTA's x themselves.  qmm_mma_kernel computes one tile of
// 128 weight rows against up to 64 rows of x: tcgen05.mma of shape M = 128
// (weight rows) x N = mpad (rows of x padded to 16) x K = 16, A (the codes)
// and D in tensor memory, B (the split x) in shared memory.  Warp roles,
// oldest first (the scheduler favours older warps, and the single-lane roles
// pace the pipeline):
//   warps 0-3             MMA issuers (NI of them): each takes every NI-th
//                         scale group, into buffers of its own, and commits the
//                         group to its D buffer (d_full) and its stage to
//                         a_done, which frees the A stage and the B slot of the
//                         same index.  The whole warp runs the loop on
//                         warp-uniform values and one elected lane issues
//                         (about 94 cycles per MMA and issuing warp, whatever N).
//   warp 4 (one lane)     streams the packed weights with one TMA bulk copy
//                         per 32-row group and 256-wide K slot into a ring of
//                         raw slots (raw_full / raw_empty);
//   warp 5 (one lane)     with split x, copies each 64-wide K block of it into
//                         a ring of B slots (b_full);
//   warps 6-13            per scale group, read D_g (tcgen05.ld; 32 columns a
//                         warp, two warps per lane quarter), free the buffer
//                         (d_empty) and add d * D_g into fp32 registers; the
//                         scale comes from the raw slot, which these warps
//                         release too.  Up to 32 rows of x one set of four
//                         warps covers the columns, so the two sets take
//                         alternate groups and add their sums at the end;
//   warps 14-17           per two 64-wide K blocks ("stages"), turn the codes
//                         of one row each into bf16 and store them to
//                         tensor-memory A stages with tcgen05.st (a_full);
//                         without split x they also fill B.
// Tensor memory: four A stages of 32 * P columns at the top, D buffers of 32
// (up to 32 rows of x) or 64 columns below them.  Consumer barriers count
// warps (one elected arrival each), and waits sleep in try_wait rather than
// spin.  When the row tiles alone do not fill the GPU, a thread-block cluster
// of ks CTAs splits K on slot boundaries; each CTA leaves its partial y in
// shared memory and, after a cluster barrier, CTA r sums columns r*mpad/ks ..
// (r+1)*mpad/ks of all ks partials in rank order through distributed shared
// memory (deterministic, no atomics).  More than 64 rows of x take
// qmm_mma_wide.cuh.  Every wait is bounded; a timeout sets the device error
// word.
#pragma once
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "debug.cuh"
#include "decode.cuh"
#include "layout.h"
#include "ptx.cuh"
#include "qmm_simt.cuh"

namespace lean {

constexpr int kMmaRows = 128;          // weight rows per tile (MMA M)
constexpr int kMmaKB = 64;             // K per stage
constexpr int kMmaSlotK = 256;         // K per raw weight slot
constexpr int kMmaSub = kMmaSlotK / kMmaKB;  // stages per raw slot
// Warp roles, oldest first: the warp scheduler favours older warps, so the
// single-thread roles that pace the pipeline come before the bulk work
// (placed after it they were measured to wait ~100 cycles per instruction).
constexpr int kMmaIssuers = 4;         // warps 0-3: issue MMAs, scale groups round robin
constexpr int kMmaWProdWarp = 4;       // weight producer
constexpr int kMmaXProdWarp = 5;       // x producer
constexpr int kMmaEpiWarp0 = 6;        // warps 6-13: scale and accumulate
constexpr int kMmaConvWarp0 = 14;      // warps 14-17: convert codes
constexpr int kMmaConvThreads = 128;
constexpr int kMmaEpiThreads = 256;
constexpr int kMmaThreads = 576;
constexpr int kMmaMaxN = 64;           // rows of x per tile (MMA N)
constexpr int kMmaMaxSplit = 8;        // CTAs of a K-splitting cluster
constexpr int kMmaMaxRaw = 8;          // raw weight slots, at most
constexpr int kMmaStages = 4;          // tensor-memory A stages (and B stages, at most)
constexpr int kMmaMaxDBufs = 12;       // tensor-memory D buffers, at most
constexpr int kMmaSmemLimit = 227 * 1024;
constexpr uint32_t kMmaTmemCols = 512;  // D buffers from column 0, then the A stages
constexpr uint64_t kMmaWaitNs = 2000000000ull;
constexpr long long kMmaWaitCycles = 4000000000ll;  // about 2 s at the top SM clock
constexpr uint32_t kMmaSleepNs = 100000;            // longest sleep of one try

constexpr unsigned kErrMmaTimeout = 4u;

// Waits of the tensor-core kernel.  One non-blocking test first; then the
// thread sleeps in try_wait (woken by the phase) instead of spinning, so that
// waiting warps leave the issue slots to the converters and the epilogue.
// Gives up after about kMmaWaitNs, or once another thread of the CTA has
// given up; either way the CTA's abort flag is set and false returned.
static __device__ __noinline__ bool mma_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort_s) {
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kMmaSleepNs)) return true;
        if (*abort_s) return false;
        if (clock64() - t0 > kMmaWaitCycles) {
            *abort_s = 1;
            return false;
        }
    }
}
__device__ __forceinline__ bool mma_wait(uint64_t *bar, uint32_t parity, volatile int *abort_s) {
    return mbar_test_wait(bar, parity) || mma_wait_slow(bar, parity, abort_s);
}

// Per format: QV packed vectors of a raw slot per 32-row group (then the
// step's scale vector), G = K elements of one D buffer (one scale; Q6_K's
// super-block scale covers four of them), P = bf16 parts of a code.
//
// A scale group never spans stages: the issuers take alternate groups, and
// with G <= 64 each A stage and B slot is always read by the same issuer (both
// issuers for G = 32), so that no issuer skips a phase of their barriers.
template <int FMT> struct MmaFmt;
template <> struct MmaFmt<Q4_0> { static constexpr int QV = 8, G = 32, P = 1; };
template <> struct MmaFmt<Q8_0> { static constexpr int QV = 16, G = 32, P = 1; };
template <> struct MmaFmt<I8_B64> { static constexpr int QV = 16, G = 64, P = 1; };
template <> struct MmaFmt<Q6_K> { static constexpr int QV = 13, G = 64, P = 2; };

template <int FMT>
__host__ __device__ constexpr int mma_raw_group_bytes() {
    return (MmaFmt<FMT>::QV + 1) * kVecBytes;
}
template <int FMT>
__host__ __device__ constexpr int mma_raw_bytes() {
    return (kMmaRows / kRowsPerGroup) * mma_raw_group_bytes<FMT>();
}

// B stage: B_hi, B_lo (mpad x 64 bf16 each) in the layout of tile_off.
__host__ __device__ inline int mma_b_bytes(int mpad) { return mpad * kMmaKB * 2; }
// B stages: as many as the A stages (x comes from L2, and a slot is refilled
// only once its stage's MMAs are done; an even count keeps each slot with one
// issuer), 64 KiB at most; the K-split partials reuse the ring (2 stages hold
// 128 x mpad fp32).
__host__ __device__ inline int mma_b_stages(int) { return kMmaStages; }
// Shared memory: 1 KiB of barriers, the B ring, then the raw ring.
__host__ __device__ inline int mma_raw_off(int mpad) {
    return 1024 + mma_b_stages(mpad) * 2 * mma_b_bytes(mpad);
}
template <int FMT>
__host__ __device__ inline int mma_raw_slots(int mpad) {
    const int s = (kMmaSmemLimit - mma_raw_off(mpad)) / mma_raw_bytes<FMT>();
    return s < kMmaMaxRaw ? s : kMmaMaxRaw;
}
template <int FMT>
__host__ __device__ inline int mma_smem_bytes(int mpad, int raw_slots) {
    return mma_raw_off(mpad) + raw_slots * mma_raw_bytes<FMT>();
}

// Split x: for each 64-row tile t of x (mpad_t rows, padded to 16) and each
// 64-wide K block kb, 2 * mpad_t * 128 bytes: the hi tile then the lo tile,
// each in the operand layout of tile_off.  Tile t starts at t * xs_tile_bytes.
__host__ __device__ inline int64_t mma_xs_tile_bytes(int nkb) {
    return (int64_t)nkb * 2 * kMmaMaxN * kMmaKB * 2;
}
inline int64_t mma_xs_bytes(int64_t M, int64_t K) {
    const int nkb = (int)((K + kMmaKB - 1) / kMmaKB);
    const int64_t full = M / kMmaMaxN, rest = M % kMmaMaxN;
    const int64_t rest_pad = (rest + 15) / 16 * 16;
    return full * mma_xs_tile_bytes(nkb) + (int64_t)nkb * 2 * rest_pad * kMmaKB * 2;
}

struct MmaArgs {
    const uint8_t *W;   // packed weights
    const float *x;     // x[M][K]
    const uint8_t *xs;  // split x, or null
    float *y;           // y[M][N]
    int N, K, M;
    int ks;             // CTAs splitting K (cluster size)
    int nkb;            // 64-wide K blocks
    int nsl;            // 256-wide K slots
    int m_base;         // first row of x of this launch
    int RS;             // raw weight slots
    int raw_off;        // byte offset of the raw ring in shared memory
    int steps, last_blocks, step_vecs;
    int64_t groups;
    int64_t group_vecs;
    int64_t xs_bytes;   // bytes of the split x (0 without)
    unsigned *err;
    Magic mg;
};

struct XsplitArgs {
    const float *x;
    uint8_t *xs;
    int M, K, nkb;
    int mtiles;
    int64_t rows;  // padded rows over all tiles
    int64_t xs_bytes;
    unsigned *err;  // device error word (LEAN_DEBUG index checks)
};

// ---- tcgen05 wrappers ------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` once every MMA issued so far by this thread has completed
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
// 32 (16) consecutive fp32 columns of one tensor-memory lane per thread; the
// caller waits with tmem_wait_ld before using them
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 16 consecutive 32-bit columns of one tensor-memory lane per thread
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of
// 8 rows x 16 bytes stored as 128 contiguous bytes; LBO = stride between the
// two core matrices along K of one MMA (128 B), SBO = stride between 8-row
// groups (256 B); bits 46-48 hold the descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) |
           ((uint64_t)(256 >> 4) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9, 10-12 = 1), both K-major, N >> 3 in bits 17-22, M >> 4 in 24-28.
__device__ __forceinline__ uint32_t mma_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kMmaRows >> 4) << 24);
}

// Byte offset of element (row r, k) of an operand tile with `rows` rows,
// k in 0..63: [16-wide K step][8-row group][8-wide K core][row % 8][k % 8].
__host__ __device__ __forceinline__ uint32_t tile_off(int rows, int r, int k) {
    return (uint32_t)((k >> 4) * (rows * 32) + (r >> 3) * 256 + ((k >> 3) & 1) * 128 +
                      (r & 7) * 16 + (k & 7) * 2);
}

// ---- bf16 helpers -------------------------------------------------------------------
// bf16 hi / lo halves of two fp32 values, packed low element first
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 bh = __floats2bfloat162_rn(a, b);
    const float2 fh = __bfloat1622float2(bh);
    const __nv_bfloat162 bl = __floats2bfloat162_rn(a - fh.x, b - fh.y);
    hi = *reinterpret_cast<const uint32_t *>(&bh);
    lo = *reinterpret_cast<const uint32_t *>(&bl);
}
// the pair (a, b) of fp32 values exact in bf16, packed low element first
__device__ __forceinline__ uint32_t bf2_exact(f32x2 v) {
    const float2 f = unpack2(v);
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t *>(&b);
}
__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// split 8 fp32 values into bf16 hi / lo halves and store 16 bytes of each
__device__ __forceinline__ void split_store8(const float *v, uint8_t *hi, uint8_t *lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) split2(v[2 * i], v[2 * i + 1], h[i], l[i]);
    *reinterpret_cast<uint4 *>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

// ---- split x ------------------------------------------------------------------------
// One thread per 8 consecutive elements of a padded row (K fastest, so the
// reads are coalesced); rows past M and elements past K are zero.
static __global__ void __launch_bounds__(256) xsplit_kernel(const XsplitArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // x may come from the previous kernel on the stream
    const int64_t per_row = (int64_t)a.nkb * 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.rows * per_row) return;
    const int64_t m = i / per_row;
    const int p = (int)(i % per_row);
    const int t = (int)(m / kMmaMaxN), mm = (int)(m % kMmaMaxN);
    const int rest = a.M - t * kMmaMaxN;
    const int mpad = t == a.mtiles - 1 ? ((rest < kMmaMaxN ? rest : kMmaMaxN) + 15) & ~15 : kMmaMaxN;
    const int kb = p >> 3, k8 = p & 7;
    const int64_t k = (int64_t)kb * kMmaKB + 8 * k8;
    float v[8];
    if (m < a.M && k < a.K && LEAN_SPAN(m * a.K + k, 8, (int64_t)a.M * a.K, a.err)) {
        const float *src = a.x + m * a.K + k;
        const float4 p0 = __ldg(reinterpret_cast<const float4 *>(src));
        const float4 p1 = __ldg(reinterpret_cast<const float4 *>(src + 4));
        v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
        v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
    }
    uint8_t *piece = a.xs + t * mma_xs_tile_bytes(a.nkb) + (int64_t)kb * 2 * mma_b_bytes(mpad);
    const uint32_t off = tile_off(mpad, mm, 8 * k8);
    if (!LEAN_SPAN(piece + mma_b_bytes(mpad) + off - a.xs, 16, a.xs_bytes, a.err)) return;
    split_store8(v, piece + off, piece + mma_b_bytes(mpad) + off);
}

// ---- weights: packed vectors -> raw slot ------------------------------------------
// Bytes of global slot gs (K range 256*gs .. 256*gs+255) of one row group,
// and, when bar is given, the TMA copies that bring them into dst: the
// slot's quant vectors at 0, the step's scale vector at QV.
template <int FMT>
__device__ __forceinline__ uint32_t raw_copy(const MmaArgs &a, int64_t gi, int64_t gs,
                                             uint8_t *dst, uint64_t *bar) {
    constexpr int VPB = BlockTraits<FMT>::VPB, QV = MmaFmt<FMT>::QV;
    // step holding the slot and the slot's first block in it
    int64_t s;
    int i0;
    if (FMT == Q4_0 || FMT == Q8_0) {
        s = gs;
        i0 = 0;
    } else if (FMT == I8_B64) {
        s = gs >> 1;
        i0 = 4 * (int)(gs & 1);
    } else {
        s = gs >> 3;
        i0 = (int)(gs & 7);
    }
    const int nblk = s == a.steps - 1 ? a.last_blocks : 8;
    const int nb = FMT == Q4_0 || FMT == Q8_0 ? nblk : FMT == I8_B64 ? min(4, nblk - i0) : 1;
    const uint32_t qbytes = (uint32_t)(nb * VPB * kVecBytes);
    {
        // both copies inside the packed matrix (else neither is made and the
        // slot's barrier does not count their bytes)
        const int64_t wbytes = a.groups * a.group_vecs * kVecBytes;
        const int64_t sbase = (gi * a.group_vecs + s * a.step_vecs) * kVecBytes;
        const bool in_q = LEAN_SPAN(sbase + (int64_t)i0 * VPB * kVecBytes, qbytes, wbytes, bar ? a.err : nullptr);
        const bool in_s = LEAN_SPAN(sbase + (int64_t)nblk * VPB * kVecBytes, kVecBytes, wbytes,
                                    bar ? a.err : nullptr);
        if (!(in_q && in_s)) return 0u;
    }
    if (bar) {
        const uint8_t *step = a.W + (gi * a.group_vecs + s * a.step_vecs) * kVecBytes;
        if ((FMT == Q4_0 || FMT == Q8_0) && nb == 8) {
            // a whole step: quant vectors and the scale vector are contiguous
            bulk_g2s(dst, step, qbytes + kVecBytes, bar);
        } else {
            bulk_g2s(dst, step + i0 * VPB * kVecBytes, qbytes, bar);
            bulk_g2s(dst + QV * kVecBytes, step + nblk * VPB * kVecBytes, kVecBytes, bar);
        }
    }
    return qbytes + kVecBytes;
}

// Scale slot, in its step's scale vector, of the scale group holding element
// 32 * c of the row (c the 32-element chunk of the row; Q6_K: 256 * ...)
template <int FMT>
__device__ __forceinline__ int scale_slot(int64_t c) {
    return FMT == Q4_0 || FMT == Q8_0 ? (int)(c & 7) : FMT == I8_B64 ? (int)((c >> 1) & 7)
                                                                      : (int)((c >> 3) & 7);
}

// Codes of one row as bf16 pairs (low element first): the 32 elements
// 32*half .. 32*half+31 of stage `sub` (0..3) of the raw slot; rv points at
// the row's 16 bytes of its group's raw slot.  Q4_0 q - 8, the int8 formats
// q (exact); Q6_K sc * (q - 32) as hi + lo (exact: at most 13 bits).
template <int FMT>
__device__ __forceinline__ void conv_codes(const uint8_t *rv, int half, int sub, const Magic &mg,
                                           uint32_t magic16, uint32_t bias16, uint32_t (&hi)[16],
                                           uint32_t (&lo)[16]) {
    if (FMT == Q4_0) {
        // block 2*sub + half of the step is vector 2*sub + half; word t holds
        // elements 8t .. 8t+7, element 8t+i in bits 4i .. 4i+3.  Pair i of a
        // word: byte i of w (low nibble) and of w >> 4 (its high nibble), each
        // put under the bf16 exponent of 128 (0x4300 | q = 128 + q), then
        // 136 subtracted exactly.
        const uint4 v = *reinterpret_cast<const uint4 *>(rv + (2 * sub + half) * kVecBytes);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t w = word_of(v, t), w4 = w >> 4;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t r = byte_perm(w, w4, 0x4040u | (uint32_t)i | ((uint32_t)(4 + i) << 8));
                hi[4 * t + i] = bf2_sub(and_or(r, 0x000F000Fu, magic16), bias16);
            }
        }
    } else if (FMT == Q8_0 || FMT == I8_B64) {
        // Q8_0: block 2*sub + half, its vectors 0, 1; I8_B64: block sub, its
        // vectors 2*half, 2*half + 1 (vector j holds elements 16j .. 16j+15)
        const int v0 = FMT == Q8_0 ? 2 * (2 * sub + half) : 4 * sub + 2 * half;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const uint4 v = *reinterpret_cast<const uint4 *>(rv + (v0 + jj) * kVecBytes);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                f32x2 p[2];
                i8_word(word_of(v, t), mg, p);
                hi[8 * jj + 2 * t] = bf2_exact(p[0]);
                hi[8 * jj + 2 * t + 1] = bf2_exact(p[1]);
            }
        }
    } else {  // Q6_K: sub-blocks 4*sub + 2*half, +1 sit in words 12*sub + 6*half .. +5
        const uint4 va = *reinterpret_cast<const uint4 *>(rv + (3 * sub + half) * kVecBytes);
        const uint4 vb = *reinterpret_cast<const uint4 *>(rv + (3 * sub + half + 1) * kVecBytes);
        const uint4 vs = *reinterpret_cast<const uint4 *>(rv + 12 * kVecBytes);
        uint32_t wd[6];
        if (half == 0) {
            wd[0] = va.x; wd[1] = va.y; wd[2] = va.z; wd[3] = va.w; wd[4] = vb.x; wd[5] = vb.y;
        } else {
            wd[0] = va.z; wd[1] = va.w; wd[2] = vb.x; wd[3] = vb.y; wd[4] = vb.z; wd[5] = vb.w;
        }
        const uint32_t scw = word_of(vs, sub);
#pragma unroll
        for (int sb = 0; sb < 2; ++sb) {
            f32x2 q6[8];
            q6_group(wd[3 * sb], wd[3 * sb + 1], wd[3 * sb + 2], mg, q6);
            const float sc = i8_byte(scw, 2 * half + sb, mg);
            const f32x2 ss = pack2(sc, sc);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 c = unpack2(mul2(q6[j], ss));  // exact: |sc (q - 32)| <= 4096
                split2(c.x, c.y, hi[8 * sb + j], lo[8 * sb + j]);
            }
        }
    }
}

// ---- the product ----------------------------------------------------------------------
// grid = (ceil(N/128) * ks, tiles of x); cluster = (ks, 1, 1); 640 threads;
// dynamic shared memory mma_smem_bytes(mpad of a full tile, a.RS).
// PRESPLIT: x comes split by xsplit_kernel (a.xs) and is copied by warp 17;
// otherwise the converter warps also split the block's x (a.x).
template <int FMT, bool PRESPLIT>
__global__ void __launch_bounds__(kMmaThreads, 1) qmm_mma_kernel(const MmaArgs a) {
    namespace cg = cooperative_groups;
    constexpr int G = MmaFmt<FMT>::G, P = MmaFmt<FMT>::P;
    constexpr int GPS = kMmaKB / G;  // scale groups per stage
    constexpr int KPG = G / 16;      // 16-wide K steps of a group
    static_assert(G == 32 || G == kMmaKB, "a scale group is half a stage or one stage");
    constexpr int RAWG = mma_raw_group_bytes<FMT>();
    extern __shared__ __align__(1024) uint8_t msm[];
    uint64_t *raw_full = reinterpret_cast<uint64_t *>(msm);
    uint64_t *raw_empty = raw_full + kMmaMaxRaw;
    uint64_t *b_full = raw_empty + kMmaMaxRaw;
    uint64_t *a_full = b_full + kMmaStages;
    uint64_t *a_done = a_full + kMmaStages;
    uint64_t *d_full = a_done + kMmaStages;
    uint64_t *d_empty = d_full + kMmaMaxDBufs;
    uint64_t *done = d_empty + kMmaMaxDBufs;
    uint32_t *taddr_s = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_s = reinterpret_cast<volatile int *>(taddr_s + 1);
    uint8_t *bring = msm + 1024;
    uint8_t *rawring = msm + a.raw_off;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RS = a.RS;
    constexpr int BS = kMmaStages;
    static_assert(kMmaSub == 4 && kMmaStages == 4, "ring indices below use & 3");
    const int rank = (int)(blockIdx.x % (unsigned)a.ks);
    const int64_t n0 = (int64_t)(blockIdx.x / (unsigned)a.ks) * kMmaRows;
    const int tile = (int)blockIdx.y + a.m_base / kMmaMaxN;
    const int m0 = tile * kMmaMaxN;
    const int mt = min(kMmaMaxN, a.M - m0);
    const int mpad = (mt + 15) & ~15;
    const int bbytes = 2 * mma_b_bytes(mpad);
    // this CTA's K range: whole 256-wide slots sl0 .. sl0+nsl_c-1
    const int sl0 = (int)((int64_t)a.nsl * rank / a.ks);
    const int nsl_c = (int)((int64_t)a.nsl * (rank + 1) / a.ks) - sl0;
    const int kb0 = sl0 * kMmaSub;
    const int nk = min(a.nkb, (sl0 + nsl_c) * kMmaSub) - kb0;  // stages
    const int ng = nk * GPS;                                   // scale groups
    // Tensor memory: the A stages (32 * P columns each) at the top, D buffers
    // of 32 or 64 columns below.  Each of the NI issuers owns KD buffers and
    // takes every NI-th group; NI divides the groups of the A ring (8 or 4), so
    // every A stage, B slot and D buffer is always read by the same issuer and
    // no issuer skips a phase of their barriers.
    const uint32_t dstride = mpad <= 32 ? 32u : 64u;
    const uint32_t acol = kMmaTmemCols - kMmaStages * 32 * P;
    const int nD = (int)(acol / dstride);            // 12, 6 (Q6_K: 8, 4)
    const int NI = nD % 4 == 0 && nD >= 8 ? 4 : 2;   // issuers
    const int KD = nD / NI;                          // buffers per issuer
    const int64_t chunks = a.K / 32;  // 32-element chunks of a row
    // Up to 32 rows of x the columns fit one set of four epilogue warps: the
    // two sets then take alternate scale groups (each D buffer read by one
    // set) and add their sums at the end.
    const bool esplit = mpad <= 32;

    // Consumer barriers count warps: each warp synchronises and one lane
    // arrives (an arrival by every thread serialises hundreds of atomic
    // updates of one shared-memory word per stage).
    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], (kMmaConvThreads + kMmaEpiThreads) / 32);
        }
        for (int s = 0; s < BS; ++s) mbar_init(&b_full[s], PRESPLIT ? 1 : kMmaConvThreads / 32);
        for (int s = 0; s < kMmaStages; ++s) {
            mbar_init(&a_full[s], kMmaConvThreads / 32);
            mbar_init(&a_done[s], GPS);  // one commit per scale group of the stage
        }
        for (int b = 0; b < nD; ++b) {
            mbar_init(&d_full[b], 1);
            mbar_init(&d_empty[b], kMmaEpiThreads / 32 / (esplit ? 2 : 1));
        }
        mbar_init(done, NI);
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(taddr_s, kMmaTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_s;

    // partial y of this CTA: row 32 * (warp & 3) + lane, columns c0 .. c0+31
    // (plain fp32 FMAs on the loaded registers: pairing them for f32x2 FMAs
    // was measured to cost more in register moves than it saved)
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    const int c0 = 32 * ((warp - kMmaEpiWarp0) >> 2);

    // Ring positions are kept as counters (slot, parity of its current use):
    // raw slot r of use u is u % RS, and a use waits on the phase of the one
    // before it.  The A stages, B slots and D buffers are rings of 4.
    // Producer and issuer warps run their loops with all 32 lanes (one lane
    // issues the copies, MMAs and commits): a warp whose other lanes sat at
    // the final barrier meanwhile was measured to run its loop several times
    // slower.
    if (warp == kMmaWProdWarp) {
        // ---------------------------------------------------- weight producer
        int issued = 0, r = 0;
        uint32_t ph = 0;
        for (int u = 0; u < nsl_c; ++u) {
            if (u >= RS && !mma_wait(&raw_empty[r], ph ^ 1u, abort_s)) break;
            if (lane == 0) {
                uint8_t *slot = rawring + r * mma_raw_bytes<FMT>();
                const int64_t gs = sl0 + u;
                uint32_t bytes = 0;
                for (int g = 0; g < kMmaRows / kRowsPerGroup; ++g) {
                    const int64_t gi = n0 / kRowsPerGroup + g;
                    if (gi < a.groups) bytes += raw_copy<FMT>(a, gi, gs, nullptr, nullptr);
                }
                mbar_arrive_expect_tx(&raw_full[r], bytes);
                for (int g = 0; g < kMmaRows / kRowsPerGroup; ++g) {
                    const int64_t gi = n0 / kRowsPerGroup + g;
                    if (gi < a.groups) raw_copy<FMT>(a, gi, gs, slot + g * RAWG, &raw_full[r]);
                }
            }
            __syncwarp();
            issued = u + 1;
            if (++r == RS) {
                r = 0;
                ph ^= 1u;
            }
        }
        // copies still in flight after an abort land before the CTA exits
        if (lane == 0)
            for (int u = issued - RS > 0 ? issued - RS : 0; u < issued; ++u)
                mbar_wait(&raw_full[u % RS], (uint32_t)((u / RS) & 1), kMmaWaitNs);
    } else if (warp == kMmaXProdWarp) {
        // --------------------------------------------------------- x producer
        if (PRESPLIT) {
            const uint8_t *xs_tile = a.xs + tile * mma_xs_tile_bytes(a.nkb);
            int issued = 0;
            for (int j = 0; j < nk; ++j) {
                // slot j & 3 was last used by stage j - 4 (the A stage of the same index)
                const int s = j & 3;
                if (j >= BS && !mma_wait(&a_done[s], ((uint32_t)(j >> 2) & 1u) ^ 1u, abort_s)) break;
                if (lane == 0) {
                    const uint8_t *src = xs_tile + (int64_t)(kb0 + j) * bbytes;
                    const bool in = LEAN_SPAN(src - a.xs, bbytes, a.xs_bytes, a.err);
                    mbar_arrive_expect_tx(&b_full[s], in ? (uint32_t)bbytes : 0u);
                    if (j == 0) pdl_wait();  // the split x comes from the kernel before
                    if (in) bulk_g2s(bring + s * bbytes, src, (uint32_t)bbytes, &b_full[s]);
                }
                __syncwarp();
                issued = j + 1;
            }
            if (lane == 0)
                for (int j = issued - BS > 0 ? issued - BS : 0; j < issued; ++j)
                    mbar_wait(&b_full[j & 3], (uint32_t)((j >> 2) & 1), kMmaWaitNs);
        }
    } else if (warp < kMmaIssuers) {
        // -------------------------------------------------------- MMA issuers
        // The whole warp runs the loop on warp-uniform values and one elected
        // lane issues: a lone lane with per-thread operands was measured to
        // need about twice as long per MMA.
        const int iss = __shfl_sync(0xffffffffu, warp, 0);
        if (iss < NI) {
            const uint32_t idesc = mma_idesc(mpad);
            // descriptors advance by adding byte offsets / 16 to the address field
            const uint64_t bdesc0 = smem_desc(smem_addr(bring));
            const uint32_t b_lo16 = (uint32_t)mma_b_bytes(mpad) >> 4, kk16 = (uint32_t)(mpad * 32) >> 4;
            int bi = 0, use = 0;  // this issuer's buffer iss + NI * bi and its use count
            for (int gi = iss; gi < ng; gi += NI) {
                const int b = iss + NI * bi;
                if (use > 0 && !__all_sync(0xffffffffu, mma_wait(&d_empty[b], (uint32_t)(use - 1) & 1u,
                                                                 abort_s)))
                    break;
                // the group's stage and its 16-wide K steps there
                const int s = gi / GPS, kk0 = (gi % GPS) * KPG;
                const int sa = s & 3;
                const uint32_t par = (uint32_t)(s >> 2) & 1u;
                if (!__all_sync(0xffffffffu, mma_wait(&a_full[sa], par, abort_s) &&
                                                 mma_wait(&b_full[sa], par, abort_s)))
                    break;
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t td = tmem + dstride * b;
                    const uint32_t ta = tmem + acol + sa * 32 * P;
                    const uint64_t bh = bdesc0 + ((uint32_t)(sa * bbytes) >> 4);
#pragma unroll
                    for (int kq = 0; kq < KPG; ++kq) {
                        const int kk = kk0 + kq;
                        const uint64_t dh = bh + kk * kk16, dl = dh + b_lo16;
                        mma_bf16_ts(td, ta + 8 * kk, dh, idesc, kq > 0 ? 1u : 0u);
                        mma_bf16_ts(td, ta + 8 * kk, dl, idesc, 1u);
                        if (P == 2) mma_bf16_ts(td, ta + 32 + 8 * kk, dh, idesc, 1u);
                    }
                    mma_commit(&a_done[sa]);
                    mma_commit(&d_full[b]);
                }
                __syncwarp();
                if (++bi == KD) {
                    bi = 0;
                    ++use;
                }
            }
            // arrives when every MMA issued above has completed
            if (elect_one()) mma_commit(done);
            __syncwarp();
        }
    } else if (warp < kMmaConvWarp0) {
        // ------------------------------------------------ scale and accumulate
        const int row = 32 * (warp & 3) + lane;
        const int q = warp & 3;
        const bool row_live = n0 / kRowsPerGroup + q < a.groups;
        const int eset = c0 / 32;                        // this warp's set of four
        const int cl0 = esplit ? 0 : c0;                 // its first column
        const int ncol = min(32, mpad - cl0);            // 32 or 16
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        // this row's scale vector in raw slot 0
        const uint8_t *sv0 = rawring + q * RAWG + (row % kRowsPerGroup) * kVec + MmaFmt<FMT>::QV * kVecBytes;
        int r = 0;
        uint32_t ph = 0;
        bool live = true;
        int ie = 0, te = 0, ue = 0;  // group gi: issuer ie, its buffer te, use ue
        for (int j0 = 0; live && j0 < nk; j0 += kMmaSub) {
            if (!mma_wait(&raw_full[r], ph, abort_s)) break;
            const unsigned short *sv =
                reinterpret_cast<const unsigned short *>(sv0 + r * mma_raw_bytes<FMT>());
            const int jn = min(nk, j0 + kMmaSub);
            for (int j = j0; j < jn; ++j) {
#pragma unroll
                for (int h = 0; h < GPS; ++h) {
                    const int b = ie + NI * te;
                    const uint32_t dpar = (uint32_t)ue & 1u;
                    if (++ie == NI) {
                        ie = 0;
                        if (++te == KD) {
                            te = 0;
                            ++ue;
                        }
                    }
                    // split sets: the other set's group (its buffer is tracked above)
                    if (esplit && ((j * GPS + h) & 1) != eset) continue;
                    // first 32-element chunk of the group in the row, and its scale
                    const int64_t c = 2 * (int64_t)(kb0 + j) + h;
                    const float d = row_live && c < chunks ? h2f(sv[scale_slot<FMT>(c)]) : 0.f;
                    if (!mma_wait(&d_full[b], dpar, abort_s)) {
                        live = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t rr[32];
                    const uint32_t td = tmem + lane_base + dstride * b + (uint32_t)cl0;
                    if (ncol == 32) tmem_ld32(td, rr);
                    else if (ncol == 16) tmem_ld16(td, rr);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&d_empty[b]);
                    if (ncol == 32) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[i] = fmaf(d, __uint_as_float(rr[i]), acc[i]);
                    } else if (ncol == 16) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[i] = fmaf(d, __uint_as_float(rr[i]), acc[i]);
                    }
                }
                if (!live) break;
            }
            if (!live) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[r]);
            if (++r == RS) {
                r = 0;
                ph ^= 1u;
            }
        }
    } else {
        // -------------------------------------------------------- converters
        const Magic mg = pin_fmt<FMT>(a.mg);
        const uint32_t magic16 = pin32(0x43004300u), bias16 = pin32(0x43084308u);  // 128, 136
        const int ct = (int)threadIdx.x - 32 * kMmaConvWarp0;  // 0 .. 127
        // a warp reaches tensor-memory lanes 32 * (warp % 4) .. + 31 only
        const int row = 32 * (warp & 3) + lane;
        const int g = row / kRowsPerGroup;
        const bool row_live = n0 / kRowsPerGroup + g < a.groups;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        // this row's 16 bytes of raw slot 0
        const uint8_t *rv0 = rawring + g * RAWG + (row % kRowsPerGroup) * kVec;
        int r = 0;
        uint32_t ph = 0;
        // two stages per iteration (both in one raw slot), for more
        // independent work between the waits
        for (int j = 0; j < nk; j += 2) {
            const int sa = j & 3;  // A stage, B slot and stage within the raw slot alike
            const int ns = j + 1 < nk ? 2 : 1;
            if (sa == 0 && !mma_wait(&raw_full[r], ph, abort_s)) break;
            if (j >= kMmaStages) {
                const uint32_t pp = ((uint32_t)(j >> 2) & 1u) ^ 1u;
                if (!mma_wait(&a_done[sa], pp, abort_s) || (ns == 2 && !mma_wait(&a_done[sa + 1], pp, abort_s)))
                    break;
            }
            tc_fence_after();
            // each stage's 64 codes of the row, one half of 32 at a time
#pragma unroll
            for (int st = 0; st < 2; ++st) {
                if (st < ns) {
                    const int64_t kb = kb0 + j + st;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t hi[16], lo[16];
                        if (row_live && 2 * kb + half < chunks) {
                            conv_codes<FMT>(rv0 + r * mma_raw_bytes<FMT>(), half, sa + st, mg, magic16, bias16,
                                            hi, lo);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) hi[i] = lo[i] = 0u;
                        }
                        const uint32_t ta = tmem + lane_base + acol + (sa + st) * 32 * P + 16 * half;
                        tmem_st16(ta, hi);
                        if (P == 2) tmem_st16(ta + 32, lo);
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&a_full[sa]);
                if (ns == 2) mbar_arrive(&a_full[sa + 1]);
            }
            const int jl = j + ns - 1;  // last stage of this iteration
            if ((jl & 3) == kMmaSub - 1 || jl == nk - 1) {
                if (lane == 0) mbar_arrive(&raw_empty[r]);
                if (++r == RS) {
                    r = 0;
                    ph ^= 1u;
                }
            }
            if (!PRESPLIT) {
                if (j == 0) pdl_wait();  // x may come from the previous kernel on the stream
            }
            for (int st = 0; !PRESPLIT && st < ns; ++st) {
                // x of stage j + st into B slot sa + st, free since its a_done was
                // waited above: item i = (row m = i % mpad, 8-wide piece i / mpad);
                // all loads first, then the splits
                const int64_t kb = kb0 + j + st;
                constexpr int XI = kMmaMaxN * 8 / kMmaConvThreads;
                uint8_t *b_hi = bring + (sa + st) * bbytes;
                float4 xv[XI][2];
#pragma unroll
                for (int qq = 0; qq < XI; ++qq) {
                    const int i = ct + qq * kMmaConvThreads;
                    const int m = i % mpad;
                    const int64_t k = kb * kMmaKB + 8 * (i / mpad);
                    if (i < mpad * 8 && m < mt && k < a.K &&
                        LEAN_SPAN((int64_t)(m0 + m) * a.K + k, 8, (int64_t)a.M * a.K, a.err)) {
                        const float *src = a.x + (int64_t)(m0 + m) * a.K + k;
                        xv[qq][0] = __ldg(reinterpret_cast<const float4 *>(src));
                        xv[qq][1] = __ldg(reinterpret_cast<const float4 *>(src + 4));
                    } else {
                        xv[qq][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                        xv[qq][1] = xv[qq][0];
                    }
                }
#pragma unroll
                for (int qq = 0; qq < XI; ++qq) {
                    const int i = ct + qq * kMmaConvThreads;
                    if (i < mpad * 8) {
                        const float v[8] = {xv[qq][0].x, xv[qq][0].y, xv[qq][0].z, xv[qq][0].w,
                                            xv[qq][1].x, xv[qq][1].y, xv[qq][1].z, xv[qq][1].w};
                        const uint32_t off = tile_off(mpad, i % mpad, 8 * (i / mpad));
                        split_store8(v, b_hi + off, b_hi + mma_b_bytes(mpad) + off);
                    }
                }
                fence_async_smem();  // the tensor cores read what the generic proxy wrote
                __syncwarp();
                if (lane == 0) mbar_arrive(&b_full[sa + st]);
            }
        }
    }

    // ------------------------------------------------------------------ epilogue
    pdl_launch_dependents();  // the next kernel may start; it waits for our completion
    const bool epi = warp >= kMmaEpiWarp0 && warp < kMmaConvWarp0;
    bool fin = true;
    if (epi) fin = mbar_wait(done, 0u, kMmaWaitNs);
    const bool ok = __syncthreads_and(fin && !*abort_s) != 0;
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(a.err, kErrMmaTimeout);
        if (epi && !fin) mbar_wait(done, 0u, kMmaWaitNs);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    }
    tc_fence_after();
    if (esplit) {
        // the second set's sums join the first set's (first + second), through
        // the raw ring, which nothing reads any more
        float *S = reinterpret_cast<float *>(rawring);
        const int row = 32 * (warp & 3) + lane;
        if (epi && c0 == 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i) S[i * kMmaRows + row] = acc[i];
        }
        __syncthreads();
        if (epi && c0 == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] += S[i * kMmaRows + row];
        }
    }
    pdl_wait();  // y is written below
    const int64_t nq = n0 + 32 * (warp & 3) + lane;
    if (a.ks == 1) {
        if (epi && nq < a.N) {
            float *yc = a.y + (int64_t)(m0 + c0) * a.N + nq;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c0 + i < mt && LEAN_IN((int64_t)(m0 + c0 + i) * a.N + nq, (int64_t)a.M * a.N, a.err))
                    yc[(int64_t)i * a.N] = acc[i];
        }
    } else {
        // partial y of this CTA into shared memory, P[m][row] (the rings are
        // free: every MMA has completed and every copy has landed)
        float *Pm = reinterpret_cast<float *>(bring);
        if (epi) {
            const int row = 32 * (warp & 3) + lane;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c0 + i < mpad) Pm[(c0 + i) * kMmaRows + row] = acc[i];
        }
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();
        // this CTA's share of the columns, summed over the cluster in rank
        // order; item = (column m, 4 consecutive rows), all ranks' loads issued
        // before the sums
        {
            const int mlo = mpad * rank / a.ks, mhi = mpad * (rank + 1) / a.ks;
            const int items = (mhi - mlo) * (kMmaRows / 4);
            const float4 *Pr[kMmaMaxSplit];
#pragma unroll
            for (int r = 0; r < kMmaMaxSplit; ++r)
                Pr[r] = reinterpret_cast<const float4 *>(cl.map_shared_rank(Pm, r < a.ks ? r : 0));
            for (int it = threadIdx.x; it < items; it += kMmaThreads) {
                const int m = mlo + it / (kMmaRows / 4), r4 = it % (kMmaRows / 4);
                const int idx = m * (kMmaRows / 4) + r4;
                float4 v[kMmaMaxSplit];
#pragma unroll
                for (int r = 0; r < kMmaMaxSplit; ++r)
                    if (r < a.ks) v[r] = Pr[r][idx];
                float4 s = v[0];
#pragma unroll
                for (int r = 1; r < kMmaMaxSplit; ++r)
                    if (r < a.ks) {
                        s.x += v[r].x;
                        s.y += v[r].y;
                        s.z += v[r].z;
                        s.w += v[r].w;
                    }
                if (m < mt) {
                    float *yr = a.y + (int64_t)(m0 + m) * a.N;
                    const int64_t nr = n0 + 4 * r4, yo = (int64_t)(m0 + m) * a.N + nr, ye = (int64_t)a.M * a.N;
                    if (nr < a.N && LEAN_IN(yo, ye, a.err)) yr[nr] = s.x;
                    if (nr + 1 < a.N && LEAN_IN(yo + 1, ye, a.err)) yr[nr + 1] = s.y;
                    if (nr + 2 < a.N && LEAN_IN(yo + 2, ye, a.err)) yr[nr + 2] = s.z;
                    if (nr + 3 < a.N && LEAN_IN(yo + 3, ye, a.err)) yr[nr + 3] = s.w;
                }
            }
        }
        cl.sync();  // no CTA leaves while others read its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kMmaTmemCols);
}

}  // namespace lean
