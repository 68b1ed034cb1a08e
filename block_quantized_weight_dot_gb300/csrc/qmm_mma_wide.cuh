// qmm_mma_wide.cuh -- the tensor-core product for more than 64 rows of x.
//
// Weights are dequantized (codes times the block scale) and split into bf16
// hi + lo on the CUDA cores, x into bf16 hi + lo, and three MMAs per 16-wide
// K step accumulate w_hi*x_hi + w_hi*x_lo + w_lo*x_hi into one fp32
// accumulator for the whole K range ("oxinfer" crate page, Platforms and
// accelerators: Browser (WebGPU), dequantized tiles in f32).  The dropped
// w_lo*x_lo and the rounding of x_lo (and of w_lo for the formats whose
// dequantized weights need more than 16 bits) are each below 2^-16 of |w*x|;
// for Q4_0 the weight split is exact, since d*(q-8) has at most 15
// significant bits.  With 256 rows of x per tile, one weight conversion
// serves four times as many MMA columns as in qmm_mma.cuh, whose per-group
// scaling costs CUDA-core work in proportion to the rows of x.
//
// Kernels: xsplit_kernel writes x as bf16 hi / lo operand tiles of 256 rows;
// qmm_mma_kernel computes D = W_tile * X^T for 128 weight rows against up to
// 256 rows of x (MMA M = 128, N = rows padded to 16, K = 16; A from tensor
// memory, B from shared memory).  Roles:
//   warp 8 (one lane)   streams the packed weights with one TMA bulk copy per
//                       32-row group and 256-wide K slot into a deep ring of
//                       raw slots (raw_full / raw_empty);
//   warp 10 (one lane)  with split x, copies each 64-wide K block of it into a
//                       ring of B stages (b_full);
//   warps 0-7           per 64-wide K block, dequantize and split the weights
//                       (thread t: row t%128, half t/128 of the block) and
//                       write them to a tensor-memory A stage with tcgen05.st
//                       (a_full); without split x they also fill B;
//   warps 9, 11-13      (one lane each) issue the block's 12 MMAs and commit
//                       them to the A stage's barrier mma_done, which frees
//                       both the A stage and the block's B stage (the B ring
//                       is no deeper than the A ring, so a B stage's last
//                       user is found on the A ring).  A warp can issue one
//                       MMA every ~55 cycles whatever N is, while the tensor
//                       core needs 128 * N / 256 cycles for one, so for small
//                       N up to four warps share the 16-wide K steps, each
//                       accumulating into its own columns of tensor memory;
//                       the epilogue adds the accumulators in a fixed order.
// When the row tiles alone do not fill the GPU, a thread-block cluster of ks
// CTAs splits K on slot boundaries; each CTA leaves its partial D in shared
// memory and, after a cluster barrier, CTA r sums columns r*mpad/ks ..
// (r+1)*mpad/ks of all ks partials in rank order through distributed shared
// memory (deterministic, no atomics).  Tiles of x beyond the first 256 rows
// are gridDim.y.  Every wait is bounded; a timeout sets the device error word.
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
namespace wide {

constexpr int kMmaRows = 128;          // weight rows per tile (MMA M)
constexpr int kMmaKB = 64;             // K per MMA stage
constexpr int kMmaSlotK = 256;         // K per raw weight slot
constexpr int kMmaSub = kMmaSlotK / kMmaKB;  // MMA stages per raw slot
constexpr int kMmaConvThreads = 256;   // warps 0-7
constexpr int kMmaThreads = 448;       // + weight producer 8, x producer 10, MMA 9, 11-13
constexpr int kMmaMaxIssuers = 4;      // warps issuing MMAs, each into its own accumulator
constexpr int kMmaMaxN = 256;          // rows of x per tile (MMA N)
constexpr int kMmaMaxSplit = 8;        // CTAs of a K-splitting cluster
constexpr int kMmaMaxRaw = 8;          // raw weight slots, at most
constexpr int kMmaMaxB = 4;            // B stages, at most (no more than A stages)
constexpr int kMmaBBudget = 32 * 1024;   // shared memory for the B ring, about
constexpr int kMmaAStages = 4;         // tensor-memory A stages
constexpr int kMmaSmemLimit = 227 * 1024;
constexpr uint32_t kMmaTmemCols = 512;  // D: columns 0..255, A stages: 256..511
constexpr uint32_t kMmaDCols = 256;
constexpr uint32_t kMmaACols = 64;      // one A stage: hi in 32 columns, lo in 32
constexpr uint64_t kMmaWaitNs = 2000000000ull;

constexpr unsigned kErrMmaTimeout = 4u;

// Raw slot of one 32-row group: QV packed vectors of the slot's 256-wide K
// range (Q6_K: the 13 of one super-block), then the step's scale vector.
template <int FMT> struct MmaRaw;
template <> struct MmaRaw<Q4_0> { static constexpr int QV = 8; };
template <> struct MmaRaw<Q8_0> { static constexpr int QV = 16; };
template <> struct MmaRaw<I8_B64> { static constexpr int QV = 16; };
template <> struct MmaRaw<Q6_K> { static constexpr int QV = 13; };
template <int FMT>
__host__ __device__ constexpr int mma_raw_group_bytes() {
    return (MmaRaw<FMT>::QV + 1) * kVecBytes;
}
template <int FMT>
__host__ __device__ constexpr int mma_raw_bytes() {
    return (kMmaRows / kRowsPerGroup) * mma_raw_group_bytes<FMT>();
}

// B stage: B_hi, B_lo (mpad x 64 bf16 each) in the layout of tile_off.
__host__ __device__ inline int mma_b_bytes(int mpad) { return mpad * kMmaKB * 2; }
// B stages: as many as fit the budget (x comes from L2, and a stage is
// refilled only once its MMAs are done), at least two (the K-split partials
// reuse the ring: 2 stages hold 128 x mpad fp32), at most the A stages.
__host__ __device__ inline int mma_b_stages(int mpad) {
    const int s = kMmaBBudget / (2 * mma_b_bytes(mpad));
    return s < 2 ? 2 : s > kMmaMaxB ? kMmaMaxB : s;
}
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

// Split x: for each 256-row tile t of x (mpad_t rows, padded to 16) and each
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
    int BS;             // B stages
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
// 32 consecutive fp32 columns of one tensor-memory lane per thread
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
// sum over the n accumulators (stride `cols` columns) of 32 fp32 columns,
// in accumulator order; zeros when !have
__device__ __forceinline__ void tmem_sum32(uint32_t taddr, int n, uint32_t cols, bool have,
                                           uint32_t (&r)[32]) {
    if (!have) {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
        return;
    }
    tmem_ld32(taddr, r);
    for (int k = 1; k < n; ++k) {
        uint32_t t[32];
        tmem_ld32(taddr + k * cols, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(t[i]));
    }
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

// bf16 hi / lo halves of two fp32 values, packed low element first
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 bh = __floats2bfloat162_rn(a, b);
    const float2 fh = __bfloat1622float2(bh);
    const __nv_bfloat162 bl = __floats2bfloat162_rn(a - fh.x, b - fh.y);
    hi = *reinterpret_cast<const uint32_t *>(&bh);
    lo = *reinterpret_cast<const uint32_t *>(&bl);
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
    constexpr int VPB = BlockTraits<FMT>::VPB, QV = MmaRaw<FMT>::QV;
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

// Dequantized weights of one row: 32 elements 32*half .. 32*half+31 of the
// 64-wide K block kb; rv points at the row's 16 bytes of its group's raw slot.
template <int FMT>
__device__ __forceinline__ void raw_chunk32(const uint8_t *rv, int half, int64_t kb,
                                            const Magic &mg, float (&w)[32]) {
    constexpr int QV = MmaRaw<FMT>::QV;
    const int sub = (int)(kb & (kMmaSub - 1));
    // scale slot of the block in its step's scale vector
    const int sidx = FMT == Q4_0 || FMT == Q8_0 ? 2 * sub + half
                     : FMT == I8_B64           ? (int)(kb & 7)
                                               : (int)((kb >> 2) & 7);
    const float d = h2f(reinterpret_cast<const unsigned short *>(rv + QV * kVecBytes)[sidx]);
    const f32x2 dd = pack2(d, d);
    if (FMT == Q4_0) {  // block 2*sub + half of the step is vector 2*sub + half
        const uint4 v = *reinterpret_cast<const uint4 *>(rv + (2 * sub + half) * kVecBytes);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            f32x2 p[4];
            q4_word(word_of(v, t), mg, p);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 q = unpack2(mul2(p[j], dd));
                w[8 * t + 2 * j] = q.x;
                w[8 * t + 2 * j + 1] = q.y;
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
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 q = unpack2(mul2(p[h], dd));
                    w[16 * jj + 4 * t + 2 * h] = q.x;
                    w[16 * jj + 4 * t + 2 * h + 1] = q.y;
                }
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
            const float dsc = d * i8_byte(scw, 2 * half + sb, mg);
            const f32x2 ds = pack2(dsc, dsc);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 q = unpack2(mul2(q6[j], ds));
                w[16 * sb + 2 * j] = q.x;
                w[16 * sb + 2 * j + 1] = q.y;
            }
        }
    }
}

// ---- the product ----------------------------------------------------------------------
// grid = (ceil(N/128) * ks, tiles of x); cluster = (ks, 1, 1); 352 threads;
// dynamic shared memory mma_smem_bytes(mpad of a full tile, a.RS).
// PRESPLIT: x comes split by xsplit_kernel (a.xs) and is copied by warp 10;
// otherwise the converter warps also split the block's x (a.x).
template <int FMT, bool PRESPLIT>
__global__ void __launch_bounds__(kMmaThreads, 1) qmm_mma_kernel(const MmaArgs a) {
    namespace cg = cooperative_groups;
    extern __shared__ __align__(1024) uint8_t msm[];
    uint64_t *raw_full = reinterpret_cast<uint64_t *>(msm);
    uint64_t *raw_empty = raw_full + kMmaMaxRaw;
    uint64_t *b_full = raw_empty + kMmaMaxRaw;
    uint64_t *a_full = b_full + kMmaMaxB;
    uint64_t *mma_done = a_full + kMmaAStages;
    uint64_t *done = mma_done + kMmaAStages;
    uint32_t *taddr_s = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_s = reinterpret_cast<volatile int *>(taddr_s + 1);
    uint8_t *bring = msm + 1024;
    uint8_t *rawring = msm + a.raw_off;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RS = a.RS, BS = a.BS;
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
    const int nk = min(a.nkb, (sl0 + nsl_c) * kMmaSub) - kb0;
    constexpr int RAWG = mma_raw_group_bytes<FMT>();
    // MMA issuers and the tensor-memory columns of each one's accumulator
    const int NI = mpad <= 64 ? 4 : mpad <= 128 ? 2 : 1;
    const uint32_t dcols = kMmaDCols / NI;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], kMmaConvThreads);
        }
        for (int s = 0; s < BS; ++s) mbar_init(&b_full[s], PRESPLIT ? 1 : kMmaConvThreads);
        for (int s = 0; s < kMmaAStages; ++s) {
            mbar_init(&a_full[s], kMmaConvThreads);
            mbar_init(&mma_done[s], NI);
        }
        mbar_init(done, NI);
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 9) tmem_alloc(taddr_s, kMmaTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_s;

    if (warp == 8) {
        // ---------------------------------------------------- weight producer
        if (lane == 0) {
            int issued = 0;
            for (int u = 0; u < nsl_c; ++u) {
                const int r = u % RS;
                if (*abort_s) break;
                if (u >= RS && !mbar_wait(&raw_empty[r], (uint32_t)(((u / RS) - 1) & 1), kMmaWaitNs)) {
                    *abort_s = 1;
                    break;
                }
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
                issued = u + 1;
            }
            // copies still in flight after an abort land before the CTA exits
            for (int u = issued - RS > 0 ? issued - RS : 0; u < issued; ++u)
                mbar_wait(&raw_full[u % RS], (uint32_t)((u / RS) & 1), kMmaWaitNs);
        }
    } else if (warp == 10) {
        // --------------------------------------------------------- x producer
        if (PRESPLIT && lane == 0) {
            const uint8_t *xs_tile = a.xs + tile * mma_xs_tile_bytes(a.nkb);
            int issued = 0;
            for (int j = 0; j < nk; ++j) {
                const int s = j % BS, jp = j - BS;  // jp: the last block that used stage s
                if (*abort_s) break;
                if (jp >= 0 && !mbar_wait(&mma_done[jp % kMmaAStages],
                                          (uint32_t)((jp / kMmaAStages) & 1), kMmaWaitNs)) {
                    *abort_s = 1;
                    break;
                }
                const uint8_t *src = xs_tile + (int64_t)(kb0 + j) * bbytes;
                const bool in = LEAN_SPAN(src - a.xs, bbytes, a.xs_bytes, a.err);
                mbar_arrive_expect_tx(&b_full[s], in ? (uint32_t)bbytes : 0u);
                if (j == 0) pdl_wait();  // the split x comes from the kernel before
                if (in) bulk_g2s(bring + s * bbytes, src, (uint32_t)bbytes, &b_full[s]);
                issued = j + 1;
            }
            for (int j = issued - BS > 0 ? issued - BS : 0; j < issued; ++j)
                mbar_wait(&b_full[j % BS], (uint32_t)((j / BS) & 1), kMmaWaitNs);
        }
    } else if (warp == 9 || warp > 10) {
        // -------------------------------------------------------- MMA issuers
        const int iss = warp == 9 ? 0 : warp - 10;  // 0 .. 3
        if (lane == 0 && iss < NI) {
            const uint32_t idesc = mma_idesc(mpad);
            const uint32_t td = tmem + iss * dcols;
            // descriptors advance by adding byte offsets / 16 to the address field
            const uint64_t bdesc0 = smem_desc(smem_addr(bring));
            const uint32_t b_lo16 = (uint32_t)mma_b_bytes(mpad) >> 4, kk16 = (uint32_t)(mpad * 32) >> 4;
            for (int j = 0; j < nk; ++j) {
                const int sa = j % kMmaAStages, sb = j % BS;
                if (*abort_s) break;
                if (!mbar_wait(&a_full[sa], (uint32_t)((j / kMmaAStages) & 1), kMmaWaitNs) ||
                    !mbar_wait(&b_full[sb], (uint32_t)((j / BS) & 1), kMmaWaitNs)) {
                    *abort_s = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t ta_hi = tmem + kMmaDCols + sa * kMmaACols;
                const uint32_t ta_lo = ta_hi + kMmaACols / 2;
                const uint64_t bh = bdesc0 + ((uint32_t)(sb * bbytes) >> 4);
                for (int kk = iss; kk < kMmaKB / 16; kk += NI) {
                    const uint64_t dh = bh + kk * kk16, dl = dh + b_lo16;
                    mma_bf16_ts(td, ta_hi + 8 * kk, dh, idesc, (j > 0 || kk > iss) ? 1u : 0u);
                    mma_bf16_ts(td, ta_hi + 8 * kk, dl, idesc, 1u);
                    mma_bf16_ts(td, ta_lo + 8 * kk, dh, idesc, 1u);
                }
                mma_commit(&mma_done[sa]);
            }
            mma_commit(done);  // arrives when every MMA issued above has completed
        }
    } else {
        // -------------------------------------------------------- converters
        const Magic mg = pin_fmt<FMT>(a.mg);
        const int row = threadIdx.x & (kMmaRows - 1), half = threadIdx.x >> 7;
        const int g = row / kRowsPerGroup;
        const bool row_live = n0 / kRowsPerGroup + g < a.groups;
        const int64_t chunks = a.K / 32;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        for (int j = 0; j < nk; ++j) {
            const int u = j / kMmaSub, r = u % RS, sa = j % kMmaAStages;
            if (*abort_s) break;
            if ((j % kMmaSub == 0 &&
                 !mbar_wait(&raw_full[r], (uint32_t)((u / RS) & 1), kMmaWaitNs)) ||
                (j >= kMmaAStages &&
                 !mbar_wait(&mma_done[sa], (uint32_t)(((j / kMmaAStages) - 1) & 1), kMmaWaitNs))) {
                *abort_s = 1;
                break;
            }
            const int64_t kb = kb0 + j;
            float w[32];
            if (row_live && 2 * kb + half < chunks) {
                raw_chunk32<FMT>(rawring + r * mma_raw_bytes<FMT>() + g * RAWG +
                                     (row % kRowsPerGroup) * kVec,
                                 half, kb, mg, w);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = 0.f;
            }
            // the block's 32 elements of this row -> A stage, columns 16*half ..
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) split2(w[2 * i], w[2 * i + 1], hi[i], lo[i]);
            tc_fence_after();
            const uint32_t ta = tmem + lane_base + kMmaDCols + sa * kMmaACols + 16 * half;
            tmem_st16(ta, hi);
            tmem_st16(ta + kMmaACols / 2, lo);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&a_full[sa]);
            if (j % kMmaSub == kMmaSub - 1 || j == nk - 1) mbar_arrive(&raw_empty[r]);
            if (!PRESPLIT) {
                // x of the block: item i = (row m = i % mpad, 8-wide piece i / mpad);
                // all loads first, then the splits
                const int sb = j % BS, jp = j - BS;  // jp: the last block that used stage sb
                if (jp >= 0 && !mbar_wait(&mma_done[jp % kMmaAStages],
                                          (uint32_t)((jp / kMmaAStages) & 1), kMmaWaitNs)) {
                    *abort_s = 1;
                    break;
                }
                if (j == 0) pdl_wait();  // x may come from the previous kernel on the stream
                constexpr int XI = kMmaMaxN * 8 / kMmaConvThreads;
                uint8_t *b_hi = bring + sb * bbytes;
                float4 xv[XI][2];
#pragma unroll
                for (int q = 0; q < XI; ++q) {
                    const int i = (int)threadIdx.x + q * kMmaConvThreads;
                    const int m = i % mpad;
                    const int64_t k = kb * kMmaKB + 8 * (i / mpad);
                    if (i < mpad * 8 && m < mt && k < a.K &&
                        LEAN_SPAN((int64_t)(m0 + m) * a.K + k, 8, (int64_t)a.M * a.K, a.err)) {
                        const float *src = a.x + (int64_t)(m0 + m) * a.K + k;
                        xv[q][0] = __ldg(reinterpret_cast<const float4 *>(src));
                        xv[q][1] = __ldg(reinterpret_cast<const float4 *>(src + 4));
                    } else {
                        xv[q][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                        xv[q][1] = xv[q][0];
                    }
                }
#pragma unroll
                for (int q = 0; q < XI; ++q) {
                    const int i = (int)threadIdx.x + q * kMmaConvThreads;
                    if (i < mpad * 8) {
                        const float v[8] = {xv[q][0].x, xv[q][0].y, xv[q][0].z, xv[q][0].w,
                                            xv[q][1].x, xv[q][1].y, xv[q][1].z, xv[q][1].w};
                        const uint32_t off = tile_off(mpad, i % mpad, 8 * (i / mpad));
                        split_store8(v, b_hi + off, b_hi + mma_b_bytes(mpad) + off);
                    }
                }
                fence_async_smem();  // the tensor cores read what the generic proxy wrote
                mbar_arrive(&b_full[sb]);
            }
        }
    }

    // ------------------------------------------------------------------ epilogue
    pdl_launch_dependents();  // the next kernel may start; it waits for our completion
    bool fin = true;
    if (warp < 8) fin = mbar_wait(done, 0u, kMmaWaitNs);
    const bool ok = __syncthreads_and(fin && !*abort_s) != 0;
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(a.err, kErrMmaTimeout);
        if (warp < 8 && !fin) mbar_wait(done, 0u, kMmaWaitNs);
    }
    tc_fence_after();
    pdl_wait();  // y is written below
    const bool have = ok && nk > 0;
    const int q = warp & 3;  // tensor-memory lanes 32q .. 32q+31 = weight rows
    const int64_t nq = n0 + 32 * q + lane;
    if (a.ks == 1) {
        if (warp < 8) {
            for (int c0 = 32 * (warp >> 2); c0 < mpad; c0 += 64) {
                uint32_t r[32];
                tmem_sum32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, NI, dcols, have, r);
                if (nq < a.N) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c0 + i < mt &&
                            LEAN_IN((int64_t)(m0 + c0 + i) * a.N + nq, (int64_t)a.M * a.N, a.err))
                            a.y[(int64_t)(m0 + c0 + i) * a.N + nq] = __uint_as_float(r[i]);
                }
            }
        }
    } else {
        // partial D of this CTA into shared memory, P[m][row] (the rings are
        // free: every MMA has completed and every copy has landed)
        float *P = reinterpret_cast<float *>(bring);
        if (warp < 8) {
            for (int c0 = 32 * (warp >> 2); c0 < mpad; c0 += 64) {
                uint32_t r[32];
                tmem_sum32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, NI, dcols, have, r);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (c0 + i < mpad) P[(c0 + i) * kMmaRows + 32 * q + lane] = __uint_as_float(r[i]);
            }
        }
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();
        // this CTA's share of the columns, summed over the cluster in rank
        // order; item = (column m, 4 consecutive rows), all ranks' loads issued
        // before the sums
        if (warp < 8) {
            const int mlo = mpad * rank / a.ks, mhi = mpad * (rank + 1) / a.ks;
            const int items = (mhi - mlo) * (kMmaRows / 4);
            const float4 *Pr[kMmaMaxSplit];
#pragma unroll
            for (int r = 0; r < kMmaMaxSplit; ++r)
                Pr[r] = reinterpret_cast<const float4 *>(cl.map_shared_rank(P, r < a.ks ? r : 0));
            for (int it = threadIdx.x; it < items; it += kMmaConvThreads) {
                const int m = mlo + it / (kMmaRows / 4), r4 = it % (kMmaRows / 4);
                const int idx = m * (kMmaRows / 4) + r4;
                float4 v[kMmaMaxSplit];
#pragma unroll
                for (int r = 0; r < kMmaMaxSplit; ++r)
                    if (r < a.ks) v[r] = Pr[r][idx];
                float4 acc = v[0];
#pragma unroll
                for (int r = 1; r < kMmaMaxSplit; ++r)
                    if (r < a.ks) {
                        acc.x += v[r].x;
                        acc.y += v[r].y;
                        acc.z += v[r].z;
                        acc.w += v[r].w;
                    }
                if (m < mt) {
                    float *yr = a.y + (int64_t)(m0 + m) * a.N;
                    const int64_t nr = n0 + 4 * r4, yo = (int64_t)(m0 + m) * a.N + nr, ye = (int64_t)a.M * a.N;
                    if (nr < a.N && LEAN_IN(yo, ye, a.err)) yr[nr] = acc.x;
                    if (nr + 1 < a.N && LEAN_IN(yo + 1, ye, a.err)) yr[nr + 1] = acc.y;
                    if (nr + 2 < a.N && LEAN_IN(yo + 2, ye, a.err)) yr[nr + 2] = acc.z;
                    if (nr + 3 < a.N && LEAN_IN(yo + 3, ye, a.err)) yr[nr + 3] = acc.w;
                }
            }
        }
        cl.sync();  // no CTA leaves while others read its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) tmem_dealloc(tmem, kMmaTmemCols);
}

}  // namespace wide
}  // namespace lean
