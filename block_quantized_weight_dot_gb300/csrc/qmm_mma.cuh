// qmm_mma.cuh -- the product for larger M on the fifth-generation tensor cores
// (tcgen05.mma with accumulators in tensor memory).
//
// With many rows of x the product is a dense contraction.  The pages' GPU
// path dequantizes weight tiles in shared memory and multiplies them there
// ("oxinfer" crate page, Platforms and accelerators: Browser (WebGPU)), in
// f32.  bf16 operands alone would miss the 1e-4 tolerance (one bf16 rounding
// is 2^-9 relative), so each operand is split into a bf16 pair, w = w_hi +
// w_lo and x = x_hi + x_lo, and three MMAs accumulate w_hi*x_hi + w_hi*x_lo +
// w_lo*x_hi in fp32.  The dropped w_lo*x_lo and the rounding of x_lo (and of
// w_lo for the formats whose dequantized weights need more than 16 bits) are
// each below 2^-16 of |w*x|; for Q4_0 the weight split is exact, since
// d*(q-8) has at most 15 significant bits.
//
// Two kernels.  xsplit_kernel writes x once as bf16 hi / lo tiles already in
// the shared-memory operand layout, one contiguous piece per (256-row tile of
// x, 64-wide K block), into a caller workspace; without one, the converter
// warps split each CTA's x themselves.  qmm_mma_kernel then computes D = W_tile * X^T for 128
// weight rows against up to 256 rows of x -- one tcgen05.mma of shape M=128
// (weight rows) x N=mpad (rows of x padded to 16) x K=16, D (= y^T) in tensor
// memory -- with three roles over an S-stage shared-memory ring:
//   warp 8 (one lane)   TMA bulk copies of the stage's packed weight vectors
//                       and of its x operand piece (complete_tx on full[s]);
//   warps 0-7           dequantize and split the weights of the stage (thread
//                       t: row t%128, half t/128 of the 64-wide block) into
//                       the A operand, then arrive on conv[s];
//   warp 9 (one lane)   issues the stage's 12 MMAs once conv[s] completes and
//                       commits them to empty[s], which frees the stage.
// When the row tiles alone do not fill the GPU, a thread-block cluster of ks
// CTAs splits K; each CTA leaves its partial D in shared memory and, after a
// cluster barrier, CTA r sums columns r*mpad/ks .. (r+1)*mpad/ks of all ks
// partials in rank order through distributed shared memory (deterministic,
// no atomics).  Tiles of x beyond the first 256 rows are gridDim.y.  Every
// wait is bounded; a timeout sets the device error word.
#pragma once
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "decode.cuh"
#include "layout.h"
#include "ptx.cuh"
#include "qmm_simt.cuh"

namespace lean {

constexpr int kMmaRows = 128;       // weight rows per tile (MMA M)
constexpr int kMmaKB = 64;          // K per pipeline stage
constexpr int kMmaConvThreads = 256;  // warps 0-7
constexpr int kMmaThreads = 320;    // + producer warp 8 + MMA warp 9
constexpr int kMmaMaxN = 256;       // rows of x per tile (MMA N)
constexpr int kMmaMaxSplit = 8;     // CTAs of a K-splitting cluster
constexpr int kMmaMaxStages = 4;
constexpr int kMmaSmemLimit = 227 * 1024;
constexpr uint64_t kMmaWaitNs = 2000000000ull;

constexpr unsigned kErrMmaTimeout = 4u;

// Packed vectors copied per 32-row group and stage: QV quant vectors, XV
// extra vectors (Q6_K sub-scales), then the step's scale vector.
template <int FMT> struct MmaRaw;
template <> struct MmaRaw<Q4_0> { static constexpr int QV = 2, XV = 0; };
template <> struct MmaRaw<Q8_0> { static constexpr int QV = 4, XV = 0; };
template <> struct MmaRaw<I8_B64> { static constexpr int QV = 4, XV = 0; };
template <> struct MmaRaw<Q6_K> { static constexpr int QV = 3, XV = 1; };
template <int FMT>
__host__ __device__ constexpr int mma_raw_group_bytes() {
    return (MmaRaw<FMT>::QV + MmaRaw<FMT>::XV + 1) * kVecBytes;
}
template <int FMT>
__host__ __device__ constexpr int mma_raw_bytes() {
    return (kMmaRows / kRowsPerGroup) * mma_raw_group_bytes<FMT>();
}

// One stage: raw weight vectors, A_hi, A_lo (128 x 64 bf16), B_hi, B_lo
// (mpad x 64 bf16).  Shared memory = 1 KiB of barriers + S stages.
__host__ __device__ constexpr int mma_a_bytes() { return kMmaRows * kMmaKB * 2; }
__host__ __device__ inline int mma_b_bytes(int mpad) { return mpad * kMmaKB * 2; }
template <int FMT>
__host__ __device__ inline int mma_stage_bytes(int mpad) {
    return mma_raw_bytes<FMT>() + 2 * mma_a_bytes() + 2 * mma_b_bytes(mpad);
}
template <int FMT>
__host__ __device__ inline int mma_stages(int mpad) {
    const int s = (kMmaSmemLimit - 1024) / mma_stage_bytes<FMT>(mpad);
    return s < kMmaMaxStages ? s : kMmaMaxStages;
}
__host__ __device__ inline uint32_t mma_tmem_cols(int mpad) {
    return mpad <= 32 ? 32u : mpad <= 64 ? 64u : mpad <= 128 ? 128u : 256u;
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
    const uint8_t *W;  // packed weights
    const float *x;    // x[M][K]
    const uint8_t *xs; // split x, or null
    float *y;          // y[M][N]
    int N, K, M;
    int ks;            // CTAs splitting K (cluster size)
    int nkb;           // 64-wide K blocks
    int m_base;        // first row of x of this launch
    int S;             // pipeline stages
    int pad;
    int64_t groups;
    int steps, last_blocks, step_vecs, pad2;
    int64_t group_vecs;
    unsigned *err;
    Magic mg;
};

struct XsplitArgs {
    const float *x;
    uint8_t *xs;
    int M, K, nkb;
    int mtiles;
    int64_t rows;  // padded rows over all tiles
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
// D[tmem] (+)= A[smem] * B[smem]^T: bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
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

// split 8 fp32 values into bf16 hi / lo halves and store 16 bytes of each
__device__ __forceinline__ void split_store8(const float *v, uint8_t *hi, uint8_t *lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 bh = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        const float2 fh = __bfloat1622float2(bh);
        const __nv_bfloat162 bl = __floats2bfloat162_rn(v[2 * i] - fh.x, v[2 * i + 1] - fh.y);
        h[i] = *reinterpret_cast<const uint32_t *>(&bh);
        l[i] = *reinterpret_cast<const uint32_t *>(&bl);
    }
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
    if (m < a.M && k < a.K) {
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
    split_store8(v, piece + off, piece + mma_b_bytes(mpad) + off);
}

// ---- weights: raw vectors in shared memory -> exact fp32 ------------------------------
// 32 elements 32*half .. 32*half+31 of the stage's 64-wide K block for one
// row; rv points at the row's 16 bytes of its group's first raw vector.
template <int FMT>
__device__ __forceinline__ void raw_chunk32(const uint8_t *rv, int half, int sidx, int64_t kb,
                                            const Magic &mg, float (&w)[32]) {
    constexpr int QV = MmaRaw<FMT>::QV, XV = MmaRaw<FMT>::XV;
    const float d = h2f(reinterpret_cast<const unsigned short *>(rv + (QV + XV) * kVecBytes)[sidx]);
    const f32x2 dd = pack2(d, d);
    if (FMT == Q4_0) {  // vector h = block 2kb + h
        const uint4 v = *reinterpret_cast<const uint4 *>(rv + half * kVecBytes);
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
    } else if (FMT == Q8_0 || FMT == I8_B64) {  // vectors 2h, 2h+1: 16 elements each
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const uint4 v = *reinterpret_cast<const uint4 *>(rv + (2 * half + jj) * kVecBytes);
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
    } else {  // Q6_K: vectors 0..2 hold sub-blocks 4p..4p+3 (p = kb % 4); this half 2 of them
        const int p = (int)(kb & 3);
        const uint4 va = *reinterpret_cast<const uint4 *>(rv + half * kVecBytes);
        const uint4 vb = *reinterpret_cast<const uint4 *>(rv + (half + 1) * kVecBytes);
        const uint4 vs = *reinterpret_cast<const uint4 *>(rv + QV * kVecBytes);
        uint32_t wd[6];
        if (half == 0) {
            wd[0] = va.x; wd[1] = va.y; wd[2] = va.z; wd[3] = va.w; wd[4] = vb.x; wd[5] = vb.y;
        } else {
            wd[0] = va.z; wd[1] = va.w; wd[2] = vb.x; wd[3] = vb.y; wd[4] = vb.z; wd[5] = vb.w;
        }
        const uint32_t scw = word_of(vs, p);
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

// Weight copies of stage kb for group gi into the raw slot of that group;
// returns the bytes they bring (0 for a group past the last one).
template <int FMT>
__device__ __forceinline__ uint32_t raw_bytes_of(const MmaArgs &a, int64_t gi, int64_t kb) {
    constexpr int VPB = BlockTraits<FMT>::VPB;
    if (gi >= a.groups) return 0;
    if (FMT == Q4_0 || FMT == Q8_0) {
        const int nb = (2 * kb + 1 < (int64_t)a.K / 32) ? 2 : 1;
        return (uint32_t)((nb * VPB + 1) * kVecBytes);
    }
    return (uint32_t)((MmaRaw<FMT>::QV + MmaRaw<FMT>::XV + 1) * kVecBytes);
}
template <int FMT>
__device__ __forceinline__ void raw_copy(const MmaArgs &a, int64_t gi, int64_t kb, uint8_t *dst,
                                         uint64_t *bar) {
    constexpr int VPB = BlockTraits<FMT>::VPB, QV = MmaRaw<FMT>::QV, XV = MmaRaw<FMT>::XV;
    const int64_t c = FMT == Q6_K ? (kb >> 2) : FMT == I8_B64 ? kb : 2 * kb;  // first block
    const int s = (int)(c >> 3), i = (int)(c & 7);
    const int nblk = s == a.steps - 1 ? a.last_blocks : 8;
    const uint8_t *step = a.W + (gi * a.group_vecs + (int64_t)s * a.step_vecs) * kVecBytes;
    if (FMT == Q4_0 || FMT == Q8_0) {
        const int nb = (2 * kb + 1 < (int64_t)a.K / 32) ? 2 : 1;
        bulk_g2s(dst, step + i * VPB * kVecBytes, nb * VPB * kVecBytes, bar);
    } else if (FMT == I8_B64) {
        bulk_g2s(dst, step + i * VPB * kVecBytes, VPB * kVecBytes, bar);
    } else {
        const int p = (int)(kb & 3);
        bulk_g2s(dst, step + (i * VPB + 3 * p) * kVecBytes, 3 * kVecBytes, bar);
        bulk_g2s(dst + QV * kVecBytes, step + (i * VPB + 12) * kVecBytes, kVecBytes, bar);
    }
    bulk_g2s(dst + (QV + XV) * kVecBytes, step + nblk * VPB * kVecBytes, kVecBytes, bar);
}

// ---- the product ----------------------------------------------------------------------
// grid = (ceil(N/128) * ks, tiles of x); cluster = (ks, 1, 1); 320 threads;
// dynamic shared memory 1024 + S * mma_stage_bytes(mpad of a full tile).
// PRESPLIT: x comes split by xsplit_kernel (a.xs) and is copied by the
// producer; otherwise the converter warps also split the stage's x (a.x).
template <int FMT, bool PRESPLIT>
__global__ void __launch_bounds__(kMmaThreads, 1) qmm_mma_kernel(const MmaArgs a) {
    namespace cg = cooperative_groups;
    extern __shared__ __align__(1024) uint8_t msm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(msm);       // [S] stage loaded
    uint64_t *conv = full + kMmaMaxStages;                   // [S] A operand written
    uint64_t *empty = conv + kMmaMaxStages;                  // [S] stage's MMAs complete
    uint64_t *done = empty + kMmaMaxStages;                  // every MMA complete
    uint32_t *taddr_s = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_s = reinterpret_cast<volatile int *>(taddr_s + 1);
    uint8_t *stages = msm + 1024;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.S;
    const int rank = (int)(blockIdx.x % (unsigned)a.ks);
    const int64_t n0 = (int64_t)(blockIdx.x / (unsigned)a.ks) * kMmaRows;
    const int tile = (int)blockIdx.y + a.m_base / kMmaMaxN;
    const int m0 = tile * kMmaMaxN;
    const int mt = min(kMmaMaxN, a.M - m0);
    const int mpad = (mt + 15) & ~15;
    const int sbytes = mma_stage_bytes<FMT>(mpad);
    const int kb0 = (int)((int64_t)a.nkb * rank / a.ks);
    const int nk = (int)((int64_t)a.nkb * (rank + 1) / a.ks) - kb0;
    const uint32_t ncols = mma_tmem_cols(mpad);
    constexpr int RAW = mma_raw_bytes<FMT>();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&conv[s], kMmaConvThreads);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 9) tmem_alloc(taddr_s, ncols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_s;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint8_t *xs_tile = a.xs + tile * mma_xs_tile_bytes(a.nkb);
            const uint32_t bbytes = (uint32_t)(2 * mma_b_bytes(mpad));
            int issued = 0;
            for (int j = 0; j < nk; ++j) {
                const int s = j % S;
                if (*abort_s) break;
                if (j >= S && !mbar_wait(&empty[s], (uint32_t)(((j / S) - 1) & 1), kMmaWaitNs)) {
                    *abort_s = 1;
                    break;
                }
                uint8_t *st = stages + s * sbytes;
                const int64_t kb = kb0 + j;
                uint32_t bytes = PRESPLIT ? bbytes : 0u;
                for (int g = 0; g < kMmaRows / kRowsPerGroup; ++g)
                    bytes += raw_bytes_of<FMT>(a, n0 / kRowsPerGroup + g, kb);
                mbar_arrive_expect_tx(&full[s], bytes);
                for (int g = 0; g < kMmaRows / kRowsPerGroup; ++g) {
                    const int64_t gi = n0 / kRowsPerGroup + g;
                    if (gi < a.groups)
                        raw_copy<FMT>(a, gi, kb, st + g * mma_raw_group_bytes<FMT>(), &full[s]);
                }
                if (PRESPLIT) {
                    if (j == 0) pdl_wait();  // the split x comes from the kernel before
                    bulk_g2s(st + RAW + 2 * mma_a_bytes(), xs_tile + kb * (int64_t)bbytes, bbytes,
                             &full[s]);
                }
                issued = j + 1;
            }
            // copies still in flight after an abort finish before the CTA exits
            for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
                mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), kMmaWaitNs);
        }
    } else if (warp == 9) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = mma_idesc(mpad);
            for (int j = 0; j < nk; ++j) {
                const int s = j % S;
                const uint32_t ph = (uint32_t)((j / S) & 1);
                if (*abort_s) break;
                if (!mbar_wait(&conv[s], ph, kMmaWaitNs) || !mbar_wait(&full[s], ph, kMmaWaitNs)) {
                    *abort_s = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t sa_hi = smem_addr(stages + s * sbytes + RAW);
                const uint32_t sa_lo = sa_hi + mma_a_bytes();
                const uint32_t sb_hi = sa_lo + mma_a_bytes();
                const uint32_t sb_lo = sb_hi + mma_b_bytes(mpad);
#pragma unroll
                for (int kk = 0; kk < kMmaKB / 16; ++kk) {
                    const uint32_t ao = kk * (kMmaRows * 32), bo = kk * (mpad * 32);
                    mma_bf16(tmem, smem_desc(sa_hi + ao), smem_desc(sb_hi + bo), idesc,
                             (j > 0 || kk > 0) ? 1u : 0u);
                    mma_bf16(tmem, smem_desc(sa_hi + ao), smem_desc(sb_lo + bo), idesc, 1u);
                    mma_bf16(tmem, smem_desc(sa_lo + ao), smem_desc(sb_hi + bo), idesc, 1u);
                }
                mma_commit(&empty[s]);
            }
            mma_commit(done);  // arrives when every MMA issued above has completed
        }
    } else {
        // -------------------------------------------------------- converters
        const Magic mg = pin(a.mg);
        const int row = threadIdx.x & (kMmaRows - 1), half = threadIdx.x >> 7;
        const int g = row / kRowsPerGroup;
        const bool row_live = n0 / kRowsPerGroup + g < a.groups;
        const int64_t chunks = a.K / 32;
        for (int j = 0; j < nk; ++j) {
            const int s = j % S;
            if (*abort_s) break;
            if (!mbar_wait(&full[s], (uint32_t)((j / S) & 1), kMmaWaitNs)) {
                *abort_s = 1;
                break;
            }
            uint8_t *st = stages + s * sbytes;
            const int64_t kb = kb0 + j;
            float w[32];
            if (row_live && 2 * kb + half < chunks) {
                // scale slot of the chunk's block within its step
                const int sidx = FMT == Q4_0 || FMT == Q8_0 ? (int)((2 * kb + half) & 7)
                                 : FMT == I8_B64           ? (int)(kb & 7)
                                                           : (int)((kb >> 2) & 7);
                raw_chunk32<FMT>(st + g * mma_raw_group_bytes<FMT>() + (row % kRowsPerGroup) * kVec,
                                 half, sidx, kb, mg, w);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = 0.f;
            }
            uint8_t *a_hi = st + RAW;
#pragma unroll
            for (int k8 = 0; k8 < 4; ++k8) {
                const uint32_t off = tile_off(kMmaRows, row, 32 * half + 8 * k8);
                split_store8(w + 8 * k8, a_hi + off, a_hi + mma_a_bytes() + off);
            }
            if (!PRESPLIT) {
                // x of the stage: item i = (row m = i % mpad, 8-wide piece i / mpad);
                // all loads first, then the splits
                if (j == 0) pdl_wait();  // x may come from the previous kernel on the stream
                constexpr int XI = kMmaMaxN * 8 / kMmaConvThreads;
                uint8_t *b_hi = a_hi + 2 * mma_a_bytes();
                float4 xv[XI][2];
#pragma unroll
                for (int u = 0; u < XI; ++u) {
                    const int i = (int)threadIdx.x + u * kMmaConvThreads;
                    const int m = i % mpad;
                    const int64_t k = kb * kMmaKB + 8 * (i / mpad);
                    if (i < mpad * 8 && m < mt && k < a.K) {
                        const float *src = a.x + (int64_t)(m0 + m) * a.K + k;
                        xv[u][0] = __ldg(reinterpret_cast<const float4 *>(src));
                        xv[u][1] = __ldg(reinterpret_cast<const float4 *>(src + 4));
                    } else {
                        xv[u][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                        xv[u][1] = xv[u][0];
                    }
                }
#pragma unroll
                for (int u = 0; u < XI; ++u) {
                    const int i = (int)threadIdx.x + u * kMmaConvThreads;
                    if (i < mpad * 8) {
                        const float v[8] = {xv[u][0].x, xv[u][0].y, xv[u][0].z, xv[u][0].w,
                                            xv[u][1].x, xv[u][1].y, xv[u][1].z, xv[u][1].w};
                        const uint32_t off = tile_off(mpad, i % mpad, 8 * (i / mpad));
                        split_store8(v, b_hi + off, b_hi + mma_b_bytes(mpad) + off);
                    }
                }
            }
            fence_async_smem();  // the tensor cores read what the generic proxy wrote
            mbar_arrive(&conv[s]);
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
                if (have) {
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, r);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
                if (nq < a.N) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c0 + i < mt)
                            a.y[(int64_t)(m0 + c0 + i) * a.N + nq] = __uint_as_float(r[i]);
                }
            }
        }
    } else {
        // partial D of this CTA into shared memory, P[m][row] (the stages are
        // free: every MMA has completed and every copy has landed)
        float *P = reinterpret_cast<float *>(stages);
        if (warp < 8) {
            for (int c0 = 32 * (warp >> 2); c0 < mpad; c0 += 64) {
                uint32_t r[32];
                if (have) {
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, r);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
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
                    const int64_t nr = n0 + 4 * r4;
                    if (nr < a.N) yr[nr] = acc.x;
                    if (nr + 1 < a.N) yr[nr + 1] = acc.y;
                    if (nr + 2 < a.N) yr[nr + 2] = acc.z;
                    if (nr + 3 < a.N) yr[nr + 3] = acc.w;
                }
            }
        }
        cl.sync();  // no CTA leaves while others read its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) tmem_dealloc(tmem, ncols);
}

}  // namespace lean
