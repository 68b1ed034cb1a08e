/*
 * lean_qmatmul.h -- C ABI of the GB300 (sm_103a) block-quantized weight x
 * activation product:  y[m][n] = sum_k w[n][k] * x[m][k].
 *
 * The operation is the linear layer of the small LLM engines described on the
 * "lean" README (llm-web), the "wgpu-llm" README and the "oxinfer" crate page:
 * during single-sequence decode every linear streams its quantized weights
 * once ("oxinfer" crate page, Performance: decode is memory-bandwidth bound),
 * so the product reads the packed blocks directly and never materialises
 * dense weights.
 *
 * Weight formats (block along K, within one output row n):
 *   LEAN_Q4_0    32 weights, fp16 scale d, 4-bit q:      w = d * (q - 8)
 *                ("oxinfer", How it works: two nibbles per byte, f16 scale;
 *                 "lean" README model table: Q4_0 weights)
 *   LEAN_Q8_0    32 weights, fp16 scale d, int8 q:       w = d * q
 *                ("lean" README: Q8_0 checkpoints; "oxinfer": 32 weights per
 *                 scale)
 *   LEAN_I8_B64  64 weights, fp16 scale d, int8 q:       w = d * q
 *                ("wgpu-llm" README, INT8 mode: symmetric, block size 64)
 *   LEAN_Q6_K   256 weights, fp16 d, 16 int8 sub-scales sc (one per 16
 *                weights), 6-bit q:                      w = d * sc * (q - 32)
 *                ("lean" README model table: Q6_K embedding)
 *
 * Two byte layouts exist:
 *   canonical  the interchange format (GGUF-style blocks, little-endian):
 *                Q4_0    [d fp16][16 B: element j<16 = low nibble of byte j,
 *                                  element j+16 = high nibble of byte j]
 *                Q8_0    [d fp16][32 x int8]
 *                I8_B64  [d fp16][64 x int8]
 *                Q6_K    [ql 128 B][qh 64 B][sc 16 x int8][d fp16]; element e:
 *                        h = e/128, g = (e%128)/32, l = e%32; low 4 bits =
 *                        nibble g/2 of ql[64h + 32(g%2) + l], high 2 bits =
 *                        bits 2g..2g+1 of qh[32h + l], sub-scale sc[e/16]
 *              A row is K / block_elems consecutive blocks; the matrix is N
 *              consecutive rows.
 *   packed     the device layout the kernels stream: a quant plane and a
 *              scale plane, as the "oxinfer" crate page keeps each quantized
 *              matrix as quant bytes plus scales "in exactly the in-memory
 *              layout of the kernels" (Pre-quantized checkpoints).  Rows are
 *              grouped by 32 and interleaved in 16-byte chunks so that one
 *              warp's load is 512 contiguous bytes.  Its size is
 *              lean_packed_bytes(); its contents are private to this library
 *              and made only by lean_pack().
 *
 * Conventions for every call:
 *   - fmt is one of the lean_fmt values (passed as int).
 *   - N, K, M > 0; K must be a multiple of lean_block_elems(fmt).
 *   - The caller owns and allocates every buffer.  Device pointers must come
 *     from the current CUDA device.  The library never allocates, frees or
 *     synchronises, and keeps no per-call state.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *     void*, NULL = the legacy default stream) and make no host read-back, so
 *     they may be captured into a CUDA graph.
 *   - Argument errors are detected on the host and returned before any launch
 *     (nothing is queued on the stream).  A failed launch returns LEAN_ERR_CUDA
 *     (cudaGetLastError is consumed).
 *   - Per-device facts (the SM count, the device addresses of the library's
 *     error word and fixed workspace, raised shared-memory limits) are looked
 *     up on a device's first use and cached by device ordinal.  The library
 *     therefore assumes each device is used through its primary context (the
 *     one the CUDA runtime and PyTorch use) and is not reset with
 *     cudaDeviceReset while the library is loaded.
 */
#ifndef LEAN_QMATMUL_H
#define LEAN_QMATMUL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LEAN_Q4_0 = 0,
    LEAN_Q8_0 = 1,
    LEAN_I8_B64 = 2,
    LEAN_Q6_K = 3
} lean_fmt;

typedef enum {
    LEAN_OK = 0,
    LEAN_ERR_FORMAT = 1, /* unknown fmt                                     */
    LEAN_ERR_SHAPE = 2,  /* N, K or M <= 0, K not a multiple of the block,
                            or a size beyond the library's limits           */
    LEAN_ERR_NULL = 3,   /* a required pointer is NULL                      */
    LEAN_ERR_ALIGN = 4,  /* a pointer is not aligned as documented          */
    LEAN_ERR_CUDA = 5,   /* the CUDA runtime reported an error              */
    LEAN_ERR_KERNEL_BOUNDS = 6, /* (lean_device_status) a kernel of a LEAN_DEBUG
                            build met an index outside its buffers          */
    LEAN_ERR_DEVICE = 7  /* (lean_device_status) a kernel reported another
                            error in the device error word                  */
} lean_status;

/* Weights per block: 32, 32, 64, 256.  0 for an unknown fmt.
 * Pages: "oxinfer" crate page, How it works (quant.rs: Q8 and Q4_0 blocks of
 * 32); "wgpu-llm" README, INT8 mode (block size 64); "lean" README, model
 * table (Q6_K). */
int lean_block_elems(int fmt);

/* Canonical bytes per block: 18, 34, 66, 210.  0 for an unknown fmt.
 * Pages: as lean_block_elems (fp16 scales: "oxinfer" crate page, How it
 * works, Q4_0 "f16 scale"; the other sizes are the same reading). */
int64_t lean_block_bytes(int fmt);

/* Canonical bytes of an N x K matrix, or -1 on a bad fmt or shape.
 * Pages: "oxinfer" crate page, Pre-quantized checkpoints (a quantized matrix
 * is its quant bytes plus its scales). */
int64_t lean_canonical_bytes(int fmt, int64_t N, int64_t K);

/* Packed (device layout) bytes of an N x K matrix, or -1 on a bad fmt or
 * shape.  Rows are padded up to a multiple of 32 and the scale plane to whole
 * 16-byte vectors, so this is a little more than lean_canonical_bytes().
 * Pages: "oxinfer" crate page, Pre-quantized checkpoints (weights kept "in
 * exactly the in-memory layout of the kernels"). */
int64_t lean_packed_bytes(int fmt, int64_t N, int64_t K);

/* Host-side repacking, canonical -> packed (pages: as lean_packed_bytes;
 * here done once at upload, as the pages' loader borrows the file's blocks
 * without copying).  canon_host holds
 * lean_canonical_bytes(fmt,N,K) bytes; packed_host receives
 * lean_packed_bytes(fmt,N,K) bytes (padding is written as zeros).  Both are
 * host pointers with no alignment requirement.  Blocks are moved bit for bit:
 * no value is rounded.  Copy the result to the device with cudaMemcpy. */
lean_status lean_pack(int fmt, const void *canon_host, void *packed_host,
                      int64_t N, int64_t K);

/* Host-side inverse of lean_pack: packed -> canonical, byte for byte (no
 * counterpart on the pages: the round trip is this library's check of its
 * own layout). */
lean_status lean_unpack_canonical(int fmt, const void *packed_host, void *canon_host,
                                  int64_t N, int64_t K);

/* Device dequantisation ("oxinfer" crate page, Performance: quantized
 * prefill dequantizes to f32; Platforms and accelerators: weights dequantized
 * to f32 in threadgroup memory): w_dev[n*K + k] = w[n][k] as fp32 (exact: every
 * weight of these formats is an fp32 value).  W_packed_dev: 16-byte aligned
 * device pointer to lean_packed_bytes() bytes made by lean_pack.  w_dev:
 * 16-byte aligned device buffer of N*K floats, overwritten. */
lean_status lean_dequant(int fmt, const void *W_packed_dev, float *w_dev,
                         int64_t N, int64_t K, void *stream);

/* Embedding lookup: the listed rows of a quantized matrix as fp32.
 * The "lean" README (model table) stores the embedding table as Q6_K, and
 * the "oxinfer" crate page (Pre-quantized checkpoints) dequantizes a
 * quantized embedding table one row per token; this is that step, for any of
 * the four formats.  out_dev[i][k] = w[ids_dev[i]][k], bit for bit what
 * lean_dequant gives for that row.
 *   W_packed_dev  device, 16-byte aligned: the N x K table packed by lean_pack
 *   ids_dev       device, 4-byte aligned, int32[n_ids], each in 0 .. N-1 (any
 *                 order, repeats allowed); read only
 *   out_dev       device, 16-byte aligned, float[n_ids][K], overwritten
 * An id outside 0 .. N-1 cannot be reported by the call (it runs on the
 * stream): its row of out_dev is filled with NaN and bit 16 of the device
 * error word is set (lean_device_error).  Host-side errors as for the other
 * calls: LEAN_ERR_FORMAT, LEAN_ERR_SHAPE (n_ids, N or K <= 0, K not a multiple
 * of the block), LEAN_ERR_NULL, LEAN_ERR_ALIGN. */
lean_status lean_embed_rows(int fmt, const void *W_packed_dev, const int32_t *ids_dev,
                            float *out_dev, int64_t n_ids, int64_t N, int64_t K, void *stream);

/* The product.  y[m][n] = sum_k w[n][k] * x[m][k], accumulated in fp32.
 * Pages: "oxinfer" crate page, Performance (decode streams every weight once
 * per token) and How it works (decode tiles over quantized rows); "wgpu-llm"
 * README, Architecture at a Glance (every layer's linears).
 *   W_packed_dev  device, 16-byte aligned, lean_packed_bytes(fmt,N,K) bytes
 *                 made by lean_pack (read only)
 *   x_dev         device, 16-byte aligned, x[M][K] fp32 row-major (read only)
 *   y_dev         device, 4-byte aligned, y[M][N] fp32 row-major, overwritten
 *   stream        cudaStream_t as void*
 * M = 1 is the decode GEMV: a product whose row groups fit the GPU in one
 * wave runs on a kernel that loads all of its weights first and reduces on
 * chip, a larger one streams its weights through a TMA ring.  From M = 2 up to
 * lean_tensor_core_min_m(fmt) - 1 rows (8; Q6_K 4) the product runs on the
 * CUDA cores with each decoded weight reused M times (when a row fits one
 * wave; else a row-tiled kernel).  From lean_tensor_core_min_m(fmt) rows on
 * it runs on the tcgen05 tensor cores, every format: up to 64 rows of x (Q6_K
 * and Q8_0: 32), the integer codes times x = x_hi + x_lo (bf16) with each
 * block scale applied after the MMAs in fp32; more rows, w = w_hi + w_lo
 * times x_hi + x_lo (three MMAs per K step).  Accuracy: |y - y_exact| <= 1e-4 * sum_k |w x| + 1e-6
 * per element.  Nothing is allocated: without a workspace (lean_qmatmul_ws)
 * the tensor-core path splits x inside each CTA. */
lean_status lean_qmatmul(int fmt, const void *W_packed_dev, const float *x_dev,
                         float *y_dev, int64_t N, int64_t K, int64_t M, void *stream);

/* Flags for lean_qmatmul_ex. */
enum {
    /* Programmatic dependent launch: the kernel may be scheduled, and may start
     * streaming W, before the preceding kernel on `stream` has finished; it
     * reads x and writes y only after that kernel has completed and its writes
     * are visible.  Consecutive products on one stream then overlap their
     * weight streaming with each other's tails, which is what a decode step
     * of many small GEMVs needs.  Set it only when the preceding kernel on the
     * stream does not write W (weights uploaded by cudaMemcpy, or resident
     * model weights, are fine). */
    LEAN_FLAG_EARLY_WEIGHTS = 1u,
    /* M = 1 with a workspace, Q4_0 / Q8_0 / I8_B64: always hand x to the
     * product as integer planes (dp4a), not only when the call streams at
     * least 32 MiB of weights.  Ignored otherwise. */
    LEAN_FLAG_X_PLANES = 2u,
    /* M = 1: use the streaming kernel (a TMA-fed ring per SM; with a
     * workspace, K split evenly over all SMs) even for products that fit the
     * GPU in one wave, which otherwise run on a kernel that loads all of its
     * weights before it waits for x and reduces on chip (the lower latency
     * for one product of up to a few tens of MB).  Large products and calls
     * that take x as planes always stream. */
    LEAN_FLAG_STREAM = 4u,
    /* M = 1 with a workspace, Q4_0 / Q8_0 / I8_B64 (LEAN_ERR_FORMAT for Q6_K
     * or M != 1, LEAN_ERR_NULL without a workspace): quantize x to int8 per
     * 32 elements and take int8 dot products, as the "oxinfer" crate page's
     * decode kernels do (How it works: per-matmul activation quantization,
     * int8 SDOT).  Rule: s = max|x| / 127 and q = round(x / s), ties away from
     * zero, both fp32 operations, q in -127..127 (s = 0, q = 0 for a block of
     * zeros).  y is then the product of w with x~ = s * q, not with x: about
     * 1e-3 .. 1e-2 of |y| away from the fp32-x result, and within 1e-4 *
     * sum_k |w x~| + 1e-6 of the exact product with x~.  x must be finite. */
    LEAN_FLAG_X_INT8 = 8u
};

/* lean_qmatmul with launch flags (LEAN_FLAG_*; unknown bits are rejected
 * with LEAN_ERR_FORMAT).  flags = 0 is exactly lean_qmatmul.  Pages: as
 * lean_qmatmul; the flags serve the decode step's chain of small products
 * ("oxinfer" crate page, How it works: ~200 small parallel regions a step). */
lean_status lean_qmatmul_ex(int fmt, const void *W_packed_dev, const float *x_dev,
                            float *y_dev, int64_t N, int64_t K, int64_t M,
                            unsigned flags, void *stream);

/* The fused gate / up projections of a decode layer's FFN, with their
 * epilogue: h[n] = silu(g[n]) * u[n], g = W_gate x, u = W_up x (M = 1),
 * silu(t) = t / (1 + e^-t).  A decode step is N x (attention + FFN) ("wgpu-llm"
 * README, Architecture at a Glance) and the FFN of the models the pages run
 * (SmolLM2, Qwen2.5, TinyLlama) feeds its down projection with silu(gate) *
 * up; this call reads x once per row group for both matrices, never stores
 * g or u, and writes the down projection's input directly, in one launch.
 *   W_gate_dev, W_up_dev  device, 16-byte aligned, both N x K of format fmt,
 *                         packed by lean_pack
 *   x_dev                 device, 16-byte aligned, x[K] fp32
 *   h_dev                 device, 4-byte aligned, h[N] fp32, overwritten; must not
 *                         overlap x or the weights
 *   flags                 0 or LEAN_FLAG_EARLY_WEIGHTS (others: LEAN_ERR_FORMAT)
 * Accuracy: g and u as lean_qmatmul's; h = fl(silu(g~)) * u~ in fp32.
 * LEAN_ERR_SHAPE for K beyond 4 x 8 x (8 Q4_0, 4 Q8_0, 2 INT8-B64, 1 Q6_K)
 * blocks (Q4_0 and Q6_K 8192, the int8 formats 4096), besides the usual shape
 * and pointer errors.  Nothing is allocated. */
lean_status lean_qmatmul_swiglu(int fmt, const void *W_gate_dev, const void *W_up_dev,
                                const float *x_dev, float *h_dev, int64_t N, int64_t K,
                                unsigned flags, void *stream);

/* Rows of x from which lean_qmatmul uses the tensor cores for format fmt: 9
 * (Q4_0, Q8_0, INT8-B64) or 5 (Q6_K); -1 for an unknown format.  The pages
 * hand matmuls of 16 or more tokens from the CPU to the GPU ("oxinfer" crate
 * page, Platforms and accelerators); on the GPU the switch from the CUDA-core
 * kernels to the tensor-core one is set where the measured times cross. */
int lean_tensor_core_min_m(int fmt);

/* Bytes of device workspace that lean_qmatmul_ws uses for this shape (0 when
 * it uses none: 2 <= M < lean_tensor_core_min_m(fmt)), or -1 on a bad fmt or
 * shape.  M = 1: stream-K partial sums and counters.  From
 * lean_tensor_core_min_m(fmt) rows on: x split into bf16 hi / lo operand
 * tiles, 4 bytes per element of x with M padded to 16 and K to 64.  (No
 * counterpart on the pages: scratch of this library's kernels.) */
int64_t lean_qmatmul_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t M);

/* lean_qmatmul_ex with a caller-owned device workspace (pages: as
 * lean_qmatmul; the workspace is this library's).  With a workspace the
 * M = 1 product splits K-steps evenly over all SMs, also inside a 32-row
 * group, and the CTA that finishes a split group last adds the parts up (in
 * a fixed order, so results stay deterministic); without one (NULL) every
 * CTA owns whole row groups, which balances well only when N/32 is much
 * larger than the SM count.
 *   workspace        device, 256-byte aligned, >= lean_qmatmul_workspace_bytes
 *                    bytes.  M = 1: it must be zeroed once (cudaMemset) before
 *                    its first use; every call that completes leaves its
 *                    arrival counters zeroed again (the rest is scratch).
 *                    After a call for which lean_device_error() reports a
 *                    timeout, counters may be left set: zero the workspace
 *                    again before its next use.  For Q4_0, Q8_0 and I8_B64
 *                    calls that stream at least 32 MiB of weights
 *                    (lean_qmatmul_batch of a whole decode step, say), or
 *                    that pass LEAN_FLAG_X_PLANES, a first kernel also writes
 *                    x there as integer planes (a power-of-two scale per 32
 *                    elements, a grid of 2^-21 or, where needed, 2^-29 of the
 *                    block's largest |x|) so that the dot products run on
 *                    dp4a.  A block of x in which even the finer grid would
 *                    move an element by more than 2^-14 of the element
 *                    itself (a small value next to an outlier channel), or
 *                    which holds an Inf or NaN, is marked and takes the exact
 *                    fp32 dot instead: every product w*x errs by at most
 *                    2^-14 * |w*x| before the fp32 sums, whatever x is.
 *                    M >= lean_tensor_core_min_m(fmt): any contents; a first
 *                    kernel writes x there as bf16 hi / lo operand tiles, once
 *                    for all CTAs, which the product then copies with TMA.
 *   workspace_bytes  its size (LEAN_ERR_SHAPE if too small).
 * Calls that may run at the same time on the GPU must not share a workspace.
 * The workspace is ignored for 2 <= M < lean_tensor_core_min_m(fmt). */
lean_status lean_qmatmul_ws(int fmt, const void *W_packed_dev, const float *x_dev,
                            float *y_dev, int64_t N, int64_t K, int64_t M,
                            unsigned flags, void *workspace, int64_t workspace_bytes,
                            void *stream);

/* Several independent M = 1 products of one format in a single launch, for a
 * decode step whose linears do not depend on each other (or one dependency
 * level of a layer, e.g. q/k/v or gate/up).  Their row-group steps are
 * concatenated and streamed by one persistent grid.  With a workspace and at
 * least three 256-row blocks per CTA of the grid (a whole decode step), the
 * CTAs take whole 256-row blocks at run time, largest first, from two
 * counters at the end of the workspace (left at zero by every call); each
 * row is still summed in one fixed order, so results do not depend on the
 * schedule. */
#define LEAN_MAX_BATCH 256
typedef struct {
    const void *W;  /* device, packed by lean_pack, 16-byte aligned         */
    const float *x; /* device, x[K] fp32, 16-byte aligned                   */
    float *y;       /* device, y[N] fp32, overwritten                       */
    int64_t N, K;
} lean_problem;

/* Workspace bytes for lean_qmatmul_batch over these problems, or -1 (no
 * counterpart on the pages). */
int64_t lean_batch_workspace_bytes(int fmt, int count, const lean_problem *problems);

/* Pages: "wgpu-llm" README, Architecture at a Glance (N x (Attn + FFN): the
 * independent linears of a layer); "oxinfer" crate page, How it works (a
 * decode step issues ~200 small parallel regions, so dispatch cost matters).
 * problems: host array of `count` (1..LEAN_MAX_BATCH) descriptors, read during
 * the call only.  workspace / workspace_bytes / flags as for lean_qmatmul_ws
 * (workspace may be NULL).  Outputs of different problems must not overlap
 * each other or any input.  On the x-plane path (Q4_0 / Q8_0 / I8_B64 with a
 * workspace and LEAN_FLAG_X_PLANES) x is read and y written only with plain
 * loads and stores, so x and y may also be pinned host memory that the
 * device addresses directly (cudaHostAlloc / cudaHostRegister under unified
 * addressing): the kernels then move them across the host link themselves.
 * W and the workspace must be device memory. */
lean_status lean_qmatmul_batch(int fmt, int count, const lean_problem *problems,
                               unsigned flags, void *workspace, int64_t workspace_bytes,
                               void *stream);

/* The M = 1 product as lean_qmatmul_ws in workspace (stream-K) mode, with no
 * allocation by the caller: its scratch is a fixed array inside this library
 * (lean_fixed_workspace_bytes() bytes, 3 MiB, held on every GPU that loads the
 * library until the process exits).  The source pages have no counterpart to
 * this entry point; it serves callers that cannot allocate device memory
 * where they run the product (code recorded by stream capture, plugins that
 * must use a host framework's pool, loops that may not risk the
 * synchronisation of cudaMalloc / cudaFree).
 *   - Accepts N up to 8388608 rows (262144 row groups); larger N returns
 *     LEAN_ERR_SHAPE.  W, x, y, flags and stream as for lean_qmatmul_ex, x in
 *     fp32 always (LEAN_FLAG_X_INT8 returns LEAN_ERR_FORMAT).
 *   - The first call on a device looks up the array's device address (and
 *     may load the library's kernels); make it before any stream capture.
 *   - Every call uses the same array: it clears the arrival counters it needs
 *     (cudaMemsetAsync on `stream`) and overwrites the partial sums, so calls
 *     that may overlap on the GPU (other streams, other threads) race and
 *     must be serialised by the caller.  Calls in order on one stream,
 *     including with LEAN_FLAG_EARLY_WEIGHTS, are safe. */
lean_status lean_qmatmul_fixed_ws(int fmt, const void *W_packed_dev, const float *x_dev,
                                  float *y_dev, int64_t N, int64_t K, unsigned flags,
                                  void *stream);

/* Size in bytes of the fixed array behind lean_qmatmul_fixed_ws (no
 * counterpart on the pages). */
int64_t lean_fixed_workspace_bytes(void);

/* No counterpart on the pages (their kernels run on the CPU, and their GPU
 * backends report through the host API): the library's own fault reporting.
 * The device error word of the current device: non-zero when a kernel gave up
 * waiting on one of its own pipeline barriers (a bounded wait timed out and
 * the kernel returned early; its outputs are then invalid) or met an index
 * out of its range.  Bits: 1 a stream consumer waited too long for a slot, 2
 * a stream producer for a free slot, 4 the tensor-core product for a stage, 8
 * lean_wait_selftest, 16 lean_embed_rows was given an id outside 0 .. N-1, 32
 * (LEAN_DEBUG builds only) a kernel computed an index outside the buffers its
 * arguments describe and skipped that access.  Reads it
 * synchronously (the device is synchronised first) and clears it when
 * `clear` is non-zero.  Returns 0xFFFFFFFF if the word cannot be read. */
unsigned lean_device_error(int clear);

/* The device error word as a status, read and cleared as lean_device_error
 * (clear non-zero): LEAN_OK when it is zero, LEAN_ERR_KERNEL_BOUNDS when bit
 * 32 is set, LEAN_ERR_DEVICE for any other bit, LEAN_ERR_CUDA when the word
 * cannot be read.  No counterpart on the pages. */
lean_status lean_device_status(int clear);

/* 1 when this library was built with LEAN_DEBUG (every kernel checks its
 * global-memory indices against the buffers its arguments describe, skips an
 * access outside them and sets bit 32 of the device error word; never a
 * trap), else 0.  No counterpart on the pages. */
int lean_debug_build(void);

/* Self-test of the bounded waits (no counterpart on the pages): launches one
 * 32-thread block on `stream`
 * that waits, with the same bounded mbarrier wait the kernels use, on a
 * barrier that nothing completes, gives up after `limit_us` microseconds
 * (1 .. 1000000) and sets bit 8 of the device error word.  The context stays
 * usable.  LEAN_ERR_SHAPE for a limit out of range. */
lean_status lean_wait_selftest(unsigned limit_us, void *stream);

/* Static description of a status code (no counterpart on the pages). */
const char *lean_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* LEAN_QMATMUL_H */
