/* lean_quant.h -- float weights to canonical Q4_0 / Q8_0 / INT8-B64 blocks.
 *
 * The load-time step before lean_pack: the pages quantize model weights into
 * these blocks when a model is loaded ("oxinfer" crate page, How it works:
 * quant.rs, Q8 blocks of 32 weights with one scale and Q4_0 with two nibbles
 * per byte and an f16 scale; "wgpu-llm" README, INT8 mode: block size 64).
 * Host code, no GPU involved.
 *
 * The pages state no rounding rule.  This one is used (per block of 32, or 64
 * for LEAN_I8_B64, along K):
 *   LEAN_Q8_0, LEAN_I8_B64: d = the binary16 value nearest to max|w| / 127
 *     (ties to even); q = the integer nearest to w / d, ties away from zero,
 *     clamped to -127..127.
 *   LEAN_Q4_0: m = the element of largest |w| (the first of equal ones);
 *     d = the binary16 value nearest to m / -8 (so m comes back exactly up
 *     to d's rounding, as d * (0 - 8)); q = (the integer nearest to w / d,
 *     ties away from zero) + 8, clamped to 0..15.
 *   A block whose d rounds to zero stores d = +0 and every value 0.
 * The results are bit-for-bit reproducible on any host.
 */
#ifndef LEAN_QUANT_H
#define LEAN_QUANT_H

#include <stdint.h>

#include "lean_qmatmul.h"

#ifdef __cplusplus
extern "C" {
#endif

/* w_host: host, fp32 w[N][K], row-major.  canon_host: host, receives
 * lean_canonical_bytes(fmt, N, K) bytes of canonical blocks (rows of K /
 * block weights), ready for lean_pack.  threads: host threads to use (0: all
 * of them).  Errors: LEAN_ERR_FORMAT for LEAN_Q6_K or an unknown format,
 * LEAN_ERR_NULL for a null pointer, LEAN_ERR_SHAPE for N or K <= 0, K not a
 * multiple of the block, threads < 0, a weight that is not finite or a block
 * whose d would exceed 65504 (canon_host is then partly written). */
lean_status lean_quantize(int fmt, const float *w_host, void *canon_host, int64_t N, int64_t K,
                          int threads);

#ifdef __cplusplus
}
#endif

#endif /* LEAN_QUANT_H */
