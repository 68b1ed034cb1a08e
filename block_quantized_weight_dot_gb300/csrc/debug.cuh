// debug.cuh -- index checks of the LEAN_DEBUG build.
//
// Built with -DLEAN_DEBUG (lean_debug_build() then returns 1), every kernel
// checks the global-memory indices it computes against the extent of the
// buffer its arguments describe, before the access.  An index outside it
// sets kErrBounds in the device error word and the access is skipped: a load
// reads zero, a store is dropped, a bulk copy is not issued (and its bytes
// are left out of the barrier's expected count, so no wait is left hanging).
// Nothing traps; lean_device_status() then returns LEAN_ERR_KERNEL_BOUNDS.
// Without LEAN_DEBUG every check is the constant true and compiles away.
#pragma once
#include <stdint.h>

#include "layout.h"

namespace lean {

#ifdef LEAN_DEBUG
// i in [0, n)
__device__ __forceinline__ bool dbg_in(int64_t i, int64_t n, unsigned *err) {
    if (i >= 0 && i < n) return true;
    if (err) atomicOr(err, kErrBounds);
    return false;
}
// [off, off + len) inside [0, n)
__device__ __forceinline__ bool dbg_span(int64_t off, int64_t len, int64_t n, unsigned *err) {
    if (off >= 0 && len >= 0 && off + len <= n) return true;
    if (err) atomicOr(err, kErrBounds);
    return false;
}
#define LEAN_IN(i, n, err) ::lean::dbg_in((int64_t)(i), (int64_t)(n), (err))
#define LEAN_SPAN(off, len, n, err) ::lean::dbg_span((int64_t)(off), (int64_t)(len), (int64_t)(n), (err))
#else
// (the operands still go through a function, so that variables which only the
// checks read count as used; their values are dead and compile away)
__device__ __forceinline__ bool dbg_none(int64_t, int64_t, int64_t, const unsigned *) { return true; }
#define LEAN_IN(i, n, err) ::lean::dbg_none((int64_t)(i), 0, (int64_t)(n), (err))
#define LEAN_SPAN(off, len, n, err) ::lean::dbg_none((int64_t)(off), (int64_t)(len), (int64_t)(n), (err))
#endif

}  // namespace lean
