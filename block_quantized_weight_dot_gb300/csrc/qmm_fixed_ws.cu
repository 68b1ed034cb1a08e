// qmm_fixed_ws.cu -- the M = 1 product in workspace (stream-K) mode with its
// scratch in a fixed device array of this library instead of caller memory.
//
// Some callers cannot allocate device memory at the point where they run the
// product: code recorded into a CUDA graph with stream capture (cudaMalloc is
// not a stream operation and is refused during capture), plugins that must
// draw every byte from a host framework's own pool, and real-time loops that
// may not call cudaMalloc / cudaFree because those can synchronise the
// device.  This entry point needs no allocation from them: the scratch is a
// file-scope __device__ array that every GPU loading the library holds until
// the process exits.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/lean_qmatmul.h"
#include "dispatch.h"
#include "layout.h"

using namespace lean;

namespace {

// Partial sums of row groups split between CTAs (2 MiB), then one arrival
// counter per row group: 1 MiB of counters, i.e. at most 262144 row groups.
constexpr int64_t kFixedWorkspaceBytes = (int64_t)3 << 20;

}  // namespace

static __device__ __align__(256) unsigned char lean_fixed_workspace[kFixedWorkspaceBytes];

namespace {

// Device address of the array on the current device, looked up once per
// device (the name is only a host-side stand-in in host code).
void *fixed_workspace() {
    static std::atomic<void *> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    void *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, lean_fixed_workspace) != cudaSuccess) return nullptr;
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" {

int64_t lean_fixed_workspace_bytes(void) { return kFixedWorkspaceBytes; }

lean_status lean_qmatmul_fixed_ws(int fmt, const void *W_packed_dev, const float *x_dev,
                                  float *y_dev, int64_t N, int64_t K, unsigned flags,
                                  void *stream) {
    if (block_elems(fmt) == 0) return LEAN_ERR_FORMAT;
    if (flags & LEAN_FLAG_X_INT8) return LEAN_ERR_FORMAT;  // no room for x codes in the array
    Geom g;
    if (!make_geom(fmt, N, K, &g)) return LEAN_ERR_SHAPE;
    const WorkspaceLayout wl = workspace_layout(g.groups);
    if (wl.total > kFixedWorkspaceBytes) return LEAN_ERR_SHAPE;  // N beyond the array's limit
    void *ws = fixed_workspace();
    if (!ws) return LEAN_ERR_CUDA;
    // The counters must start at zero; a call that gave up on a timeout could
    // have left some set, so the call clears the ones it uses (after its
    // arguments have been checked).  x stays fp32 here: the array has no room
    // for the x planes of every K.
    return qmatmul_m1_ws(fmt, W_packed_dev, x_dev, y_dev, N, K, flags, ws, wl.total, false, true,
                         (cudaStream_t)stream);
}

}  // extern "C"
