// qmm_q4_0.cu -- Q4_0 instantiation of the product and dequantisation kernels.
#include "launch.cuh"

namespace lean {
LEAN_INSTANTIATE(Q4_0)
}  // namespace lean
