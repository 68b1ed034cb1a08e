// qmm_q8_0.cu -- Q8_0 instantiation of the product and dequantisation kernels.
#include "launch.cuh"

namespace lean {
LEAN_INSTANTIATE(Q8_0)
}  // namespace lean
