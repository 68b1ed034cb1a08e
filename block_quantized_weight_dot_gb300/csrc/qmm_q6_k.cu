// qmm_q6_k.cu -- Q6_K instantiation of the product and dequantisation kernels.
#include "launch.cuh"

namespace lean {
LEAN_INSTANTIATE(Q6_K)
}  // namespace lean
