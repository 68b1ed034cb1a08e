// qmm_i8_b64.cu -- I8_B64 instantiation of the product and dequantisation kernels.
#include "launch.cuh"

namespace lean {
LEAN_INSTANTIATE(I8_B64)
}  // namespace lean
