// qmm_q4_0.cu -- Q4_0 instantiation of the CUDA-core product and dequant kernels.
#include "simt_launch.cuh"

namespace lean {
template lean_status qmm_fmt<Q4_0>(const Geom &, const uint8_t *, const float *, float *, int64_t,
                                 unsigned, cudaStream_t);
template lean_status dequant_fmt<Q4_0>(const Geom &, const uint8_t *, float *, cudaStream_t);
}  // namespace lean
