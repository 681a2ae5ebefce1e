// Explicit-mask kernel instantiations for f16 IO (forward and backward).
#include "gtms_explicit.cuh"

namespace gtms {
template cudaError_t launch_forward_explicit<__half>(int, const void*, void*, const uint8_t*, int32_t, const Geom&, float,
                                          cudaStream_t);
template cudaError_t launch_backward_explicit<__half>(int, const void*, const void*, void*, const uint8_t*, int32_t,
                                           const Geom&, float, cudaStream_t);
}  // namespace gtms
