// Backward kernel instantiations: f16 IO, mask kind 0 (tril).
#include "gtms_launch.cuh"

namespace gtms {
template cudaError_t launch_backward<__half, 0>(int, const void*, const void*, void*, const int32_t*, const Geom&, float,
                                         cudaStream_t);
}  // namespace gtms
