// Backward kernel instantiations: f32 IO, mask kind 1 (length).
#include "gtms_launch.cuh"

namespace gtms {
template cudaError_t launch_backward<float, 1>(int, const void*, const void*, void*, const int32_t*, const Geom&, float,
                                         cudaStream_t);
}  // namespace gtms
