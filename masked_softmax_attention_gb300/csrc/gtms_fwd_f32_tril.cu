// Forward kernel instantiations: f32 IO, mask kind 0 (tril).
#include "gtms_launch.cuh"

namespace gtms {
template cudaError_t launch_forward<float, 0>(int, const void*, void*, const int32_t*, const Geom&, float, cudaStream_t);
}  // namespace gtms
