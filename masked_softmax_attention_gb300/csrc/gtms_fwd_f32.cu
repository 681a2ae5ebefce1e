// Forward kernel instantiations for f32 IO.
#include "gtms_launch.cuh"

namespace gtms {
template void launch_forward<float>(int, const void*, void*, const int32_t*, const Geom&, float, cudaStream_t);
}  // namespace gtms
