// Backward kernel instantiations for f16 IO.
#include "gtms_launch.cuh"

namespace gtms {
template void launch_backward<__half>(int, const void*, const void*, void*, const int32_t*, const Geom&, float,
                                   cudaStream_t);
}  // namespace gtms
