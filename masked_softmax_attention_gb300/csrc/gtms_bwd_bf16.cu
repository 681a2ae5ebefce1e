// Backward kernel instantiations for bf16 IO.
#include "gtms_launch.cuh"

namespace gtms {
template void launch_backward<__nv_bfloat16>(int, const void*, const void*, void*, const int32_t*, const Geom&, float,
                                   cudaStream_t);
}  // namespace gtms
