// Instantiations of the fused attention-backward step (bf16 / fp16, head dim 64 / 128).
#include "gtms_attn_bwd.cuh"

namespace gtms {
template cudaError_t launch_attn_dscores<__nv_bfloat16, 64>(const void*, const void*, const void*, void*,
                                                            const int32_t*, int64_t, int64_t, int64_t, float,
                                                            int32_t*, cudaStream_t, uint64_t);
template cudaError_t launch_attn_dscores<__nv_bfloat16, 128>(const void*, const void*, const void*, void*,
                                                             const int32_t*, int64_t, int64_t, int64_t, float,
                                                             int32_t*, cudaStream_t, uint64_t);
template cudaError_t launch_attn_dscores<__half, 64>(const void*, const void*, const void*, void*, const int32_t*,
                                                     int64_t, int64_t, int64_t, float, int32_t*, cudaStream_t, uint64_t);
template cudaError_t launch_attn_dscores<__half, 128>(const void*, const void*, const void*, void*, const int32_t*,
                                                      int64_t, int64_t, int64_t, float, int32_t*, cudaStream_t, uint64_t);
}  // namespace gtms
