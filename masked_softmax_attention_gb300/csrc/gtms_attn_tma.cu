// Instantiations of the TMA-fed fused attention-backward step (bf16 / fp16, head dim 64 / 128).
#include "gtms_attn_tma.cuh"

namespace gtms {
#define GTMS_ATTN_TMA(T, D)                                                                                      \
    template cudaError_t launch_attn_dscores_tma<T, D>(const void*, const void*, const void*, void*,            \
                                                       const int32_t*, int64_t, int64_t, int64_t, float,        \
                                                       int32_t*, cudaStream_t, uint64_t);
GTMS_ATTN_TMA(__nv_bfloat16, 64)
GTMS_ATTN_TMA(__nv_bfloat16, 128)
GTMS_ATTN_TMA(__half, 64)
GTMS_ATTN_TMA(__half, 128)
#undef GTMS_ATTN_TMA
}  // namespace gtms
