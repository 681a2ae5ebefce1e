// Staged-forward instantiations (grouped tril mask; fp32, bf16, fp16).
#include "gtms_dispatch.h"
#include "gtms_staged.cuh"

namespace gtms {

template <typename T>
cudaError_t launch_forward_staged(int id, const void* x, void* y, const int32_t* seq_lens, const Geom& g, float scale,
                                  cudaStream_t st)
{
#define GTMS_STAGED_CASE(vid, tw, nv, ns, mb) \
    case vid: return launch_fwd_staged<T, kMaskGroupedTril, tw, nv, ns, mb>(x, y, seq_lens, g, scale, st, kAttnWaitNs);
    if constexpr (sizeof(T) == 4) {
        switch (id) { GTMS_FWD_STAGED4(GTMS_STAGED_CASE) default: break; }
    } else {
        switch (id) { GTMS_FWD_STAGED2(GTMS_STAGED_CASE) default: break; }
    }
#undef GTMS_STAGED_CASE
    return cudaErrorInvalidValue;   // no kernel for this variant id
}

template cudaError_t launch_forward_staged<float>(int, const void*, void*, const int32_t*, const Geom&, float,
                                                  cudaStream_t);
template cudaError_t launch_forward_staged<__nv_bfloat16>(int, const void*, void*, const int32_t*, const Geom&, float,
                                                          cudaStream_t);
template cudaError_t launch_forward_staged<__half>(int, const void*, void*, const int32_t*, const Geom&, float,
                                                   cudaStream_t);

}  // namespace gtms
