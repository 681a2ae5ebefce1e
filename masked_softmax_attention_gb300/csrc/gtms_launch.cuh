// gtms_launch.cuh -- launchers that map a variant index to a kernel instantiation.
#pragma once

#include <cuda_runtime.h>

#include "gtms_dispatch.h"
#include "gtms_kernels.cuh"

namespace gtms {

// Grid: one team per row, capped; the kernels stride over any remaining rows.
template <int TW>
inline unsigned grid_for(int64_t rows)
{
    const int64_t teams_per_cta = TW == 32 ? kWarpTeamBlock / 32 : 1;
    int64_t ctas = (rows + teams_per_cta - 1) / teams_per_cta;
    const int64_t cap = 1 << 30;
    if (ctas > cap)
        ctas = cap;
    return static_cast<unsigned>(ctas);
}

template <typename T, bool VEC, int TW, int NV>
inline void launch_fwd_v(const void* x, void* y, const int32_t* seq_lens, const Geom& g, float scale,
                         cudaStream_t st)
{
    gtms_fwd_kernel<T, VEC, TW, NV><<<grid_for<TW>(g.rows), TW == 32 ? kWarpTeamBlock : TW, 0, st>>>(
        static_cast<const T*>(x), static_cast<T*>(y), seq_lens, g, scale);
}

template <typename T, bool VEC, int TW, int NV>
inline void launch_bwd_v(const void* y, const void* dy, void* dx, const int32_t* seq_lens, const Geom& g,
                         float scale, cudaStream_t st)
{
    gtms_bwd_kernel<T, VEC, TW, NV><<<grid_for<TW>(g.rows), TW == 32 ? kWarpTeamBlock : TW, 0, st>>>(
        static_cast<const T*>(y), static_cast<const T*>(dy), static_cast<T*>(dx), seq_lens, g, scale);
}

// The case labels follow kVecVariants then kElemVariants in gtms_dispatch.h.
constexpr bool variant_is(int i, bool vec, int tw, int nv)
{
    return (i < kNumVec ? kVecVariants[i] : kElemVariants[i - kNumVec]).vec16 == vec &&
           (i < kNumVec ? kVecVariants[i] : kElemVariants[i - kNumVec]).team == tw &&
           (i < kNumVec ? kVecVariants[i] : kElemVariants[i - kNumVec]).per_thread == nv;
}
static_assert(kNumVec == 7 && kNumElem == 6, "variant table and switch out of step");
static_assert(variant_is(0, true, 32, 1) && variant_is(1, true, 32, 2) && variant_is(2, true, 32, 4) &&
                  variant_is(3, true, 32, 8) && variant_is(4, true, 128, 4) && variant_is(5, true, 256, 4) &&
                  variant_is(6, true, 512, 4) && variant_is(7, false, 32, 1) && variant_is(8, false, 32, 4) &&
                  variant_is(9, false, 32, 16) && variant_is(10, false, 32, 32) &&
                  variant_is(11, false, 128, 32) && variant_is(12, false, 256, 32),
              "variant table and switch out of step");
#define GTMS_VARIANT_CASES(CALL)        \
    case 0: CALL(true, 32, 1); break;   \
    case 1: CALL(true, 32, 2); break;   \
    case 2: CALL(true, 32, 4); break;   \
    case 3: CALL(true, 32, 8); break;   \
    case 4: CALL(true, 128, 4); break;  \
    case 5: CALL(true, 256, 4); break;  \
    case 6: CALL(true, 512, 4); break;  \
    case 7: CALL(false, 32, 1); break;  \
    case 8: CALL(false, 32, 4); break;  \
    case 9: CALL(false, 32, 16); break; \
    case 10: CALL(false, 32, 32); break; \
    case 11: CALL(false, 128, 32); break; \
    case 12: CALL(false, 256, 32); break;

template <typename T>
void launch_forward(int variant, const void* x, void* y, const int32_t* seq_lens, const Geom& g, float scale,
                    cudaStream_t st)
{
#define GTMS_FWD_CALL(V, TW, NV) launch_fwd_v<T, V, TW, NV>(x, y, seq_lens, g, scale, st)
    switch (variant) { GTMS_VARIANT_CASES(GTMS_FWD_CALL) default: break; }
#undef GTMS_FWD_CALL
}

template <typename T>
void launch_backward(int variant, const void* y, const void* dy, void* dx, const int32_t* seq_lens,
                     const Geom& g, float scale, cudaStream_t st)
{
#define GTMS_BWD_CALL(V, TW, NV) launch_bwd_v<T, V, TW, NV>(y, dy, dx, seq_lens, g, scale, st)
    switch (variant) { GTMS_VARIANT_CASES(GTMS_BWD_CALL) default: break; }
#undef GTMS_BWD_CALL
}

}  // namespace gtms
