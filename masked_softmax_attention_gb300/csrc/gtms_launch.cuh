// gtms_launch.cuh -- map a variant id (gtms_dispatch.h) to a kernel instantiation.
#pragma once

#include <cuda_runtime.h>

#include "gtms_dispatch.h"
#include "gtms_kernels.cuh"
#include "gtms_band.cuh"
#include "gtms_stream.cuh"

namespace gtms {

// Grid: one team per row (capped); the kernels stride over any remaining rows.
template <int TW>
inline unsigned grid_for(int64_t rows)
{
    const int64_t teams_per_cta = TW == 32 ? kWarpTeamBlock / 32 : 1;
    int64_t ctas = (rows + teams_per_cta - 1) / teams_per_cta;
    const int64_t cap = int64_t(1) << 30;
    return static_cast<unsigned>(ctas > cap ? cap : ctas);
}

template <int TW>
constexpr int block_for() { return TW == 32 ? kWarpTeamBlock : TW; }

template <typename T, int MK>
cudaError_t launch_forward_mk(int id, const void* x, void* y, const int32_t* seq_lens, const Geom& g, float scale,
                              cudaStream_t st)
{
    const T* xp = static_cast<const T*>(x);
    T* yp = static_cast<T*>(y);
    const int64_t pairs = g.rows / (g.rows_per_b / g.S);   // (batch, row) pairs: the heads kernels' teams
// (16-bit CTA-team rows launch as heads kernels, so their per-row form is not instantiated.)
#define GTMS_FWD_VEC_CASE(vid, tw, nv, mb)                                                                        \
    case vid:                                                                                                     \
        if constexpr (sizeof(T) == 4 || tw == 32)                                                                 \
            return launch_kernel(gtms_fwd_vec_kernel<T, MK, tw, nv, mb>, grid_for<tw>(g.rows), block_for<tw>(), 0, \
                                 st, xp, yp, seq_lens, g, scale);                                                 \
        break;
#define GTMS_FWD_ELEM_CASE(vid, tw, nv)                                                                               \
    case kElemBase + vid:                                                                                             \
        return launch_kernel(gtms_fwd_elem_kernel<T, MK, tw, nv>, grid_for<tw>(g.rows), block_for<tw>(), 0, st, xp, yp, \
                             seq_lens, g, scale);
#define GTMS_FWD_HEADS_CASE(vid, tw, nv, mb)                                                                         \
    case kHeadsBase + vid:                                                                                           \
        return launch_kernel(gtms_fwd_heads_kernel<T, MK, tw, nv, mb>, grid_for<tw>(pairs), block_for<tw>(), 0, st, \
                             xp, yp, seq_lens, g, scale);
    if constexpr (sizeof(T) == 2) {
        switch (id) { GTMS_FWD_HEADS2(GTMS_FWD_HEADS_CASE) default: break; }
    }
#undef GTMS_FWD_HEADS_CASE
#define GTMS_FWD_BAND_CASE(vid, nv, mb)                                                                          \
    case kBandBase + vid:                                                                                        \
        return launch_kernel(gtms_fwd_band_kernel<T, nv, mb>, grid_for<32>(g.rows), block_for<32>(), 0, st, xp, yp, \
                             seq_lens, g, scale);
    if constexpr (MK == kMaskWindow) {
        switch (id) { GTMS_FWD_BAND(GTMS_FWD_BAND_CASE) default: break; }
    }
#undef GTMS_FWD_BAND_CASE
#define GTMS_FWD_ST_CASE(vid, tw, nv, mb, mu)                                                                  \
    case kStreamBase + vid:                                                                                    \
        return launch_kernel(gtms_fwd_stream_kernel<T, MK, tw, nv, mb>, grid_for<tw>(g.rows), tw, 0, st, xp, yp, \
                             seq_lens, g, scale);
    if constexpr (sizeof(T) == 4) {
        switch (id) { GTMS_FWD_VEC4(GTMS_FWD_VEC_CASE) GTMS_ELEM(GTMS_FWD_ELEM_CASE)
                      GTMS_FWD_ST4(GTMS_FWD_ST_CASE) default: break; }
    } else {
        switch (id) { GTMS_FWD_VEC2(GTMS_FWD_VEC_CASE) GTMS_ELEM(GTMS_FWD_ELEM_CASE)
                      GTMS_FWD_ST2(GTMS_FWD_ST_CASE) default: break; }
    }
#undef GTMS_FWD_VEC_CASE
#undef GTMS_FWD_ELEM_CASE
#undef GTMS_FWD_ST_CASE
    return cudaErrorInvalidValue;   // no kernel for this variant id
}

template <typename T, int MK>
cudaError_t launch_backward_mk(int id, const void* y, const void* dy, void* dx, const int32_t* seq_lens, const Geom& g,
                               float scale, cudaStream_t st)
{
    const T* yp = static_cast<const T*>(y);
    const T* gp = static_cast<const T*>(dy);
    T* dp = static_cast<T*>(dx);
#define GTMS_BWD_VEC_CASE(vid, tw, nv, mb)                                                                          \
    case vid:                                                                                                       \
        return launch_kernel(gtms_bwd_vec_kernel<T, MK, tw, nv, mb>, grid_for<tw>(g.rows), block_for<tw>(), 0, st, \
                             yp, gp, dp, seq_lens, g, scale);
#define GTMS_BWD_ELEM_CASE(vid, tw, nv)                                                                           \
    case kElemBase + vid:                                                                                         \
        return launch_kernel(gtms_bwd_elem_kernel<T, MK, tw, nv>, grid_for<tw>(g.rows), block_for<tw>(), 0, st, yp, \
                             gp, dp, seq_lens, g, scale);
#define GTMS_BWD_BAND_CASE(vid, nv, mb)                                                                          \
    case kBandBase + vid:                                                                                        \
        return launch_kernel(gtms_bwd_band_kernel<T, nv, mb>, grid_for<32>(g.rows), block_for<32>(), 0, st, yp, gp, \
                             dp, seq_lens, g, scale);
    if constexpr (MK == kMaskWindow) {
        switch (id) { GTMS_BWD_BAND(GTMS_BWD_BAND_CASE) default: break; }
    }
#undef GTMS_BWD_BAND_CASE
#define GTMS_BWD_ST_CASE(vid, tw, nv, mb, mu)                                                                  \
    case kStreamBase + vid:                                                                                    \
        return launch_kernel(gtms_bwd_stream_kernel<T, MK, tw, nv, mb>, grid_for<tw>(g.rows), tw, 0, st, yp, gp, \
                             dp, seq_lens, g, scale);
    if constexpr (sizeof(T) == 4) {
        switch (id) { GTMS_BWD_VEC4(GTMS_BWD_VEC_CASE) GTMS_ELEM(GTMS_BWD_ELEM_CASE)
                      GTMS_BWD_ST4(GTMS_BWD_ST_CASE) default: break; }
    } else {
        switch (id) { GTMS_BWD_VEC2(GTMS_BWD_VEC_CASE) GTMS_ELEM(GTMS_BWD_ELEM_CASE)
                      GTMS_BWD_ST2(GTMS_BWD_ST_CASE) default: break; }
    }
#undef GTMS_BWD_VEC_CASE
#undef GTMS_BWD_ELEM_CASE
#undef GTMS_BWD_ST_CASE
    return cudaErrorInvalidValue;   // no kernel for this variant id
}

// One translation unit instantiates one mask kind of one dtype and direction.
template <typename T, int MK>
cudaError_t launch_forward(int id, const void* x, void* y, const int32_t* seq_lens, const Geom& g, float scale,
                           cudaStream_t st)
{
    return launch_forward_mk<T, MK>(id, x, y, seq_lens, g, scale, st);
}

template <typename T, int MK>
cudaError_t launch_backward(int id, const void* y, const void* dy, void* dx, const int32_t* seq_lens, const Geom& g,
                            float scale, cudaStream_t st)
{
    return launch_backward_mk<T, MK>(id, y, dy, dx, seq_lens, g, scale, st);
}

}  // namespace gtms
