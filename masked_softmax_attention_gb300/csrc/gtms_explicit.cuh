// gtms_explicit.cuh -- masked softmax with an explicit keep mask
// ("优化ScaledMaskSoftmax算子", sections 2.2 and 3.1: the op takes the input, a
// mask tensor and the scale; section 4.1: a row with nothing kept is zero).
//
// The mask is uint8 [mask_batches, S, S] (mask_batches 1 or B), shared by the M
// heads; a nonzero byte keeps the entry. Kept entries of a row need not be
// contiguous, so every unit is masked per element. A team takes one (batch,
// row) pair and its M heads: each thread loads the mask bytes of its 16-byte
// units once (4 bytes per fp32 unit, 8 per 16-bit unit) and keeps the bits
// for every head; a unit with no kept element loads no x and is stored as
// +0.0, so masked inputs are still never read. The forward loads the next
// head's kept units as soon as it has decoded the current head's, so those
// loads are in flight through the current head's two reductions and its
// stores. The arithmetic is the vector kernels' (fp32 pairs, one
// ex2.approx.f32 per kept element, float-float backward dot).
#pragma once

#include "gtms_kernels.cuh"

namespace gtms {

// Keep bits (bit e = element e kept) of the EPU mask bytes of one unit.
template <int EPU>
__device__ __forceinline__ uint32_t keep_bits(const uint8_t* mrow, int j)
{
    if constexpr (EPU == 4) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(mrow + 4 * j);
        uint32_t bits = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            bits |= ((w >> (8 * e)) & 0xffu) ? (1u << e) : 0u;
        return bits;
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(mrow + 8 * j);
        uint32_t bits = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bits |= ((w.x >> (8 * e)) & 0xffu) ? (1u << e) : 0u;
            bits |= ((w.y >> (8 * e)) & 0xffu) ? (1u << (e + 4)) : 0u;
        }
        return bits;
    }
}

__device__ __forceinline__ const uint8_t* explicit_mask_row(const uint8_t* mask, int32_t mask_batches, int32_t b,
                                                            int32_t r, int32_t S)
{
    const int64_t mb = mask_batches == 1 ? 0 : b;
    return mask + (mb * S + r) * static_cast<int64_t>(S);
}

template <typename T, int TW, int NV, int MINB>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW, MINB)
gtms_fwd_explicit_kernel(const T* x, T* y, const uint8_t* __restrict__ mask, int32_t mask_batches, Geom g,
                         float scale)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs, EPU = 2 * PPU;
    __shared__ float red[TW > 32 ? 2 * (TW / 32) : 1];
    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    const float neutral = use_max ? -INFINITY : INFINITY;
    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);

    // A team takes one (batch, row) pair and all M heads of it: the row's mask
    // bits are read once and serve every head.
    const int32_t M = static_cast<int32_t>(g.rows_per_b / g.S);
    for (int64_t qm = team; qm < g.rows / M; qm += nteams) {
        const int32_t b = static_cast<int32_t>(qm / g.S), r = static_cast<int32_t>(qm % g.S);
        const uint8_t* mrow = explicit_mask_row(mask, mask_batches, b, r, g.S);
        uint32_t kb[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            kb[k] = j < g.units ? keep_bits<EPU>(mrow, j) : 0u;
        }
        // Head 0's kept units; each head then loads the next head's units as
        // soon as it has decoded its own, so those loads overlap its reductions.
        Unit16 raw[NV];
        {
            const char* x0 = reinterpret_cast<const char*>(x + (static_cast<int64_t>(b) * M * g.S + r) * g.S);
#pragma unroll
            for (int k = 0; k < NV; ++k)
                if (kb[k])
                    raw[k] = load16(x0 + 16 * (tid + k * TW));
        }
      for (int32_t m = 0; m < M; ++m) {
        const int64_t q = (static_cast<int64_t>(b) * M + m) * g.S + r;
        char* yr = reinterpret_cast<char*>(y + q * g.S);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (!kb[k] && j < g.units)
                store16(yr + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
        }

        float2 v[NV][PPU];
        float ext = neutral;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (kb[k]) {
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    v[k][p] = IO::get(raw[k], p);
                    if (!(kb[k] & (1u << (2 * p))))
                        v[k][p].x = neutral;
                    if (!(kb[k] & (2u << (2 * p))))
                        v[k][p].y = neutral;
                    ext = use_max ? max3(ext, v[k][p].x, v[k][p].y) : min3(ext, v[k][p].x, v[k][p].y);
                }
            }
        }
        if (m + 1 < M) {   // the next head's row is S rows further on
            const char* xn = reinterpret_cast<const char*>(x + (q + g.S) * g.S);
#pragma unroll
            for (int k = 0; k < NV; ++k)
                if (kb[k])
                    raw[k] = load16(xn + 16 * (tid + k * TW));
        }
        ext = use_max ? team_max<TW>(ext, red) : -team_max<TW>(-ext, red);

        const float2 shift = splat2(-ext), c2 = splat2(c);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (kb[k]) {
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    const float2 t = __fmul2_rn(__fadd2_rn(v[k][p], shift), c2);
                    v[k][p].x = (kb[k] & (1u << (2 * p))) ? ex2(t.x) : 0.0f;
                    v[k][p].y = (kb[k] & (2u << (2 * p))) ? ex2(t.y) : 0.0f;
                    acc = __fadd2_rn(acc, v[k][p]);
                }
            }
        }
        const float s = team_sum<TW>(__fadd_rn(acc.x, acc.y), red + (TW > 32 ? TW / 32 : 0));
        // A row with nothing kept has s == 0 and has already been stored as zeros.
        const float2 inv = splat2(s > 0.0f ? __frcp_rn(s) : 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (kb[k]) {
                Unit16 o;
#pragma unroll
                for (int p = 0; p < PPU; ++p)
                    IO::put(o, p, __fmul2_rn(v[k][p], inv));
                store16(yr + 16 * j, o);
            }
        }
      }
    }
}

template <typename T, int TW, int NV, int MINB>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW, MINB)
gtms_bwd_explicit_kernel(const T* y, const T* dy, T* dx, const uint8_t* __restrict__ mask, int32_t mask_batches,
                         Geom g, float scale)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs, EPU = 2 * PPU;
    __shared__ float red[2][TW > 32 ? 2 * (TW / 32) : 1];
    int par = 0;
    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);
    const float2 sc = splat2(scale);

    // A team takes one (batch, row) pair and all M heads of it (mask bits read once).
    const int32_t M = static_cast<int32_t>(g.rows_per_b / g.S);
    for (int64_t qm = team; qm < g.rows / M; qm += nteams) {
        const int32_t b = static_cast<int32_t>(qm / g.S), r = static_cast<int32_t>(qm % g.S);
        const uint8_t* mrow = explicit_mask_row(mask, mask_batches, b, r, g.S);
        uint32_t kb[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            kb[k] = j < g.units ? keep_bits<EPU>(mrow, j) : 0u;
        }
      for (int32_t m = 0; m < M; ++m) {
        const int64_t q = (static_cast<int64_t>(b) * M + m) * g.S + r;
        const char* yr = reinterpret_cast<const char*>(y + q * g.S);
        const char* gr = reinterpret_cast<const char*>(dy + q * g.S);
        char* dr = reinterpret_cast<char*>(dx + q * g.S);
        Unit16 ry[NV], rg[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (kb[k]) {
                ry[k] = load16(yr + 16 * j);
                rg[k] = load16(gr + 16 * j);
            } else if (j < g.units) {
                store16(dr + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
            }
        }

        float2 hi2 = make_float2(0.0f, 0.0f), lo2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (kb[k]) {
                IO::clear_unkept(ry[k], kb[k]);   // masked elements (and any NaN there) become 0
                IO::clear_unkept(rg[k], kb[k]);
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    const float2 a = IO::get(ry[k], p), cdy = IO::get(rg[k], p);
                    const float2 pr = __fmul2_rn(a, cdy);
                    const float2 s = __fadd2_rn(hi2, pr);
                    const float2 bb = __fadd2_rn(s, neg2(hi2));
                    const float2 e = __fadd2_rn(__fadd2_rn(hi2, neg2(__fadd2_rn(s, neg2(bb)))),
                                                __fadd2_rn(pr, neg2(bb)));
                    if constexpr (IO::kExactProducts) {
                        lo2 = __fadd2_rn(lo2, e);
                    } else {
                        const float2 pe = __ffma2_rn(a, cdy, neg2(pr));
                        lo2 = __fadd2_rn(lo2, __fadd2_rn(e, pe));
                    }
                    hi2 = s;
                }
            }
        }
        float hi, lo, e0;
        two_sum(hi2.x, hi2.y, hi, e0);
        lo = __fadd_rn(__fadd_rn(lo2.x, lo2.y), e0);
        team_ff_sum<TW>(hi, lo, red[par]);
        par ^= 1;
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));
        const float2 ndh = splat2(-dh), ndl = splat2(-dl);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (kb[k]) {
                Unit16 o;
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    const float2 a = IO::get(ry[k], p), cdy = IO::get(rg[k], p);
                    IO::put(o, p, __fmul2_rn(__fmul2_rn(a, __fadd2_rn(__fadd2_rn(cdy, ndh), ndl)), sc));
                }
                IO::clear_unkept(o, kb[k]);   // masked outputs are +0.0 bits
                store16(dr + 16 * j, o);
            }
        }
      }
    }
}

}  // namespace gtms

#include "gtms_dispatch.h"
#include "gtms_launch.cuh"

namespace gtms {

// Explicit-mask launchers: the per-row vector variants of gtms_dispatch.h (the
// forward with its own register caps, GTMS_EXF_VEC*).
template <typename T>
cudaError_t launch_forward_explicit(int id, const void* x, void* y, const uint8_t* mask, int32_t mask_batches,
                                    const Geom& g, float scale, cudaStream_t st)
{
    const T* xp = static_cast<const T*>(x);
    T* yp = static_cast<T*>(y);
    const int64_t pairs = g.rows / (g.rows_per_b / g.S);   // (batch, row) pairs: one team each
#define GTMS_EX_FWD_CASE(vid, tw, nv, mb)                                                                          \
    case vid:                                                                                                      \
        return launch_kernel(gtms_fwd_explicit_kernel<T, tw, nv, mb>, grid_for<tw>(pairs), block_for<tw>(), 0, st, \
                             xp, yp, mask, mask_batches, g, scale);
    if constexpr (sizeof(T) == 4) {
        switch (id) { GTMS_EXF_VEC4(GTMS_EX_FWD_CASE) default: break; }
    } else {
        switch (id) { GTMS_EXF_VEC2(GTMS_EX_FWD_CASE) default: break; }
    }
#undef GTMS_EX_FWD_CASE
    return cudaErrorInvalidValue;   // no kernel for this variant id
}

template <typename T>
cudaError_t launch_backward_explicit(int id, const void* y, const void* dy, void* dx, const uint8_t* mask,
                                     int32_t mask_batches, const Geom& g, float scale, cudaStream_t st)
{
    const T* yp = static_cast<const T*>(y);
    const T* gp = static_cast<const T*>(dy);
    T* dp = static_cast<T*>(dx);
    const int64_t pairs = g.rows / (g.rows_per_b / g.S);
#define GTMS_EX_BWD_CASE(vid, tw, nv, mb)                                                                          \
    case vid:                                                                                                      \
        return launch_kernel(gtms_bwd_explicit_kernel<T, tw, nv, mb>, grid_for<tw>(pairs), block_for<tw>(), 0, st, \
                             yp, gp, dp, mask, mask_batches, g, scale);
    if constexpr (sizeof(T) == 4) {
        switch (id) { GTMS_BWD_VEC4(GTMS_EX_BWD_CASE) default: break; }
    } else {
        switch (id) { GTMS_BWD_VEC2(GTMS_EX_BWD_CASE) default: break; }
    }
#undef GTMS_EX_BWD_CASE
    return cudaErrorInvalidValue;   // no kernel for this variant id
}

}  // namespace gtms
