// gtms_band.cuh -- sliding-window rows whose window is far narrower than the row.
//
// The sliding causal window ("优化ScaledMaskSoftmax算子", section 6, local
// window) keeps at most w contiguous columns of a row. When those fit in one
// warp's slots but the row does not, the per-row kernels of gtms_kernels.cuh
// spread the row over a CTA team whose warps mostly hold no kept element, and
// pay two CTA-wide reductions per row for it. Here a warp owns a row: its
// lanes take the kept units in KV slots counted from the window's first unit
// (slot k of lane l is unit u0 + l + 32 k), store the zeros of the rest of the
// row in a strided loop, and reduce with shuffles only. Arithmetic, masking of
// the partial end units and the stored bits are those of the vector kernels.
#pragma once

#include "gtms_kernels.cuh"

namespace gtms {

// Zero stores of every unit of a row outside [u0, u1), by the 32 lanes of a warp.
__device__ __forceinline__ void band_zero_fill(char* row, const UnitRange& ur, int units, int lane)
{
    for (int j = lane; j < ur.u0; j += 32)
        store16(row + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
    for (int j = ur.u1 + lane; j < units; j += 32)
        store16(row + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
}

template <typename T, int KV, int MINB>
__global__ void __launch_bounds__(kWarpTeamBlock, MINB)
gtms_fwd_band_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    int lane;
    int64_t team, nteams;
    team_coords<32>(lane, team, nteams);

    for (int64_t q = team; q < g.rows; q += nteams) {
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<kMaskWindow>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const auto unit_of = [lane, u0 = ur.u0](int k) { return u0 + lane + 32 * k; };
        const char* xr = reinterpret_cast<const char*>(x + q * g.S);
        char* yr = reinterpret_cast<char*>(y + q * g.S);

        Unit16 raw[KV];
        load_kept<KV>(xr, ur, unit_of, raw);
        band_zero_fill(yr, ur, g.units, lane);
        if (c1 <= c0)
            continue;   // uniform across the warp

        float2 v[KV][Pairs<T>::kPairs];
        float ext = fwd_decode_extreme<T, KV>(raw, v, ur, unit_of, use_max);
        ext = use_max ? team_max<32>(ext, nullptr) : -team_max<32>(-ext, nullptr);
        const float s = team_sum<32>(fwd_exp_sum<T, KV>(v, ur, unit_of, ext, c), nullptr);
        fwd_store<T, KV>(yr, v, ur, unit_of, __frcp_rn(s));
    }
}

template <typename T, int KV, int MINB>
__global__ void __launch_bounds__(kWarpTeamBlock, MINB)
gtms_bwd_band_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    int lane;
    int64_t team, nteams;
    team_coords<32>(lane, team, nteams);

    for (int64_t q = team; q < g.rows; q += nteams) {
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<kMaskWindow>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const auto unit_of = [lane, u0 = ur.u0](int k) { return u0 + lane + 32 * k; };
        const char* yr = reinterpret_cast<const char*>(y + q * g.S);
        const char* gr = reinterpret_cast<const char*>(dy + q * g.S);
        char* dr = reinterpret_cast<char*>(dx + q * g.S);

        Unit16 ry[KV], rg[KV];
        load_kept<KV>(yr, ur, unit_of, ry);
        load_kept<KV>(gr, ur, unit_of, rg);
        band_zero_fill(dr, ur, g.units, lane);
        if (c1 <= c0)
            continue;

        float hi, lo;
        bwd_dot<T, KV>(ry, rg, ur, unit_of, hi, lo);
        team_ff_sum<32>(hi, lo, nullptr);
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));
        bwd_store<T, KV>(dr, ry, rg, ur, unit_of, dh, dl, scale);
    }
}

}  // namespace gtms
