// gtms_cluster.cuh -- split-row kernels for rows longer than one CTA holds
// (8192 < S <= 65536): a thread-block cluster of C CTAs owns one row.
//
// Each CTA keeps a chunk of the row in registers. The chunks interleave in
// blocks of 32 sixteen-byte units (512 bytes, one warp instruction's worth),
// round robin over the cluster's CTAs, so every warp still loads and stores
// 512 contiguous bytes and the kept prefix -- always at the start of the row --
// spreads over all CTAs. Each CTA reduces its own chunk, publishes one partial
// result in its shared memory and, after one cluster barrier, reads the
// partials of every CTA of the cluster through distributed shared memory and
// folds them in the same order, so all CTAs agree bit for bit.
//
// Forward partials are (local extreme m_i, local sum l_i of exponentials taken
// against m_i). They merge the way split-KV flash decoding merges its
// per-split results (ColossalAI flash_decoding.py, the reduce kernel): with
// M the global extreme, L = sum_i l_i * 2^((m_i - M) * c) and each CTA scales
// its exponentials by 2^((m_i - M) * c) / L. Only one exchange per row is
// needed. Backward partials are the float-float dot products of each chunk.
//
// Every mask family of gtms_kernels.cuh is supported (template parameter MK).
//
// The exchange slots alternate per reduced row: a CTA writes the slot of row
// k+2 only after passing the barrier of row k+1, which every peer reaches only
// after reading row k's slots. A final cluster barrier keeps every CTA's shared
// memory alive until its peers are done reading it.
#pragma once

#include <cooperative_groups.h>

#include "gtms_kernels.cuh"

namespace gtms {

namespace cg = cooperative_groups;

// Row unit handled by local slot (tid, k) of CTA `rank` in a cluster of C CTAs.
template <int TW, int C>
__device__ __forceinline__ int cluster_unit(int tid, int k, int rank)
{
    const int u = tid + k * TW;
    return ((u >> 5) * C + rank) * 32 + (u & 31);
}

template <typename T, int MK, int C, int TW, int NV, int MINB>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(TW, MINB)
gtms_fwd_cluster_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    __shared__ float red[2 * (TW / 32)];
    __shared__ float2 slot[2];

    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    const int64_t ncl = gridDim.x / C;
    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    const auto unit_of = [tid, rank](int k) { return cluster_unit<TW, C>(tid, k, rank); };
    int par = 0;

    for (int64_t q = blockIdx.x / C; q < g.rows; q += ncl) {
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const char* xr = reinterpret_cast<const char*>(x + q * g.S);
        char* yr = reinterpret_cast<char*>(y + q * g.S);

        Unit16 raw[NV];
        load_kept<NV>(xr, ur, unit_of, raw);
        store_zeros<NV>(yr, ur, g.units, unit_of);
        if (c1 <= c0)
            continue;   // uniform across the cluster

        float2 v[NV][Pairs<T>::kPairs];
        float ext = fwd_decode_extreme<T, NV>(raw, v, ur, unit_of, use_max);
        ext = use_max ? team_max<TW>(ext, red) : -team_max<TW>(-ext, red);
        const float l = team_sum<TW>(fwd_exp_sum<T, NV>(v, ur, unit_of, ext, c), red + TW / 32);

        if (tid == 0)
            slot[par] = make_float2(ext, l);
        cl.sync();
        float2 part[C];
#pragma unroll
        for (int i = 0; i < C; ++i)
            part[i] = *cl.map_shared_rank(&slot[par], i);
        par ^= 1;
        // A CTA whose chunk holds no kept element reports l = 0 and takes no part.
        float gext = use_max ? -INFINITY : INFINITY;
#pragma unroll
        for (int i = 0; i < C; ++i)
            if (part[i].y > 0.0f)
                gext = use_max ? fmaxf(gext, part[i].x) : fminf(gext, part[i].x);
        float L = 0.0f;
#pragma unroll
        for (int i = 0; i < C; ++i)
            if (part[i].y > 0.0f)
                L = __fadd_rn(L, __fmul_rn(part[i].y, ex2(__fmul_rn(__fsub_rn(part[i].x, gext), c))));
        const float f = l > 0.0f ? __fmul_rn(ex2(__fmul_rn(__fsub_rn(ext, gext), c)), __frcp_rn(L)) : 0.0f;
        fwd_store<T, NV>(yr, v, ur, unit_of, f);
    }
    cl.sync();
}

template <typename T, int MK, int C, int TW, int NV, int MINB>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(TW, MINB)
gtms_bwd_cluster_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    __shared__ float red[2][2 * (TW / 32)];
    __shared__ float2 slot[2];

    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    const int64_t ncl = gridDim.x / C;
    const auto unit_of = [tid, rank](int k) { return cluster_unit<TW, C>(tid, k, rank); };
    int par = 0;

    for (int64_t q = blockIdx.x / C; q < g.rows; q += ncl) {
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const char* yr = reinterpret_cast<const char*>(y + q * g.S);
        const char* gr = reinterpret_cast<const char*>(dy + q * g.S);
        char* dr = reinterpret_cast<char*>(dx + q * g.S);

        Unit16 ry[NV], rg[NV];
        load_kept<NV>(yr, ur, unit_of, ry);
        load_kept<NV>(gr, ur, unit_of, rg);
        store_zeros<NV>(dr, ur, g.units, unit_of);
        if (c1 <= c0)
            continue;

        float hi, lo;
        bwd_dot<T, NV>(ry, rg, ur, unit_of, hi, lo);
        team_ff_sum<TW>(hi, lo, red[par]);

        if (tid == 0)
            slot[par] = make_float2(hi, lo);
        cl.sync();
        float2 part[C];
#pragma unroll
        for (int i = 0; i < C; ++i)
            part[i] = *cl.map_shared_rank(&slot[par], i);
        par ^= 1;
        hi = part[0].x;
        lo = part[0].y;
#pragma unroll
        for (int i = 1; i < C; ++i)
            ff_merge(hi, lo, part[i].x, part[i].y);
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));
        bwd_store<T, NV>(dr, ry, rg, ur, unit_of, dh, dl, scale);
    }
    cl.sync();
}

}  // namespace gtms
