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

template <typename T, int C, int TW, int NV, int MINB>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(TW, MINB)
gtms_fwd_cluster_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs;
    constexpr int EPU = 2 * PPU;
    __shared__ float red[2 * (TW / 32)];
    __shared__ float2 slot[2];

    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    const int64_t ncl = gridDim.x / C;
    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    int par = 0;

    for (int64_t q = blockIdx.x / C; q < g.rows; q += ncl) {
        int32_t b, r;
        g.locate(q, b, r);
        const int32_t n = kept_prefix(seq_lens, b, r, g.S);
        const int32_t nu = (n + EPU - 1) / EPU;
        const char* xr = reinterpret_cast<const char*>(x + q * g.S);
        char* yr = reinterpret_cast<char*>(y + q * g.S);

        Unit16 raw[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j < nu)
                raw[k] = load16(xr + 16 * j);
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j >= nu && j < g.units)
                store16(yr + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
        }
        if (n == 0)
            continue;   // uniform across the cluster

        float2 v[NV][PPU];
        float ext = use_max ? -INFINITY : INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j < nu) {
#pragma unroll
                for (int p = 0; p < PPU; ++p)
                    v[k][p] = IO::get(raw[k], p);
                if (j == nu - 1) {
                    const int vc = n - j * EPU;
#pragma unroll
                    for (int p = 0; p < PPU; ++p) {
                        if (2 * p >= vc)
                            v[k][p].x = v[k][0].x;
                        if (2 * p + 1 >= vc)
                            v[k][p].y = v[k][0].x;
                    }
                }
                if (use_max) {
#pragma unroll
                    for (int p = 0; p < PPU; ++p)
                        ext = max3(ext, v[k][p].x, v[k][p].y);
                } else {
#pragma unroll
                    for (int p = 0; p < PPU; ++p)
                        ext = min3(ext, v[k][p].x, v[k][p].y);
                }
            }
        }
        ext = use_max ? team_max<TW>(ext, red) : -team_max<TW>(-ext, red);

        const float2 shift = splat2(-ext), c2 = splat2(c);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j < nu) {
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    const float2 t = __fmul2_rn(__fadd2_rn(v[k][p], shift), c2);
                    v[k][p] = make_float2(ex2(t.x), ex2(t.y));
                }
                if (j == nu - 1) {
                    const int vc = n - j * EPU;
#pragma unroll
                    for (int p = 0; p < PPU; ++p) {
                        if (2 * p >= vc)
                            v[k][p].x = 0.0f;
                        if (2 * p + 1 >= vc)
                            v[k][p].y = 0.0f;
                    }
                }
#pragma unroll
                for (int p = 0; p < PPU; ++p)
                    acc = __fadd2_rn(acc, v[k][p]);
            }
        }
        const float l = team_sum<TW>(__fadd_rn(acc.x, acc.y), red + TW / 32);

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
        const float2 f2 = splat2(f);

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j < nu) {
                Unit16 o;
#pragma unroll
                for (int p = 0; p < PPU; ++p)
                    IO::put(o, p, __fmul2_rn(v[k][p], f2));
                store16(yr + 16 * j, o);
            }
        }
    }
    cl.sync();
}

template <typename T, int C, int TW, int NV, int MINB>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(TW, MINB)
gtms_bwd_cluster_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs;
    constexpr int EPU = 2 * PPU;
    __shared__ float red[2][2 * (TW / 32)];
    __shared__ float2 slot[2];

    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    const int64_t ncl = gridDim.x / C;
    const float2 sc = splat2(scale);
    int par = 0;

    for (int64_t q = blockIdx.x / C; q < g.rows; q += ncl) {
        int32_t b, r;
        g.locate(q, b, r);
        const int32_t n = kept_prefix(seq_lens, b, r, g.S);
        const int32_t nu = (n + EPU - 1) / EPU;
        const char* yr = reinterpret_cast<const char*>(y + q * g.S);
        const char* gr = reinterpret_cast<const char*>(dy + q * g.S);
        char* dr = reinterpret_cast<char*>(dx + q * g.S);

        Unit16 ry[NV], rg[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j < nu) {
                ry[k] = load16(yr + 16 * j);
                rg[k] = load16(gr + 16 * j);
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j >= nu && j < g.units)
                store16(dr + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
        }
        if (n == 0)
            continue;

        float2 hi2 = make_float2(0.0f, 0.0f), lo2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j < nu) {
                if (j == nu - 1) {
                    const int vc = n - j * EPU;
                    IO::clear_from(ry[k], vc);
                    IO::clear_from(rg[k], vc);
                }
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
        const float2 ndh = splat2(-dh), ndl = splat2(-dl);

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = cluster_unit<TW, C>(tid, k, rank);
            if (j < nu) {
                Unit16 o;
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    const float2 a = IO::get(ry[k], p), cdy = IO::get(rg[k], p);
                    const float2 diff = __fadd2_rn(__fadd2_rn(cdy, ndh), ndl);
                    IO::put(o, p, __fmul2_rn(__fmul2_rn(a, diff), sc));
                }
                if (j == nu - 1)
                    IO::clear_from(o, n - j * EPU);
                store16(dr + 16 * j, o);
            }
        }
    }
    cl.sync();
}

}  // namespace gtms
