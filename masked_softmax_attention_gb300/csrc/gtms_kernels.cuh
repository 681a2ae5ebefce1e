// gtms_kernels.cuh -- sm_103a kernels of the grouped-tril masked softmax.
//
// One "team" of threads owns one row of X[B,M,S,S] at a time: a warp for rows
// of up to 4 KB, a whole CTA for longer rows. The kept set of row r in batch b
// is the prefix [0, n) with n = r + 1 if r < L_b else 0, L_b = clamp(seq_lens[b],
// 0, S) ("Attention-Mask-Optimization" README, operator behaviour: kept iff
// r < L, c < L and c <= r; c <= r < L already implies c < L). The mask is this
// one comparison per row; no mask tensor exists ("实现思路": compute instead
// of loading).
//
// Per row, a team
//   1. issues 16-byte loads of only the units that cover [0, n)  (padded rows: none),
//   2. issues the zero stores of every unit past the kept prefix right away --
//      they depend on no load, so they overlap the load latency,
//   3. reduces (max, then sum of exp) in fp32 with warp shuffles and, for CTA
//      teams, one shared-memory exchange per reduction,
//   4. writes the kept units (the masked elements of the last, partial unit
//      as +0.0).
// Every unit is loaded and stored by the same thread, so y may alias x exactly.
//
// The backward forms d = sum_c dy_c * y_c as a float-float (TwoSum, Knuth /
// Moller) sum so that dy - d keeps full fp32 accuracy under cancellation, then
// writes dx = scale * y * ((dy - d_hi) - d_lo)  ("ops(8): self-attention 的 CUDA
// 实现及优化 (下)", section 2.1 Jacobian y_i (delta_ij - y_j), chain rule through
// scale * x). All rounding steps use the explicit _rn intrinsics so that no
// multiply-add is contracted behind the compensated arithmetic.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gtms {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpTeamBlock = 128;   // threads per CTA when a warp owns a row (4 rows per CTA)

// Row geometry shared by all kernels.
struct Geom {
    int64_t rows;         // B * M * S
    int64_t rows_per_b;   // M * S
    int32_t S;
    int32_t units;        // access units per row (16-byte vectors, or elements)
    int32_t small;        // rows fits in 32 bits: use 32-bit division

    __device__ __forceinline__ void locate(int64_t q, int32_t& b, int32_t& r) const
    {
        if (small) {
            const uint32_t qq = static_cast<uint32_t>(q);
            b = static_cast<int32_t>(qq / static_cast<uint32_t>(rows_per_b));
            r = static_cast<int32_t>(qq % static_cast<uint32_t>(S));
        } else {
            b = static_cast<int32_t>(q / rows_per_b);
            r = static_cast<int32_t>(q % S);
        }
    }
};

// ---------------------------------------------------------------------------
// Access units: a 16-byte vector (VEC) or one element, and the element <-> fp32
// conversions of each IO dtype. Conversions to the IO dtype round to nearest even.
// ---------------------------------------------------------------------------
template <typename T, bool VEC> struct Unit;

__device__ __forceinline__ uint32_t word_of(const uint4& r, int i)
{
    return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}

template <> struct Unit<float, true> {
    using Raw = uint4;
    static constexpr int EPU = 4;
    __device__ static float get(const Raw& r, int i) { return __uint_as_float(word_of(r, i)); }
    __device__ static Raw pack(const float (&o)[EPU])
    {
        return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                          __float_as_uint(o[3]));
    }
};

template <> struct Unit<__nv_bfloat16, true> {
    using Raw = uint4;
    static constexpr int EPU = 8;
    __device__ static float get(const Raw& r, int i)
    {
        const uint32_t w = word_of(r, i >> 1);
        return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    __device__ static uint32_t pair(float lo, float hi)
    {
        const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&p);
    }
    __device__ static Raw pack(const float (&o)[EPU])
    {
        return make_uint4(pair(o[0], o[1]), pair(o[2], o[3]), pair(o[4], o[5]), pair(o[6], o[7]));
    }
};

template <> struct Unit<__half, true> {
    using Raw = uint4;
    static constexpr int EPU = 8;
    __device__ static float get(const Raw& r, int i)
    {
        const uint32_t w = word_of(r, i >> 1);
        return __half2float(__ushort_as_half(static_cast<unsigned short>((i & 1) ? (w >> 16) : (w & 0xffffu))));
    }
    __device__ static uint32_t pair(float lo, float hi)
    {
        const __half2 p = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&p);
    }
    __device__ static Raw pack(const float (&o)[EPU])
    {
        return make_uint4(pair(o[0], o[1]), pair(o[2], o[3]), pair(o[4], o[5]), pair(o[6], o[7]));
    }
};

template <> struct Unit<float, false> {
    using Raw = uint32_t;
    static constexpr int EPU = 1;
    __device__ static float get(const Raw& r, int) { return __uint_as_float(r); }
    __device__ static Raw pack(const float (&o)[EPU]) { return __float_as_uint(o[0]); }
};

template <> struct Unit<__nv_bfloat16, false> {
    using Raw = unsigned short;
    static constexpr int EPU = 1;
    __device__ static float get(const Raw& r, int) { return __uint_as_float(static_cast<uint32_t>(r) << 16); }
    __device__ static Raw pack(const float (&o)[EPU]) { return __bfloat16_as_ushort(__float2bfloat16_rn(o[0])); }
};

template <> struct Unit<__half, false> {
    using Raw = unsigned short;
    static constexpr int EPU = 1;
    __device__ static float get(const Raw& r, int) { return __half2float(__ushort_as_half(r)); }
    __device__ static Raw pack(const float (&o)[EPU]) { return __half_as_ushort(__float2half_rn(o[0])); }
};

// ---------------------------------------------------------------------------
// Team reductions. TW == 32: one warp, shuffles only. TW > 32: the team is the
// whole CTA; warp results meet in shared memory and every thread folds them in
// the same order, so all threads hold the identical value.
// ---------------------------------------------------------------------------
template <int TW>
__device__ __forceinline__ float team_max(float v, float* smem)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if constexpr (TW > 32) {
        if ((threadIdx.x & 31) == 0)
            smem[threadIdx.x >> 5] = v;
        __syncthreads();
        v = smem[0];
#pragma unroll
        for (int w = 1; w < TW / 32; ++w)
            v = fmaxf(v, smem[w]);
    }
    return v;
}

template <int TW>
__device__ __forceinline__ float team_sum(float v, float* smem)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if constexpr (TW > 32) {
        if ((threadIdx.x & 31) == 0)
            smem[threadIdx.x >> 5] = v;
        __syncthreads();
        v = smem[0];
#pragma unroll
        for (int w = 1; w < TW / 32; ++w)
            v = __fadd_rn(v, smem[w]);
    }
    return v;
}

// TwoSum (Knuth): s + e == a + b exactly, s = fl(a + b).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += (ohi, olo), float-float.
__device__ __forceinline__ void ff_merge(float& hi, float& lo, float ohi, float olo)
{
    float s, e;
    two_sum(hi, ohi, s, e);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, olo), e);
}

template <int TW>
__device__ __forceinline__ void team_ff_sum(float& hi, float& lo, float* smem)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ohi = __shfl_xor_sync(0xffffffffu, hi, o);
        const float olo = __shfl_xor_sync(0xffffffffu, lo, o);
        ff_merge(hi, lo, ohi, olo);
    }
    if constexpr (TW > 32) {
        constexpr int W = TW / 32;
        if ((threadIdx.x & 31) == 0) {
            smem[threadIdx.x >> 5] = hi;
            smem[W + (threadIdx.x >> 5)] = lo;
        }
        __syncthreads();
        hi = smem[0];
        lo = smem[W];
#pragma unroll
        for (int w = 1; w < W; ++w)
            ff_merge(hi, lo, smem[w], smem[W + w]);
    }
}

template <int TW>
__device__ __forceinline__ void team_coords(int& tid, int64_t& team, int64_t& nteams)
{
    if constexpr (TW == 32) {
        tid = threadIdx.x & 31;
        team = static_cast<int64_t>(blockIdx.x) * (kWarpTeamBlock / 32) + (threadIdx.x >> 5);
        nteams = static_cast<int64_t>(gridDim.x) * (kWarpTeamBlock / 32);
    } else {
        tid = threadIdx.x;
        team = blockIdx.x;
        nteams = gridDim.x;
    }
}

__device__ __forceinline__ int32_t kept_prefix(const int32_t* __restrict__ seq_lens, int32_t b, int32_t r,
                                               int32_t S)
{
    int32_t L = __ldg(seq_lens + b);
    L = L < 0 ? 0 : (L > S ? S : L);
    return r < L ? r + 1 : 0;
}

// ---------------------------------------------------------------------------
// Forward: y = masked softmax(scale * x).
// ---------------------------------------------------------------------------
template <typename T, bool VEC, int TW, int NV>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW)
gtms_fwd_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using U = Unit<T, VEC>;
    using Raw = typename U::Raw;
    constexpr int EPU = U::EPU;
    __shared__ float red[TW > 32 ? 2 * (TW / 32) : 1];

    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);

    for (int64_t q = team; q < g.rows; q += nteams) {
        int32_t b, r;
        g.locate(q, b, r);
        const int32_t n = kept_prefix(seq_lens, b, r, g.S);
        const int32_t nu = (n + EPU - 1) / EPU;
        const Raw* xr = reinterpret_cast<const Raw*>(x + q * g.S);
        Raw* yr = reinterpret_cast<Raw*>(y + q * g.S);

        Raw v[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu)
                v[k] = xr[j];
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= nu && j < g.units)
                yr[j] = Raw{};
        }
        if (n == 0)
            continue;   // uniform across the team

        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
#pragma unroll
                for (int i = 0; i < EPU; ++i)
                    if (j * EPU + i < n)
                        m = fmaxf(m, __fmul_rn(U::get(v[k], i), scale));
            }
        }
        m = team_max<TW>(m, red);

        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
#pragma unroll
                for (int i = 0; i < EPU; ++i)
                    if (j * EPU + i < n)
                        s = __fadd_rn(s, exp2f(__fmul_rn(__fsub_rn(__fmul_rn(U::get(v[k], i), scale), m), kLog2e)));
            }
        }
        s = team_sum<TW>(s, red + (TW > 32 ? TW / 32 : 0));
        const float inv = __frcp_rn(s);

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
                float o[EPU];
#pragma unroll
                for (int i = 0; i < EPU; ++i)
                    o[i] = (j * EPU + i < n)
                               ? __fmul_rn(exp2f(__fmul_rn(__fsub_rn(__fmul_rn(U::get(v[k], i), scale), m), kLog2e)), inv)
                               : 0.0f;
                yr[j] = U::pack(o);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Backward: dx = scale * y * (dy - rowsum(dy * y)).
// ---------------------------------------------------------------------------
template <typename T, bool VEC, int TW, int NV>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW)
gtms_bwd_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using U = Unit<T, VEC>;
    using Raw = typename U::Raw;
    constexpr int EPU = U::EPU;
    // Two buffers, alternating per reduced row: with a single exchange per row a
    // fast warp could otherwise overwrite a slot that a slow warp is still reading.
    __shared__ float red[2][TW > 32 ? 2 * (TW / 32) : 1];
    int par = 0;

    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);

    for (int64_t q = team; q < g.rows; q += nteams) {
        int32_t b, r;
        g.locate(q, b, r);
        const int32_t n = kept_prefix(seq_lens, b, r, g.S);
        const int32_t nu = (n + EPU - 1) / EPU;
        const Raw* yr = reinterpret_cast<const Raw*>(y + q * g.S);
        const Raw* gr = reinterpret_cast<const Raw*>(dy + q * g.S);
        Raw* dr = reinterpret_cast<Raw*>(dx + q * g.S);

        Raw vy[NV], vg[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
                vy[k] = yr[j];
                vg[k] = gr[j];
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= nu && j < g.units)
                dr[j] = Raw{};
        }
        if (n == 0)
            continue;

        // d = sum dy*y as float-float: each product split exactly by an FMA
        // (zero error term for bf16/fp16 inputs, whose products are exact in fp32).
        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
#pragma unroll
                for (int i = 0; i < EPU; ++i)
                    if (j * EPU + i < n) {
                        const float a = U::get(vy[k], i), c = U::get(vg[k], i);
                        const float p = __fmul_rn(a, c);
                        const float pe = __fmaf_rn(a, c, -p);
                        float s, e;
                        two_sum(hi, p, s, e);
                        hi = s;
                        lo = __fadd_rn(lo, __fadd_rn(e, pe));
                    }
            }
        }
        team_ff_sum<TW>(hi, lo, red[par]);
        par ^= 1;
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
                float o[EPU];
#pragma unroll
                for (int i = 0; i < EPU; ++i) {
                    const float a = U::get(vy[k], i), c = U::get(vg[k], i);
                    o[i] = (j * EPU + i < n) ? __fmul_rn(__fmul_rn(a, __fsub_rn(__fsub_rn(c, dh), dl)), scale) : 0.0f;
                }
                dr[j] = U::pack(o);
            }
        }
    }
}

}  // namespace gtms
