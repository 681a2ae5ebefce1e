// gtms_kernels.cuh -- sm_103a kernels of the grouped-tril masked softmax.
//
// One "team" of threads owns one row of X[B,M,S,S] at a time: a warp for short
// rows, a whole CTA for long ones. The kept set of row r in batch b is the
// prefix [0, n) with n = r + 1 if r < L_b else 0, L_b = clamp(seq_lens[b], 0, S)
// ("Attention-Mask-Optimization" README, operator behaviour: kept iff r < L,
// c < L and c <= r; c <= r < L already implies c < L). The mask is this one
// comparison per row; no mask tensor exists ("实现思路": compute instead of
// loading).
//
// Per row, a team
//   1. issues loads of only the access units that cover [0, n) (padded rows: none),
//   2. issues the zero stores of every unit past the kept prefix right away --
//      they depend on no load, so they overlap the load latency,
//   3. reduces in fp32 with warp shuffles and, for CTA teams, one shared-memory
//      exchange per reduction,
//   4. writes the kept units (the masked elements of the last, partial unit as +0.0).
// Every unit is loaded and stored by the same thread, so an output may alias its
// input exactly.
//
// Two kernel families:
//   * vector kernels (16-byte units, rows whose byte length is a multiple of 16):
//     elements are handled as fp32 pairs with the packed f32x2 instructions of
//     sm_100+ (__fadd2_rn / __fmul2_rn / __ffma2_rn); the exponential is one
//     ex2.approx.f32 per kept element, kept in registers between the sum and
//     the store; masking touches only the row's last, partial unit;
//   * element kernels (one element per unit) for rows that are not 16-byte
//     multiples or buffers that are only element-aligned.
//
// The backward forms d = sum_c dy_c * y_c as a float-float (TwoSum, Knuth) sum,
// each product split exactly by an FMA (the split is zero for bf16 / fp16 inputs,
// whose products are exact in fp32), so that dy - d keeps full fp32 accuracy
// under cancellation; then dx = scale * y * ((dy - d_hi) - d_lo)
// ("ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1 Jacobian
// y_i (delta_ij - y_j); chain rule through scale * x). All rounding steps are
// explicit _rn intrinsics, so no multiply-add is contracted behind the
// compensated arithmetic.
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

__device__ __forceinline__ int32_t kept_prefix(const int32_t* __restrict__ seq_lens, int32_t b, int32_t r,
                                               int32_t S)
{
    int32_t L = __ldg(seq_lens + b);
    L = L < 0 ? 0 : (L > S ? S : L);
    return r < L ? r + 1 : 0;
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

// ---------------------------------------------------------------------------
// Team reductions. TW == 32: one warp, butterfly shuffles (every lane ends with
// the same value). TW > 32: the team is the whole CTA; warp results meet in
// shared memory and every thread folds them in the same order.
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

// ---------------------------------------------------------------------------
// Packed fp32 pair helpers (sm_100+ f32x2 instructions) and the exponential.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }

// 2^t, the MUFU approximation (no flush of subnormal results).
__device__ __forceinline__ float ex2(float t)
{
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float min3(float a, float b, float c)
{
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ---------------------------------------------------------------------------
// 16-byte access units as element pairs. Element e of a unit is pair e / 2,
// half e % 2 (x = lower address).
// ---------------------------------------------------------------------------
struct Unit16 {
    uint32_t w[4];
};

__device__ __forceinline__ Unit16 load16(const void* p)
{
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    return Unit16{{v.x, v.y, v.z, v.w}};
}

__device__ __forceinline__ void store16(void* p, const Unit16& u)
{
    *reinterpret_cast<uint4*>(p) = make_uint4(u.w[0], u.w[1], u.w[2], u.w[3]);
}

template <typename T> struct Pairs;

template <> struct Pairs<float> {
    static constexpr int kPairs = 2;   // 4 floats per 16 bytes
    static constexpr bool kExactProducts = false;
    __device__ static float2 get(const Unit16& u, int p)
    {
        return make_float2(__uint_as_float(u.w[2 * p]), __uint_as_float(u.w[2 * p + 1]));
    }
    __device__ static void put(Unit16& u, int p, float2 v)
    {
        u.w[2 * p] = __float_as_uint(v.x);
        u.w[2 * p + 1] = __float_as_uint(v.y);
    }
    // Zero the raw bits of elements e >= vc.
    __device__ static void clear_from(Unit16& u, int vc)
    {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e >= vc)
                u.w[e] = 0u;
    }
};

template <> struct Pairs<__nv_bfloat16> {
    static constexpr int kPairs = 4;   // 8 bf16 per 16 bytes
    static constexpr bool kExactProducts = true;
    __device__ static float2 get(const Unit16& u, int p)
    {
        return make_float2(__uint_as_float(u.w[p] << 16), __uint_as_float(u.w[p] & 0xffff0000u));
    }
    __device__ static void put(Unit16& u, int p, float2 v)
    {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
        u.w[p] = *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static void clear_from(Unit16& u, int vc)
    {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e >= vc)
                u.w[e >> 1] &= (e & 1) ? 0x0000ffffu : 0xffff0000u;
    }
};

template <> struct Pairs<__half> {
    static constexpr int kPairs = 4;   // 8 fp16 per 16 bytes
    static constexpr bool kExactProducts = true;
    __device__ static float2 get(const Unit16& u, int p)
    {
        return __half22float2(*reinterpret_cast<const __half2*>(&u.w[p]));
    }
    __device__ static void put(Unit16& u, int p, float2 v)
    {
        const __half2 h = __floats2half2_rn(v.x, v.y);
        u.w[p] = *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static void clear_from(Unit16& u, int vc)
    {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e >= vc)
                u.w[e >> 1] &= (e & 1) ? 0x0000ffffu : 0xffff0000u;
    }
};

// ---------------------------------------------------------------------------
// Vector forward: y = masked softmax(scale * x).
//
// t = (x - x_ext) * (scale * log2 e) with x_ext the row max (scale >= 0) or min
// (scale < 0): t <= 0 everywhere and exactly 0 at the extreme element, so a
// one-element row gives exp = 1, sum = 1, y = 1.
// Masked elements of the partial unit are first set to element 0 of that unit
// (which is kept), so they cannot move the extreme, then their exponentials are
// set to 0 before the sum.
// ---------------------------------------------------------------------------
template <typename T, int TW, int NV, int MINB>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW, MINB)
gtms_fwd_vec_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs;
    constexpr int EPU = 2 * PPU;
    __shared__ float red[TW > 32 ? 2 * (TW / 32) : 1];

    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);

    for (int64_t q = team; q < g.rows; q += nteams) {
        int32_t b, r;
        g.locate(q, b, r);
        const int32_t n = kept_prefix(seq_lens, b, r, g.S);
        const int32_t nu = (n + EPU - 1) / EPU;
        const char* xr = reinterpret_cast<const char*>(x + q * g.S);
        char* yr = reinterpret_cast<char*>(y + q * g.S);

        Unit16 raw[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu)
                raw[k] = load16(xr + 16 * j);
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= nu && j < g.units)
                store16(yr + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
        }
        if (n == 0)
            continue;   // uniform across the team

        float2 v[NV][PPU];
        float ext = use_max ? -INFINITY : INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
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
            const int j = tid + k * TW;
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
        const float s = team_sum<TW>(__fadd_rn(acc.x, acc.y), red + (TW > 32 ? TW / 32 : 0));
        const float2 inv = splat2(__frcp_rn(s));

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
                Unit16 o;
#pragma unroll
                for (int p = 0; p < PPU; ++p)
                    IO::put(o, p, __fmul2_rn(v[k][p], inv));
                store16(yr + 16 * j, o);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Vector backward: dx = scale * y * (dy - rowsum(dy * y)).
// The raw units of y and dy stay in registers (masked elements of the partial
// unit zeroed, which also neutralises any NaN there); each pass decodes them.
// ---------------------------------------------------------------------------
template <typename T, int TW, int NV, int MINB>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW, MINB)
gtms_bwd_vec_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs;
    constexpr int EPU = 2 * PPU;
    // Two buffers, alternating per reduced row: with a single exchange per row a
    // fast warp could otherwise overwrite a slot that a slow warp is still reading.
    __shared__ float red[2][TW > 32 ? 2 * (TW / 32) : 1];
    int par = 0;

    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);
    const float2 sc = splat2(scale);

    for (int64_t q = team; q < g.rows; q += nteams) {
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
            const int j = tid + k * TW;
            if (j < nu) {
                ry[k] = load16(yr + 16 * j);
                rg[k] = load16(gr + 16 * j);
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= nu && j < g.units)
                store16(dr + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
        }
        if (n == 0)
            continue;

        float2 hi2 = make_float2(0.0f, 0.0f), lo2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
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
        par ^= 1;
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));
        const float2 ndh = splat2(-dh), ndl = splat2(-dl);

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < nu) {
                Unit16 o;
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    const float2 a = IO::get(ry[k], p), cdy = IO::get(rg[k], p);
                    const float2 diff = __fadd2_rn(__fadd2_rn(cdy, ndh), ndl);
                    IO::put(o, p, __fmul2_rn(__fmul2_rn(a, diff), sc));
                }
                if (j == nu - 1)
                    IO::clear_from(o, n - j * EPU);   // masked outputs are +0.0 bits
                store16(dr + 16 * j, o);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Element kernels: one element per access unit, any alignment of the row start.
// ---------------------------------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<float> {
    using Raw = uint32_t;
    __device__ static float get(Raw r) { return __uint_as_float(r); }
    __device__ static Raw put(float v) { return __float_as_uint(v); }
};

template <> struct Elem<__nv_bfloat16> {
    using Raw = unsigned short;
    __device__ static float get(Raw r) { return __uint_as_float(static_cast<uint32_t>(r) << 16); }
    __device__ static Raw put(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
};

template <> struct Elem<__half> {
    using Raw = unsigned short;
    __device__ static float get(Raw r) { return __half2float(__ushort_as_half(r)); }
    __device__ static Raw put(float v) { return __half_as_ushort(__float2half_rn(v)); }
};

template <typename T, int TW, int NV>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW)
gtms_fwd_elem_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using E = Elem<T>;
    using Raw = typename E::Raw;
    __shared__ float red[TW > 32 ? 2 * (TW / 32) : 1];
    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;

    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);

    for (int64_t q = team; q < g.rows; q += nteams) {
        int32_t b, r;
        g.locate(q, b, r);
        const int32_t n = kept_prefix(seq_lens, b, r, g.S);
        const Raw* xr = reinterpret_cast<const Raw*>(x + q * g.S);
        Raw* yr = reinterpret_cast<Raw*>(y + q * g.S);

        float v[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < n)
                v[k] = E::get(xr[j]);
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= n && j < g.S)
                yr[j] = Raw(0);
        }
        if (n == 0)
            continue;

        float ext = use_max ? -INFINITY : INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (tid + k * TW < n)
                ext = use_max ? fmaxf(ext, v[k]) : fminf(ext, v[k]);
        ext = use_max ? team_max<TW>(ext, red) : -team_max<TW>(-ext, red);

        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (tid + k * TW < n) {
                v[k] = ex2(__fmul_rn(__fsub_rn(v[k], ext), c));
                s = __fadd_rn(s, v[k]);
            }
        s = team_sum<TW>(s, red + (TW > 32 ? TW / 32 : 0));
        const float inv = __frcp_rn(s);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < n)
                yr[j] = E::put(__fmul_rn(v[k], inv));
        }
    }
}

template <typename T, int TW, int NV>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW)
gtms_bwd_elem_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    using E = Elem<T>;
    using Raw = typename E::Raw;
    __shared__ float red[2][TW > 32 ? 2 * (TW / 32) : 1];
    int par = 0;

    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);

    for (int64_t q = team; q < g.rows; q += nteams) {
        int32_t b, r;
        g.locate(q, b, r);
        const int32_t n = kept_prefix(seq_lens, b, r, g.S);
        const Raw* yr = reinterpret_cast<const Raw*>(y + q * g.S);
        const Raw* gr = reinterpret_cast<const Raw*>(dy + q * g.S);
        Raw* dr = reinterpret_cast<Raw*>(dx + q * g.S);

        float vy[NV], vg[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < n) {
                vy[k] = E::get(yr[j]);
                vg[k] = E::get(gr[j]);
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= n && j < g.S)
                dr[j] = Raw(0);
        }
        if (n == 0)
            continue;

        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (tid + k * TW < n) {
                const float p = __fmul_rn(vy[k], vg[k]);
                const float pe = __fmaf_rn(vy[k], vg[k], -p);
                float s, e;
                two_sum(hi, p, s, e);
                hi = s;
                lo = __fadd_rn(lo, __fadd_rn(e, pe));
            }
        team_ff_sum<TW>(hi, lo, red[par]);
        par ^= 1;
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j < n)
                dr[j] = E::put(__fmul_rn(__fmul_rn(vy[k], __fsub_rn(__fsub_rn(vg[k], dh), dl)), scale));
        }
    }
}

}  // namespace gtms
