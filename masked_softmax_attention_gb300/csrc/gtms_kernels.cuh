// gtms_kernels.cuh -- sm_103a kernels of the grouped-tril masked softmax.
//
// One "team" of threads owns one row of X[B,M,S,S] at a time: a warp for short
// rows, a whole CTA for long ones (rows of 32 KB and more go to the two-pass
// stream kernels of gtms_stream.cuh; the 16-bit forward's CTA teams run the M
// heads of one (batch, row) pair in turn, gtms_fwd_heads_kernel below; narrow
// sliding windows go to the band kernels of gtms_band.cuh). The kept set of row r in batch b is a
// contiguous column range [c0, c1) computed from (r, L_b, mask kind), with
// L_b = clamp(seq_lens[b], 0, S). For the default op ("Attention-Mask-
// Optimization" README, operator behaviour: kept iff r < L, c < L and c <= r)
// it is the prefix [0, r + 1) of rows r < L, since c <= r < L already implies
// c < L. The mask is this computation per row; no mask tensor exists
// ("实现思路": compute instead of loading).
//
// Per row, a team
//   1. issues loads of only the access units that cover [c0, c1) (padded rows: none),
//   2. issues the zero stores of every unit outside them right away -- they
//      depend on no load, so they overlap the load latency,
//   3. reduces in fp32 with warp shuffles and, for CTA teams, one shared-memory
//      exchange per reduction,
//   4. writes the kept units (the masked elements of the first and last,
//      partial units as +0.0).
// Every unit is loaded and stored by the same thread, so an output may alias its
// input exactly.
//
// Two kernel families:
//   * vector kernels (16-byte units, rows whose byte length is a multiple of 16):
//     elements are handled as fp32 pairs with the packed f32x2 instructions of
//     sm_100+ (__fadd2_rn / __fmul2_rn / __ffma2_rn); the exponential is one
//     ex2.approx.f32 per kept element, kept in registers between the sum and
//     the store; masking touches only the partial units at the range's ends;
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

// Launch through cudaLaunchKernelEx and return that launch's own status. (A
// triple-chevron launch reports only through cudaGetLastError, which would also
// return, and clear, an error left behind by earlier unrelated work on the thread.)
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                                 Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Time bounds of the waits on mbarriers, in nanoseconds of the GPU's global
// timer. kAttnWaitNs bounds a wait in the main loop: one that runs out means
// another role stopped making progress, and the kernel gives up (the host
// entry point passes it; a test build passes a short one). kAttnDrainWaitNs
// bounds, after giving up, each wait for a copy or an MMA already issued; those
// complete unless the hardware itself failed, and a CTA whose drain wait runs
// out exits with that operation still outstanding.
constexpr uint64_t kAttnWaitNs = 1000000000ull;        // 1 s
constexpr uint64_t kAttnDrainWaitNs = 2000000000ull;   // 2 s

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpTeamBlock = 128;   // threads per CTA when a warp owns a row (4 rows per CTA)

// Row geometry shared by all kernels.
struct Geom {
    int64_t rows;         // B * M * S
    int64_t rows_per_b;   // M * S
    int32_t S;
    int32_t units;        // access units per row (16-byte vectors, or elements)
    int32_t small;        // rows fits in 32 bits: use 32-bit division
    int32_t window;       // width of the sliding causal window (mask kind 2)

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

// Mask families: every kind keeps a contiguous column range [c0, c1) of a row
// r < L and nothing of the rows r >= L ("优化ScaledMaskSoftmax算子", section 6,
// lists the length mask and the local window besides the default):
//   kMaskGroupedTril (0): [0, r + 1)                 -- the README's operator
//   kMaskLength      (1): [0, L)                     -- padded keys and queries
//   kMaskWindow      (2): [max(0, r - w + 1), r + 1) -- causal band of width w
constexpr int kMaskGroupedTril = 0;
constexpr int kMaskLength = 1;
constexpr int kMaskWindow = 2;

template <int MK>
__device__ __forceinline__ void kept_range(const int32_t* __restrict__ seq_lens, int32_t b, int32_t r,
                                           const Geom& g, int32_t& c0, int32_t& c1)
{
    int32_t L = __ldg(seq_lens + b);
    L = L < 0 ? 0 : (L > g.S ? g.S : L);
    c0 = 0;
    c1 = 0;
    if (r < L) {
        if constexpr (MK == kMaskLength) {
            c1 = L;
        } else {
            c1 = r + 1;
            if constexpr (MK == kMaskWindow)
                c0 = r - g.window + 1 > 0 ? r - g.window + 1 : 0;
        }
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

// Softmax statistics of a row over a CTA team in one shared-memory exchange.
// Each warp has reduced, with shuffles, its extreme e_w (max, or min when the
// scale is negative) and its sum s_w of 2^((x - e_w) c) over its kept
// elements. The warps' pairs meet once in `smem` (2 * TW / 32 floats; callers
// alternate two buffers per row). Lane l of every warp then takes pair l, and
// two butterflies give the row's extreme E and sum S = sum_w s_w 2^((e_w - E) c)
// (the same operations in every warp, so every thread gets the same E and S).
// A warp with no kept element, or whose kept inputs are all infinite on the
// far side of the extreme, has s_w == 0 and takes no part (a NaN sum still
// propagates). Returns E in `ext` and 1 / S in `inv`: an output is then
// 2^((x - E) c) / S, the formula of the per-row kernels.
template <int TW>
__device__ __forceinline__ void team_softmax_stats(float e_w, float s_w, float c, bool use_max, float* smem,
                                                   float& ext, float& inv)
{
    constexpr int NW = TW / 32;
    const int l = threadIdx.x & 31;
    if (l == 0) {
        smem[threadIdx.x >> 5] = e_w;
        smem[NW + (threadIdx.x >> 5)] = s_w;
    }
    __syncthreads();
    const float e_l = l < NW ? smem[l] : 0.0f, s_l = l < NW ? smem[NW + l] : 0.0f;
    const bool has = s_l != 0.0f;
    float E = has ? e_l : (use_max ? -INFINITY : INFINITY);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float other = __shfl_xor_sync(0xffffffffu, E, o);
        E = use_max ? fmaxf(E, other) : fminf(E, other);
    }
    float S = has ? __fmul_rn(s_l, ex2(__fmul_rn(__fsub_rn(e_l, E), c))) : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        S = __fadd_rn(S, __shfl_xor_sync(0xffffffffu, S, o));
    ext = E;
    inv = __frcp_rn(S);
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

// 16-byte load and store under an L2 cache policy (createpolicy): data read
// again soon can be kept (evict_last), data not read again let go first.
__device__ __forceinline__ Unit16 load16_hint(const void* p, uint64_t pol)
{
    Unit16 u;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(u.w[0]), "=r"(u.w[1]), "=r"(u.w[2]), "=r"(u.w[3])
                 : "l"(p), "l"(pol)
                 : "memory");
    return u;
}

__device__ __forceinline__ void store16_hint(void* p, const Unit16& u, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :: "l"(p), "r"(u.w[0]), "r"(u.w[1]), "r"(u.w[2]), "r"(u.w[3]), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
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
    // Zero the raw bits of elements outside [lo, hi).
    __device__ static void clear_outside(Unit16& u, int lo, int hi)
    {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e < lo || e >= hi)
                u.w[e] = 0u;
    }
    // Zero the raw bits of elements whose keep bit is 0.
    __device__ static void clear_unkept(Unit16& u, uint32_t keep)
    {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (!(keep & (1u << e)))
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
    __device__ static void clear_outside(Unit16& u, int lo, int hi)
    {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < lo || e >= hi)
                u.w[e >> 1] &= (e & 1) ? 0x0000ffffu : 0xffff0000u;
    }
    __device__ static void clear_unkept(Unit16& u, uint32_t keep)
    {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (!(keep & (1u << e)))
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
    __device__ static void clear_outside(Unit16& u, int lo, int hi)
    {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < lo || e >= hi)
                u.w[e >> 1] &= (e & 1) ? 0x0000ffffu : 0xffff0000u;
    }
    __device__ static void clear_unkept(Unit16& u, uint32_t keep)
    {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (!(keep & (1u << e)))
                u.w[e >> 1] &= (e & 1) ? 0x0000ffffu : 0xffff0000u;
    }
};

// ---------------------------------------------------------------------------
// Unit range of a kept column range: units [u0, u1) hold kept elements; only
// the first and the last of them can be partial (element e of unit j is kept
// iff lo <= e < hi with lo = c0 - j*EPU, hi = c1 - j*EPU).
// ---------------------------------------------------------------------------
struct UnitRange {
    int32_t c0, c1, u0, u1;

    template <int EPU>
    __device__ __forceinline__ static UnitRange of(int32_t c0, int32_t c1)
    {
        UnitRange u{c0, c1, c0 / EPU, (c1 + EPU - 1) / EPU};
        if (c1 <= c0)
            u.u0 = u.u1 = 0;
        return u;
    }
    __device__ __forceinline__ bool kept(int j) const { return j >= u0 && j < u1; }
};

// ---------------------------------------------------------------------------
// Row stages shared by the per-row vector kernels and the stream kernels. A
// thread holds NV slots; unit_of(k) is the row unit of slot k (row units are
// 16 bytes; UnitOf differs only in which units a thread's slots cover).
// ---------------------------------------------------------------------------

// Loads of the kept units only.
template <int NV, typename UnitOf>
__device__ __forceinline__ void load_kept(const char* row, const UnitRange& ur, UnitOf unit_of, Unit16 (&raw)[NV])
{
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (ur.kept(j))
            raw[k] = load16(row + 16 * j);
    }
}

// +0.0 stores of every unit of the row that holds no kept element.
template <int NV, typename UnitOf>
__device__ __forceinline__ void store_zeros(char* row, const UnitRange& ur, int units, UnitOf unit_of)
{
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (j < units && !ur.kept(j))
            store16(row + 16 * j, Unit16{{0u, 0u, 0u, 0u}});
    }
}

// Decode the kept units into fp32 pairs and return this thread's extreme (max
// when use_max, else min). Masked elements of a partial unit become the
// neutral value (-inf / +inf), so they can never be the extreme.
template <typename T, int NV, typename UnitOf>
__device__ __forceinline__ float fwd_decode_extreme(const Unit16 (&raw)[NV], float2 (&v)[NV][Pairs<T>::kPairs],
                                                    const UnitRange& ur, UnitOf unit_of, bool use_max)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs, EPU = 2 * PPU;
    const float neutral = use_max ? -INFINITY : INFINITY;
    float ext = neutral;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (ur.kept(j)) {
#pragma unroll
            for (int p = 0; p < PPU; ++p)
                v[k][p] = IO::get(raw[k], p);
            const int lo = ur.c0 - j * EPU, hi = ur.c1 - j * EPU;
            if (lo > 0 || hi < EPU) {
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    if (2 * p < lo || 2 * p >= hi)
                        v[k][p].x = neutral;
                    if (2 * p + 1 < lo || 2 * p + 1 >= hi)
                        v[k][p].y = neutral;
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
    return ext;
}

// Replace the pairs by 2^((x - ext) * c) (masked elements 0) and return this
// thread's sum of them.
template <typename T, int NV, typename UnitOf>
__device__ __forceinline__ float fwd_exp_sum(float2 (&v)[NV][Pairs<T>::kPairs], const UnitRange& ur, UnitOf unit_of,
                                             float ext, float c)
{
    constexpr int PPU = Pairs<T>::kPairs, EPU = 2 * PPU;
    const float2 shift = splat2(-ext), c2 = splat2(c);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (ur.kept(j)) {
#pragma unroll
            for (int p = 0; p < PPU; ++p) {
                const float2 t = __fmul2_rn(__fadd2_rn(v[k][p], shift), c2);
                v[k][p] = make_float2(ex2(t.x), ex2(t.y));
            }
            const int lo = ur.c0 - j * EPU, hi = ur.c1 - j * EPU;
            if (lo > 0 || hi < EPU) {
#pragma unroll
                for (int p = 0; p < PPU; ++p) {
                    if (2 * p < lo || 2 * p >= hi)
                        v[k][p].x = 0.0f;
                    if (2 * p + 1 < lo || 2 * p + 1 >= hi)
                        v[k][p].y = 0.0f;
                }
            }
#pragma unroll
            for (int p = 0; p < PPU; ++p)
                acc = __fadd2_rn(acc, v[k][p]);
        }
    }
    return __fadd_rn(acc.x, acc.y);
}

// Store y = e * f for the kept units (masked elements of partial units are
// already 0, so they store as +0.0).
template <typename T, int NV, typename UnitOf>
__device__ __forceinline__ void fwd_store(char* row, const float2 (&v)[NV][Pairs<T>::kPairs], const UnitRange& ur,
                                          UnitOf unit_of, float f)
{
    using IO = Pairs<T>;
    const float2 f2 = splat2(f);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (ur.kept(j)) {
            Unit16 o;
#pragma unroll
            for (int p = 0; p < IO::kPairs; ++p)
                IO::put(o, p, __fmul2_rn(v[k][p], f2));
            store16(row + 16 * j, o);
        }
    }
}

// Backward: zero the masked elements of partial units (also clears any NaN
// there), then return this thread's float-float dot sum(dy * y) in (hi, lo).
template <typename T, int NV, typename UnitOf>
__device__ __forceinline__ void bwd_dot(Unit16 (&ry)[NV], Unit16 (&rg)[NV], const UnitRange& ur, UnitOf unit_of,
                                        float& hi, float& lo)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs, EPU = 2 * PPU;
    float2 hi2 = make_float2(0.0f, 0.0f), lo2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (ur.kept(j)) {
            const int lo_e = ur.c0 - j * EPU, hi_e = ur.c1 - j * EPU;
            if (lo_e > 0 || hi_e < EPU) {
                IO::clear_outside(ry[k], lo_e, hi_e);
                IO::clear_outside(rg[k], lo_e, hi_e);
            }
#pragma unroll
            for (int p = 0; p < PPU; ++p) {
                const float2 a = IO::get(ry[k], p), cdy = IO::get(rg[k], p);
                const float2 pr = __fmul2_rn(a, cdy);
                const float2 s = __fadd2_rn(hi2, pr);
                const float2 bb = __fadd2_rn(s, neg2(hi2));
                const float2 e = __fadd2_rn(__fadd2_rn(hi2, neg2(__fadd2_rn(s, neg2(bb)))), __fadd2_rn(pr, neg2(bb)));
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
    float e0;
    two_sum(hi2.x, hi2.y, hi, e0);
    lo = __fadd_rn(__fadd_rn(lo2.x, lo2.y), e0);
}

// Backward: store dx = scale * y * ((dy - dh) - dl) for the kept units, +0.0
// bits at masked elements.
template <typename T, int NV, typename UnitOf>
__device__ __forceinline__ void bwd_store(char* row, const Unit16 (&ry)[NV], const Unit16 (&rg)[NV],
                                          const UnitRange& ur, UnitOf unit_of, float dh, float dl, float scale,
                                          uint64_t pol = 0, bool hint = false)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs, EPU = 2 * PPU;
    const float2 ndh = splat2(-dh), ndl = splat2(-dl), sc = splat2(scale);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (ur.kept(j)) {
            Unit16 o;
#pragma unroll
            for (int p = 0; p < PPU; ++p) {
                const float2 a = IO::get(ry[k], p), cdy = IO::get(rg[k], p);
                const float2 diff = __fadd2_rn(__fadd2_rn(cdy, ndh), ndl);
                IO::put(o, p, __fmul2_rn(__fmul2_rn(a, diff), sc));
            }
            const int lo_e = ur.c0 - j * EPU, hi_e = ur.c1 - j * EPU;
            if (lo_e > 0 || hi_e < EPU)
                IO::clear_outside(o, lo_e, hi_e);
            if (hint)
                store16_hint(row + 16 * j, o, pol);
            else
                store16(row + 16 * j, o);
        }
    }
}

// ---------------------------------------------------------------------------
// Vector forward: y = masked softmax(scale * x), one team per row.
//
// t = (x - x_ext) * (scale * log2 e) with x_ext the row max (scale >= 0) or min
// (scale < 0): t <= 0 everywhere and exactly 0 at the extreme element, so a
// one-element row gives exp = 1, sum = 1, y = 1.
// ---------------------------------------------------------------------------
template <typename T, int MK, int TW, int NV, int MINB>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW, MINB)
gtms_fwd_vec_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    // Per-warp slots of the max and of the sum. A warp writes the max slots of
    // row k + 1 only after the sum barrier of row k, which every warp reaches
    // after reading row k's max slots (and likewise for the sum slots).
    __shared__ float red[TW > 32 ? 2 * (TW / 32) : 1];
    float* red_max = red;
    float* red_sum = TW > 32 ? red + TW / 32 : red;

    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);
    const auto unit_of = [tid](int k) { return tid + k * TW; };

    for (int64_t q = team; q < g.rows; q += nteams) {
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
            continue;   // uniform across the team

        float2 v[NV][Pairs<T>::kPairs];
        float ext = fwd_decode_extreme<T, NV>(raw, v, ur, unit_of, use_max);
        ext = use_max ? team_max<TW>(ext, red_max) : -team_max<TW>(-ext, red_max);
        const float s = team_sum<TW>(fwd_exp_sum<T, NV>(v, ur, unit_of, ext, c), red_sum);
        fwd_store<T, NV>(yr, v, ur, unit_of, __frcp_rn(s));
    }
}

// ---------------------------------------------------------------------------
// Heads forward: the vector forward with a team per (batch, row) pair that
// runs the pair's M heads in turn. The heads share the row's kept range, so a
// team loads head m + 1's kept units right after decoding head m's, and those
// loads are in flight through head m's two reductions and its stores. Same
// arithmetic in the same order as gtms_fwd_vec_kernel, so the same bits.
// ---------------------------------------------------------------------------
template <typename T, int MK, int TW, int NV, int MINB>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW, MINB)
gtms_fwd_heads_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    __shared__ float red[TW > 32 ? 2 * (TW / 32) : 1];
    float* red_max = red;
    float* red_sum = TW > 32 ? red + TW / 32 : red;
    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);
    const auto unit_of = [tid](int k) { return tid + k * TW; };
    const int32_t M = static_cast<int32_t>(g.rows_per_b / g.S);

    for (int64_t qm = team; qm < g.rows / M; qm += nteams) {
        const int32_t b = static_cast<int32_t>(qm / g.S), r = static_cast<int32_t>(qm % g.S);
        int32_t c0, c1;
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const int64_t q0 = static_cast<int64_t>(b) * M * g.S + r;
        Unit16 raw[NV];
        load_kept<NV>(reinterpret_cast<const char*>(x + q0 * g.S), ur, unit_of, raw);
        for (int32_t m = 0; m < M; ++m) {
            const int64_t q = q0 + static_cast<int64_t>(m) * g.S;
            char* yr = reinterpret_cast<char*>(y + q * g.S);
            store_zeros<NV>(yr, ur, g.units, unit_of);
            if (c1 <= c0)
                continue;
            float2 v[NV][Pairs<T>::kPairs];
            float ext = fwd_decode_extreme<T, NV>(raw, v, ur, unit_of, use_max);
            if (m + 1 < M)
                load_kept<NV>(reinterpret_cast<const char*>(x + (q + g.S) * g.S), ur, unit_of, raw);
            ext = use_max ? team_max<TW>(ext, red_max) : -team_max<TW>(-ext, red_max);
            const float s = team_sum<TW>(fwd_exp_sum<T, NV>(v, ur, unit_of, ext, c), red_sum);
            fwd_store<T, NV>(yr, v, ur, unit_of, __frcp_rn(s));
        }
    }
}

// ---------------------------------------------------------------------------
// Vector backward: dx = scale * y * (dy - rowsum(dy * y)), one team per row.
// The raw units of y and dy stay in registers; each pass decodes them.
// ---------------------------------------------------------------------------
template <typename T, int MK, int TW, int NV, int MINB>
__global__ void __launch_bounds__(TW == 32 ? kWarpTeamBlock : TW, MINB)
gtms_bwd_vec_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    // Two buffers, alternating per reduced row: with a single exchange per row a
    // fast warp could otherwise overwrite a slot that a slow warp is still reading.
    __shared__ float red[2][TW > 32 ? 2 * (TW / 32) : 1];
    int par = 0;

    int tid;
    int64_t team, nteams;
    team_coords<TW>(tid, team, nteams);
    const auto unit_of = [tid](int k) { return tid + k * TW; };

    for (int64_t q = team; q < g.rows; q += nteams) {
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
        par ^= 1;
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));
        bwd_store<T, NV>(dr, ry, rg, ur, unit_of, dh, dl, scale);
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

template <typename T, int MK, int TW, int NV>
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
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const Raw* xr = reinterpret_cast<const Raw*>(x + q * g.S);
        Raw* yr = reinterpret_cast<Raw*>(y + q * g.S);

        float v[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= c0 && j < c1)
                v[k] = E::get(xr[j]);
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if ((j < c0 || j >= c1) && j < g.S)
                yr[j] = Raw(0);
        }
        if (c1 <= c0)
            continue;

        float ext = use_max ? -INFINITY : INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= c0 && j < c1)
                ext = use_max ? fmaxf(ext, v[k]) : fminf(ext, v[k]);
        }
        ext = use_max ? team_max<TW>(ext, red) : -team_max<TW>(-ext, red);

        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= c0 && j < c1) {
                v[k] = ex2(__fmul_rn(__fsub_rn(v[k], ext), c));
                s = __fadd_rn(s, v[k]);
            }
        }
        s = team_sum<TW>(s, red + (TW > 32 ? TW / 32 : 0));
        const float inv = __frcp_rn(s);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= c0 && j < c1)
                yr[j] = E::put(__fmul_rn(v[k], inv));
        }
    }
}

template <typename T, int MK, int TW, int NV>
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
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const Raw* yr = reinterpret_cast<const Raw*>(y + q * g.S);
        const Raw* gr = reinterpret_cast<const Raw*>(dy + q * g.S);
        Raw* dr = reinterpret_cast<Raw*>(dx + q * g.S);

        float vy[NV], vg[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= c0 && j < c1) {
                vy[k] = E::get(yr[j]);
                vg[k] = E::get(gr[j]);
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if ((j < c0 || j >= c1) && j < g.S)
                dr[j] = Raw(0);
        }
        if (c1 <= c0)
            continue;

        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= c0 && j < c1) {
                const float p = __fmul_rn(vy[k], vg[k]);
                const float pe = __fmaf_rn(vy[k], vg[k], -p);
                float s, e;
                two_sum(hi, p, s, e);
                hi = s;
                lo = __fadd_rn(lo, __fadd_rn(e, pe));
            }
        }
        team_ff_sum<TW>(hi, lo, red[par]);
        par ^= 1;
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = tid + k * TW;
            if (j >= c0 && j < c1)
                dr[j] = E::put(__fmul_rn(__fmul_rn(vy[k], __fsub_rn(__fsub_rn(vg[k], dh), dl)), scale));
        }
    }
}

}  // namespace gtms
