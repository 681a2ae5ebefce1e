// gtms_stream.cuh -- long rows streamed in two passes by one CTA.
//
// A row held whole in registers caps the rows in flight per SM: at S = 32768
// (16-bit) a 1024-thread CTA holds one row and the SM holds one such CTA, so
// the SM idles while that row reduces. The stream kernels hold only a batch of
// U units per thread and walk the row's kept units twice, TW * U units at a
// time:
//   pass 1 loads a batch and folds it into the thread's running extreme m and
//          running sum l of 2^((x - m) c); when the extreme moves, l is first
//          rescaled by 2^((m_old - m_new) c) (the online normaliser of
//          Milakov and Gimelshein, "Online normalizer calculation for
//          softmax", 2018);
//   the threads' (m, l) merge, first per warp into (e_w, s_w), then in one
//          exchange across the warps into the row's extreme E and sum S, as a
//          split-KV reduction merges partial softmax results (ColossalAI
//          flash_decoding.py, the reduce kernel);
//   pass 2 walks the batches in reverse order, so the units read last in
//          pass 1 -- the ones most likely still in L2 -- are read first, and
//          stores 2^((x - E) c) / S.
// The backward is the same walk with the float-float dot of gtms_kernels.cuh
// in pass 1 and dx = scale * y * (dy - d) in pass 2.
//
// The kept units of a row are read twice; the second read is meant to hit L2
// (the rows in flight hold far less than its 129 MB), so DRAM still sees each
// kept byte about once. Cache policies make it so at the longest rows: pass 1
// reads with evict_last, pass 2 reads and every store (zeros and outputs) with
// evict_first, so the output stream does not push pass 1's lines out of L2
// (measured on GB300 at S = 65536: forward 0.95 -> 0.99 and backward 0.91 ->
// 0.96 of the copy rate in bf16, 1.00 -> 1.04 and 0.93 -> 0.98 in fp32).
// Zero stores of the masked units are issued first, as in the other kernels.
// Every unit is loaded and stored by the same thread, so an output may alias
// its input exactly.
#pragma once

#include "gtms_kernels.cuh"

namespace gtms {

// Units of batch i of a thread: base(i) + tid + k * TW, k < U, clipped to [u0, u1).
template <int TW, int U>
struct StreamBatch {
    int32_t first;   // first unit of the batch for this thread (slot 0)
    __device__ __forceinline__ int operator()(int k) const { return first + k * TW; }
};

// Element e of unit j lies in the kept range iff lo <= e < hi (lo = c0 - j*EPU,
// hi = c1 - j*EPU); only the first and last kept units are partial.
__device__ __forceinline__ bool in_range(int e, int lo, int hi) { return e >= lo && e < hi; }

// Loads of the kept units of one batch under an L2 policy.
template <int NV, typename UnitOf>
__device__ __forceinline__ void load_kept_hint(const char* row, const UnitRange& ur, UnitOf unit_of, Unit16 (&raw)[NV],
                                               uint64_t pol)
{
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = unit_of(k);
        if (ur.kept(j))
            raw[k] = load16_hint(row + 16 * j, pol);
    }
}

// Pass 1 of one batch: fold the kept elements of the units at(k) into the
// running extreme m and sum l. Values are decoded from the raw units twice (for
// the extreme, then for the exponentials) rather than held as fp32.
template <typename T, int U, typename At>
__device__ __forceinline__ void stream_fold(const Unit16 (&raw)[U], const UnitRange& ur, At at, float c,
                                            bool use_max, float& m, float& l)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs, EPU = 2 * PPU;
    const float neutral = use_max ? -INFINITY : INFINITY;
    float mb = neutral;
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const int j = at(k);
        if (ur.kept(j)) {
            const int lo = ur.c0 - j * EPU, hi = ur.c1 - j * EPU;
            const bool partial = lo > 0 || hi < EPU;
#pragma unroll
            for (int p = 0; p < PPU; ++p) {
                float2 v = IO::get(raw[k], p);
                if (partial) {
                    if (!in_range(2 * p, lo, hi))
                        v.x = neutral;
                    if (!in_range(2 * p + 1, lo, hi))
                        v.y = neutral;
                }
                mb = use_max ? max3(mb, v.x, v.y) : min3(mb, v.x, v.y);
            }
        }
    }
    if (mb == neutral)
        return;   // no kept element of this thread in the batch
    const float mn = use_max ? fmaxf(m, mb) : fminf(m, mb);
    // Rescale only a non-empty sum whose extreme moved: an empty sum has no
    // extreme yet (m is still the neutral infinity), and an unmoved extreme
    // would cost an exponential for a factor of 1 -- or give NaN from
    // inf - inf when the extreme is an infinite input.
    if (l != 0.0f && m != mn)
        l = __fmul_rn(l, ex2(__fmul_rn(__fsub_rn(m, mn), c)));
    m = mn;
    const float2 shift = splat2(-mn), c2 = splat2(c);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const int j = at(k);
        if (ur.kept(j)) {
            const int lo = ur.c0 - j * EPU, hi = ur.c1 - j * EPU;
            const bool partial = lo > 0 || hi < EPU;
#pragma unroll
            for (int p = 0; p < PPU; ++p) {
                const float2 t = __fmul2_rn(__fadd2_rn(IO::get(raw[k], p), shift), c2);
                float2 e = make_float2(ex2(t.x), ex2(t.y));
                if (partial) {
                    if (!in_range(2 * p, lo, hi))
                        e.x = 0.0f;
                    if (!in_range(2 * p + 1, lo, hi))
                        e.y = 0.0f;
                }
                acc = __fadd2_rn(acc, e);
            }
        }
    }
    l = __fadd_rn(l, __fadd_rn(acc.x, acc.y));
}

// Pass 2 of one batch: store y = 2^((x - e) c) * f for the kept units (e the
// row's extreme, f = 1 / sum; masked elements of partial units as +0.0).
template <typename T, int U, typename At>
__device__ __forceinline__ void stream_store(char* row, const Unit16 (&raw)[U], const UnitRange& ur, At at, float e,
                                             float c, float f, uint64_t pol)
{
    using IO = Pairs<T>;
    constexpr int PPU = IO::kPairs, EPU = 2 * PPU;
    const float2 shift = splat2(-e), c2 = splat2(c), f2 = splat2(f);
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const int j = at(k);
        if (ur.kept(j)) {
            const int lo = ur.c0 - j * EPU, hi = ur.c1 - j * EPU;
            const bool partial = lo > 0 || hi < EPU;
            Unit16 o;
#pragma unroll
            for (int p = 0; p < PPU; ++p) {
                const float2 t = __fmul2_rn(__fadd2_rn(IO::get(raw[k], p), shift), c2);
                float2 y = make_float2(ex2(t.x), ex2(t.y));
                if (partial) {
                    if (!in_range(2 * p, lo, hi))
                        y.x = 0.0f;
                    if (!in_range(2 * p + 1, lo, hi))
                        y.y = 0.0f;
                }
                IO::put(o, p, __fmul2_rn(y, f2));
            }
            store16_hint(row + 16 * j, o, pol);
        }
    }
}

template <typename T, int MK, int TW, int U, int MINB>
__global__ void __launch_bounds__(TW, MINB)
gtms_fwd_stream_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    // L2 policies: pass 1's reads stay for pass 2; pass 2's reads and every store go first.
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    constexpr int kBatch = TW * U;
    __shared__ float red[2][2 * (TW / 32)];
    int par = 0;

    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    const int tid = threadIdx.x;

    for (int64_t q = blockIdx.x; q < g.rows; q += gridDim.x) {
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const char* xr = reinterpret_cast<const char*>(x + q * g.S);
        char* yr = reinterpret_cast<char*>(y + q * g.S);

        for (int j = tid; j < ur.u0; j += TW)
            store16_hint(yr + 16 * j, Unit16{{0u, 0u, 0u, 0u}}, drop);
        for (int j = ur.u1 + tid; j < g.units; j += TW)
            store16_hint(yr + 16 * j, Unit16{{0u, 0u, 0u, 0u}}, drop);
        if (c1 <= c0)
            continue;   // uniform across the CTA

        // Pass 1: running extreme and rescaled sum.
        float m = use_max ? -INFINITY : INFINITY, l = 0.0f;
        const int nb = (ur.u1 - ur.u0 + kBatch - 1) / kBatch;
        for (int i = 0; i < nb; ++i) {
            const StreamBatch<TW, U> at{ur.u0 + i * kBatch + tid};
            Unit16 raw[U];
            load_kept_hint<U>(xr, ur, at, raw, keep);
            stream_fold<T, U>(raw, ur, at, c, use_max, m, l);
        }

        // Merge (m, l) over the warp, then over the CTA, into the row's extreme
        // E and 1 / sum. (Pass 2 exponentiates against E, not against a warp's
        // own extreme: a warp whose kept inputs are all -inf has e_w = -inf, and
        // x - e_w would be NaN there.)
        const float e_w = use_max ? team_max<32>(m, nullptr) : -team_max<32>(-m, nullptr);
        const float part = l != 0.0f ? __fmul_rn(l, ex2(__fmul_rn(__fsub_rn(m, e_w), c))) : 0.0f;
        const float s_w = team_sum<32>(part, nullptr);
        float E, inv;
        team_softmax_stats<TW>(e_w, s_w, c, use_max, red[par], E, inv);
        par ^= 1;

        // Pass 2, batches in reverse order.
        for (int i = nb - 1; i >= 0; --i) {
            const StreamBatch<TW, U> at{ur.u0 + i * kBatch + tid};
            Unit16 raw[U];
            load_kept_hint<U>(xr, ur, at, raw, drop);
            stream_store<T, U>(yr, raw, ur, at, E, c, inv, drop);
        }
    }
}

template <typename T, int MK, int TW, int U, int MINB>
__global__ void __launch_bounds__(TW, MINB)
gtms_bwd_stream_kernel(const T* y, const T* dy, T* dx, const int32_t* __restrict__ seq_lens, Geom g, float scale)
{
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    constexpr int kBatch = TW * U;
    __shared__ float red[2][2 * (TW / 32)];
    int par = 0;
    const int tid = threadIdx.x;

    for (int64_t q = blockIdx.x; q < g.rows; q += gridDim.x) {
        int32_t b, r, c0, c1;
        g.locate(q, b, r);
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const char* yr = reinterpret_cast<const char*>(y + q * g.S);
        const char* gr = reinterpret_cast<const char*>(dy + q * g.S);
        char* dr = reinterpret_cast<char*>(dx + q * g.S);

        for (int j = tid; j < ur.u0; j += TW)
            store16_hint(dr + 16 * j, Unit16{{0u, 0u, 0u, 0u}}, drop);
        for (int j = ur.u1 + tid; j < g.units; j += TW)
            store16_hint(dr + 16 * j, Unit16{{0u, 0u, 0u, 0u}}, drop);
        if (c1 <= c0)
            continue;

        // Pass 1: float-float dot over the batches.
        float hi = 0.0f, lo = 0.0f;
        const int nb = (ur.u1 - ur.u0 + kBatch - 1) / kBatch;
        for (int i = 0; i < nb; ++i) {
            const StreamBatch<TW, U> at{ur.u0 + i * kBatch + tid};
            Unit16 ry[U], rg[U];
            load_kept_hint<U>(yr, ur, at, ry, keep);
            load_kept_hint<U>(gr, ur, at, rg, keep);
            float bh, bl;
            bwd_dot<T, U>(ry, rg, ur, at, bh, bl);
            ff_merge(hi, lo, bh, bl);
        }
        team_ff_sum<TW>(hi, lo, red[par]);
        par ^= 1;
        const float dh = __fadd_rn(hi, lo);
        const float dl = __fsub_rn(lo, __fsub_rn(dh, hi));

        // Pass 2, batches in reverse order.
        for (int i = nb - 1; i >= 0; --i) {
            const StreamBatch<TW, U> at{ur.u0 + i * kBatch + tid};
            Unit16 ry[U], rg[U];
            load_kept_hint<U>(yr, ur, at, ry, drop);
            load_kept_hint<U>(gr, ur, at, rg, drop);
            bwd_store<T, U>(dr, ry, rg, ur, at, dh, dl, scale, drop, true);
        }
    }
}

}  // namespace gtms
