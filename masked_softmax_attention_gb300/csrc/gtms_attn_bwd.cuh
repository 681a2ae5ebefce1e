// gtms_attn_bwd.cuh -- the attention-backward step around the masked softmax,
// fused with its GEMM on the sm_100+ tensor cores.
//
// "ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1: with P the masked
// softmax, O = P V and upstream gradient dO, the backward forms dP = dO V^T and
// then dS = softmax-backward(dP, P) = scale * P * (dP - rowsum(dP * P)) -- the
// softmax backward of this library with dY = dP. Here dP never goes to memory:
// a CTA owns 128 rows of one (b, m) slice, keeps their 128 rows of dO in shared
// memory and, for each 128-column tile that holds kept entries (the grouped
// tril mask keeps c <= r < L, so only tiles up to the diagonal), computes the
// dP tile with tcgen05.mma into tensor memory:
//   pass 1 reads each dP tile back and forms the row sum d_r = sum_c dP_rc P_rc
//          over kept columns: each 16-byte unit's 8 products summed in fp32, the
//          unit sums accumulated as a float-float pair;
//   pass 2 recomputes the same tiles and writes dS = scale * P * ((dP - d_hi) - d_lo),
//          +0.0 at masked entries.
// Recomputing the K = d GEMM costs far less than sending dP through HBM, which
// a one-pass version would need: a 128-row dP block of a long row does not fit
// in the 512 tensor-memory columns. Columns past the diagonal tile and padded
// row blocks are written as +0.0 without any GEMM.
//
// Pipeline (256 threads, two CTAs per SM). Each tile iteration has a stage in
// shared memory: the V tile (the MMA's B operand) and the P tile. Both are
// fetched with cp.async one iteration ahead, into the other stage, so the
// loads of the next tile overlap the MMA, the read-back and the stores of
// this one. Warp w reads tensor-memory lanes 32 (w % 4) .. + 31 (its rows) and
// columns 64 (w / 4) .. + 63 of the tile. The P tile is stored as two
// 128-row x 128-byte halves in the 128-byte swizzle pattern (16-byte chunk j
// of row r at chunk j ^ (r % 8)), so both the row-per-thread read-back and the
// coalesced row-major copies are free of bank conflicts. Pass 2 writes dS over
// P in the same stage, and the CTA then stores the tile with 16-byte stores
// that are contiguous along each row.
//
// Only 16-byte units of P that hold a kept element are fetched. Every wait on
// the MMA's mbarrier is bounded in time; if one runs out the kernel ORs
// GTMS_ERR_TIMEOUT into the caller's status word, skips the remaining work,
// frees its tensor memory and returns.
#pragma once

#include <cstdint>
#include <type_traits>

#include "gtms.h"
#include "gtms_kernels.cuh"
#include "gtms_tcgen05.cuh"

namespace gtms {

constexpr int kAttnRows = 128;      // rows per CTA (the MMA's M) and columns per tile (its N)
constexpr int kAttnThreads = 256;
constexpr uint32_t kAttnPTileBytes = kAttnRows * 256;   // one 128 x 128 tile of 16-bit P or dS

template <int D>
struct AttnSmem {
    static constexpr uint32_t op = kAttnRows * D * 2;              // 128 rows of dO or V
    static constexpr uint32_t stage = op + kAttnPTileBytes;        // V tile + P tile
    static constexpr uint32_t total = op + 2 * stage;              // dO + two stages
    static constexpr uint32_t sbo = (D / 8) * 128;                 // core-matrix stride along rows
};

// Byte offset of 16-byte chunk c16 (0..15) of tile row `row` in a P / dS stage.
__device__ __forceinline__ uint32_t p_chunk_offset(int row, int c16)
{
    return (c16 >> 3) * (kAttnRows * 128) + row * 128 + ((((c16 & 7) ^ (row & 7))) << 4);
}

// Fetch rows [row0, row0 + 128) of a [S, D] matrix into the no-swizzle K-major
// core-matrix layout (LBO = 128 bytes along K, SBO = D * 16 bytes along rows);
// rows >= S become zero. Eight consecutive threads take one 16-byte column
// chunk of eight consecutive rows, so a warp reads 8 rows x 64 contiguous
// bytes and writes 512 contiguous bytes of shared memory. Chunk q of the copy
// is (row group q / (8 D / 8), column chunk (q / 8) % (D / 8), row q % 8); a
// thread takes q = tid + 256 k.
template <int D>
__device__ __forceinline__ void fetch_operand(uint32_t dst, const uint8_t* mat, int32_t row0, int32_t S)
{
    constexpr int kc_n = D / 8;
    constexpr int per_thread = kAttnRows * kc_n / kAttnThreads;
    constexpr int groups_per_k = kAttnThreads / (8 * kc_n);   // row groups advanced per k
    const int tid = threadIdx.x;
    const int n_lo = tid & 7, kc = (tid >> 3) % kc_n, n_hi0 = tid / (8 * kc_n);
    const uint32_t soff = dst + n_hi0 * AttnSmem<D>::sbo + kc * 128 + n_lo * 16;
    const int32_t row_t = row0 + n_hi0 * 8 + n_lo;
#pragma unroll
    for (int k = 0; k < per_thread; ++k) {
        const int32_t row = row_t + k * groups_per_k * 8;
        const bool in = row < S;
        tc::cp_async16(soff + k * groups_per_k * AttnSmem<D>::sbo,
                       mat + static_cast<int64_t>(in ? row : 0) * (D * 2) + kc * 16, in ? 16u : 0u);
    }
}

// A thread's share of copying one 128 x 128 tile between global memory and a
// P / dS stage: 16-byte column chunk c16 = tid % 16 of tile rows row0 + 16 k
// (row0 = tid / 16, k = 0..7), so sixteen consecutive threads cover one
// 256-byte tile row. In the stage, row + 16 k lies 16 k * 128 bytes further.
struct TileLane {
    int c16, row0;
    uint32_t soff;
    __device__ __forceinline__ TileLane()
        : c16(threadIdx.x & 15), row0(threadIdx.x >> 4), soff(p_chunk_offset(threadIdx.x >> 4, threadIdx.x & 15))
    {
    }
};

// Fetch the units of the P tile at columns [tc0, tc0 + 128) that hold a kept
// element (row r live, first column <= r).
template <typename T>
__device__ __forceinline__ void fetch_p_tile(uint32_t dst, const TileLane& tl, const T* p_slice, int32_t S, int32_t r0,
                                             int32_t L, int32_t tc0)
{
    const int32_t c = tc0 + tl.c16 * 8;
    const int32_t r_first = r0 + tl.row0;
    const T* src = p_slice + static_cast<int64_t>(r_first) * S + c;
#pragma unroll
    for (int k = 0; k < kAttnRows / 16; ++k) {
        const int32_t r = r_first + 16 * k;
        if (r < L && c <= r)   // (r < L <= S, so the unit lies inside the row)
            tc::cp_async16(dst + tl.soff + k * 2048, src + static_cast<int64_t>(16 * k) * S, 16u);
    }
}

// Store the units of a finished dS tile (columns [tc0, tc0 + 128)) of the live rows.
template <typename T>
__device__ __forceinline__ void store_ds_tile(const uint8_t* stage, const TileLane& tl, T* ds_slice, int32_t S,
                                              int32_t r0, int32_t L, int32_t tc0)
{
    const int32_t c = tc0 + tl.c16 * 8;
    if (c >= S)
        return;
    const int32_t r_first = r0 + tl.row0;
    T* dst = ds_slice + static_cast<int64_t>(r_first) * S + c;
#pragma unroll
    for (int k = 0; k < kAttnRows / 16; ++k) {
        if (r_first + 16 * k < L)
            *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(16 * k) * S) =
                *reinterpret_cast<const uint4*>(stage + tl.soff + k * 2048);
    }
}

// Zero-fill columns [c_from, S) of rows [row0, row1) of one [S, S] slice with
// 16-byte stores, `nthreads` threads (this one is number t) walking the
// region's units in row-major order (S % 8 == 0). The lines are marked to
// leave L2 first: nothing reads them again.
template <typename T>
__device__ __forceinline__ void zero_region(T* slice, int32_t S, int32_t row0, int32_t row1, int32_t c_from,
                                            int t = threadIdx.x, int nthreads = kAttnThreads)
{
    const int32_t units = (S - c_from) / 8;   // per row
    if (units <= 0 || row1 <= row0)
        return;
    const uint64_t pol = tc::policy_evict_first();
    int32_t r = row0, u = t;
    while (u >= units) {
        u -= units;
        ++r;
    }
    uint4* row_ptr = reinterpret_cast<uint4*>(slice + static_cast<int64_t>(r) * S + c_from);
    const int32_t row_units = S / 8;
    while (r < row1) {
        tc::st_global_zero16(row_ptr + u, pol);
        u += nthreads;
        while (u >= units) {
            u -= units;
            ++r;
            row_ptr += row_units;
        }
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kAttnThreads, 2)
gtms_attn_dscores_kernel(const T* P, const T* dO, const T* V, T* dS, const int32_t* __restrict__ seq_lens,
                         int32_t M, int32_t S, int32_t n_row_blocks, float scale, int32_t* status,
                         uint64_t wait_ns)
{
    using IO = Pairs<T>;
    using SM = AttnSmem<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t mbar;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int64_t slice = blockIdx.x / n_row_blocks;          // b * M + m
    const int32_t r0 = (blockIdx.x % n_row_blocks) * kAttnRows;
    const int32_t b = static_cast<int32_t>(slice / M);
    int32_t L = __ldg(seq_lens + b);
    L = L < 0 ? 0 : (L > S ? S : L);
    const int32_t r_end = r0 + kAttnRows < S ? r0 + kAttnRows : S;   // rows of this block
    T* ds_slice = dS + slice * static_cast<int64_t>(S) * S;

    if (r0 >= L) {   // padded row block: all zero, no GEMM
        zero_region(ds_slice, S, r0, r_end, 0);
        return;
    }
    // Kept columns satisfy c <= r < r0 + 128: tiles 0 .. r0 / 128 (the diagonal tile).
    const int32_t n_tiles = r0 / kAttnRows + 1;
    const int32_t n_iter = 2 * n_tiles;                       // pass 1, then pass 2
    const int64_t slice_rows = slice * static_cast<int64_t>(S);
    const T* p_slice = P + slice_rows * S;
    const uint8_t* do_mat = reinterpret_cast<const uint8_t*>(dO + slice_rows * D);
    const uint8_t* v_mat = reinterpret_cast<const uint8_t*>(V + slice_rows * D);
    const uint32_t s_a = tc::smem_u32(smem);
    const uint32_t s_stage0 = s_a + SM::op;

    // Prologue: dO, and the first tile's V and P, in flight while the zero regions are stored.
    const TileLane tl;
    fetch_operand<D>(s_a, do_mat, r0, S);
    fetch_operand<D>(s_stage0, v_mat, 0, S);
    fetch_p_tile<T>(s_stage0 + SM::op, tl, p_slice, S, r0, L, 0);
    tc::cp_async_commit();

    const int32_t c_tiles_end = n_tiles * kAttnRows < S ? n_tiles * kAttnRows : S;
    const int32_t live_end = L < r_end ? L : r_end;
    zero_region(ds_slice, S, r0, live_end, c_tiles_end);   // live rows: right of the diagonal tile
    zero_region(ds_slice, S, live_end, r_end, 0);          // padded rows of this block: whole rows

    if (warp == 0)
        tc::tmem_alloc<kAttnRows>(&tmem_slot);
    if (tid == 0)
        tc::mbar_init(&mbar, 1);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tmem_mine = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * 64;
    constexpr uint32_t idesc = tc::idesc_f16<T>(kAttnRows, kAttnRows);

    const int row = quarter * 32 + lane;             // this thread's row in the block
    const int32_t r = r0 + row;
    const bool live = r < L;                          // (L <= S, so live rows are in range)
    float dot_hi = 0.0f, dot_lo = 0.0f, dh = 0.0f, dl = 0.0f;
    uint32_t phase = 0;
    bool failed = false;

    for (int32_t i = 0; i < n_iter; ++i) {
        const bool pass2 = i >= n_tiles;
        const int32_t tc0 = (pass2 ? i - n_tiles : i) * kAttnRows;
        const uint32_t st_v = s_stage0 + (i & 1) * SM::stage, st_p = st_v + SM::op;
        uint8_t* p_tile = smem + (st_p - s_a);

        tc::cp_async_wait_all();       // this iteration's V and P (fetched one iteration ago)
        tc::fence_smem_for_async();    // ... visible to the tensor core
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_f16(tmem, tc::smem_desc(s_a + ks * 256, 128, SM::sbo), tc::smem_desc(st_v + ks * 256, 128, SM::sbo),
                            idesc, ks > 0 ? 1u : 0u);
            tc::commit(&mbar);
        }
        if (i + 1 < n_iter) {          // next iteration's tile into the other stage
            const int32_t i1 = i + 1;
            const int32_t tn = (i1 >= n_tiles ? i1 - n_tiles : i1) * kAttnRows;
            const uint32_t nx_v = s_stage0 + (i1 & 1) * SM::stage;
            fetch_operand<D>(nx_v, v_mat, tn, S);
            fetch_p_tile<T>(nx_v + SM::op, tl, p_slice, S, r0, L, tn);
            tc::cp_async_commit();
        }
        const bool ok = tc::mbar_wait(&mbar, phase, wait_ns);
        phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc::fence_after_sync();
        float dp[64];
        tc::tmem_ld64(tmem_mine, dp);   // warp-collective: every thread takes part
        if (live) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c16 = half * 8 + u;
                const int32_t c = tc0 + c16 * 8;
                uint4* cell = reinterpret_cast<uint4*>(p_tile + p_chunk_offset(row, c16));
                if (c >= S)
                    continue;
                if (c > r) {                           // no kept element in this unit
                    if (pass2)
                        *cell = make_uint4(0u, 0u, 0u, 0u);
                    continue;
                }
                const uint4 raw = *cell;
                Unit16 pu{{raw.x, raw.y, raw.z, raw.w}};
                const bool diag = c + 7 > r;           // the unit holding the diagonal
                if (diag) {   // masked P and dP read as +0.0 (dP may be infinite where P is masked)
                    IO::clear_outside(pu, 0, r - c + 1);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dp[u * 8 + e] = c + e <= r ? dp[u * 8 + e] : 0.0f;
                }
                if (!pass2) {
                    // Unit sum in fp32 (two FMA chains), then into the float-float row sum.
                    float2 acc = __fmul2_rn(IO::get(pu, 0), make_float2(dp[u * 8], dp[u * 8 + 1]));
#pragma unroll
                    for (int q = 1; q < 4; ++q)
                        acc = __ffma2_rn(IO::get(pu, q), make_float2(dp[u * 8 + 2 * q], dp[u * 8 + 2 * q + 1]), acc);
                    float s, e;
                    two_sum(dot_hi, __fadd_rn(acc.x, acc.y), s, e);
                    dot_hi = s;
                    dot_lo = __fadd_rn(dot_lo, e);
                } else {
                    const float2 ndh = make_float2(-dh, -dh), ndl = make_float2(-dl, -dl);
                    const float2 sc = make_float2(scale, scale);
                    Unit16 o;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 g = make_float2(dp[u * 8 + 2 * q], dp[u * 8 + 2 * q + 1]);
                        const float2 t = __fadd2_rn(__fadd2_rn(g, ndh), ndl);
                        IO::put(o, q, __fmul2_rn(__fmul2_rn(IO::get(pu, q), t), sc));
                    }
                    if (diag)
                        IO::clear_outside(o, 0, r - c + 1);   // masked entries are +0.0 bits
                    *cell = make_uint4(o.w[0], o.w[1], o.w[2], o.w[3]);
                }
            }
        }
        tc::fence_before_sync();
        __syncthreads();   // tensor memory read back; the dS tile is complete in shared memory

        if (!pass2 && i == n_tiles - 1) {
            // Merge the two column halves' float-float sums (scratch: this stage's V
            // tile, whose MMA has completed and which is refilled only next iteration).
            float* red = reinterpret_cast<float*>(smem + (st_v - s_a));
            if (half == 1) {
                red[row] = dot_hi;
                red[kAttnRows + row] = dot_lo;
            }
            __syncthreads();
            if (half == 0) {
                float s, e;
                two_sum(dot_hi, red[row], s, e);
                const float lo = __fadd_rn(__fadd_rn(dot_lo, red[kAttnRows + row]), e);
                dh = __fadd_rn(s, lo);
                dl = __fsub_rn(lo, __fsub_rn(dh, s));
                red[2 * kAttnRows + row] = dh;
                red[3 * kAttnRows + row] = dl;
            }
            __syncthreads();
            if (half == 1) {
                dh = red[2 * kAttnRows + row];
                dl = red[3 * kAttnRows + row];
            }
        }
        if (pass2)   // the live rows' units of this tile, 256 contiguous bytes per row
            store_ds_tile<T>(p_tile, tl, ds_slice, S, r0, L, tc0);
    }

    tc::cp_async_wait_all();
    if (failed) {
        if (tid == 0 && status)
            atomicOr(status, GTMS_ERR_TIMEOUT);
        tc::mbar_wait(&mbar, phase ^ 1u, kAttnDrainWaitNs);   // one more bounded wait for the MMA in flight
        tc::fence_before_sync();
        __syncthreads();
    }
    if (warp == 0)
        tc::tmem_free<kAttnRows>(tmem);
}

// Launch over B * M slices of ceil(S / 128) row blocks; dynamic shared memory
// holds dO and two stages of (V tile, P tile).
template <typename T, int D>
cudaError_t launch_attn_dscores(const void* P, const void* dO, const void* V, void* dS, const int32_t* seq_lens,
                                int64_t B, int64_t M, int64_t S, float scale, int32_t* status, cudaStream_t st,
                                uint64_t wait_ns = kAttnWaitNs)
{
    constexpr int smem = static_cast<int>(AttnSmem<D>::total);
    auto* kern = gtms_attn_dscores_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    const int32_t nrb = static_cast<int32_t>((S + kAttnRows - 1) / kAttnRows);
    const int64_t grid = B * M * nrb;
    return launch_kernel(kern, static_cast<unsigned>(grid), kAttnThreads, smem, st, static_cast<const T*>(P),
                         static_cast<const T*>(dO), static_cast<const T*>(V), static_cast<T*>(dS), seq_lens,
                         static_cast<int32_t>(M), static_cast<int32_t>(S), nrb, scale, status, wait_ns);
}

}  // namespace gtms
