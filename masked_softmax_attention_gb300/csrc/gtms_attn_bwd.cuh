// gtms_attn_bwd.cuh -- the attention-backward step around the masked softmax,
// fused with its GEMM on the sm_100+ tensor cores.
//
// "ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1: with P the masked
// softmax, O = P V and upstream gradient dO, the backward forms dP = dO V^T and
// then dS = softmax-backward(dP, P) = scale * P * (dP - rowsum(dP * P)) -- the
// softmax backward of this library with dY = dP. Here dP never goes to memory:
// a CTA owns 128 rows of one (b, m) slice, keeps its 128 rows of dO in shared
// memory and, for each 128-column tile that holds kept entries (the grouped
// tril mask keeps c <= r < L, so only tiles up to the diagonal), computes the
// dP tile with tcgen05.mma into tensor memory:
//   pass 1 reads each dP tile back row by row (one thread per row) and forms
//          the float-float row sum  d_r = sum_c dP_rc P_rc  over kept columns;
//   pass 2 recomputes the same tiles and writes dS = scale * P * ((dP - d_hi) - d_lo),
//          +0.0 at masked entries.
// Recomputing the K = d GEMM costs far less than sending dP through HBM, which
// a one-pass version would need: a 128-row dP block of a long row does not fit
// in the 512 tensor-memory columns. Columns past the diagonal tile and padded
// row blocks are written as +0.0 without any GEMM.
//
// P is loaded only in the 16-byte units that hold a kept element, as in the
// softmax kernels. Every wait on the MMA's mbarrier is bounded; if one runs out
// the kernel ORs 1 into the caller's status word, skips the remaining work,
// frees its tensor memory and returns.
#pragma once

#include <cstdint>
#include <type_traits>

#include "gtms_kernels.cuh"
#include "gtms_tcgen05.cuh"

namespace gtms {

constexpr int kAttnRows = 128;     // rows per CTA (the MMA's M) and columns per tile (its N)
constexpr int kAttnWaitLimit = 1 << 24;

// Copy rows [row0, row0 + 128) of a [S, D] matrix into the core-matrix layout
// (LBO = 128 bytes along K, SBO = D * 16 bytes along rows); rows >= S become 0.
template <int D>
__device__ __forceinline__ void load_rows_km(uint8_t* smem, const void* mat, int32_t row0, int32_t S)
{
    constexpr uint32_t SBO = (D / 8) * 128;
    const int t = threadIdx.x;
    const int32_t row = row0 + t;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(mat) +
                                                      static_cast<int64_t>(row) * D * 2);
#pragma unroll
    for (int kc = 0; kc < D / 8; ++kc) {
        const uint4 v = row < S ? src[kc] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + (t / 8) * SBO + kc * 128 + (t % 8) * 16) = v;
    }
}

// Zero-fill columns [c_from, S) of rows [row0, row1) of one [S, S] slice, the
// CTA's 128 threads cooperating along each row (16-byte stores; S % 8 == 0).
template <typename T>
__device__ __forceinline__ void zero_region(T* slice, int32_t S, int32_t row0, int32_t row1, int32_t c_from)
{
    const int32_t units = (S - c_from) / 8;
    for (int32_t r = row0; r < row1; ++r) {
        uint4* dst = reinterpret_cast<uint4*>(slice + static_cast<int64_t>(r) * S + c_from);
        for (int32_t u = threadIdx.x; u < units; u += kAttnRows)
            dst[u] = make_uint4(0u, 0u, 0u, 0u);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kAttnRows)
gtms_attn_dscores_kernel(const T* P, const T* dO, const T* V, T* dS, const int32_t* __restrict__ seq_lens,
                         int32_t M, int32_t S, int32_t n_row_blocks, float scale, int32_t* status)
{
    using IO = Pairs<T>;
    constexpr uint32_t SBO = (D / 8) * 128;
    extern __shared__ __align__(1024) uint8_t smem_tiles[];
    uint8_t* sA = smem_tiles;                       // 128 rows of dO
    uint8_t* sB = smem_tiles + kAttnRows * D * 2;   // 128 rows of V
    __shared__ __align__(8) uint64_t mbar;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5;
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
    const int32_t c_tiles_end = n_tiles * kAttnRows < S ? n_tiles * kAttnRows : S;
    const int32_t live_end = L < r_end ? L : r_end;
    zero_region(ds_slice, S, r0, live_end, c_tiles_end);   // live rows: right of the diagonal tile
    zero_region(ds_slice, S, live_end, r_end, 0);          // padded rows of this block: whole rows

    const int64_t slice_rows = slice * static_cast<int64_t>(S);
    load_rows_km<D>(sA, dO + slice_rows * D, r0, S);
    if (warp == 0)
        tc::tmem_alloc<kAttnRows>(&tmem_slot);
    if (tid == 0)
        tc::mbar_init(&mbar, 1);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tmem_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    constexpr uint32_t idesc = tc::idesc_f16<T>(kAttnRows, kAttnRows);

    const int32_t r = r0 + tid;                      // this thread's row
    const bool live = r < L;                         // (L <= S, so live rows are in range)
    const T* p_row = P + (slice_rows + r) * S;
    T* ds_row = ds_slice + static_cast<int64_t>(r) * S;
    float dot_hi = 0.0f, dot_lo = 0.0f, dh = 0.0f, dl = 0.0f;
    uint32_t phase = 0;
    bool failed = false;

    for (int pass = 0; pass < 2 && !failed; ++pass) {
        for (int32_t t = 0; t < n_tiles; ++t) {
            const int32_t tc0 = t * kAttnRows;
            load_rows_km<D>(sB, V + slice_rows * D, tc0, S);
            tc::fence_smem_for_async();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                const uint32_t a0 = tc::smem_u32(sA), b0 = tc::smem_u32(sB);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_f16(tmem, tc::smem_desc(a0 + ks * 256, 128, SBO), tc::smem_desc(b0 + ks * 256, 128, SBO),
                                idesc, ks > 0 ? 1u : 0u);
                tc::commit(&mbar);
            }
            const bool ok = tc::mbar_wait(&mbar, phase, kAttnWaitLimit);
            phase ^= 1u;
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
#pragma unroll 1
            for (int ch = 0; ch < kAttnRows / 32; ++ch) {
                float dp[32];
                tc::tmem_ld32(tmem_row + ch * 32, dp);   // warp-collective: every thread takes part
                if (!live)
                    continue;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int32_t c = tc0 + ch * 32 + u * 8;
                    if (c >= S)
                        continue;
                    if (c > r) {                           // no kept element in this unit
                        if (pass == 1)
                            store16(ds_row + c, Unit16{{0u, 0u, 0u, 0u}});
                        continue;
                    }
                    const Unit16 pu = load16(p_row + c);
                    if (pass == 0) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 pv = IO::get(pu, q);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                if (c + 2 * q + h <= r) {
                                    const float a = h ? pv.y : pv.x, g = dp[u * 8 + 2 * q + h];
                                    const float pr = __fmul_rn(a, g), pe = __fmaf_rn(a, g, -pr);
                                    float s, e;
                                    two_sum(dot_hi, pr, s, e);
                                    dot_hi = s;
                                    dot_lo = __fadd_rn(dot_lo, __fadd_rn(e, pe));
                                }
                            }
                        }
                    } else {
                        Unit16 o;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 pv = IO::get(pu, q);
                            float2 out;
                            out.x = (c + 2 * q <= r)
                                        ? __fmul_rn(__fmul_rn(pv.x, __fsub_rn(__fsub_rn(dp[u * 8 + 2 * q], dh), dl)), scale)
                                        : 0.0f;
                            out.y = (c + 2 * q + 1 <= r)
                                        ? __fmul_rn(__fmul_rn(pv.y, __fsub_rn(__fsub_rn(dp[u * 8 + 2 * q + 1], dh), dl)), scale)
                                        : 0.0f;
                            IO::put(o, q, out);
                        }
                        IO::clear_outside(o, 0, r - c + 1);   // masked entries are +0.0 bits
                        store16(ds_row + c, o);
                    }
                }
            }
            tc::fence_before_sync();
            __syncthreads();   // TMEM and sB are rewritten by the next tile
        }
        if (pass == 0) {
            dh = __fadd_rn(dot_hi, dot_lo);
            dl = __fsub_rn(dot_lo, __fsub_rn(dh, dot_hi));
        }
    }

    if (failed) {
        if (tid == 0 && status)
            atomicOr(status, 1);
        tc::mbar_wait(&mbar, phase ^ 1u, kAttnWaitLimit);   // one more bounded wait for the MMA in flight
        tc::fence_before_sync();
        __syncthreads();
    }
    if (warp == 0)
        tc::tmem_free<kAttnRows>(tmem);
}

// Launch over B * M slices of ceil(S / 128) row blocks; dynamic shared memory
// holds the dO and V tiles (2 * 128 * D * 2 bytes).
template <typename T, int D>
cudaError_t launch_attn_dscores(const void* P, const void* dO, const void* V, void* dS, const int32_t* seq_lens,
                                int64_t B, int64_t M, int64_t S, float scale, int32_t* status, cudaStream_t st)
{
    constexpr int smem = 2 * kAttnRows * D * 2;
    auto* kern = gtms_attn_dscores_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    const int32_t nrb = static_cast<int32_t>((S + kAttnRows - 1) / kAttnRows);
    const int64_t grid = B * M * nrb;
    kern<<<static_cast<unsigned>(grid), kAttnRows, smem, st>>>(
        static_cast<const T*>(P), static_cast<const T*>(dO), static_cast<const T*>(V), static_cast<T*>(dS), seq_lens,
        static_cast<int32_t>(M), static_cast<int32_t>(S), nrb, scale, status);
    return cudaGetLastError();
}

}  // namespace gtms
