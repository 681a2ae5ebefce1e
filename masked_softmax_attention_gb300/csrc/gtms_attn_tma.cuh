// gtms_attn_tma.cuh -- the fused attention-backward step (dS from P, dO, V; see
// gtms_attn_bwd.cuh for the arithmetic) as a warp-specialised, TMA-fed,
// persistent kernel for operands in device memory.
//
// "ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1:
//   dP = dO V^T,  dS = scale * P * (dP - rowsum(dP * P))  over the kept set c <= r < L.
//
// Pass 1 forms the row sum. For the tiles left of the diagonal tile every entry
// is kept, and sum_c dP_rc P_rc = dO_r . sum_c P_rc V_c, so those tiles go to the
// tensor cores alone: O = P V accumulates in tensor memory (P the A operand
// straight from its TMA stage, V the B operand read MN-major), with no epilogue
// work per tile. Only the diagonal tile, whose masked entries must not be used
// (they may hold anything), goes through the per-element row sum of dP * P.
// The row sum is then D_r = (diagonal tile's sum) + dO_r . O_r. Pass 2
// recomputes dP tile by tile and writes dS.
//
// One CTA per SM walks the (slice, 128-row block) work items (see attn_item
// for their order). Its warps:
//   producer (1 lane)  TMA loads, per tile iteration, the P tile into a ring of
//                      NP stages (two 64-column boxes, 128-byte swizzle) and
//                      the V tile into a ring of NV stages; once per work item
//                      the dO rows (at head dim 64 two buffers, so the next
//                      item's can land early; one at 128); and at head dim 64
//                      an L2 prefetch of the next P tile. V and dO travel as
//                      8-column boxes without swizzle at head dim 64, and as
//                      64-column boxes with the 128-byte swizzle at 128 (see
//                      AttnTma). A tile left of the diagonal whose P stage
//                      last held a dP tile gets its V only once that stage is
//                      free, so that the MMA, which waits on the stage's P
//                      barrier for such tiles, never polls it a phase behind;
//   MMA (1 lane)       pass-1 tiles left of the diagonal: O += P . V into the
//                      O columns of tensor memory, committed to the barriers
//                      that free the P and V stages; the diagonal tile and the
//                      pass-2 tiles: dP = dO . V^T into one of two accumulators,
//                      committed to the barriers that hand it to the epilogue;
//   epilogue (16 warps) first zero each block's columns right of its diagonal
//                      tile (while the tensor cores run the tiles left of it);
//                      then warp w reads lanes 32 (w % 4) .. + 31 (its rows)
//                      and columns 32 (w / 4) .. + 31 of an accumulator: the
//                      diagonal tile's row sums and, after it, its quarter of
//                      O dotted with dO (pass 1), or dS written over P in the
//                      stage (pass 2);
//   store (1 lane)     TMA-stores each finished dS tile (rows past the tensor
//                      are dropped by the TMA unit) and returns the stage;
//   zero (2 warps)     zero-fill whole padded row blocks.
// Every hand-off is an mbarrier; every wait is bounded in time (kAttnWaitNs,
// gtms_kernels.cuh). If a wait runs out, the kernel ORs GTMS_ERR_TIMEOUT into
// the caller's status word, every role leaves its loop, the copies and MMAs
// already issued are waited for (bounded by kAttnDrainWaitNs) and the tensor
// memory is freed.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gtms_attn_bwd.cuh"
#include "gtms_tcgen05.cuh"

namespace gtms {

constexpr int kTmaEpiWarps = 16;                          // 4 lane quarters x 4 column quarters
constexpr int kWarpProducer = 16, kWarpMma = 17, kWarpStore = 18, kWarpZero0 = 19, kZeroWarps = 2;
constexpr int kTmaThreads = 32 * (kWarpZero0 + kZeroWarps);
// Tile iterations by which the L2 prefetch of P runs ahead of the TMA loads
// (measured on GB300 at head dim 64: 0-2 is best, 6 and more lose to L2
// thrashing). At head dim 128 the prefetch costs time (1.308 ms without it,
// 1.328 one tile ahead, 1.359 two ahead), so that kernel does not prefetch.
constexpr uint32_t kPrefetchAhead = 1;

// Test builds only: with GTMS_ATTN_TMA_NO_LOADS defined to 1 (a separate library
// that the test suite compiles; never libgtms) the producer issues no copies, so
// the consumers' waits run out and the kernel takes its give-up path.
#ifndef GTMS_ATTN_TMA_NO_LOADS
#define GTMS_ATTN_TMA_NO_LOADS 0
#endif
constexpr bool kAttnNoLoads = GTMS_ATTN_TMA_NO_LOADS != 0;

template <int D>
struct AttnTma {
    // Stages of the P / dS ring, of the V ring and dO buffers: 213 KB of shared
    // memory in all for head dim 64, 197 KB for 128. At 128 a V or dO tile is
    // 32 KB, and one dO buffer buys a third P stage (measured on GB300 at
    // [32,16,2048^2] fp16: 1.568 -> 1.539 ms).
    static constexpr int NP = D == 64 ? 4 : 3;
    static constexpr int NV = D == 64 ? 3 : 2;
    static constexpr int ND = D == 64 ? 2 : 1;
    // V and dO as 64-column boxes with the 128-byte swizzle (one TMA row of 128
    // bytes per tile row and box) instead of 8-column boxes of 16-byte rows.
    // With 128 columns the 8-column boxes make 2048 TMA rows per V tile and
    // limit the kernel: swizzled, 1.539 -> 1.333 ms. At 64 columns the
    // swizzled form measured 3 % slower, so head dim 64 keeps the 8-column boxes.
    static constexpr bool swizzled = D == 128;
    static constexpr bool prefetch = D == 64;                       // L2 prefetch of P (kPrefetchAhead)
    static constexpr uint32_t op = kAttnRows * D * 2;               // 128 rows of dO or V
    static constexpr uint32_t off_p = 0;                            // NP P / dS tiles (1024-aligned)
    static constexpr uint32_t off_v = NP * kAttnPTileBytes;         // NV V tiles
    static constexpr uint32_t off_do = off_v + NV * op;             // ND dO tiles
    static constexpr uint32_t off_red = off_do + ND * op;           // 8 x 128 floats: row-sum exchange
    static constexpr uint32_t bytes = off_red + 8 * kAttnRows * 4 + 1024;   // + slack to align the base
    static constexpr uint32_t lbo = kAttnRows * 16;                 // K-adjacent core matrices (one 8-column box)
    static constexpr uint32_t sbo = 128;                            // row-adjacent core matrices
    static constexpr uint32_t box = kAttnRows * 128;                // one swizzled 64-column box (16 KB)

    // TMA load of 128 rows of dO or V (row0 .. row0 + 127 of slice z) into dst.
    __device__ static __forceinline__ void load_rows(uint32_t dst, const CUtensorMap* map, int32_t row0, int32_t z,
                                                     uint64_t* bar)
    {
        if constexpr (swizzled) {
            for (int kc = 0; kc < D / 64; ++kc)
                tc::tma_load_3d(dst + kc * box, map, kc * 64, row0, z, bar);
        } else {
            for (int kc = 0; kc < D / 8; ++kc)
                tc::tma_load_3d(dst + kc * lbo, map, kc * 8, row0, z, bar);
        }
    }
};

constexpr int kAttnTmemCols = 512;          // two 128-column dP accumulators, then O (64 or 128 columns)
constexpr uint32_t kAttnOCol = 2 * kAttnRows;

struct AttnShared {
    uint64_t pfull[4], dsready[4];              // per P stage: loaded; dS written into it
    uint64_t pepi[4], pmma[4];                  // per P stage: freed by the epilogue / store lane, or by the MMA
    uint64_t vfull[3], vempty[3];               // per V stage
    uint64_t tfull[2], tempty[2];               // per dP accumulator
    uint64_t ofull, oempty;                     // the O accumulator (once per work item)
    uint64_t dofull[2], doempty[2];             // per dO buffer
    uint64_t red_in, red_out;                   // row-sum exchange between the column quarters
    uint64_t mma_done;                          // every MMA issued has completed (before TMEM is freed)
    uint32_t tmem_slot;
    int abort_flag;
};

__device__ __forceinline__ bool attn_aborted(const AttnShared& sh)
{
    return *reinterpret_cast<const volatile int*>(&sh.abort_flag) != 0;
}

__device__ __forceinline__ void attn_abort(AttnShared& sh, int32_t* status)
{
    *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
    if (status)
        atomicOr(status, GTMS_ERR_TIMEOUT);
}

// All 32 lanes wait; the verdict is the warp's (so that warp-collective
// instructions that follow stay converged).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, limit_ns)) != 0;
}

struct AttnItem {
    int64_t slice;
    int32_t r0, L, n_tiles;
};

// Work item `item`: the slices are taken in groups of `group` (the last group
// may be smaller); inside a group, row-block-major with the costliest row
// blocks first: row block nrb - 1 - j / k of slice group_start + j % k, for
// item = group_start * nrb + j and k the group's size. A CTA takes items
// blockIdx.x + n * gridDim.x, so every CTA meets every row block about equally
// often (the CTAs finish together), and at any time the CTAs work on the rows
// of one group of slices only (few pages of P and dS in use at once).
__device__ __forceinline__ AttnItem attn_item(int64_t item, int64_t n_slices, int64_t group, int32_t nrb, int32_t M,
                                              int32_t S, const int32_t* __restrict__ seq_lens)
{
    AttnItem it;
    const int64_t gi = item / (group * nrb), j = item % (group * nrb);
    const int64_t k = n_slices - gi * group < group ? n_slices - gi * group : group;
    it.slice = gi * group + j % k;
    it.r0 = (nrb - 1 - static_cast<int32_t>(j / k)) * kAttnRows;
    int32_t L = __ldg(seq_lens + static_cast<int32_t>(it.slice / M));
    it.L = L < 0 ? 0 : (L > S ? S : L);
    it.n_tiles = it.r0 < it.L ? it.r0 / kAttnRows + 1 : 0;   // 0: padded block, no GEMM
    return it;
}

template <typename T, int D>
__global__ void __launch_bounds__(kTmaThreads, 1)
gtms_attn_dscores_tma_kernel(const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_ds,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                             T* dS, const int32_t* __restrict__ seq_lens, int32_t M, int32_t S, int32_t nrb,
                             int64_t n_slices, int64_t group, float scale, int32_t* status, uint64_t wait_ns)
{
    using IO = Pairs<T>;
    using TL = AttnTma<D>;
    constexpr int NP = TL::NP, NV = TL::NV;
    static_assert(NP <= 4 && NV <= 3 && TL::ND <= 2 && TL::ND >= 1,
                  "AttnShared holds barriers for at most 4 P stages, 3 V stages and 2 dO buffers");
    static_assert(TL::bytes <= 227 * 1024 - sizeof(AttnShared), "shared memory of one CTA");
    constexpr int DQ = D / 4;   // O columns per epilogue column quarter
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ AttnShared sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_items = n_slices * nrb;
    const uint32_t raw_u32 = tc::smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;              // 1024-aligned for the 128-byte swizzle
    uint8_t* smem = smem_raw + (base - raw_u32);

    if (tid == 0) {
        for (int s = 0; s < NP; ++s) {
            tc::mbar_init(&sh.pfull[s], 1);
            tc::mbar_init(&sh.dsready[s], kTmaEpiWarps);
            tc::mbar_init(&sh.pepi[s], kTmaEpiWarps);   // 16 epilogue warps, or the store lane x 16
            tc::mbar_init(&sh.pmma[s], 1);              // the MMA's commit
        }
        for (int s = 0; s < NV; ++s) {
            tc::mbar_init(&sh.vfull[s], 1);
            tc::mbar_init(&sh.vempty[s], 1);   // the MMA's commit
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&sh.tfull[a], 1);
            tc::mbar_init(&sh.tempty[a], kTmaEpiWarps);
            tc::mbar_init(&sh.dofull[a], 1);
            tc::mbar_init(&sh.doempty[a], 1);
        }
        tc::mbar_init(&sh.ofull, 1);
        tc::mbar_init(&sh.oempty, kTmaEpiWarps);
        tc::mbar_init(&sh.red_in, 3 * kAttnRows);   // the threads of column quarters 1..3
        tc::mbar_init(&sh.red_out, kAttnRows);      // the threads of column quarter 0
        tc::mbar_init(&sh.mma_done, 1);
        sh.abort_flag = 0;
    }
    if (warp == kWarpMma) {
        __syncwarp();
        tc::tmem_alloc<kAttnTmemCols>(&sh.tmem_slot);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh.tmem_slot;

    if (warp == kWarpProducer) {
        if (lane == 0) {
            uint32_t g = 0, itm = 0, gv = 0, gp = 0, gd = 0;   // iterations, work items; V, P, dO loads issued
            // Which barrier frees each P stage's latest tile (bit s set: the MMA's pmma[s], else pepi[s]),
            // and the parity of the next phase to wait for on each.
            uint32_t by_mma = 0, par_epi = 0, par_mma = 0;
            bool ok = true;
            // A second cursor walks the same iterations kPrefetchAhead ahead of the
            // loads and prefetches the P tiles of pass 1 into L2, so that the TMA
            // loads into the ring find them there (head dim 64 only: TL::prefetch).
            const uint64_t pol_keep = tc::policy_evict_last();
            int64_t pf_item = blockIdx.x;
            AttnItem pf{};
            int32_t pf_i = 0;
            uint32_t pf_g = 0;
            auto pf_seek = [&]() {   // the cursor's next work item that has tiles
                for (; pf_item < n_items; pf_item += gridDim.x) {
                    pf = attn_item(pf_item, n_slices, group, nrb, M, S, seq_lens);
                    if (pf.n_tiles > 0)
                        return true;
                }
                return false;
            };
            bool pf_live = TL::prefetch && pf_seek();
            for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const AttnItem it = attn_item(item, n_slices, group, nrb, M, S, seq_lens);
                if (it.n_tiles == 0)
                    continue;
                const int32_t z = static_cast<int32_t>(it.slice);
                const uint32_t p = itm % TL::ND;
                ok = tc::mbar_wait(&sh.doempty[p], ((itm / TL::ND) & 1u) ^ 1u, wait_ns) && !attn_aborted(sh);
                if (!ok)
                    break;
                if constexpr (!kAttnNoLoads) {
                    tc::mbar_arrive_expect_tx(&sh.dofull[p], TL::op);
                    TL::load_rows(base + TL::off_do + p * TL::op, &tm_do, it.r0, z, &sh.dofull[p]);
                    gd = itm + 1;
                }
                for (int32_t i = 0; i < 2 * it.n_tiles; ++i, ++g) {
                    const uint32_t sv = g % NV, phv = (g / NV) & 1u, sp = g % NP, bit = 1u << sp;
                    const int32_t tc0 = (i < it.n_tiles ? i : i - it.n_tiles) * kAttnRows;
                    while (pf_live && pf_g <= g + kPrefetchAhead) {
                        if (pf_i < pf.n_tiles) {
                            const int32_t zf = static_cast<int32_t>(pf.slice);
                            tc::tma_prefetch_3d(&tm_p, pf_i * kAttnRows, pf.r0, zf, pol_keep);
                            if (pf_i * kAttnRows + 64 < S)
                                tc::tma_prefetch_3d(&tm_p, pf_i * kAttnRows + 64, pf.r0, zf, pol_keep);
                        }
                        ++pf_g;
                        if (++pf_i == 2 * pf.n_tiles) {
                            pf_i = 0;
                            pf_item += gridDim.x;
                            pf_live = pf_seek();
                        }
                    }
                    // A tile left of the diagonal whose P stage last held a dP tile waits for
                    // that stage before its V is issued: the MMA then waits on the stage's
                    // P barrier, and must not find it a phase behind. Every other tile
                    // issues its V first.
                    const bool v_first = !(i < it.n_tiles - 1 && g >= static_cast<uint32_t>(NP) && !(by_mma & bit));
                    if (v_first) {
                        ok = tc::mbar_wait(&sh.vempty[sv], phv ^ 1u, wait_ns) && !attn_aborted(sh);
                        if (!ok)
                            break;
                        if constexpr (!kAttnNoLoads) {
                            tc::mbar_arrive_expect_tx(&sh.vfull[sv], TL::op);
                            TL::load_rows(base + TL::off_v + sv * TL::op, &tm_v, tc0, z, &sh.vfull[sv]);
                            ++gv;
                        }
                    }
                    // The P stage: wait until its previous tile (g - NP) has been freed.
                    if (g >= static_cast<uint32_t>(NP)) {
                        if (by_mma & bit) {
                            ok = tc::mbar_wait(&sh.pmma[sp], (par_mma >> sp) & 1u, wait_ns);
                            par_mma ^= bit;
                        } else {
                            ok = tc::mbar_wait(&sh.pepi[sp], (par_epi >> sp) & 1u, wait_ns);
                            par_epi ^= bit;
                        }
                        if (!(ok = ok && !attn_aborted(sh)))
                            break;
                    }
                    by_mma = i < it.n_tiles - 1 ? by_mma | bit : by_mma & ~bit;   // tiles left of the diagonal
                    if (!v_first) {
                        ok = tc::mbar_wait(&sh.vempty[sv], phv ^ 1u, wait_ns) && !attn_aborted(sh);
                        if (!ok)
                            break;
                        if constexpr (!kAttnNoLoads) {
                            tc::mbar_arrive_expect_tx(&sh.vfull[sv], TL::op);
                            TL::load_rows(base + TL::off_v + sv * TL::op, &tm_v, tc0, z, &sh.vfull[sv]);
                            ++gv;
                        }
                    }
                    if constexpr (!kAttnNoLoads) {
                        tc::mbar_arrive_expect_tx(&sh.pfull[sp], kAttnPTileBytes);
                        ++gp;
                        const uint32_t pt = base + TL::off_p + sp * kAttnPTileBytes;
                        // Pass 1 keeps the P tile in L2 for pass 2, which is its last read.
                        const uint64_t pol = i < it.n_tiles ? tc::policy_evict_last() : tc::policy_evict_first();
                        tc::tma_load_3d(pt, &tm_p, tc0, it.r0, z, &sh.pfull[sp], pol);
                        tc::tma_load_3d(pt + kAttnRows * 128, &tm_p, tc0 + 64, it.r0, z, &sh.pfull[sp], pol);
                    }
                }
                ++itm;
            }
            if (!ok) {
                attn_abort(sh, status);
                // Let the copies already issued land before the CTA can exit.
                for (uint32_t k = 0; k < static_cast<uint32_t>(NV) && k < gv; ++k) {
                    const uint32_t gk = gv - 1 - k;
                    tc::mbar_wait(&sh.vfull[gk % NV], (gk / NV) & 1u, kAttnDrainWaitNs);
                }
                for (uint32_t k = 0; k < static_cast<uint32_t>(NP) && k < gp; ++k) {
                    const uint32_t gk = gp - 1 - k;
                    tc::mbar_wait(&sh.pfull[gk % NP], (gk / NP) & 1u, kAttnDrainWaitNs);
                }
                if (gd > 0)
                    tc::mbar_wait(&sh.dofull[(gd - 1) % TL::ND], ((gd - 1) / TL::ND) & 1u, kAttnDrainWaitNs);
            }
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            constexpr uint32_t idesc_dp = tc::idesc_f16<T>(kAttnRows, kAttnRows);
            constexpr uint32_t idesc_o = tc::idesc_f16<T>(kAttnRows, D) | tc::kIdescBMnMajor;
            uint32_t g = 0, ga = 0, itm = 0;   // tile iterations, dP accumulations, work items
            bool ok = true, issued = false;
            for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const AttnItem it = attn_item(item, n_slices, group, nrb, M, S, seq_lens);
                if (it.n_tiles == 0)
                    continue;
                const uint32_t p = itm % TL::ND;
                ok = tc::mbar_wait(&sh.dofull[p], (itm / TL::ND) & 1u, wait_ns) &&
                     (itm == 0 || tc::mbar_wait(&sh.oempty, (itm - 1) & 1u, wait_ns)) && !attn_aborted(sh);
                if (!ok)
                    break;
                const uint32_t a_base = base + TL::off_do + p * TL::op;
                for (int32_t i = 0; i < 2 * it.n_tiles; ++i, ++g) {
                    const uint32_t sv = g % NV, phv = (g / NV) & 1u, sp = g % NP, php = (g / NP) & 1u;
                    const uint32_t v_base = base + TL::off_v + sv * TL::op;
                    if (i < it.n_tiles - 1) {
                        // O += P . V: K = the tile's 128 columns, 8 steps of 16 (32 bytes of a
                        // swizzled P row; 16 V rows, two core-matrix groups of 128 bytes).
                        ok = tc::mbar_wait(&sh.vfull[sv], phv, wait_ns) && tc::mbar_wait(&sh.pfull[sp], php, wait_ns) &&
                             !attn_aborted(sh);
                        if (!ok)
                            break;
                        tc::fence_after_sync();
                        const uint32_t p_base = base + TL::off_p + sp * kAttnPTileBytes;
#pragma unroll
                        for (int ks = 0; ks < kAttnRows / 16; ++ks) {
                            // V is the MN-major B operand: 16 V rows per K step, 256 bytes of 8-column boxes,
                            // or 2048 bytes (two 8-row swizzle atoms) of the swizzled boxes.
                            const uint64_t b_desc = TL::swizzled ? tc::smem_desc_sw128_mn(v_base + ks * 2048, TL::box)
                                                                 : tc::smem_desc(v_base + ks * 256, 128, TL::lbo);
                            tc::mma_f16(tmem + kAttnOCol,
                                        tc::smem_desc_sw128(p_base + (ks >> 2) * (kAttnRows * 128) + (ks & 3) * 32, 1024),
                                        b_desc, idesc_o, (i > 0 || ks > 0) ? 1u : 0u);
                        }
                        tc::commit(&sh.pmma[sp]);
                        tc::commit(&sh.vempty[sv]);
                    } else {
                        // dP = dO . V^T into accumulator ga % 2.
                        const uint32_t acc = ga & 1u, pha = (ga >> 1) & 1u;
                        ok = tc::mbar_wait(&sh.tempty[acc], pha ^ 1u, wait_ns) &&
                             tc::mbar_wait(&sh.vfull[sv], phv, wait_ns) && !attn_aborted(sh);
                        if (!ok)
                            break;
                        tc::fence_after_sync();
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            // dO (A) and V (B) both K-major: a K step is 32 bytes of a swizzled 128-byte row
                            // (the next box after four steps), or two 8-column boxes.
                            const uint32_t koff = (ks >> 2) * TL::box + (ks & 3) * 32;
                            const uint64_t a_desc = TL::swizzled ? tc::smem_desc_sw128(a_base + koff, 1024)
                                                                 : tc::smem_desc(a_base + ks * 2 * TL::lbo, TL::lbo, TL::sbo);
                            const uint64_t b_desc = TL::swizzled ? tc::smem_desc_sw128(v_base + koff, 1024)
                                                                 : tc::smem_desc(v_base + ks * 2 * TL::lbo, TL::lbo, TL::sbo);
                            tc::mma_f16(tmem + acc * kAttnRows, a_desc, b_desc, idesc_dp, ks > 0 ? 1u : 0u);
                        }
                        tc::commit(&sh.tfull[acc]);
                        tc::commit(&sh.vempty[sv]);
                        if (i == it.n_tiles - 1)
                            tc::commit(&sh.ofull);   // every O product of the item precedes this commit
                        ++ga;
                    }
                    issued = true;
                }
                if (!ok)
                    break;
                tc::commit(&sh.doempty[p]);
                ++itm;
            }
            if (!ok)
                attn_abort(sh, status);
            if (issued) {   // every MMA must complete before the tensor memory is freed
                tc::commit(&sh.mma_done);
                tc::mbar_wait(&sh.mma_done, 0, kAttnDrainWaitNs);
            }
        }
    } else if (warp == kWarpStore) {
        if (lane == 0) {
            uint32_t g = 0, ds_par = 0;
            bool ok = true;
            for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const AttnItem it = attn_item(item, n_slices, group, nrb, M, S, seq_lens);
                const int32_t z = static_cast<int32_t>(it.slice);
                for (int32_t i = 0; i < 2 * it.n_tiles; ++i, ++g) {
                    if (i < it.n_tiles)
                        continue;
                    const uint32_t s = g % NP;
                    ok = tc::mbar_wait(&sh.dsready[s], (ds_par >> s) & 1u, wait_ns) && !attn_aborted(sh);
                    if (!ok)
                        break;
                    ds_par ^= 1u << s;
                    const int32_t tc0 = (i - it.n_tiles) * kAttnRows;
                    const uint32_t pt = base + TL::off_p + s * kAttnPTileBytes;
                    const uint64_t pol = tc::policy_evict_first();   // dS is not read again here
                    tc::tma_store_3d(&tm_ds, tc0, it.r0, z, pt, pol);
                    if (tc0 + 64 < S)   // (a box wholly past the last column is not issued)
                        tc::tma_store_3d(&tm_ds, tc0 + 64, it.r0, z, pt + kAttnRows * 128, pol);
                    tc::bulk_commit();
                    tc::bulk_wait_read_all();
                    tc::mbar_arrive(&sh.pepi[s], kTmaEpiWarps);
                }
            }
            if (!ok)
                attn_abort(sh, status);
            tc::bulk_wait_all();
        }
    } else if (warp >= kWarpZero0) {
        // Zero-fill warps: whole padded row blocks (the epilogue warps zero the
        // columns right of the diagonal tile of the blocks that have tiles).
        const int zt = tid - kWarpZero0 * 32;
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
            if (attn_aborted(sh))
                break;
            const AttnItem it = attn_item(item, n_slices, group, nrb, M, S, seq_lens);
            if (it.n_tiles > 0)
                continue;
            const int32_t r_end = it.r0 + kAttnRows < S ? it.r0 + kAttnRows : S;
            zero_region(dS + it.slice * static_cast<int64_t>(S) * S, S, it.r0, r_end, 0, zt, kZeroWarps * 32);
        }
    } else {
        // Epilogue warps 0..15: rows 32 (w % 4) + lane, columns 32 (w / 4) .. + 31 of each dP tile
        // (and O columns DQ (w / 4) .. + DQ - 1).
        const int quarter = warp & 3, colq = warp >> 2;
        const int row = quarter * 32 + lane;
        float* red = reinterpret_cast<float*>(smem + TL::off_red);
        const uint32_t row_off = TL::off_p + (colq >> 1) * (kAttnRows * 128) + row * 128;
        const int chunk0 = (colq & 1) * 4, rx = row & 7;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t g = 0, ga = 0, itm = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const AttnItem it = attn_item(item, n_slices, group, nrb, M, S, seq_lens);
            if (it.n_tiles == 0)
                continue;
            // The block's columns right of its diagonal tile, zeroed by all 512 epilogue
            // threads while the tensor cores run the tiles left of the diagonal.
            {
                const int32_t r_end = it.r0 + kAttnRows < S ? it.r0 + kAttnRows : S;
                const int32_t c_from = it.n_tiles * kAttnRows < S ? it.n_tiles * kAttnRows : S;
                zero_region(dS + it.slice * static_cast<int64_t>(S) * S, S, it.r0, r_end, c_from, tid,
                            kTmaEpiWarps * 32);
            }
            const int32_t r = it.r0 + row;
            const bool live = r < it.L;
            float dot_hi = 0.0f, dot_lo = 0.0f, dh = 0.0f, dl = 0.0f;
            for (int32_t i = 0; i < 2 * it.n_tiles; ++i, ++g) {
                if (i < it.n_tiles - 1)
                    continue;   // O tiles: tensor cores only
                const bool pass2 = i >= it.n_tiles;
                const int32_t tc0 = (pass2 ? i - it.n_tiles : i) * kAttnRows;
                // Kept elements of this thread's 32 columns: the first `kept` of them.
                const int32_t lim = live ? r - (tc0 + colq * 32) + 1 : 0;
                const int kept = lim < 0 ? 0 : (lim > 32 ? 32 : lim);
                const uint32_t s = g % NP, ph = (g / NP) & 1u, acc = ga & 1u, pha = (ga >> 1) & 1u;
                ++ga;
                ok = warp_wait(&sh.tfull[acc], pha, wait_ns) && !attn_aborted(sh);
                if (!ok)
                    break;
                tc::fence_after_sync();
                float dp[32];
                tc::tmem_ld32(tmem + lane_base + acc * kAttnRows + colq * 32, dp);
                if (pass2) {
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        tc::mbar_arrive(&sh.tempty[acc]);
                }
                ok = warp_wait(&sh.pfull[s], ph, wait_ns);   // the P tile
                if (!ok)
                    break;
                uint8_t* p_row = smem + row_off + s * kAttnPTileBytes;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4* cell = reinterpret_cast<uint4*>(p_row + (((chunk0 + u) ^ rx) << 4));
                    const int n_in = kept - u * 8;   // kept elements in this unit, if < 8
                    if (n_in <= 0) {                  // nothing kept in this unit
                        if (pass2)
                            *cell = make_uint4(0u, 0u, 0u, 0u);
                        continue;
                    }
                    const uint4 raw = *cell;          // (kept columns lie inside the tensor)
                    Unit16 pu{{raw.x, raw.y, raw.z, raw.w}};
                    if (n_in < 8) {   // masked P and dP read as +0.0 (dP may be infinite where P is masked)
                        IO::clear_outside(pu, 0, n_in);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dp[u * 8 + e] = e < n_in ? dp[u * 8 + e] : 0.0f;
                    }
                    if (!pass2) {
                        float2 a2 = __fmul2_rn(IO::get(pu, 0), make_float2(dp[u * 8], dp[u * 8 + 1]));
#pragma unroll
                        for (int q = 1; q < 4; ++q)
                            a2 = __ffma2_rn(IO::get(pu, q), make_float2(dp[u * 8 + 2 * q], dp[u * 8 + 2 * q + 1]), a2);
                        float sum, err;
                        two_sum(dot_hi, __fadd_rn(a2.x, a2.y), sum, err);
                        dot_hi = sum;
                        dot_lo = __fadd_rn(dot_lo, err);
                    } else {
                        const float2 ndh = make_float2(-dh, -dh), ndl = make_float2(-dl, -dl);
                        const float2 sc = make_float2(scale, scale);
                        Unit16 o;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 gq = make_float2(dp[u * 8 + 2 * q], dp[u * 8 + 2 * q + 1]);
                            const float2 t = __fadd2_rn(__fadd2_rn(gq, ndh), ndl);
                            IO::put(o, q, __fmul2_rn(__fmul2_rn(IO::get(pu, q), t), sc));
                        }
                        if (n_in < 8)
                            IO::clear_outside(o, 0, n_in);   // masked entries are +0.0 bits
                        *cell = make_uint4(o.w[0], o.w[1], o.w[2], o.w[3]);
                    }
                }
                if (!pass2) {
                    // The diagonal tile (the last of pass 1): its P stage is free again.
                    __syncwarp();
                    if (lane == 0)
                        tc::mbar_arrive(&sh.pepi[s]);
                    // The tiles left of it: dO_r . O_r over this warp's DQ columns of O.
                    ok = warp_wait(&sh.ofull, itm & 1u, wait_ns) && !attn_aborted(sh);
                    if (!ok)
                        break;
                    tc::fence_after_sync();
                    if (it.n_tiles > 1) {
                        float o[DQ];
                        if constexpr (DQ == 16)
                            tc::tmem_ld16(tmem + lane_base + kAttnOCol + colq * DQ, o);
                        else
                            tc::tmem_ld32(tmem + lane_base + kAttnOCol + colq * DQ, o);
                        if (live) {
                            const uint8_t* do_tile = smem + TL::off_do + (itm % TL::ND) * TL::op;
                            float acc_o = 0.0f;
#pragma unroll
                            for (int j = 0; j < DQ / 8; ++j) {
                                const int k = colq * (DQ / 8) + j;   // 16-byte chunk of the dO row
                                const uint32_t off = TL::swizzled ? (k >> 3) * TL::box + row * 128 + (((k & 7) ^ rx) << 4)
                                                                  : k * TL::lbo + row * 16;
                                const uint4 raw = *reinterpret_cast<const uint4*>(do_tile + off);
                                const Unit16 du{{raw.x, raw.y, raw.z, raw.w}};
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const float2 d2 = IO::get(du, q);
                                    acc_o = __fmaf_rn(d2.x, o[j * 8 + 2 * q], acc_o);
                                    acc_o = __fmaf_rn(d2.y, o[j * 8 + 2 * q + 1], acc_o);
                                }
                            }
                            float sum, err;
                            two_sum(dot_hi, acc_o, sum, err);
                            dot_hi = sum;
                            dot_lo = __fadd_rn(dot_lo, err);
                        }
                    }
                    // O and dO read: the MMA may overwrite O, and reach the end of the item
                    // (which frees the dO buffer) only after this accumulator is returned.
                    // That order rests on two accumulators: in an item of n >= 2 tiles the
                    // second pass-2 dP product reuses this one, so the item's dO buffer is
                    // committed free only after this read (n == 1 reads no dO). With a third
                    // accumulator the next item's dO could land over this one first.
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(&sh.oempty);
                        tc::mbar_arrive(&sh.tempty[acc]);
                    }
                    // Merge the four column quarters' row sums.
                    const uint32_t rp = itm & 1u;
                    if (colq != 0) {
                        red[(colq - 1) * 2 * kAttnRows + row] = dot_hi;
                        red[(colq - 1) * 2 * kAttnRows + kAttnRows + row] = dot_lo;
                        tc::mbar_arrive(&sh.red_in);
                        ok = warp_wait(&sh.red_out, rp, wait_ns);
                        dh = red[6 * kAttnRows + row];
                        dl = red[7 * kAttnRows + row];
                    } else {
                        ok = warp_wait(&sh.red_in, rp, wait_ns);
                        float hi = dot_hi, lo = dot_lo;
#pragma unroll
                        for (int k = 0; k < 3; ++k) {
                            float sum, err;
                            two_sum(hi, red[k * 2 * kAttnRows + row], sum, err);
                            hi = sum;
                            lo = __fadd_rn(__fadd_rn(lo, red[k * 2 * kAttnRows + kAttnRows + row]), err);
                        }
                        dh = __fadd_rn(hi, lo);
                        dl = __fsub_rn(lo, __fsub_rn(dh, hi));
                        red[6 * kAttnRows + row] = dh;
                        red[7 * kAttnRows + row] = dl;
                        tc::mbar_arrive(&sh.red_out);
                    }
                    if (!ok)
                        break;
                } else {
                    tc::fence_smem_for_async();   // dS in the stage, visible to the TMA store
                    __syncwarp();
                    if (lane == 0)
                        tc::mbar_arrive(&sh.dsready[s]);
                }
            }
            ++itm;
        }
        if (!ok && lane == 0)
            attn_abort(sh, status);
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kWarpMma) {
        __syncwarp();
        tc::tmem_free<kAttnTmemCols>(tmem);
    }
}

// The driver's tensor-map encoder, looked up once through the runtime.
using TensorMapEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                       const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline TensorMapEncodeFn tensor_map_encoder()
{
    static TensorMapEncodeFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<TensorMapEncodeFn>(f);
    }();
    return fn;
}

// 3-D map of 16-bit elements [n2][n1][n0] (n0 contiguous) with box {b0, b1, 1}.
inline bool encode_map_3d(CUtensorMap* map, const void* ptr, uint64_t n0, uint64_t n1, uint64_t n2, uint32_t b0,
                          uint32_t b1, CUtensorMapSwizzle swz)
{
    const TensorMapEncodeFn enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {n0, n1, n2};
    const cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

// Persistent launch: one CTA per SM (at most one per work item).
template <typename T, int D>
cudaError_t launch_attn_dscores_tma(const void* P, const void* dO, const void* V, void* dS, const int32_t* seq_lens,
                                    int64_t B, int64_t M, int64_t S, float scale, int32_t* status, cudaStream_t st,
                                    uint64_t wait_ns = kAttnWaitNs)
{
    const uint64_t slices = static_cast<uint64_t>(B) * M;
    CUtensorMap tm_p, tm_ds, tm_v, tm_do;
    if (!encode_map_3d(&tm_p, P, S, S, slices, 64, kAttnRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_3d(&tm_ds, dS, S, S, slices, 64, kAttnRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_3d(&tm_v, V, D, S, slices, AttnTma<D>::swizzled ? 64 : 8, kAttnRows,
                       AttnTma<D>::swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map_3d(&tm_do, dO, D, S, slices, AttnTma<D>::swizzled ? 64 : 8, kAttnRows,
                       AttnTma<D>::swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    constexpr int smem = static_cast<int>(AttnTma<D>::bytes);
    auto* kern = gtms_attn_dscores_tma_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    const int32_t nrb = static_cast<int32_t>((S + kAttnRows - 1) / kAttnRows);
    const int64_t n_items = static_cast<int64_t>(slices) * nrb;
    const int nsm = sm_count();
    if (nsm <= 0)
        return cudaErrorUnknown;
    const int64_t grid = n_items < nsm ? n_items : nsm;
    const int64_t group = (4 * grid + nrb - 1) / nrb;   // slices whose items make about 4 per CTA
    return launch_kernel(kern, static_cast<unsigned>(grid), kTmaThreads, smem, st, tm_p, tm_ds, tm_v, tm_do,
                         static_cast<T*>(dS), seq_lens, static_cast<int32_t>(M), static_cast<int32_t>(S), nrb,
                         static_cast<int64_t>(slices), group, scale, status, wait_ns);
}

}  // namespace gtms
