// gtms_staged.cuh -- the forward with each row's kept units staged in shared
// memory by a TMA bulk copy, one CTA team per row.
//
// The per-row kernels of gtms_kernels.cuh load a row's kept units into
// registers; how many rows are in flight per SM then follows from the registers
// a team holds. Here the loads leave the registers: a persistent CTA team takes
// the M heads of one (batch, row) pair after another (the heads share the kept
// range), and one thread issues, for each live row, a single untiled bulk copy
// ("cp.async.bulk", global -> shared) of the row's kept units into a ring of NS
// row slots. The copies run NS rows ahead of the rows being reduced, and each
// completes on its slot's mbarrier. This is the block-per-row layout of
// "优化ScaledMaskSoftmax算子" (sections 2.2 and 4.2: a block per row, the row
// staged in shared memory) with the copy engine, instead of the threads, moving
// the row.
//
// A team's row: zero stores of the masked units first (they depend on nothing),
// then the wait for the row's slot, the kept units from the slot into registers
// and the arithmetic of gtms_fwd_vec_kernel (same steps in the same order, so
// the same bits). Right after the first CTA-wide reduction every thread has read
// the slot, and the issuing thread refills it with the row NS places further on.
//
// Every wait on a slot is bounded (wait_ns of the GPU's global timer). A thread
// whose wait runs out reads that row from global memory instead, which gives
// the same values; if the issuing thread's own wait ran out, the team stops
// staging and reads every later row from global memory, and before the CTA exits
// the issuing thread waits (bounded by kAttnDrainWaitNs) for the copies still
// outstanding. A slow copy therefore costs time, never a wrong result or a hang.
#pragma once

#include "gtms_kernels.cuh"
#include "gtms_tcgen05.cuh"

namespace gtms {

// Test builds only: with GTMS_STAGED_NO_COPIES defined to 1 (a separate library
// that the test suite compiles; never libgtms) no copy is issued, so every wait
// runs out and the kernel takes its give-up path.
#ifndef GTMS_STAGED_NO_COPIES
#define GTMS_STAGED_NO_COPIES 0
#endif
constexpr bool kStagedNoCopies = GTMS_STAGED_NO_COPIES != 0;

// The issuing thread's cursor over its CTA's live rows, in the order the team
// takes them: copy k goes to slot k % NS and completes phase (k / NS) & 1. It
// lives in shared memory, so that the other threads hold no registers for it,
// and it advances without divisions: the CTA's pairs are blockIdx.x + i *
// gridDim.x, so (b, r) moves by gridDim.x rows a step.
struct StagedCursor {
    int32_t b, r;      // (batch, row) pair of the next copy (b == B: none left)
    int32_t m;         // its head
    int32_t u0, u1;    // its kept units
    int32_t L;         // clamped length of batch b
    uint32_t issued;   // copies issued
    uint32_t waited;   // copies the issuing thread has seen complete
};

template <int MK>
__device__ __forceinline__ void staged_set_range(StagedCursor& cur, const int32_t* __restrict__ seq_lens,
                                                 const Geom& g, int epu)
{
    int32_t c0 = 0, c1 = 0;
    if (cur.r < cur.L) {
        if constexpr (MK == kMaskLength) {
            c1 = cur.L;
        } else {
            c1 = cur.r + 1;
            if constexpr (MK == kMaskWindow)
                c0 = cur.r - g.window + 1 > 0 ? cur.r - g.window + 1 : 0;
        }
    }
    cur.u0 = c0 / epu;
    cur.u1 = c1 > c0 ? (c1 + epu - 1) / epu : cur.u0;
}

template <int MK>
__device__ __forceinline__ void staged_step_pair(StagedCursor& cur, const int32_t* __restrict__ seq_lens,
                                                 const Geom& g, int32_t B, int epu)
{
    cur.r += gridDim.x;
    bool new_batch = false;
    while (cur.r >= g.S && cur.b < B) {
        cur.r -= g.S;
        ++cur.b;
        new_batch = true;
    }
    if (cur.b >= B)
        return;
    if (new_batch) {
        const int32_t L = __ldg(seq_lens + cur.b);
        cur.L = L < 0 ? 0 : (L > g.S ? g.S : L);
    }
    staged_set_range<MK>(cur, seq_lens, g, epu);
}

// Issue the copy of the next live row into its slot (none once the CTA's rows
// run out).
template <typename T, int MK, int NS>
__device__ __forceinline__ void staged_issue_next(StagedCursor& cur, const T* x, const int32_t* __restrict__ seq_lens,
                                                  const Geom& g, int32_t M, int32_t B, uint32_t stage_u32,
                                                  uint32_t slot_bytes, uint64_t* full)
{
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    while (cur.b < B && cur.u1 <= cur.u0)   // padded pairs need no copy
        staged_step_pair<MK>(cur, seq_lens, g, B, EPU);
    if (cur.b >= B)
        return;
    const int64_t q = (static_cast<int64_t>(cur.b) * M + cur.m) * g.S + cur.r;
    const uint32_t s = cur.issued % NS, bytes = 16u * static_cast<uint32_t>(cur.u1 - cur.u0);
    if constexpr (!kStagedNoCopies) {
        tc::mbar_arrive_expect_tx(&full[s], bytes);
        tc::bulk_load_1d(stage_u32 + s * slot_bytes + 16u * cur.u0,
                         reinterpret_cast<const char*>(x + q * g.S) + 16 * cur.u0, bytes, &full[s],
                         tc::policy_evict_first());   // x is read once
        ++cur.issued;
    }
    if (++cur.m == M) {
        cur.m = 0;
        staged_step_pair<MK>(cur, seq_lens, g, B, EPU);
    }
}

template <typename T, int MK, int TW, int NV, int NS, int MINB>
__global__ void __launch_bounds__(TW, MINB)
gtms_fwd_staged_kernel(const T* x, T* y, const int32_t* __restrict__ seq_lens, Geom g, float scale, uint64_t wait_ns)
{
    static_assert(TW > 32 && TW % 32 == 0, "a CTA team");
    constexpr int EPU = 2 * Pairs<T>::kPairs;
    extern __shared__ __align__(128) uint8_t stage[];   // NS slots of g.units 16-byte units
    __shared__ __align__(8) uint64_t full[NS];
    __shared__ float red[2 * (TW / 32)];
    __shared__ StagedCursor cur;
    __shared__ int staging_off;
    float* red_max = red;
    float* red_sum = red + TW / 32;

    const float c = __fmul_rn(scale, kLog2e);
    const bool use_max = scale >= 0.0f;
    const int tid = threadIdx.x;
    const auto unit_of = [tid](int k) { return tid + k * TW; };
    const int32_t M = static_cast<int32_t>(g.rows_per_b / g.S);
    const int64_t n_items = g.rows / M;                       // (batch, row) pairs
    const uint32_t slot_bytes = static_cast<uint32_t>(g.units) * 16u;
    const uint32_t stage_u32 = tc::smem_u32(stage);

    const int32_t B = static_cast<int32_t>(n_items / g.S);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s)
            tc::mbar_init(&full[s], 1);
        staging_off = 0;
        cur.b = static_cast<int32_t>(blockIdx.x / g.S);
        cur.r = static_cast<int32_t>(blockIdx.x % g.S);
        cur.m = 0;
        cur.issued = cur.waited = 0;
        if (cur.b < B) {
            const int32_t L = __ldg(seq_lens + cur.b);
            cur.L = L < 0 ? 0 : (L > g.S ? g.S : L);
            staged_set_range<MK>(cur, seq_lens, g, EPU);
        }
        for (int k = 0; k < NS; ++k)
            staged_issue_next<T, MK, NS>(cur, x, seq_lens, g, M, B, stage_u32, slot_bytes, full);
    }
    __syncthreads();

    uint32_t live = 0;   // live rows taken so far (every thread counts them)
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int32_t b = static_cast<int32_t>(item / g.S), r = static_cast<int32_t>(item % g.S);
        int32_t c0, c1;
        kept_range<MK>(seq_lens, b, r, g, c0, c1);
        const UnitRange ur = UnitRange::of<EPU>(c0, c1);
        const int64_t q0 = static_cast<int64_t>(b) * M * g.S + r;
        for (int32_t m = 0; m < M; ++m) {
            const int64_t q = q0 + static_cast<int64_t>(m) * g.S;
            char* yr = reinterpret_cast<char*>(y + q * g.S);
            store_zeros<NV>(yr, ur, g.units, unit_of);
            if (c1 <= c0)
                continue;   // uniform across the team

            const uint32_t s = live % NS;
            const char* src = reinterpret_cast<const char*>(x + q * g.S);
            if (!*reinterpret_cast<volatile int*>(&staging_off)) {
                if (tc::mbar_wait(&full[s], (live / NS) & 1u, wait_ns)) {
                    src = reinterpret_cast<const char*>(stage + s * slot_bytes);
                    if (tid == 0)
                        ++cur.waited;
                } else if (tid == 0) {
                    *reinterpret_cast<volatile int*>(&staging_off) = 1;
                }
            }
            Unit16 raw[NV];
            load_kept<NV>(src, ur, unit_of, raw);
            float2 v[NV][Pairs<T>::kPairs];
            float ext = fwd_decode_extreme<T, NV>(raw, v, ur, unit_of, use_max);
            ext = use_max ? team_max<TW>(ext, red_max) : -team_max<TW>(-ext, red_max);
            // Every thread has read slot s: refill it with the row NS places on.
            if (tid == 0 && !*reinterpret_cast<volatile int*>(&staging_off)) {
                tc::fence_smem_for_async();
                staged_issue_next<T, MK, NS>(cur, x, seq_lens, g, M, B, stage_u32, slot_bytes, full);
            }
            const float sum = team_sum<TW>(fwd_exp_sum<T, NV>(v, ur, unit_of, ext, c), red_sum);
            fwd_store<T, NV>(yr, v, ur, unit_of, __frcp_rn(sum));
            ++live;
        }
    }

    // After a give-up, the copies issued but never seen complete must land
    // before the CTA's shared memory can be handed to another CTA.
    if (tid == 0)
        for (uint32_t k = cur.waited; k < cur.issued; ++k)
            tc::mbar_wait(&full[k % NS], (k / NS) & 1u, kAttnDrainWaitNs);
}

// Persistent launch: as many CTAs as fit on the device at once (at most one per
// (batch, row) pair); NS row slots of dynamic shared memory per CTA.
template <typename T, int MK, int TW, int NV, int NS, int MINB>
cudaError_t launch_fwd_staged(const void* x, void* y, const int32_t* seq_lens, const Geom& g, float scale,
                              cudaStream_t st, uint64_t wait_ns)
{
    auto* kern = gtms_fwd_staged_kernel<T, MK, TW, NV, NS, MINB>;
    const size_t smem = static_cast<size_t>(NS) * g.units * 16;
    cudaError_t e = cudaSuccess;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
        cudaSuccess)
        return e;
    int dev = 0, nsm = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, TW, smem)) != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t items = g.rows / (g.rows_per_b / g.S);
    const int64_t resident = static_cast<int64_t>(per_sm) * nsm;
    const unsigned grid = static_cast<unsigned>(items < resident ? items : resident);
    return launch_kernel(kern, grid, TW, smem, st, static_cast<const T*>(x), static_cast<T*>(y), seq_lens, g, scale,
                         wait_ns);
}

}  // namespace gtms
