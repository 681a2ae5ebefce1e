// gtms_tcgen05.cuh -- the few sm_100+ tensor-core (tcgen05), tensor-memory,
// mbarrier and asynchronous-copy instructions the fused attention-backward step
// uses, as inline PTX.
//
// Operands live in shared memory in the canonical K-major layout without
// swizzle: the matrix is cut into core matrices of 8 rows x 16 bytes (8 x 8
// 16-bit elements), each stored as 128 contiguous bytes (row after row). The
// shared-memory descriptor gives the byte stride between core matrices that
// are neighbours along K (leading dimension, LBO) and along M / N (stride
// dimension, SBO). One MMA of kind::f16 consumes K = 16, i.e. two core
// matrices along K, so successive K steps advance the start address by 2 * LBO.
// The fp32 accumulator of an M = 128 MMA sits in tensor memory with row i in
// lane i and column j in column j.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gtms {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor (no swizzle): start address >> 4 in bits 0-13,
// LBO >> 4 in bits 16-29, SBO >> 4 in bits 32-45, descriptor version 1 at bit 46.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16) |
           (static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Shared-memory matrix descriptor of a K-major operand stored with the 128-byte
// swizzle (the layout a TMA load with SWIZZLE_128B writes): rows of 128 bytes,
// 16-byte chunk j of row r at chunk j ^ (r % 8), 8-row groups `sbo` bytes apart;
// layout type 2 (128-byte swizzle) in bits 61-63. The atom base must be
// 1024-byte aligned; a K step inside the 128-byte row advances the start address.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t sbo)
{
    return smem_desc(addr, 16, sbo) | (static_cast<uint64_t>(2) << 61);
}

// Shared-memory matrix descriptor of an MN-major operand stored with the 128-byte
// swizzle: each K row holds 64 16-bit MN elements in 128 bytes (chunks swizzled as
// above), 8 K rows make a 1024-byte atom and the next 8 K rows follow it (SBO =
// 1024); `lbo` is the byte stride between 64-element boxes along MN. A K step of
// 16 advances the start address by 2048 bytes. (Checked on GB300 with a one-tile
// product against a CPU reference, for N = 64 and 128.)
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t addr, uint32_t lbo)
{
    return smem_desc(addr, lbo, 1024) | (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and B
// of the same 16-bit type (bits 7-9 and 10-12: 0 = fp16, 1 = bf16), both
// K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28. (Bit 16 set makes B
// MN-major: see kIdescBMnMajor.)
template <typename T>
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N)
{
    constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction-descriptor bit of a B operand stored MN-major (N contiguous in
// each 16-byte row of a core matrix). In the no-swizzle MN-major layout the
// descriptor's LBO is then the byte stride between core matrices adjacent
// along K, and SBO between those adjacent along N (checked on GB300 with a
// one-tile product against a CPU reference).
constexpr uint32_t kIdescBMnMajor = 1u << 16;

// D (tensor memory) = A * B^T (+ D when accumulate != 0); issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(tmem_d), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// The mbarrier receives one arrival once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t* mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(mbar)) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Make this thread's generic-proxy writes to shared memory visible to the tensor core.
__device__ __forceinline__ void fence_smem_for_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Warp-collective: allocate / free `ncols` tensor-memory columns (power of 2, >= 32).
template <int NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(slot)), "n"(NCOLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int NCOLS>
__device__ __forceinline__ void tmem_free(uint32_t taddr)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "n"(NCOLS) : "memory");
}

// Warp-collective: 16 consecutive fp32 columns of this thread's lane, then wait
// (load and wait in one statement, so no use of the values can move above the wait).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j)
        v[j] = __uint_as_float(r[j]);
}

// Warp-collective: 32 consecutive fp32 columns of this thread's lane, then wait
// (load and wait in one statement, so no use of the values can move above the wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j)
        v[j] = __uint_as_float(r[j]);
}

// 16-byte global -> shared copy that completes asynchronously (cp.async, cached
// in L2 only). src_bytes < 16 zero-fills the rest of the destination; with 0 the
// source is not read.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Warp-collective: 64 consecutive fp32 columns of this thread's lane, then wait
// (load and wait in one statement, so no use of the values can move above the wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64])
{
    uint32_t r[64];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
                 "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                   "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
                   "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
                   "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                   "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
                   "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int j = 0; j < 64; ++j)
        v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(mbar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive on the mbarrier and raise its expected transaction count by `bytes`
// (the bytes that the TMA copies signalling it will deliver).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_u32(mbar)), "r"(bytes) : "memory");
}

// `count` arrivals on the mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* mbar, uint32_t count = 1)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" :: "r"(smem_u32(mbar)), "r"(count) : "memory");
}

// TMA: box of a 3-D tensor map at element coordinates (x, y, z) into shared
// memory; completion is signalled on the mbarrier as transaction bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint64_t* mbar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(mbar))
                 : "memory");
}

// L2 cache policies for the hinted copies below: keep the lines (data that is
// read again soon) or evict them first (data that is not read again).
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// tma_load_3d with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint64_t* mbar, uint64_t pol)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%2, %3, %4}], [%5], %6;"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(mbar)),
                    "l"(pol)
                 : "memory");
}

// tma_store_3d with an L2 cache policy.
__device__ __forceinline__ void tma_store_3d(const void* tmap, int32_t x, int32_t y, int32_t z, uint32_t src,
                                             uint64_t pol)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2, %3}], [%4], %5;"
                 :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(src), "l"(pol) : "memory");
}

// Untiled bulk copy (TMA) of `bytes` bytes from global memory into this CTA's
// shared memory, under an L2 cache policy; completion is signalled on the
// mbarrier as transaction bytes. Both addresses 16-byte aligned, `bytes` a
// multiple of 16.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint64_t* mbar,
                                             uint64_t pol)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(smem_u32(mbar)), "l"(pol) : "memory");
}

// TMA: prefetch the box of a 3-D tensor map at (x, y, z) into L2 (no shared
// memory, no completion signal), under an L2 cache policy.
__device__ __forceinline__ void tma_prefetch_3d(const void* tmap, int32_t x, int32_t y, int32_t z, uint64_t pol)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile.L2::cache_hint [%0, {%1, %2, %3}], %4;"
                 :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "l"(pol) : "memory");
}

// 16 zero bytes to global memory under an L2 cache policy.
__device__ __forceinline__ void st_global_zero16(void* p, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %1, %1, %1}, %2;" :: "l"(p), "r"(0u), "l"(pol) : "memory");
}

// TMA: shared memory into the box of a 3-D tensor map at (x, y, z) (elements
// outside the tensor are not written); tracked by the bulk async-group.
__device__ __forceinline__ void tma_store_3d(const void* tmap, int32_t x, int32_t y, int32_t z, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                 :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(src) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the committed bulk stores have finished reading shared memory / have completed.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* mbar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
    return done != 0;
}

// Wait until the mbarrier's phase `parity` has completed, giving up once
// `limit_ns` nanoseconds of the global timer have passed since the first poll
// failed (each poll may itself suspend the thread for a short, hardware-chosen
// time). Returns false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(mbar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    do {
        if (mbar_try_wait(mbar, parity))
            return true;
    } while (globaltimer_ns() - t0 < limit_ns);
    return false;
}

}  // namespace tc
}  // namespace gtms
