// gtms_dispatch.h -- host-side choice of kernel variant for a row length, dtype
// and direction.
//
// Vector variants (16-byte units; the row's byte length is a multiple of 16 and
// every buffer is 16-byte aligned) are listed per direction and element size,
// smallest row capacity first. The forward holds up to 16 (fp32) or 32 (16-bit)
// kept elements per thread as fp32 exponentials; the backward holds up to 8
// raw 16-byte units of y and of dy per thread. Rows too long for one warp take a
// CTA of 64..1024 threads, up to 64 KB rows. The last number is the minimum number of CTAs per SM
// requested from the compiler (__launch_bounds__): it caps registers so that
// enough rows are in flight per SM. These choices come from a sweep on GB300 of
// team size, units per thread, register cap and grid shape over the
// S = 1000 / 2048 / 4096 / 8192 workloads.
//
// Element variants (one element per unit) serve rows that are not 16-byte
// multiples, and element-aligned buffers, up to S = 8192.
//
// Cluster variants serve 16-byte-unit rows longer than the largest CTA variant
// (64 KB: fp32 S > 16384, 16-bit S > 32768), up to S = 65536: a cluster of 2 or
// 4 CTAs owns one row (gtms_cluster.cuh). Measured on GB300, one 512- or
// 1024-thread CTA per row beats a cluster for rows that still fit one CTA
// (S = 16384 bf16: 5.2 vs 3.1 TB/s forward, 6.1 vs 4.3 backward): the
// cluster barrier per row costs more than the larger CTA's block barriers.
#pragma once

#include <cstdint>

//                       id  team  units/thread  min CTAs/SM (0: no register cap)
#define GTMS_FWD_VEC4(X) X(0, 32, 1, 8) X(1, 32, 2, 8) X(2, 32, 4, 8) X(3, 64, 4, 0) \
                         X(4, 128, 4, 0) X(5, 256, 4, 0) X(6, 512, 4, 0) X(7, 1024, 4, 0)
#define GTMS_FWD_VEC2(X) X(0, 32, 1, 8) X(1, 32, 2, 8) X(2, 32, 4, 6) X(3, 64, 4, 16) \
                         X(4, 128, 4, 8) X(5, 256, 4, 4) X(6, 512, 4, 2) X(7, 1024, 4, 0)
#define GTMS_BWD_VEC4(X) X(0, 32, 1, 4) X(1, 32, 2, 4) X(2, 32, 4, 4) X(3, 32, 8, 5) \
                         X(4, 64, 8, 0) X(5, 128, 8, 0) X(6, 256, 8, 0) X(7, 512, 8, 0)
#define GTMS_BWD_VEC2(X) X(0, 32, 1, 4) X(1, 32, 2, 4) X(2, 32, 4, 4) X(3, 32, 8, 5) \
                         X(4, 64, 8, 0) X(5, 128, 8, 0) X(6, 256, 8, 0) X(7, 512, 8, 0)
//                       id  team  elements/thread
#define GTMS_ELEM(X) X(0, 32, 1) X(1, 32, 4) X(2, 32, 16) X(3, 32, 32) X(4, 128, 32) X(5, 256, 32)
// Cluster variants (rows longer than one CTA holds, 16-byte units only):
//                      id  CTAs/cluster  team  units/thread  min CTAs/SM
#define GTMS_FWD_CL4(X) X(0, 2, 1024, 4, 0) X(1, 4, 1024, 4, 0)
#define GTMS_FWD_CL2(X) X(0, 2, 1024, 4, 0)
#define GTMS_BWD_CL4(X) X(0, 2, 512, 8, 0) X(1, 4, 512, 8, 0)
#define GTMS_BWD_CL2(X) X(0, 2, 512, 8, 0)

namespace gtms {

struct Variant {
    int team;         // threads per row (per CTA for clusters): 32 = one warp, otherwise the whole CTA
    int per_thread;   // access units held per thread
    int min_ctas;     // __launch_bounds__ minimum CTAs per SM (0: none)
    bool vec16;       // 16-byte units (else one element per unit)
    int max_units;    // cluster * team * per_thread
    int cluster;      // CTAs per row (1: no cluster)
};

#define GTMS_VEC_ROW(id, tw, nv, mb) {tw, nv, mb, true, (tw) * (nv), 1},
#define GTMS_ELEM_ROW(id, tw, nv) {tw, nv, 0, false, (tw) * (nv), 1},
#define GTMS_CL_ROW(id, cl, tw, nv, mb) {tw, nv, mb, true, (cl) * (tw) * (nv), cl},
constexpr Variant kFwdVec4[] = {GTMS_FWD_VEC4(GTMS_VEC_ROW)};
constexpr Variant kFwdVec2[] = {GTMS_FWD_VEC2(GTMS_VEC_ROW)};
constexpr Variant kBwdVec4[] = {GTMS_BWD_VEC4(GTMS_VEC_ROW)};
constexpr Variant kBwdVec2[] = {GTMS_BWD_VEC2(GTMS_VEC_ROW)};
constexpr Variant kElem[] = {GTMS_ELEM(GTMS_ELEM_ROW)};
constexpr Variant kFwdCl4[] = {GTMS_FWD_CL4(GTMS_CL_ROW)};
constexpr Variant kFwdCl2[] = {GTMS_FWD_CL2(GTMS_CL_ROW)};
constexpr Variant kBwdCl4[] = {GTMS_BWD_CL4(GTMS_CL_ROW)};
constexpr Variant kBwdCl2[] = {GTMS_BWD_CL2(GTMS_CL_ROW)};
#undef GTMS_VEC_ROW
#undef GTMS_ELEM_ROW
#undef GTMS_CL_ROW

template <typename V, int N>
constexpr int count_of(const V (&)[N]) { return N; }

constexpr int kElemBase = 100;      // variant ids in [kElemBase, kClusterBase) are element variants
constexpr int kClusterBase = 200;   // variant ids >= kClusterBase are cluster variants

struct VariantTable {
    const Variant* rows;
    int count;
};

inline VariantTable vec_table(int direction, int elem_bytes)
{
    if (direction == 0)
        return elem_bytes == 4 ? VariantTable{kFwdVec4, count_of(kFwdVec4)} : VariantTable{kFwdVec2, count_of(kFwdVec2)};
    return elem_bytes == 4 ? VariantTable{kBwdVec4, count_of(kBwdVec4)} : VariantTable{kBwdVec2, count_of(kBwdVec2)};
}

inline VariantTable cluster_table(int direction, int elem_bytes)
{
    if (direction == 0)
        return elem_bytes == 4 ? VariantTable{kFwdCl4, count_of(kFwdCl4)} : VariantTable{kFwdCl2, count_of(kFwdCl2)};
    return elem_bytes == 4 ? VariantTable{kBwdCl4, count_of(kBwdCl4)} : VariantTable{kBwdCl2, count_of(kBwdCl2)};
}

// Variant id for (direction, S, element size, all buffers 16-byte aligned), or -1.
inline int pick_variant(int direction, int64_t S, int elem_bytes, bool aligned16)
{
    if (S <= 0)
        return -1;
    if (aligned16 && (S * elem_bytes) % 16 == 0) {
        const int64_t units = S * elem_bytes / 16;
        const VariantTable t = vec_table(direction, elem_bytes);
        for (int i = 0; i < t.count; ++i)
            if (units <= t.rows[i].max_units)
                return i;
        const VariantTable c = cluster_table(direction, elem_bytes);
        for (int i = 0; i < c.count; ++i)
            if (units <= c.rows[i].max_units)
                return kClusterBase + i;
        return -1;
    }
    for (int i = 0; i < count_of(kElem); ++i)
        if (S <= kElem[i].max_units)
            return kElemBase + i;
    return -1;
}

inline Variant variant_at(int direction, int elem_bytes, int id)
{
    if (id >= kClusterBase)
        return cluster_table(direction, elem_bytes).rows[id - kClusterBase];
    if (id >= kElemBase)
        return kElem[id - kElemBase];
    return vec_table(direction, elem_bytes).rows[id];
}

}  // namespace gtms
