// gtms_dispatch.h -- host-side choice of kernel variant for a row length, dtype
// and direction.
//
// Vector variants (16-byte units; the row's byte length is a multiple of 16 and
// every buffer is 16-byte aligned) are listed per direction and element size,
// smallest row capacity first. The forward holds up to 16 (fp32) or 32 (16-bit)
// kept elements per thread as fp32 exponentials; the backward holds up to 8
// raw 16-byte units of y and of dy per thread. Rows too long for one warp take a
// CTA of 64..512 threads. The last number is the minimum number of CTAs per SM
// requested from the compiler (__launch_bounds__): it caps registers so that
// enough rows are in flight per SM. These choices come from a sweep on GB300 of
// team size, units per thread, register cap and grid shape over the
// S = 1000 / 2048 / 4096 / 8192 workloads.
//
// Element variants (one element per unit) serve rows that are not 16-byte
// multiples, and element-aligned buffers, up to S = 8192.
//
// Stream variants serve 16-byte-unit rows of 32 KB and more (fp32 S >= 8192,
// 16-bit S >= 16384) up to S = 65536: one CTA per row walks the kept units
// twice, a batch of units per thread at a time (gtms_stream.cuh), so the row
// length no longer bounds the rows in flight per SM. Measured on GB300 against
// a 512- or 1024-thread CTA holding the whole row (S = 16384 bf16: 6.4 vs 5.2
// TB/s forward; S = 32768 bf16: 6.9 vs 4.8) and against a cluster of 2 or 4
// CTAs splitting the row over distributed shared memory (S = 65536 bf16: 6.2
// vs 2.5 TB/s forward, 5.8 vs 3.9 backward). Below 32 KB the rows held in
// registers stay faster (S = 8192 fp16 forward: 5.7 vs 4.6 TB/s).
#pragma once

#include <cstdint>

//                       id  team  units/thread  min CTAs/SM (0: no register cap)
#define GTMS_FWD_VEC4(X) X(0, 32, 1, 8) X(1, 32, 2, 8) X(2, 32, 4, 8) X(3, 64, 4, 0) \
                         X(4, 128, 4, 0) X(5, 256, 4, 0) X(6, 512, 4, 0)
#define GTMS_FWD_VEC2(X) X(0, 32, 1, 8) X(1, 32, 2, 8) X(2, 32, 4, 6) X(3, 64, 4, 16) \
                         X(4, 128, 4, 8) X(5, 256, 4, 4) X(6, 512, 4, 2)
#define GTMS_BWD_VEC4(X) X(0, 32, 1, 4) X(1, 32, 2, 4) X(2, 32, 4, 4) X(3, 32, 8, 5) \
                         X(4, 64, 8, 0) X(5, 128, 8, 0) X(6, 256, 8, 0)
#define GTMS_BWD_VEC2(X) X(0, 32, 1, 4) X(1, 32, 2, 4) X(2, 32, 4, 4) X(3, 32, 8, 5) \
                         X(4, 64, 8, 0) X(5, 128, 8, 0) X(6, 256, 8, 0)
// 16-bit forward rows served by a CTA team run as heads kernels (a team per
// (batch, row) pair, next head's loads issued early; gtms_kernels.cuh), with
// their own register caps. Measured on GB300 against one row per team: S = 2048
// bf16 5.86 -> 6.40 TB/s, S = 4096 bf16 5.82 -> 6.49, S = 8192 fp16 5.66 ->
// 6.41; for fp32 rows (S = 1000: 6.53 -> 6.21) one row per team stays ahead.
//                         id  team  units/thread  min CTAs/SM  (ids of GTMS_FWD_VEC2)
#define GTMS_FWD_HEADS2(X) X(3, 64, 4, 12) X(4, 128, 4, 6) X(5, 256, 4, 3) X(6, 512, 4, 1)
// The explicit-mask forward (gtms_explicit.cuh) takes the same rows with its own
// register caps: it holds the next head's units besides the current head's
// exponentials (fp32 warp teams 80 registers, 16-bit teams 78-127).
#define GTMS_EXF_VEC4(X) X(0, 32, 1, 8) X(1, 32, 2, 8) X(2, 32, 4, 6) X(3, 64, 4, 0) \
                         X(4, 128, 4, 0) X(5, 256, 4, 0) X(6, 512, 4, 1)
#define GTMS_EXF_VEC2(X) X(0, 32, 1, 8) X(1, 32, 2, 8) X(2, 32, 4, 5) X(3, 64, 4, 12) \
                         X(4, 128, 4, 6) X(5, 256, 4, 3) X(6, 512, 4, 1)
//                       id  team  elements/thread
#define GTMS_ELEM(X) X(0, 32, 1) X(1, 32, 4) X(2, 32, 16) X(3, 32, 32) X(4, 128, 32) X(5, 256, 32)
// Band variants (sliding-window rows whose window spans at most 32 * KV units,
// in rows longer than one warp's 128 units; 16-byte units only, below the
// stream rows): a warp owns a row and holds only the window (gtms_band.cuh).
//                        id  units/lane  min CTAs/SM
#define GTMS_FWD_BAND(X) X(0, 1, 8) X(1, 2, 8) X(2, 4, 6)
#define GTMS_BWD_BAND(X) X(0, 1, 4) X(1, 2, 4) X(2, 4, 4) X(3, 8, 5)
// Stream variants (rows of at least kStreamFromBytes, 16-byte units only):
//                      id  team  units/thread per batch  min CTAs/SM  max row units
#define GTMS_FWD_ST4(X) X(0, 128, 4, 8, 4095) X(1, 256, 4, 4, INT32_MAX)
#define GTMS_FWD_ST2(X) X(0, 128, 4, 8, 4095) X(1, 256, 4, 4, INT32_MAX)
#define GTMS_BWD_ST4(X) X(0, 256, 2, 4, INT32_MAX)
#define GTMS_BWD_ST2(X) X(0, 256, 2, 4, INT32_MAX)

// Staged forward (gtms_forward_staged, gtms_staged.cuh): a persistent CTA team per
// row, the row's kept units brought into shared memory by one TMA bulk copy,
// NS row slots per CTA. Rows of 16-byte units below the stream rows. Measured on
// GB300 against the default forward (TB/s): S = 1000 fp32 5.58 vs 6.55, S = 2048
// bf16 5.63 vs 6.43, S = 4096 bf16 6.03 vs 6.55, S = 8192 fp16 6.01 vs 6.46.
//                            id  team  units/thread  slots  min CTAs/SM
#define GTMS_FWD_STAGED4(X) X(0, 64, 4, 6, 12) X(1, 128, 4, 2, 5) X(2, 256, 4, 2, 3)
#define GTMS_FWD_STAGED2(X) X(0, 64, 4, 2, 10) X(1, 128, 4, 2, 5) X(2, 256, 4, 2, 3)

namespace gtms {

struct Variant {
    int team;         // threads per row: 32 = one warp, otherwise the whole CTA
    int per_thread;   // access units held per thread (stream variants: per batch)
    int min_ctas;     // __launch_bounds__ minimum CTAs per SM (0: none)
    bool vec16;       // 16-byte units (else one element per unit)
    int max_units;    // longest row served, in units (team * per_thread for the per-row variants)
};

#define GTMS_VEC_ROW(id, tw, nv, mb) {tw, nv, mb, true, (tw) * (nv)},
#define GTMS_ELEM_ROW(id, tw, nv) {tw, nv, 0, false, (tw) * (nv)},
#define GTMS_ST_ROW(id, tw, nv, mb, mu) {tw, nv, mb, true, mu},
#define GTMS_BAND_ROW(id, nv, mb) {32, nv, mb, true, 32 * (nv)},
constexpr Variant kFwdVec4[] = {GTMS_FWD_VEC4(GTMS_VEC_ROW)};
constexpr Variant kFwdVec2[] = {GTMS_FWD_VEC2(GTMS_VEC_ROW)};
constexpr Variant kBwdVec4[] = {GTMS_BWD_VEC4(GTMS_VEC_ROW)};
constexpr Variant kBwdVec2[] = {GTMS_BWD_VEC2(GTMS_VEC_ROW)};
constexpr Variant kElem[] = {GTMS_ELEM(GTMS_ELEM_ROW)};
#define GTMS_HEADS_ROW(id, tw, nv, mb) {tw, nv, mb, true, (tw) * (nv)},
constexpr Variant kFwdHeads2[] = {GTMS_FWD_HEADS2(GTMS_HEADS_ROW)};
#undef GTMS_HEADS_ROW
#define GTMS_HEADS_ID(id, tw, nv, mb) id,
constexpr int kFwdHeads2Ids[] = {GTMS_FWD_HEADS2(GTMS_HEADS_ID)};
#undef GTMS_HEADS_ID
constexpr Variant kFwdBand[] = {GTMS_FWD_BAND(GTMS_BAND_ROW)};
constexpr Variant kBwdBand[] = {GTMS_BWD_BAND(GTMS_BAND_ROW)};
constexpr Variant kExFwdVec4[] = {GTMS_EXF_VEC4(GTMS_VEC_ROW)};
constexpr Variant kExFwdVec2[] = {GTMS_EXF_VEC2(GTMS_VEC_ROW)};
constexpr Variant kFwdSt4[] = {GTMS_FWD_ST4(GTMS_ST_ROW)};
constexpr Variant kFwdSt2[] = {GTMS_FWD_ST2(GTMS_ST_ROW)};
constexpr Variant kBwdSt4[] = {GTMS_BWD_ST4(GTMS_ST_ROW)};
constexpr Variant kBwdSt2[] = {GTMS_BWD_ST2(GTMS_ST_ROW)};
#undef GTMS_VEC_ROW
#undef GTMS_ELEM_ROW
#undef GTMS_ST_ROW
#undef GTMS_BAND_ROW

template <typename V, int N>
constexpr int count_of(const V (&)[N]) { return N; }

constexpr int kElemBase = 100;     // variant ids in [kElemBase, kStreamBase) are element variants
constexpr int kStreamBase = 300;   // variant ids in [kStreamBase, kBandBase) are stream variants
constexpr int kBandBase = 400;     // variant ids in [kBandBase, kHeadsBase) are band variants
constexpr int kHeadsBase = 500;    // variant id kHeadsBase + v: the heads form of 16-bit forward row v

// Row byte length from which the stream variants serve a row, per direction
// (forward, backward).
constexpr int64_t kStreamFromBytes[2] = {32768, 32768};

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

constexpr bool same_shapes(const Variant* a, const Variant* b, int n)
{
    for (int i = 0; i < n; ++i)
        if (a[i].team != b[i].team || a[i].per_thread != b[i].per_thread)
            return false;
    return true;
}
static_assert(count_of(kExFwdVec4) == count_of(kFwdVec4) && same_shapes(kExFwdVec4, kFwdVec4, count_of(kFwdVec4)) &&
                  count_of(kExFwdVec2) == count_of(kFwdVec2) && same_shapes(kExFwdVec2, kFwdVec2, count_of(kFwdVec2)),
              "explicit-mask forward rows must match the vector rows id for id");

constexpr bool heads_rows_match()
{
    for (int i = 0; i < count_of(kFwdHeads2Ids); ++i) {
        const Variant& v = kFwdVec2[kFwdHeads2Ids[i]];
        if (v.team != kFwdHeads2[i].team || v.per_thread != kFwdHeads2[i].per_thread || v.team == 32)
            return false;
    }
    return true;
}
static_assert(heads_rows_match(), "heads rows must match the 16-bit forward CTA-team rows they replace");

// Variant table of the explicit-mask kernels (same ids as vec_table).
inline VariantTable explicit_table(int direction, int elem_bytes)
{
    if (direction == 0)
        return elem_bytes == 4 ? VariantTable{kExFwdVec4, count_of(kExFwdVec4)}
                               : VariantTable{kExFwdVec2, count_of(kExFwdVec2)};
    return vec_table(direction, elem_bytes);
}

inline VariantTable stream_table(int direction, int elem_bytes)
{
    if (direction == 0)
        return elem_bytes == 4 ? VariantTable{kFwdSt4, count_of(kFwdSt4)} : VariantTable{kFwdSt2, count_of(kFwdSt2)};
    return elem_bytes == 4 ? VariantTable{kBwdSt4, count_of(kBwdSt4)} : VariantTable{kBwdSt2, count_of(kBwdSt2)};
}

// Variant id for (direction, S, element size, all buffers 16-byte aligned), or
// -1. `allow_stream` false keeps to the per-row vector variants (the explicit-
// mask kernels have no other form).
inline int pick_variant(int direction, int64_t S, int elem_bytes, bool aligned16, bool allow_stream = true)
{
    if (S <= 0)
        return -1;
    if (aligned16 && (S * elem_bytes) % 16 == 0) {
        const int64_t units = S * elem_bytes / 16;
        if (allow_stream && S * elem_bytes >= kStreamFromBytes[direction]) {
            const VariantTable t = stream_table(direction, elem_bytes);
            for (int i = 0; i < t.count; ++i)
                if (units <= t.rows[i].max_units)
                    return kStreamBase + i;
            return -1;
        }
        const VariantTable t = vec_table(direction, elem_bytes);
        for (int i = 0; i < t.count; ++i)
            if (units <= t.rows[i].max_units)
                return i;
        return -1;
    }
    for (int i = 0; i < count_of(kElem); ++i)
        if (S <= kElem[i].max_units)
            return kElemBase + i;
    return -1;
}

inline VariantTable heads_table() { return VariantTable{kFwdHeads2, count_of(kFwdHeads2)}; }

// The heads variant that replaces per-row vector variant `vec_id` of the 16-bit
// forward, or -1.
inline int heads_variant(int direction, int elem_bytes, int vec_id)
{
    if (direction != 0 || elem_bytes != 2)
        return -1;
    for (int i = 0; i < count_of(kFwdHeads2Ids); ++i)
        if (kFwdHeads2Ids[i] == vec_id)
            return kHeadsBase + vec_id;
    return -1;
}

// Row of heads variant id (kHeadsBase + vector row id).
inline Variant heads_row(int id)
{
    for (int i = 0; i < count_of(kFwdHeads2Ids); ++i)
        if (kHeadsBase + kFwdHeads2Ids[i] == id)
            return kFwdHeads2[i];
    return kFwdHeads2[0];
}

inline VariantTable band_table(int direction)
{
    return direction == 0 ? VariantTable{kFwdBand, count_of(kFwdBand)} : VariantTable{kBwdBand, count_of(kBwdBand)};
}

// Band variant id for a sliding window of `window` columns, or -1 when the
// row-length variant (pick_variant) serves the row better: the window must fit
// a warp's slots, and the row must be a 16-byte-unit row longer than 128 units
// that is not a stream row.
inline int pick_band_variant(int direction, int64_t S, int elem_bytes, bool aligned16, int64_t window)
{
    if (S <= 0 || window < 1 || !aligned16 || (S * elem_bytes) % 16 != 0)
        return -1;
    const int64_t units = S * elem_bytes / 16;
    if (units <= 128 || S * elem_bytes >= kStreamFromBytes[direction])
        return -1;
    const int64_t epu = 16 / elem_bytes;
    const int64_t w = window < S ? window : S;
    const int64_t spanned = (w + 2 * epu - 2) / epu;   // units a run of w columns can touch
    if (2 * spanned > units)
        return -1;
    const VariantTable t = band_table(direction);
    for (int i = 0; i < t.count; ++i)
        if (spanned <= t.rows[i].max_units)
            return kBandBase + i;
    return -1;
}

// Variant id that gtms_forward_masked / gtms_backward_masked launch for a
// row-length choice: pick_variant, with the heads rows in place of the 16-bit
// forward's CTA-team rows.
inline int pick_launch_variant(int direction, int64_t S, int elem_bytes, bool aligned16)
{
    const int v = pick_variant(direction, S, elem_bytes, aligned16);
    const int h = v >= 0 ? heads_variant(direction, elem_bytes, v) : -1;
    return h >= 0 ? h : v;
}

struct StagedVariant {
    int team, per_thread, slots, min_ctas;
};
#define GTMS_STAGED_ROW(id, tw, nv, ns, mb) {tw, nv, ns, mb},
constexpr StagedVariant kFwdStaged4[] = {GTMS_FWD_STAGED4(GTMS_STAGED_ROW)};
constexpr StagedVariant kFwdStaged2[] = {GTMS_FWD_STAGED2(GTMS_STAGED_ROW)};
#undef GTMS_STAGED_ROW

// Staged-forward variant id for (S, element size, all buffers 16-byte aligned), or
// -1: rows of 16-byte units, shorter than the stream rows, that a row of the table holds.
inline int pick_staged_variant(int64_t S, int elem_bytes, bool aligned16)
{
    if (S <= 0 || !aligned16 || (S * elem_bytes) % 16 != 0 || S * elem_bytes >= kStreamFromBytes[0])
        return -1;
    const int64_t units = S * elem_bytes / 16;
    const StagedVariant* t = elem_bytes == 4 ? kFwdStaged4 : kFwdStaged2;
    const int n = elem_bytes == 4 ? count_of(kFwdStaged4) : count_of(kFwdStaged2);
    for (int i = 0; i < n; ++i)
        if (units <= static_cast<int64_t>(t[i].team) * t[i].per_thread)
            return i;
    return -1;
}

static_assert(count_of(kFwdStaged4) == 3 && count_of(kFwdStaged2) == 3, "three staged rows per element size");

inline StagedVariant staged_at(int elem_bytes, int id)
{
    return elem_bytes == 4 ? kFwdStaged4[id] : kFwdStaged2[id];
}

inline Variant variant_at(int direction, int elem_bytes, int id)
{
    if (id >= kHeadsBase)
        return heads_row(id);
    if (id >= kBandBase)
        return band_table(direction).rows[id - kBandBase];
    if (id >= kStreamBase)
        return stream_table(direction, elem_bytes).rows[id - kStreamBase];
    if (id >= kElemBase)
        return kElem[id - kElemBase];
    return vec_table(direction, elem_bytes).rows[id];
}

}  // namespace gtms
