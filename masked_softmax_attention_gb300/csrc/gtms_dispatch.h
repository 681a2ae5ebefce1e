// gtms_dispatch.h -- host-side choice of kernel variant (team size, units per
// thread, 16-byte or element access) for a row length and dtype.
#pragma once

#include <cstdint>

namespace gtms {

struct Variant {
    int team;          // threads per row: 32 = one warp, otherwise the whole CTA
    int per_thread;    // access units held per thread
    bool vec16;        // 16-byte vector units (else one element per unit)
    int max_units;     // team * per_thread
};

// 16-byte vectors: every row starts on a 16-byte boundary and all buffers are
// 16-byte aligned. Row capacity in vectors, smallest first.
constexpr Variant kVecVariants[] = {
    {32, 1, true, 32},      // rows <= 512 B
    {32, 2, true, 64},      // <= 1 KB
    {32, 4, true, 128},     // <= 2 KB
    {32, 8, true, 256},     // <= 4 KB   (fp32 S = 1000, bf16 S = 2048)
    {128, 4, true, 512},    // <= 8 KB
    {256, 4, true, 1024},   // <= 16 KB  (fp16 / bf16 S = 8192)
    {512, 4, true, 2048},   // <= 32 KB  (fp32 S = 8192)
};

// Element units: rows whose byte length is not a multiple of 16, or buffers
// that are only element-aligned.
constexpr Variant kElemVariants[] = {
    {32, 1, false, 32},
    {32, 4, false, 128},
    {32, 16, false, 512},
    {32, 32, false, 1024},
    {128, 32, false, 4096},
    {256, 32, false, 8192},
};

constexpr int kNumVec = sizeof(kVecVariants) / sizeof(kVecVariants[0]);
constexpr int kNumElem = sizeof(kElemVariants) / sizeof(kElemVariants[0]);

// Index into kVecVariants (0..kNumVec-1) or kElemVariants (kNumVec..), or -1.
inline int pick_variant(int64_t S, int elem_bytes, bool aligned16)
{
    if (S <= 0)
        return -1;
    const bool vec = aligned16 && ((S * elem_bytes) % 16 == 0);
    if (vec) {
        const int64_t units = S * elem_bytes / 16;
        for (int i = 0; i < kNumVec; ++i)
            if (units <= kVecVariants[i].max_units)
                return i;
        return -1;
    }
    for (int i = 0; i < kNumElem; ++i)
        if (S <= kElemVariants[i].max_units)
            return kNumVec + i;
    return -1;
}

inline const Variant& variant_at(int idx)
{
    return idx < kNumVec ? kVecVariants[idx] : kElemVariants[idx - kNumVec];
}

}  // namespace gtms
