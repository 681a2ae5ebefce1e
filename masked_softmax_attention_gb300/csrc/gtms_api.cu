// gtms_api.cu -- the C ABI declared in include/gtms.h: host-side argument
// checks, variant choice and kernel launch. No allocation, no synchronisation,
// no host read of device memory.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gtms.h"
#include "gtms_dispatch.h"
#include "gtms_kernels.cuh"

#define GTMS_EXPORT extern "C" __attribute__((visibility("default")))

namespace gtms {
template <typename T, int MK>
cudaError_t launch_forward(int, const void*, void*, const int32_t*, const Geom&, float, cudaStream_t);
template <typename T, int MK>
cudaError_t launch_backward(int, const void*, const void*, void*, const int32_t*, const Geom&, float, cudaStream_t);
// Instantiated one per translation unit (gtms_{fwd,bwd}_<dtype>_<mask>.cu).
#define GTMS_EXTERN_FOR(T, MK) \
    extern template cudaError_t launch_forward<T, MK>(int, const void*, void*, const int32_t*, const Geom&, float,   \
                                                      cudaStream_t);                                               \
    extern template cudaError_t launch_backward<T, MK>(int, const void*, const void*, void*, const int32_t*,        \
                                                       const Geom&, float, cudaStream_t);
GTMS_EXTERN_FOR(float, 0)
GTMS_EXTERN_FOR(float, 1)
GTMS_EXTERN_FOR(float, 2)
GTMS_EXTERN_FOR(__nv_bfloat16, 0)
GTMS_EXTERN_FOR(__nv_bfloat16, 1)
GTMS_EXTERN_FOR(__nv_bfloat16, 2)
GTMS_EXTERN_FOR(__half, 0)
GTMS_EXTERN_FOR(__half, 1)
GTMS_EXTERN_FOR(__half, 2)
#undef GTMS_EXTERN_FOR
template <typename T>
cudaError_t launch_forward_explicit(int, const void*, void*, const uint8_t*, int32_t, const Geom&, float, cudaStream_t);
template <typename T>
cudaError_t launch_backward_explicit(int, const void*, const void*, void*, const uint8_t*, int32_t, const Geom&, float,
                                     cudaStream_t);
#define GTMS_EXTERN_EXPLICIT(T)                                                                                     \
    extern template cudaError_t launch_forward_explicit<T>(int, const void*, void*, const uint8_t*, int32_t,        \
                                                           const Geom&, float, cudaStream_t);                      \
    extern template cudaError_t launch_backward_explicit<T>(int, const void*, const void*, void*, const uint8_t*,   \
                                                            int32_t, const Geom&, float, cudaStream_t);
GTMS_EXTERN_EXPLICIT(float)
GTMS_EXTERN_EXPLICIT(__nv_bfloat16)
GTMS_EXTERN_EXPLICIT(__half)
#undef GTMS_EXTERN_EXPLICIT
template <typename T, int D>
cudaError_t launch_attn_dscores(const void*, const void*, const void*, void*, const int32_t*, int64_t, int64_t,
                                int64_t, float, int32_t*, cudaStream_t, uint64_t);
extern template cudaError_t launch_attn_dscores<__nv_bfloat16, 64>(const void*, const void*, const void*, void*,
                                                                   const int32_t*, int64_t, int64_t, int64_t, float,
                                                                   int32_t*, cudaStream_t, uint64_t);
extern template cudaError_t launch_attn_dscores<__nv_bfloat16, 128>(const void*, const void*, const void*, void*,
                                                                    const int32_t*, int64_t, int64_t, int64_t, float,
                                                                    int32_t*, cudaStream_t, uint64_t);
extern template cudaError_t launch_attn_dscores<__half, 64>(const void*, const void*, const void*, void*,
                                                            const int32_t*, int64_t, int64_t, int64_t, float,
                                                            int32_t*, cudaStream_t, uint64_t);
extern template cudaError_t launch_attn_dscores<__half, 128>(const void*, const void*, const void*, void*,
                                                             const int32_t*, int64_t, int64_t, int64_t, float,
                                                             int32_t*, cudaStream_t, uint64_t);
template <typename T, int D>
cudaError_t launch_attn_dscores_tma(const void*, const void*, const void*, void*, const int32_t*, int64_t, int64_t,
                                    int64_t, float, int32_t*, cudaStream_t, uint64_t);
#define GTMS_EXTERN_ATTN_TMA(T, D)                                                                              \
    extern template cudaError_t launch_attn_dscores_tma<T, D>(const void*, const void*, const void*, void*,     \
                                                              const int32_t*, int64_t, int64_t, int64_t, float, \
                                                              int32_t*, cudaStream_t, uint64_t);
GTMS_EXTERN_ATTN_TMA(__nv_bfloat16, 64)
GTMS_EXTERN_ATTN_TMA(__nv_bfloat16, 128)
GTMS_EXTERN_ATTN_TMA(__half, 64)
GTMS_EXTERN_ATTN_TMA(__half, 128)
#undef GTMS_EXTERN_ATTN_TMA
template <typename T>
cudaError_t launch_forward_staged(int, const void*, void*, const int32_t*, const Geom&, float, cudaStream_t);
extern template cudaError_t launch_forward_staged<float>(int, const void*, void*, const int32_t*, const Geom&, float,
                                                         cudaStream_t);
extern template cudaError_t launch_forward_staged<__nv_bfloat16>(int, const void*, void*, const int32_t*, const Geom&,
                                                                 float, cudaStream_t);
extern template cudaError_t launch_forward_staged<__half>(int, const void*, void*, const int32_t*, const Geom&, float,
                                                          cudaStream_t);
}  // namespace gtms

namespace {

// True for memory the CUDA runtime reports as device memory (not mapped host
// memory, managed memory or an unknown pointer).
bool in_device_memory(const void* ptr)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice;
}

int elem_bytes(int dtype)
{
    switch (dtype) {
    case GTMS_F32: return 4;
    case GTMS_BF16:
    case GTMS_F16: return 2;
    default: return 0;
    }
}

struct Checked {
    int status;
    int64_t rows;
    uint64_t bytes;   // bytes of one [B,M,S,S] tensor
};

// Shape, scale and dtype checks shared by both directions.
Checked check_shape(int64_t B, int64_t M, int64_t S, float scale, int dtype)
{
    Checked c{GTMS_OK, 0, 0};
    if (B < 0 || M < 0 || S < 0 || !std::isfinite(scale)) {
        c.status = GTMS_ERR_INVALID_ARG;
        return c;
    }
    const int e = elem_bytes(dtype);
    if (e == 0 || S > GTMS_MAX_S) {
        c.status = GTMS_ERR_UNSUPPORTED;
        return c;
    }
    int64_t rows = 0, elems = 0, bytes = 0;
    if (__builtin_mul_overflow(B, M, &rows) || __builtin_mul_overflow(rows, S, &rows) ||
        __builtin_mul_overflow(rows, S, &elems) || __builtin_mul_overflow(elems, static_cast<int64_t>(e), &bytes) ||
        B > INT32_MAX) {
        c.status = GTMS_ERR_INVALID_ARG;
        return c;
    }
    c.rows = rows;
    c.bytes = static_cast<uint64_t>(bytes);
    return c;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, uint64_t an, const void* b, uint64_t bn)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

// An output may equal an input exactly; any other overlap is rejected.
bool bad_alias(const void* out, const void* in, uint64_t bytes)
{
    return out != in && overlaps(out, bytes, in, bytes);
}

gtms::Geom make_geom(int direction, int64_t rows, int64_t M, int64_t S, int variant, int e, int64_t window)
{
    const gtms::Variant v = gtms::variant_at(direction, e, variant);
    gtms::Geom g;
    g.rows = rows;
    g.rows_per_b = M * S;
    g.S = static_cast<int32_t>(S);
    g.units = static_cast<int32_t>(v.vec16 ? S * e / 16 : S);
    g.small = rows <= static_cast<int64_t>(UINT32_MAX) ? 1 : 0;
    g.window = static_cast<int32_t>(window < S ? window : S);
    return g;
}

// Mask kind and window: kinds 0..2; the sliding window needs a width >= 1.
int check_mask(int mask_kind, int64_t window)
{
    if (mask_kind < 0 || mask_kind > 2)
        return GTMS_ERR_UNSUPPORTED;
    if (mask_kind == 2 && window < 1)
        return GTMS_ERR_INVALID_ARG;
    return GTMS_OK;
}

template <typename T>
cudaError_t run_forward(int kind, int variant, const void* x, void* y, const int32_t* seq_lens, const gtms::Geom& g,
                        float scale, cudaStream_t st)
{
    switch (kind) {
    case 0: return gtms::launch_forward<T, 0>(variant, x, y, seq_lens, g, scale, st);
    case 1: return gtms::launch_forward<T, 1>(variant, x, y, seq_lens, g, scale, st);
    default: return gtms::launch_forward<T, 2>(variant, x, y, seq_lens, g, scale, st);
    }
}

template <typename T>
cudaError_t run_backward(int kind, int variant, const void* y, const void* dy, void* dx, const int32_t* seq_lens,
                         const gtms::Geom& g, float scale, cudaStream_t st)
{
    switch (kind) {
    case 0: return gtms::launch_backward<T, 0>(variant, y, dy, dx, seq_lens, g, scale, st);
    case 1: return gtms::launch_backward<T, 1>(variant, y, dy, dx, seq_lens, g, scale, st);
    default: return gtms::launch_backward<T, 2>(variant, y, dy, dx, seq_lens, g, scale, st);
    }
}

// Status of a launch from the launch call's own return value. A failed launch
// also leaves its error as the thread's last error, which is cleared here: it
// has been reported through the returned code.
int launch_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return GTMS_OK;
    cudaGetLastError();
    return GTMS_ERR_CUDA;
}

}  // namespace

GTMS_EXPORT int gtms_forward_masked(const void* x, void* y, const int32_t* seq_lens, int64_t B, int64_t M,
                                    int64_t S, float scale, int mask_kind, int64_t window, int dtype, void* stream)
{
    const Checked c = check_shape(B, M, S, scale, dtype);
    if (c.status != GTMS_OK)
        return c.status;
    const int mc = check_mask(mask_kind, window);
    if (mc != GTMS_OK || c.rows == 0)
        return mc;
    const int e = elem_bytes(dtype);
    if (!x || !y || !seq_lens)
        return GTMS_ERR_INVALID_ARG;
    if (!aligned_to(x, e) || !aligned_to(y, e) || !aligned_to(seq_lens, 4))
        return GTMS_ERR_INVALID_ARG;
    const uint64_t lens_bytes = static_cast<uint64_t>(B) * 4;
    if (bad_alias(y, x, c.bytes) || overlaps(y, c.bytes, seq_lens, lens_bytes))
        return GTMS_ERR_INVALID_ARG;

    const bool a16 = aligned_to(x, 16) && aligned_to(y, 16);
    const int band = mask_kind == GTMS_MASK_SLIDING_WINDOW ? gtms::pick_band_variant(0, S, e, a16, window) : -1;
    const int variant = band >= 0 ? band : gtms::pick_launch_variant(0, S, e, a16);
    if (variant < 0)
        return GTMS_ERR_UNSUPPORTED;
    const gtms::Geom g = make_geom(0, c.rows, M, S, variant, e, window);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case GTMS_F32: return launch_status(run_forward<float>(mask_kind, variant, x, y, seq_lens, g, scale, st));
    case GTMS_BF16: return launch_status(run_forward<__nv_bfloat16>(mask_kind, variant, x, y, seq_lens, g, scale, st));
    default: return launch_status(run_forward<__half>(mask_kind, variant, x, y, seq_lens, g, scale, st));
    }
}

GTMS_EXPORT int gtms_forward(const void* x, void* y, const int32_t* seq_lens, int64_t B, int64_t M, int64_t S,
                             float scale, int dtype, void* stream)
{
    return gtms_forward_masked(x, y, seq_lens, B, M, S, scale, GTMS_MASK_GROUPED_TRIL, 0, dtype, stream);
}

GTMS_EXPORT int gtms_forward_staged(const void* x, void* y, const int32_t* seq_lens, int64_t B, int64_t M,
                                    int64_t S, float scale, int dtype, void* stream)
{
    const Checked c = check_shape(B, M, S, scale, dtype);
    if (c.status != GTMS_OK || c.rows == 0)
        return c.status;
    const int e = elem_bytes(dtype);
    if (!x || !y || !seq_lens)
        return GTMS_ERR_INVALID_ARG;
    if (!aligned_to(x, e) || !aligned_to(y, e) || !aligned_to(seq_lens, 4))
        return GTMS_ERR_INVALID_ARG;
    if (bad_alias(y, x, c.bytes) || overlaps(y, c.bytes, seq_lens, static_cast<uint64_t>(B) * 4))
        return GTMS_ERR_INVALID_ARG;
    const int variant = gtms::pick_staged_variant(S, e, aligned_to(x, 16) && aligned_to(y, 16));
    if (variant < 0)
        return GTMS_ERR_UNSUPPORTED;
    gtms::Geom g;
    g.rows = c.rows;
    g.rows_per_b = M * S;
    g.S = static_cast<int32_t>(S);
    g.units = static_cast<int32_t>(S * e / 16);
    g.small = c.rows <= static_cast<int64_t>(UINT32_MAX) ? 1 : 0;
    g.window = static_cast<int32_t>(S);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case GTMS_F32: return launch_status(gtms::launch_forward_staged<float>(variant, x, y, seq_lens, g, scale, st));
    case GTMS_BF16:
        return launch_status(gtms::launch_forward_staged<__nv_bfloat16>(variant, x, y, seq_lens, g, scale, st));
    default: return launch_status(gtms::launch_forward_staged<__half>(variant, x, y, seq_lens, g, scale, st));
    }
}

GTMS_EXPORT int gtms_backward_masked(const void* y, const void* dy, void* dx, const int32_t* seq_lens, int64_t B,
                                     int64_t M, int64_t S, float scale, int mask_kind, int64_t window, int dtype,
                                     void* stream)
{
    const Checked c = check_shape(B, M, S, scale, dtype);
    if (c.status != GTMS_OK)
        return c.status;
    const int mc = check_mask(mask_kind, window);
    if (mc != GTMS_OK || c.rows == 0)
        return mc;
    const int e = elem_bytes(dtype);
    if (!y || !dy || !dx || !seq_lens)
        return GTMS_ERR_INVALID_ARG;
    if (!aligned_to(y, e) || !aligned_to(dy, e) || !aligned_to(dx, e) || !aligned_to(seq_lens, 4))
        return GTMS_ERR_INVALID_ARG;
    const uint64_t lens_bytes = static_cast<uint64_t>(B) * 4;
    if (bad_alias(dx, y, c.bytes) || bad_alias(dx, dy, c.bytes) || overlaps(dx, c.bytes, seq_lens, lens_bytes))
        return GTMS_ERR_INVALID_ARG;

    const bool a16 = aligned_to(y, 16) && aligned_to(dy, 16) && aligned_to(dx, 16);
    const int band = mask_kind == GTMS_MASK_SLIDING_WINDOW ? gtms::pick_band_variant(1, S, e, a16, window) : -1;
    const int variant = band >= 0 ? band : gtms::pick_launch_variant(1, S, e, a16);
    if (variant < 0)
        return GTMS_ERR_UNSUPPORTED;
    const gtms::Geom g = make_geom(1, c.rows, M, S, variant, e, window);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case GTMS_F32: return launch_status(run_backward<float>(mask_kind, variant, y, dy, dx, seq_lens, g, scale, st));
    case GTMS_BF16:
        return launch_status(run_backward<__nv_bfloat16>(mask_kind, variant, y, dy, dx, seq_lens, g, scale, st));
    default: return launch_status(run_backward<__half>(mask_kind, variant, y, dy, dx, seq_lens, g, scale, st));
    }
}

GTMS_EXPORT int gtms_backward(const void* y, const void* dy, void* dx, const int32_t* seq_lens, int64_t B, int64_t M,
                              int64_t S, float scale, int dtype, void* stream)
{
    return gtms_backward_masked(y, dy, dx, seq_lens, B, M, S, scale, GTMS_MASK_GROUPED_TRIL, 0, dtype, stream);
}

// Shared checks of the explicit-mask entry points: everything gtms_forward
// checks, plus the mask (non-null, 8-byte aligned, mask_batches 1 or B, no
// overlap with the output) and the 16-byte row layout the kernels need.
namespace {
int check_explicit(const Checked& c, int64_t B, int64_t S, int e, const uint8_t* mask, int64_t mask_batches,
                   const void* out, bool a16)
{
    if (!mask || (mask_batches != 1 && mask_batches != B) || !aligned_to(mask, 8))
        return GTMS_ERR_INVALID_ARG;
    const uint64_t mask_bytes = static_cast<uint64_t>(mask_batches) * S * S;
    if (overlaps(out, c.bytes, mask, mask_bytes))
        return GTMS_ERR_INVALID_ARG;
    if (!a16 || (S * e) % 16 != 0 || S > 8192)
        return GTMS_ERR_UNSUPPORTED;
    return GTMS_OK;
}
}  // namespace

GTMS_EXPORT int gtms_forward_explicit(const void* x, void* y, const uint8_t* mask, int64_t mask_batches, int64_t B,
                                      int64_t M, int64_t S, float scale, int dtype, void* stream)
{
    const Checked c = check_shape(B, M, S, scale, dtype);
    if (c.status != GTMS_OK || c.rows == 0)
        return c.status;
    const int e = elem_bytes(dtype);
    if (!x || !y || !aligned_to(x, e) || !aligned_to(y, e) || bad_alias(y, x, c.bytes))
        return GTMS_ERR_INVALID_ARG;
    const int ce = check_explicit(c, B, S, e, mask, mask_batches, y, aligned_to(x, 16) && aligned_to(y, 16));
    if (ce != GTMS_OK)
        return ce;
    const int variant = gtms::pick_variant(0, S, e, true, false);
    const gtms::Geom g = make_geom(0, c.rows, M, S, variant, e, 0);
    const int32_t mb = static_cast<int32_t>(mask_batches);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case GTMS_F32: return launch_status(gtms::launch_forward_explicit<float>(variant, x, y, mask, mb, g, scale, st));
    case GTMS_BF16:
        return launch_status(gtms::launch_forward_explicit<__nv_bfloat16>(variant, x, y, mask, mb, g, scale, st));
    default: return launch_status(gtms::launch_forward_explicit<__half>(variant, x, y, mask, mb, g, scale, st));
    }
}

GTMS_EXPORT int gtms_backward_explicit(const void* y, const void* dy, void* dx, const uint8_t* mask,
                                       int64_t mask_batches, int64_t B, int64_t M, int64_t S, float scale, int dtype,
                                       void* stream)
{
    const Checked c = check_shape(B, M, S, scale, dtype);
    if (c.status != GTMS_OK || c.rows == 0)
        return c.status;
    const int e = elem_bytes(dtype);
    if (!y || !dy || !dx || !aligned_to(y, e) || !aligned_to(dy, e) || !aligned_to(dx, e) ||
        bad_alias(dx, y, c.bytes) || bad_alias(dx, dy, c.bytes))
        return GTMS_ERR_INVALID_ARG;
    const bool a16 = aligned_to(y, 16) && aligned_to(dy, 16) && aligned_to(dx, 16);
    const int ce = check_explicit(c, B, S, e, mask, mask_batches, dx, a16);
    if (ce != GTMS_OK)
        return ce;
    const int variant = gtms::pick_variant(1, S, e, true, false);
    const gtms::Geom g = make_geom(1, c.rows, M, S, variant, e, 0);
    const int32_t mb = static_cast<int32_t>(mask_batches);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case GTMS_F32: return launch_status(gtms::launch_backward_explicit<float>(variant, y, dy, dx, mask, mb, g, scale, st));
    case GTMS_BF16:
        return launch_status(gtms::launch_backward_explicit<__nv_bfloat16>(variant, y, dy, dx, mask, mb, g, scale, st));
    default: return launch_status(gtms::launch_backward_explicit<__half>(variant, y, dy, dx, mask, mb, g, scale, st));
    }
}

GTMS_EXPORT int gtms_attention_softmax_backward(const void* p, const void* dout, const void* v, void* ds,
                                                const int32_t* seq_lens, int64_t B, int64_t M, int64_t S,
                                                int64_t head_dim, float scale, int dtype, int32_t* status,
                                                void* stream)
{
    const Checked c = check_shape(B, M, S, scale, dtype);
    if (c.status != GTMS_OK)
        return c.status;
    if (head_dim < 0)
        return GTMS_ERR_INVALID_ARG;
    if (dtype == GTMS_F32 || (head_dim != 64 && head_dim != 128) || S % 8 != 0)
        return GTMS_ERR_UNSUPPORTED;
    if (c.rows == 0)
        return GTMS_OK;
    const int64_t nrb = (S + 127) / 128;
    if (B * M > INT32_MAX / nrb)
        return GTMS_ERR_UNSUPPORTED;
    if (!p || !dout || !v || !ds || !seq_lens)
        return GTMS_ERR_INVALID_ARG;
    if (!aligned_to(p, 16) || !aligned_to(dout, 16) || !aligned_to(v, 16) || !aligned_to(ds, 16) ||
        !aligned_to(seq_lens, 4) || (status && !aligned_to(status, 4)))
        return GTMS_ERR_INVALID_ARG;
    const uint64_t ob = static_cast<uint64_t>(B) * M * S * head_dim * 2;   // dO and V bytes
    if (bad_alias(ds, p, c.bytes) || overlaps(ds, c.bytes, dout, ob) || overlaps(ds, c.bytes, v, ob) ||
        overlaps(ds, c.bytes, seq_lens, static_cast<uint64_t>(B) * 4) || (status && overlaps(ds, c.bytes, status, 4)))
        return GTMS_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Operands in device memory take the TMA-fed persistent kernel; any in
    // mapped host memory, the kernel that copies with cp.async.
    const bool tma = in_device_memory(p) && in_device_memory(dout) && in_device_memory(v) && in_device_memory(ds);
    cudaError_t e;
    if (dtype == GTMS_BF16) {
        if (tma)
            e = head_dim == 64 ? gtms::launch_attn_dscores_tma<__nv_bfloat16, 64>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs)
                               : gtms::launch_attn_dscores_tma<__nv_bfloat16, 128>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs);
        else
            e = head_dim == 64 ? gtms::launch_attn_dscores<__nv_bfloat16, 64>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs)
                               : gtms::launch_attn_dscores<__nv_bfloat16, 128>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs);
    } else {
        if (tma)
            e = head_dim == 64 ? gtms::launch_attn_dscores_tma<__half, 64>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs)
                               : gtms::launch_attn_dscores_tma<__half, 128>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs);
        else
            e = head_dim == 64 ? gtms::launch_attn_dscores<__half, 64>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs)
                               : gtms::launch_attn_dscores<__half, 128>(p, dout, v, ds, seq_lens, B, M, S, scale, status, st, gtms::kAttnWaitNs);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GTMS_ERR_CUDA;
    }
    return GTMS_OK;
}

GTMS_EXPORT int gtms_device_pointer_of_host(const void* host, void** device)
{
    if (!host || !device)
        return GTMS_ERR_INVALID_ARG;
    void* d = nullptr;
    const cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void*>(host), 0);
    if (e == cudaErrorInvalidValue) {
        cudaGetLastError();
        return GTMS_ERR_INVALID_ARG;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GTMS_ERR_CUDA;
    }
    *device = d;
    return GTMS_OK;
}

GTMS_EXPORT const char* gtms_status_string(int status)
{
    switch (status) {
    case GTMS_OK: return "GTMS_OK";
    case GTMS_ERR_INVALID_ARG: return "GTMS_ERR_INVALID_ARG";
    case GTMS_ERR_UNSUPPORTED: return "GTMS_ERR_UNSUPPORTED";
    case GTMS_ERR_CUDA: return "GTMS_ERR_CUDA";
    case GTMS_ERR_TIMEOUT: return "GTMS_ERR_TIMEOUT";
    default: return "GTMS_UNKNOWN_STATUS";
    }
}

GTMS_EXPORT int gtms_version(void) { return GTMS_VERSION; }

namespace {

// Names of every kernel variant, filled once (thread-safe static init):
// [direction][dtype][mask kind][slot], slot = table row + kSlots * family
// (per-row vector, element, stream, band, heads). Mask kinds 1 and 2 append
// ",maskK".
struct KernelNames {
    static constexpr int kSlots = 16;
    char text[2][3][3][5 * kSlots][96];

    KernelNames()
    {
        static const char* const kDtype[3] = {"f32", "bf16", "f16"};
        for (int d = 0; d < 2; ++d)
            for (int t = 0; t < 3; ++t)
                for (int mk = 0; mk < 3; ++mk) {
                    char suffix[16] = "";
                    if (mk != 0)
                        std::snprintf(suffix, sizeof suffix, ",mask%d", mk);
                    const char* dir = d == 0 ? "fwd" : "bwd";
                    const int e = t == 0 ? 4 : 2;
                    const gtms::VariantTable vt = gtms::vec_table(d, e);
                    for (int i = 0; i < vt.count && i < kSlots; ++i)
                        std::snprintf(text[d][t][mk][i], 96, "gtms_%s_vec_kernel<%s,team%d,x%d,minb%d%s>", dir,
                                      kDtype[t], vt.rows[i].team, vt.rows[i].per_thread, vt.rows[i].min_ctas, suffix);
                    for (int i = 0; i < gtms::count_of(gtms::kElem) && i < kSlots; ++i)
                        std::snprintf(text[d][t][mk][kSlots + i], 96, "gtms_%s_elem_kernel<%s,team%d,x%d%s>", dir,
                                      kDtype[t], gtms::kElem[i].team, gtms::kElem[i].per_thread, suffix);
                    const gtms::VariantTable st = gtms::stream_table(d, e);
                    for (int i = 0; i < st.count && i < kSlots; ++i)
                        std::snprintf(text[d][t][mk][2 * kSlots + i], 96, "gtms_%s_stream_kernel<%s,team%d,x%d,minb%d%s>",
                                      dir, kDtype[t], st.rows[i].team, st.rows[i].per_thread, st.rows[i].min_ctas,
                                      suffix);
                    const gtms::VariantTable ht = gtms::heads_table();
                    for (int i = 0; i < ht.count && gtms::kFwdHeads2Ids[i] < kSlots; ++i)
                        std::snprintf(text[d][t][mk][4 * kSlots + gtms::kFwdHeads2Ids[i]], 96,
                                      "gtms_%s_heads_kernel<%s,team%d,x%d,minb%d%s>", dir, kDtype[t], ht.rows[i].team,
                                      ht.rows[i].per_thread, ht.rows[i].min_ctas, suffix);
                    const gtms::VariantTable bt = gtms::band_table(d);
                    for (int i = 0; i < bt.count && i < kSlots; ++i)
                        std::snprintf(text[d][t][mk][3 * kSlots + i], 96, "gtms_%s_band_kernel<%s,x%d,minb%d>", dir,
                                      kDtype[t], bt.rows[i].per_thread, bt.rows[i].min_ctas);
                }
    }

    const char* of(int direction, int dtype, int mask_kind, int variant) const
    {
        int slot;
        if (variant >= gtms::kHeadsBase)
            slot = 4 * kSlots + variant - gtms::kHeadsBase;
        else if (variant >= gtms::kBandBase)
            slot = 3 * kSlots + variant - gtms::kBandBase;
        else if (variant >= gtms::kStreamBase)
            slot = 2 * kSlots + variant - gtms::kStreamBase;
        else if (variant >= gtms::kElemBase)
            slot = kSlots + variant - gtms::kElemBase;
        else
            slot = variant;
        return text[direction][dtype][mask_kind][slot];
    }
};

const KernelNames& kernel_names()
{
    static const KernelNames names;
    return names;
}

}  // namespace

GTMS_EXPORT const char* gtms_kernel_name(int direction, int64_t S, int dtype, int aligned16)
{
    if (direction == 2) {   // gtms_forward_staged
        static const char* const kDtype[3] = {"f32", "bf16", "f16"};
        struct Names {
            char text[3][8][80];
            Names()
            {
                for (int t = 0; t < 3; ++t)
                    for (int i = 0; i < 3; ++i) {
                        const gtms::StagedVariant v = gtms::staged_at(t == 0 ? 4 : 2, i);
                        std::snprintf(text[t][i], sizeof text[t][i], "gtms_fwd_staged_kernel<%s,team%d,x%d,slots%d,minb%d>",
                                      kDtype[t], v.team, v.per_thread, v.slots, v.min_ctas);
                    }
            }
        };
        static const Names names;
        const int e = elem_bytes(dtype);
        const int v = e == 0 ? -1 : gtms::pick_staged_variant(S, e, aligned16 != 0);
        return v < 0 ? "none" : names.text[dtype][v];
    }
    return gtms_kernel_name_masked(direction, S, dtype, aligned16, GTMS_MASK_GROUPED_TRIL, 0);
}

GTMS_EXPORT const char* gtms_kernel_name_masked(int direction, int64_t S, int dtype, int aligned16, int mask_kind,
                                                int64_t window)
{
    const int e = elem_bytes(dtype);
    if ((direction != 0 && direction != 1) || e == 0 || S < 1 || S > GTMS_MAX_S || check_mask(mask_kind, window))
        return "none";
    int v = mask_kind == GTMS_MASK_SLIDING_WINDOW ? gtms::pick_band_variant(direction, S, e, aligned16 != 0, window)
                                                  : -1;
    if (v < 0)
        v = gtms::pick_launch_variant(direction, S, e, aligned16 != 0);
    return v < 0 ? "none" : kernel_names().of(direction, dtype, mask_kind, v);
}

GTMS_EXPORT const char* gtms_kernel_name_explicit(int direction, int64_t S, int dtype)
{
    static const char* const kDtype[3] = {"f32", "bf16", "f16"};
    constexpr int kMaxRows = 16;
    struct Names {
        char text[2][3][kMaxRows][80];
        Names()
        {
            for (int d = 0; d < 2; ++d)
                for (int t = 0; t < 3; ++t) {
                    const gtms::VariantTable vt = gtms::explicit_table(d, t == 0 ? 4 : 2);
                    for (int i = 0; i < vt.count && i < kMaxRows; ++i)
                        std::snprintf(text[d][t][i], sizeof text[d][t][i],
                                      "gtms_%s_explicit_kernel<%s,team%d,x%d,minb%d>", d == 0 ? "fwd" : "bwd",
                                      kDtype[t], vt.rows[i].team, vt.rows[i].per_thread, vt.rows[i].min_ctas);
                }
        }
    };
    static const Names names;
    const int e = elem_bytes(dtype);
    if ((direction != 0 && direction != 1) || e == 0 || S < 1 || S > 8192 || (S * e) % 16 != 0)
        return "none";
    const int v = gtms::pick_variant(direction, S, e, true, false);
    return v < 0 || v >= kMaxRows ? "none" : names.text[direction][dtype][v];
}
