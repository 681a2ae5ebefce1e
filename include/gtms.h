/*
 * gtms.h -- C ABI of libgtms: the grouped-tril masked softmax over attention
 * scores, forward and backward, as hand-written CUDA kernels for sm_103a.
 *
 * The operation ("Attention-Mask-Optimization" README, section
 * "算子行为（融合下面的计算）", operator behaviour, and its printed worked
 * example): X is a contiguous row-major [B, M, S, S] tensor of attention
 * scores (B batches, M heads, S x S scores per head). For batch b with
 * valid length L = seq_lens[b], entry (r, c) is kept iff r < L, c < L and
 * c <= r; the same mask applies to every head. The kept entries of each row
 * are passed through a softmax of scale * x ("优化ScaledMaskSoftmax算子",
 * section 4.1: the scale sits inside the exponent); every masked entry is
 * written as +0.0, and rows r >= L are all +0.0. The mask is computed from
 * (r, c, seq_lens[b]) inside the kernel and never read from memory (the
 * README's implementation idea, "实现思路"); masked inputs are never loaded.
 *
 * The backward ("ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1,
 * Softmax 求导: dy_i/dx_j = y_i (delta_ij - y_j); section 2.2 applies the scale
 * in the softmax backward) is dx = scale * y * (dy - rowsum(dy * y)) on kept
 * entries and +0.0 on masked ones.
 *
 * Values of seq_lens outside [0, S] are clamped to that range in the kernel.
 * Arithmetic is fp32 for every IO dtype; outputs are rounded to the IO dtype
 * to nearest, ties to even.
 *
 * Ownership and threading. The caller owns every buffer. All tensor
 * pointers are addresses the current CUDA device can dereference: device
 * memory, or page-locked host memory mapped with gtms_device_pointer_of_host;
 * seq_lens is an int32[B] array in such memory. The library allocates
 * nothing, keeps no per-call state, is safe to call from several host
 * threads, and never synchronises: work is enqueued on `stream` (a
 * cudaStream_t passed as void*; NULL is the legacy default stream) and the
 * call returns at once. The host never reads seq_lens.
 *
 * Aliasing. Outputs may alias an input exactly (y == x; dx == dy or
 * dx == y): each row is read before that row is written. Partial overlap of
 * an output with any input, or of seq_lens with an output, is rejected.
 *
 * Errors are returned, never raised, trapped or printed:
 *   GTMS_OK              work enqueued (or nothing to do: B*M*S == 0).
 *   GTMS_ERR_INVALID_ARG null pointer with B*M*S > 0, B/M/S < 0, a size whose
 *                        byte count overflows, a non-finite scale, a pointer
 *                        not aligned to its element size, partial overlap.
 *   GTMS_ERR_UNSUPPORTED unknown dtype; S > GTMS_MAX_S; or S > 8192 with a row
 *                        whose byte length is not a multiple of 16 or a buffer
 *                        that is not 16-byte aligned (long rows are streamed
 *                        in 16-byte units only).
 *   GTMS_ERR_CUDA        the kernel launch failed (the status the launch call
 *                        itself returned; an error left behind by earlier,
 *                        unrelated work on the thread is not reported here).
 *   GTMS_ERR_TIMEOUT     never returned by a call, which returns before its
 *                        kernel runs: it is the code that the attention step's
 *                        kernel writes into the caller's status word when one of
 *                        its bounded internal waits ran out (see
 *                        gtms_attention_softmax_backward).
 * All argument checks run on the host before anything is enqueued; a call
 * that returns an error has enqueued nothing.
 */
#ifndef GTMS_H
#define GTMS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GTMS_VERSION 1
#define GTMS_MAX_S 65536

typedef enum { GTMS_F32 = 0, GTMS_BF16 = 1, GTMS_F16 = 2 } gtms_dtype;

/*
 * Mask families ("优化ScaledMaskSoftmax算子", section 6, lists a local window
 * mask and a length mask next to the default). Each keeps a contiguous column
 * range of a row r < L = clamp(seq_lens[b], 0, S) and nothing of rows r >= L:
 *   GTMS_MASK_GROUPED_TRIL   c <= r                (the operator above)
 *   GTMS_MASK_LENGTH         c < L                 (padded keys and queries)
 *   GTMS_MASK_SLIDING_WINDOW r - window < c <= r   (causal band, window >= 1;
 *                            the section's garbled local-window snippet is read
 *                            as this band)
 */
typedef enum {
    GTMS_MASK_GROUPED_TRIL = 0,
    GTMS_MASK_LENGTH = 1,
    GTMS_MASK_SLIDING_WINDOW = 2
} gtms_mask_kind;

typedef enum {
    GTMS_OK = 0,
    GTMS_ERR_INVALID_ARG = 1,
    GTMS_ERR_UNSUPPORTED = 2,
    GTMS_ERR_CUDA = 3,
    GTMS_ERR_TIMEOUT = 4
} gtms_status;

/*
 * Forward: y = grouped-tril masked softmax(scale * x).
 *   x        device, [B, M, S, S] of `dtype`, read-only; only the kept prefix
 *            x[b, m, r, 0 : min(r + 1, L)] of rows r < L is loaded.
 *   y        device, [B, M, S, S] of `dtype`, every element written.
 *   seq_lens device, int32[B].
 *   scale    finite float, applied inside the exponent.
 *   dtype    gtms_dtype of x and y.
 *   stream   cudaStream_t or NULL.
 */
int gtms_forward(const void* x, void* y, const int32_t* seq_lens,
                 int64_t B, int64_t M, int64_t S, float scale, int dtype, void* stream);

/*
 * Backward: dx = scale * y * (dy - rowsum(dy * y)) under the same mask.
 *   y, dy    device, [B, M, S, S] of `dtype`, read-only (y is the forward
 *            output); only the kept prefix of each live row is loaded.
 *   dx       device, [B, M, S, S] of `dtype`, every element written.
 *   Other arguments as in gtms_forward.
 */
int gtms_backward(const void* y, const void* dy, void* dx, const int32_t* seq_lens,
                  int64_t B, int64_t M, int64_t S, float scale, int dtype, void* stream);

/*
 * gtms_forward computed by the staged kernel: the block-per-row design of
 * "优化ScaledMaskSoftmax算子" (sections 2.2 and 4.2: a thread block per row,
 * the row staged in shared memory), with each live row's kept units brought
 * into shared memory by one TMA bulk copy, several rows ahead of the row being
 * reduced. Same operation, arguments and errors as gtms_forward, and the same
 * output values within the parity tolerances. On GB300 it measured slower than
 * gtms_forward (S = 2048 bf16: 5.6 against 6.4 TB/s), which stays the fast
 * path; this entry point is kept for comparison and for other parts.
 * GTMS_ERR_UNSUPPORTED beyond gtms_forward's cases: rows whose byte length is
 * not a multiple of 16 or is 32 KB or more, buffers not 16-byte aligned.
 * A copy that does not arrive within 1 s of GPU time is given up on: the row is
 * then read straight from x (same result), never waited on forever.
 */
int gtms_forward_staged(const void* x, void* y, const int32_t* seq_lens,
                        int64_t B, int64_t M, int64_t S, float scale, int dtype, void* stream);

/*
 * Device address of a page-locked host buffer (allocated with cudaHostAlloc
 * or registered with cudaHostRegister), for passing host-resident tensors
 * straight to gtms_forward / gtms_backward: the kernels then read the kept
 * inputs from, and write every output to, host memory over the host link
 * (NVLink-C2C on Grace-Blackwell), with no staging copy.
 *   host     pointer into a page-locked host allocation.
 *   device   out: the address the current device uses for it.
 * Returns GTMS_ERR_INVALID_ARG for null arguments or for memory the CUDA
 * runtime cannot map for the current device, GTMS_ERR_CUDA for other runtime
 * errors. (Where the device reads pageable host memory through the host's page
 * tables, as on Grace-Blackwell, the runtime maps pageable memory as well;
 * page-locked memory is still what the transfer rate assumes.) Host-only,
 * enqueues nothing, allocates nothing.
 */
int gtms_device_pointer_of_host(const void* host, void** device);

/*
 * gtms_forward / gtms_backward with another mask family (gtms_mask_kind).
 * `window` is the band width of GTMS_MASK_SLIDING_WINDOW (>= 1; widths >= S
 * give the grouped-tril op) and is ignored by the other kinds. An unknown kind
 * is GTMS_ERR_UNSUPPORTED, a sliding window narrower than 1
 * GTMS_ERR_INVALID_ARG; everything else is as for gtms_forward / gtms_backward
 * (gtms_forward is gtms_forward_masked with GTMS_MASK_GROUPED_TRIL).
 */
int gtms_forward_masked(const void* x, void* y, const int32_t* seq_lens, int64_t B, int64_t M, int64_t S,
                        float scale, int mask_kind, int64_t window, int dtype, void* stream);
int gtms_backward_masked(const void* y, const void* dy, void* dx, const int32_t* seq_lens, int64_t B, int64_t M,
                         int64_t S, float scale, int mask_kind, int64_t window, int dtype, void* stream);

/*
 * Masked softmax with an explicit keep mask ("优化ScaledMaskSoftmax算子",
 * sections 2.2 and 3.1: input, mask, scale; section 4.1: a row with nothing
 * kept is zero). y[b, m, r, c] = softmax over {c' : mask[b', r, c'] != 0} of
 * scale * x[b, m, r, c'] at kept entries, +0.0 elsewhere; b' = 0 when
 * mask_batches == 1, else b. The backward is dx = scale * y * (dy - rowsum(dy * y))
 * over the same kept set.
 *   mask         device uint8 [mask_batches, S, S], 8-byte aligned, read-only,
 *                shared by the M heads; nonzero = keep.
 *   mask_batches 1 or B.
 * Masked inputs are not loaded: each 16-byte unit of x (or of y and dy) is
 * read only if its mask bytes keep at least one element.
 * GTMS_ERR_INVALID_ARG also covers a null or misaligned mask, mask_batches
 * other than 1 or B, and a mask overlapping the output. GTMS_ERR_UNSUPPORTED:
 * S > 8192, rows that are not 16-byte multiples, or buffers not 16-byte aligned.
 */
int gtms_forward_explicit(const void* x, void* y, const uint8_t* mask, int64_t mask_batches, int64_t B, int64_t M,
                          int64_t S, float scale, int dtype, void* stream);
int gtms_backward_explicit(const void* y, const void* dy, void* dx, const uint8_t* mask, int64_t mask_batches,
                           int64_t B, int64_t M, int64_t S, float scale, int dtype, void* stream);

/*
 * Attention-backward step around the masked softmax, fused with its GEMM on the
 * tensor cores ("ops(8): self-attention 的 CUDA 实现及优化 (下)", section 2.1: with
 * P the softmax output, O = P V and upstream gradient dO, the backward forms
 * dP = dO V^T and then the softmax backward of dP):
 *   dS[b,m,r,c] = scale * P[b,m,r,c] * (dP[r,c] - sum_c' dP[r,c'] P[b,m,r,c'])
 * on the grouped-tril kept entries (c <= r < L), +0.0 elsewhere, with
 * dP[r,c] = sum_k dO[b,m,r,k] V[b,m,c,k] accumulated in fp32 and never
 * written to memory.
 *   p        [B,M,S,S] of `dtype` (the forward output), read-only. Masked
 *            entries are never used (NaN there does not reach ds); tiles
 *            right of the diagonal and padded row blocks are not read.
 *   dout, v  [B,M,S,head_dim] of `dtype`, read-only.
 *   ds       [B,M,S,S] of `dtype`, every element written; may equal p.
 * The four tensors are device-addressable: when all four are device memory
 * the call runs a persistent TMA-fed kernel (one CTA per SM); otherwise
 * (mapped page-locked host memory, see gtms_device_pointer_of_host) a kernel
 * that copies with cp.async and reads P only in 16-byte units that hold a
 * kept entry.
 *   seq_lens device int32[B]; scale finite.
 *   head_dim 64 or 128; dtype GTMS_BF16 or GTMS_F16; S a multiple of 8.
 *   status   NULL, or a device-addressable int32 that the kernel ORs
 *            GTMS_ERR_TIMEOUT into when one of its internal waits (a hand-off
 *            between its warps, each bounded to 1 s of GPU time) ran out; the
 *            kernel then stops early and its results are incomplete. The
 *            caller clears the word before the call and reads it after
 *            synchronising with `stream`: 0, or GTMS_ERR_TIMEOUT.
 * All pointers 16-byte aligned (status 4-byte). GTMS_ERR_UNSUPPORTED: fp32,
 * other head dims, S not a multiple of 8, S > GTMS_MAX_S. Otherwise as
 * gtms_backward.
 */
int gtms_attention_softmax_backward(const void* p, const void* dout, const void* v, void* ds, const int32_t* seq_lens,
                                    int64_t B, int64_t M, int64_t S, int64_t head_dim, float scale, int dtype,
                                    int32_t* status, void* stream);

/* Static, NUL-terminated name of a status code ("GTMS_OK", ...). */
const char* gtms_status_string(int status);

/* GTMS_VERSION of the built library. */
int gtms_version(void);

/*
 * Name of the kernel variant that gtms_forward (direction 0), gtms_backward
 * (direction 1) or gtms_forward_staged (direction 2) launches for this row
 * length, dtype and alignment (aligned16 != 0: every pointer is 16-byte
 * aligned). Static string; "none" for unsupported arguments. Host-only,
 * enqueues nothing.
 */
const char* gtms_kernel_name(int direction, int64_t S, int dtype, int aligned16);

/*
 * Name of the kernel variant that gtms_forward_masked (direction 0) or
 * gtms_backward_masked (direction 1) launches for this row length, dtype,
 * alignment, mask kind and window. Mask kinds 1 and 2 append ",maskK" to the
 * per-row kernel's name; a narrow sliding window may take a band kernel
 * instead. Static string; "none" for unsupported arguments. Host-only,
 * enqueues nothing.
 */
const char* gtms_kernel_name_masked(int direction, int64_t S, int dtype, int aligned16, int mask_kind,
                                    int64_t window);

/*
 * Name of the kernel variant that gtms_forward_explicit (direction 0) or
 * gtms_backward_explicit (direction 1) launches for this row length and dtype
 * (16-byte-aligned buffers). Static string; "none" for arguments those calls
 * reject. Host-only, enqueues nothing.
 */
const char* gtms_kernel_name_explicit(int direction, int64_t S, int dtype);

#ifdef __cplusplus
}
#endif

#endif /* GTMS_H */
