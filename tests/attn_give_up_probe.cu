// Test-only library (built by tests/test_parity_gpu.py, never part of libgtms):
// the TMA-fed attention-backward kernel compiled with GTMS_ATTN_TMA_NO_LOADS, so
// its producer issues no copies. No consumer wait can then complete: each runs
// out after `wait_ns` nanoseconds, and the kernel must record GTMS_ERR_TIMEOUT in
// the status word, leave its loops, free its tensor memory and return.
#define GTMS_ATTN_TMA_NO_LOADS 1
#include "gtms_attn_tma.cuh"

extern "C" __attribute__((visibility("default"))) int gtms_test_attn_no_loads(
    const void* p, const void* dout, const void* v, void* ds, const int32_t* seq_lens, int64_t B, int64_t M,
    int64_t S, float scale, int32_t* status, void* stream, uint64_t wait_ns)
{
    const cudaError_t e = gtms::launch_attn_dscores_tma<__nv_bfloat16, 64>(
        p, dout, v, ds, seq_lens, B, M, S, scale, status, static_cast<cudaStream_t>(stream), wait_ns);
    return e == cudaSuccess ? 0 : static_cast<int>(e);
}
