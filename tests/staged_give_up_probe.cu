// Test-only library (built by tests/test_parity_gpu.py, never part of libgtms):
// the staged forward compiled with GTMS_STAGED_NO_COPIES, so that no bulk copy is
// ever issued. Every wait for a row's slot then runs out after `wait_ns`
// nanoseconds, the team gives up on staging and reads the rows from global
// memory: the output must still be exact, and the kernel must end.
#define GTMS_STAGED_NO_COPIES 1
#include "gtms_dispatch.h"
#include "gtms_staged.cuh"

extern "C" __attribute__((visibility("default"))) int gtms_test_staged_no_copies(
    const void* x, void* y, const int32_t* seq_lens, int64_t B, int64_t M, int64_t S, float scale, int dtype,
    void* stream, uint64_t wait_ns)
{
    const int e = dtype == 0 ? 4 : 2;
    gtms::Geom g;
    g.rows = B * M * S;
    g.rows_per_b = M * S;
    g.S = static_cast<int32_t>(S);
    g.units = static_cast<int32_t>(S * e / 16);
    g.small = 1;
    g.window = static_cast<int32_t>(S);
    if (gtms::pick_staged_variant(S, e, true) != 0)
        return -1;   // the probe instantiates the first table row only
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t r;
    switch (dtype) {
    case 0: r = gtms::launch_fwd_staged<float, gtms::kMaskGroupedTril, 64, 4, 6, 12>(x, y, seq_lens, g, scale, st, wait_ns); break;
    case 1: r = gtms::launch_fwd_staged<__nv_bfloat16, gtms::kMaskGroupedTril, 64, 4, 2, 10>(x, y, seq_lens, g, scale, st, wait_ns); break;
    default: r = gtms::launch_fwd_staged<__half, gtms::kMaskGroupedTril, 64, 4, 2, 10>(x, y, seq_lens, g, scale, st, wait_ns); break;
    }
    return r == cudaSuccess ? 0 : static_cast<int>(r);
}
