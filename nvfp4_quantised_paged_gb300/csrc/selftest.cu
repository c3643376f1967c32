// selftest.cu -- exercises the bounded-wait failure path of the kernels on the GPU.
//
// The decode kernel waits on mbarriers that bulk copies complete; if a copy
// never completed, the wait gives up after its poll limit, records
// kErrTimeout in the device error word and the kernel returns, leaving the
// context usable.  That path cannot be reached with real copies without
// breaking the hardware, so this kernel reproduces it with a barrier that
// nothing completes: it uses the same wait routine and the same error word.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4kv {

namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int arrive, uint32_t poll_limit, int *result,
                                                          unsigned *err) {
    __shared__ uint64_t bar;
    const int lane = threadIdx.x;
    if (lane == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (arrive && lane == 0) mbar_arrive(&bar);  // completes phase 0
    __syncwarp();
    const bool ok = mbar_wait_bounded(&bar, 0, poll_limit, nullptr);
    if (lane == 0) {
        *result = ok ? 0 : 1;
        if (!ok) flag_error(err, kErrTimeout);
    }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int arrive, uint32_t poll_limit, int *result, unsigned *err,
                                         cudaStream_t stream) {
    bounded_wait_kernel<<<1, 32, 0, stream>>>(arrive, poll_limit, result, err);
    return cudaGetLastError();
}

}  // namespace nvfp4kv
