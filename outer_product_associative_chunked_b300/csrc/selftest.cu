// Self-test of the bounded mbarrier wait that every tensor-core kernel uses:
// one warp whose lane 0 waits on a barrier that completes only if `arrive` is
// set.  Otherwise the wait runs out after `limit` cycles and sets a bit in the
// caller's status word (the head of the workspace it was given), which
// opam_check_device_error reports as a timeout.  Nothing here can hang or
// fault: the wait is bounded and the kernel touches only its own shared
// memory and that one word.
#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

__global__ void bounded_wait_selftest_kernel(int arrive, long long limit, unsigned int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        if (arrive) mbar_arrive(&bar);
        if (!mbar_wait_for(&bar, 0, limit)) atomicOr(status, kStatusSelfTest);
    }
    __syncwarp();
}

// Every thread checks threadIdx.x < n through the debug-bounds index check;
// with n below the block size some checks fail, which in a debug-bounds
// build sets kStatusBounds (and in a normal build does nothing).  No memory
// is accessed either way.
__global__ void bounds_selftest_kernel(int n, unsigned int *status) {
    if (OPAM_BOUNDS(threadIdx.x < (unsigned)n, status)) {
    }
}

}  // namespace

int bounds_selftest(int n, unsigned int *status, cudaStream_t s) {
    bounds_selftest_kernel<<<1, 32, 0, s>>>(n, status);
    return launched("bounds_selftest");
}

int bounded_wait_selftest(int arrive, long long limit, unsigned int *status, cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(arrive, limit, status);
    return launched("bounded_wait_selftest");
}

}  // namespace opam
