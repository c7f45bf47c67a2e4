// Self-test of the bounded mbarrier wait that every tensor-core kernel uses:
// one warp whose lane 0 waits on a barrier that completes only if `arrive` is
// set.  Otherwise the wait runs out after `limit` cycles and sets this file's
// status word, which opam_device_status reports as a timeout.  Nothing here
// can hang or fault: the wait is bounded and the kernel touches only its own
// shared memory.
#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

__device__ unsigned int g_status = 0;
constexpr unsigned int kStSelfTest = 1u;  // the wait ran out

__global__ void bounded_wait_selftest_kernel(int arrive, long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        if (arrive) mbar_arrive(&bar);
        if (!mbar_wait_for(&bar, 0, limit)) atomicOr(&g_status, kStSelfTest);
    }
    __syncwarp();
}

}  // namespace

int bounded_wait_selftest(int arrive, long long limit, cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(arrive, limit);
    return launched("bounded_wait_selftest");
}

unsigned int bounded_wait_selftest_status(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (clear && v) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_status, &z, sizeof z);
    }
    return v;
}

}  // namespace opam
