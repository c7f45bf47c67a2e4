// Tensor Cache prefill for callers that cannot allocate device memory.
//
// Some hosts hand a library only the input and output buffers and do not let
// it allocate: plugins inside an application that owns every byte of device
// memory through its own allocator, and services that forbid allocation
// after start-up because cudaMalloc can block, synchronise the device or fail
// once the memory pool is reserved.  tc_layer_forward needs scratch memory
// (the per-chunk L2 states), which its caller normally passes in.  This entry
// point takes that scratch from a fixed array compiled into the library
// instead, so the caller passes inputs and outputs only and nothing is
// allocated during the call.
//
// Properties a caller must know:
//  - The array below is OPAM_STATIC_SCRATCH_BYTES long and lives on every
//    GPU that loads this library, for as long as the process runs.
//  - Problems whose scratch need (tc_layer_forward_workspace_size) exceeds it
//    are rejected with OPAM_ERR_WORKSPACE and a message naming both sizes.
//  - The first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make
//    that first call before any stream capture.
//  - All calls on a device share the one array, and it keeps the previous
//    call's contents.  Every kernel writes each scratch element before it
//    reads it, so stale contents never reach a result; but calls that
//    overlap on the GPU (different streams, or different host threads)
//    race on the array and must be serialised by the caller.
#include <mutex>

#include "opam_internal.cuh"

namespace {

// Host code sees only a stand-in for this symbol: its device address comes
// from cudaGetSymbolAddress, never from taking &g_static_scratch on the host.
static __device__ __align__(256) unsigned char g_static_scratch[OPAM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the static scratch on the current device (set up once).
int static_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return opam::cuda_fail(e, "tc_layer_forward_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        opam::set_error("tc_layer_forward_noalloc: device %d above the supported %d", dev, kMaxDevices);
        return OPAM_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return opam::cuda_fail(e, "tc_layer_forward_noalloc: cudaGetSymbolAddress");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return OPAM_OK;
}

}  // namespace

extern "C" int tc_layer_forward_noalloc(const void *q, const void *k, const void *v, int dtype, int B,
                                        int H, int T, int d_k, int d_v, int W, const float *lambda,
                                        const float *eta, const float *gate, float softmax_scale,
                                        void *y, opam_tc_state *state_out, void *stream) {
    const size_t need = tc_layer_forward_workspace_size(B, H, T, d_k, d_v, W, dtype);
    if (need > (size_t)OPAM_STATIC_SCRATCH_BYTES) {
        opam::set_error(
            "tc_layer_forward_noalloc: this problem needs %zu bytes of scratch but the built-in "
            "scratch holds %zu; call tc_layer_forward with a caller-provided workspace instead",
            need, (size_t)OPAM_STATIC_SCRATCH_BYTES);
        return OPAM_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    if (need > 0)  // need == 0: invalid arguments, reported by tc_layer_forward below
        if (int rc = static_scratch(&scratch)) return rc;
    return tc_layer_forward(q, k, v, dtype, B, H, T, d_k, d_v, W, lambda, eta, gate, softmax_scale, y,
                            state_out, scratch, (size_t)OPAM_STATIC_SCRATCH_BYTES, stream);
}
