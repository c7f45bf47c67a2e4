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
//  - A call made outside stream capture looks up the array's device address
//    (cudaGetSymbolAddress, with the call's device current) and remembers it
//    per device; a call under stream capture uses the remembered address.
//    So the first call on each device, and the first after a device reset
//    (which reloads the module and may move the array), must come before any
//    capture.
//  - All calls on a device share the one array, and it keeps the previous
//    call's contents.  The head of the array is the call's status block,
//    which the call zeroes first; every kernel writes each other scratch
//    element before it reads it, so stale contents never reach a result.
//    Calls that overlap on the GPU (different streams, or different host
//    threads) race on the array and must be serialised by the caller.
#include <mutex>

#include "opam_internal.cuh"

namespace {

// Host code sees only a stand-in for this symbol: its device address comes
// from cudaGetSymbolAddress, never from taking &g_static_scratch on the host.
static __device__ __align__(256) unsigned char g_static_scratch[OPAM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int current_device(int *dev, const char *fn) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return opam::cuda_fail(e, fn);
    if (*dev < 0 || *dev >= kMaxDevices) {
        opam::set_error("%s: device %d above the supported %d", fn, *dev, kMaxDevices);
        return OPAM_ERR_UNSUPPORTED;
    }
    return OPAM_OK;
}

// Device address of the static scratch on the current device: looked up
// afresh unless `stream` is capturing, in which case the last address found
// on this device is used.
int static_scratch(cudaStream_t stream, void **out) {
    const char *fn = "tc_layer_forward_noalloc";
    int dev = -1;
    if (int rc = current_device(&dev, fn)) return rc;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return opam::cuda_fail(e, "tc_layer_forward_noalloc: cudaStreamIsCapturing");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cs == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return opam::cuda_fail(e, "tc_layer_forward_noalloc: cudaGetSymbolAddress");
        g_scratch_ptr[dev] = p;
    } else if (!g_scratch_ptr[dev]) {
        opam::set_error("%s: first call on device %d is under stream capture; make one call on this "
                        "device outside capture first", fn, dev);
        return OPAM_ERR_INVALID_ARG;
    }
    *out = g_scratch_ptr[dev];
    return OPAM_OK;
}

}  // namespace

namespace opam {

void *noalloc_scratch_if_ready() {
    int dev = -1;
    if (current_device(&dev, "opam_check_device_error") != OPAM_OK) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) return nullptr;
    // Look it up again, in case the device was reset since the last call.
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
    return p;
}

}  // namespace opam

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
        if (int rc = static_scratch((cudaStream_t)stream, &scratch)) return rc;
    return tc_layer_forward(q, k, v, dtype, B, H, T, d_k, d_v, W, lambda, eta, gate, softmax_scale, y,
                            state_out, scratch, (size_t)OPAM_STATIC_SCRATCH_BYTES, stream);
}
