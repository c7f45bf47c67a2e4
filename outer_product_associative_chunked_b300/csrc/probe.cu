// FP32 fused multiply-add rate of the device, for the roofline of the
// float32 paths (whose bound is the CUDA cores' FFMA pipe, not the tensor
// cores).  Every thread runs kChains independent FMA chains for `iters`
// rounds, so the pipe always has independent work; the chains' sum is
// stored so the compiler keeps every FMA.  Work per launch:
//   blocks * threads * iters * kChains FMAs = twice that many flops.
#include "opam_internal.cuh"

namespace opam {
namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) fp32_fma_probe_kernel(float *out, int iters, float a, float b) {
    float x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = (float)(threadIdx.x + c);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) x[c] = fmaf(x[c], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += x[c];
    out[blockIdx.x * kThreads + threadIdx.x] = s;
}

}  // namespace

double kChainsTotal(int blocks, int iters) { return (double)blocks * kThreads * (double)iters * kChains; }

int fp32_fma_probe(float *out, int blocks, int iters, cudaStream_t s) {
    fp32_fma_probe_kernel<<<blocks, kThreads, 0, s>>>(out, iters, 0.999f, 0.001f);
    return launched("fp32_fma_probe");
}

}  // namespace opam

extern "C" int opam_fp32_fma_probe(float *out, int blocks, int iters, double *flops, void *stream) {
    if (!out || blocks < 1 || iters < 1) {
        opam::set_error("opam_fp32_fma_probe: out must be non-NULL, blocks and iters positive");
        return OPAM_ERR_INVALID_ARG;
    }
    if (flops) *flops = 2.0 * opam::kChainsTotal(blocks, iters);
    return opam::fp32_fma_probe(out, blocks, iters, (cudaStream_t)stream);
}
