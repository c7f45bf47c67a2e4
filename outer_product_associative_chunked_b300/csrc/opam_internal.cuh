// Internal declarations shared by the libopam translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "opam.h"

namespace opam {

// ---------------------------------------------------------------- errors
void set_error(const char *fmt, ...);
int cuda_fail(cudaError_t e, const char *where);
// Raise a kernel's dynamic shared-memory limit to `bytes` (once per kernel
// and device; later calls that need no more are free).
int set_smem_limit(const void *func, int bytes, const char *where);
// Number of SMs of the current device (cached).
int device_sm_count();

// ---------------------------------------------------------------- instrumentation
// count_launch(): one kernel enqueued.  prof_begin / prof_end bracket the
// dominant kernel of an entry point with the caller's events, if any.
void count_launch(int n = 1);
void prof_begin(cudaStream_t s);
void prof_end(cudaStream_t s);
// After a kernel launch: count it and turn a launch error into OPAM_ERR_CUDA.
inline int launched(const char *what) {
    count_launch();
    return cuda_fail(cudaGetLastError(), what);
}

// ---------------------------------------------------------------- element I/O
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) {
        *p = __float2bfloat16_rn(x);
    }
};

__device__ __forceinline__ float logistic(float x) { return 1.0f / (1.0f + __expf(-x)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// ---------------------------------------------------------------- device status
// Every workspace begins with an OPAM_STATUS_BYTES block whose first
// kStatusWords words hold the call's device status: zero, or (OR-ed over the
// words) the bits below, set by a bounded wait that ran out.  Each call zeroes
// the words in stream order before they can be set -- with clear_status, or
// inside its own first kernel where that is race-free -- and
// opam_check_device_error reads them.
constexpr unsigned int kStatusTcPrefill = 1u << 0;   // 7 bits: Tensor Cache prefill kernels
constexpr unsigned int kStatusDelta = 1u << 8;       // 5 bits: DeltaNet tensor-core kernels
constexpr unsigned int kStatusTcBackward = 1u << 13;  // 3 bits: Tensor Cache backward tensor-core kernel
constexpr unsigned int kStatusSelfTest = 1u << 16;   // the bounded-wait self-test
constexpr unsigned int kStatusSparse = 1u << 17;     // 2 bits: BDH lists from the dense rows
constexpr unsigned int kStatusKeygen = 1u << 20;     // 3 bits: BDH key generation
constexpr unsigned int kStatusBounds = 1u << 24;     // an index check failed (debug-bounds builds)
constexpr int kStatusWords = 4;

// Index checks of a debug-bounds build (compiled with -DOPAM_DEBUG_BOUNDS):
// OPAM_BOUNDS(cond, status) is false, and sets kStatusBounds in *status, when
// `cond` fails, so the caller skips the access; it never traps.  In a normal
// build it is `true` and costs nothing.
#ifdef OPAM_DEBUG_BOUNDS
#define OPAM_BOUNDS(cond, status) ((cond) ? true : (atomicOr((status), ::opam::kStatusBounds), false))
#else
#define OPAM_BOUNDS(cond, status) true
#endif
inline unsigned int *status_word(void *ws) { return (unsigned int *)ws; }
inline void *status_body(void *ws) { return ws ? (char *)ws + OPAM_STATUS_BYTES : nullptr; }
// Zero the status words on the call's stream (enqueued before its kernels).
int clear_status(void *ws, cudaStream_t s);
// Device address of the built-in scratch of tc_layer_forward_noalloc on the
// current device, or NULL if no call has set it up there.
void *noalloc_scratch_if_ready();

// Finite stand-in for -infinity in running maxima (keeps exp() finite).
constexpr float kNegBig = -1.0e30f;

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- launchers
// Tensor Cache prefill, CUDA-core path (any supported head size / dtype).
size_t tc_prefill_simt_workspace(int BH, int T, int dk, int dv, int W);
// l2 = false: window only (the L1 ring); lam, eta, gate, A_final and ws are
// then unused and may be NULL.
int tc_prefill_simt(const void *q, const void *k, const void *v, int dtype, int B, int H,
                    int T, int dk, int dv, int W, const float *lam, const float *eta,
                    const float *gate, float scale, void *y, float *A_final,
                    void *ws, cudaStream_t s, bool l2 = true);
// Ring / pos export after a prefill (A is written by the prefill itself).
int tc_export_ring(const void *k, const void *v, int dtype, int B, int H, int T, int dk,
                   int dv, int W, void *ring_k, void *ring_v, int64_t *pos, cudaStream_t s);

// Tensor Cache prefill, tensor-core path (bf16 inputs, d_k, d_v in {64, 128}).
bool tc_prefill_tcgen05_supported(int dtype, int dk, int dv);
size_t tc_prefill_tcgen05_workspace(int BH, int T, int dk, int dv);
int tc_prefill_tcgen05(const void *q, const void *k, const void *v, int B, int H, int T, int dk,
                       int dv, int W, const float *lam, const float *eta, const float *gate,
                       float scale, void *y, float *A_final, void *ws, unsigned int *status,
                       cudaStream_t s, bool l2 = true);
// Self-test of the bounded mbarrier wait (sets kStatusSelfTest in *status
// when it runs out).
int bounded_wait_selftest(int arrive, long long limit, unsigned int *status, cudaStream_t s);
// Self-test of the debug-bounds index check (sets kStatusBounds in *status in
// a debug-bounds build when n < 32).
int bounds_selftest(int n, unsigned int *status, cudaStream_t s);

// Tensor Cache layer backward (CUDA cores; bf16 or fp32 inputs).
// Window part of the Tensor Cache backward's dK and dV on the tensor cores
// (bf16, d_k = d_v = 64); LSE and D rows at stride lstride (a multiple of 128).
bool tcb_window_dkdv_tcgen05_supported(int dtype, int dk, int dv);
// Window dQ with the softmax statistics it writes (LSE, D at stride lstride),
// on the tensor cores for the same sizes.
int tcb_window_dq_tcgen05(const void *q, const void *k, const void *v, const void *dy, int BH, int Tn, int W,
                          float scale, float *lse, float *D, int lstride, float *dQ, unsigned int *status,
                          cudaStream_t st);
int tcb_window_dkdv_tcgen05(const void *q, const void *k, const void *v, const void *dy, int BH, int Tn, int W,
                            float scale, const float *lse, const float *D, int lstride, float *dK, float *dV,
                            unsigned int *status, cudaStream_t st);
size_t tc_backward_workspace(int BH, int T, int dk, int dv);
int tc_backward(const void *q, const void *k, const void *v, int dtype, int B, int H, int T, int dk, int dv, int W,
                const float *lam, const float *eta, const float *gate, float scale, const void *dy, void *dq,
                void *dkk, void *dvv, float *dlam, float *deta, float *dgate, void *ws, unsigned int *status,
                cudaStream_t s);

size_t tc_decode_workspace(int S, int H, int dk, int dv, int W);
int tc_decode(const opam_tc_state *st, const void *q, const void *k, const void *v,
              const float *lam, const float *eta, const float *gate, float scale, void *y,
              void *ws, unsigned int *status, cudaStream_t s);

size_t delta_simt_workspace(int BH, int T, int dk, int dv, int C);
int delta_simt(const void *q, const void *k, const void *v, const float *beta, int dtype,
               int B, int H, int T, int dk, int dv, int C, const float *S0, float *S_out,
               void *y, void *ws, cudaStream_t s);

// DeltaNet, tensor-core path (bf16, d_k in {64, 128}, d_v = 128, chunk 64).
bool delta_tcgen05_supported(int dtype, int dk, int dv, int chunk);
size_t delta_tcgen05_workspace(int BH, int T, int dk);
int delta_tcgen05(const void *q, const void *k, const void *v, const float *beta, int B, int H, int T,
                  int dk, int dv, const float *S0, float *S_out, void *y, void *ws, unsigned int *status,
                  cudaStream_t s);

// DeltaNet backward (CUDA cores, per-token reverse recurrence).
size_t delta_backward_workspace(int BH, int T, int dv);
int delta_backward(const void *q, const void *k, const void *v, const float *beta, int dtype, int B, int H, int T,
                   int dkk, int dvv, const float *S0, const void *dy, const float *dST, void *dq, void *dk,
                   void *dv, float *dbeta, float *dS0, void *ws, unsigned int *status, cudaStream_t s);

// DeltaNet single-token decode (state updated in place, no scratch).
int delta_decode(float *S, const void *q, const void *k, const void *v, const float *beta, int dtype,
                 int B, int H, int dk, int dv, void *y, cudaStream_t s);

// FP32 FMA rate probe (instrumentation): FMAs one launch performs, and the launch.
double kChainsTotal(int blocks, int iters);
int fp32_fma_probe(float *out, int blocks, int iters, cudaStream_t s);

// BDH key generation fused with support compaction (bf16 x and U, fp32
// accumulation): writes the per-row support lists of q and k.
bool bdh_keygen_supported(int R, int N);
// With coff == NULL it writes the per-row lists (recurrent form); otherwise
// the coordinate-major lists of each 128-token block (pairwise form).
int bdh_keygen(const void *xq, const void *xk, const void *U, float theta, int B, int H, int T, int R, int N,
               int *kidx, float *kval, int *kcnt, int *qidx, float *qval, int *qcnt, int *coff, uint8_t *ct,
               float *cv, unsigned int *status, cudaStream_t s);

size_t sparse_workspace(int BH, int T, int N, int dv, bool need_state);
int sparse_forward(const float *q, const float *k, const float *v, int B, int H, int T, int N,
                   int dv, const float *S0, float *S_out, float *y, void *ws, unsigned int *status,
                   cudaStream_t s);
// The same attention with q and k generated on chip from x and U_h.
int sparse_keygen_forward(const void *xq, const void *xk, const void *U, float theta, const float *v, int B,
                          int H, int T, int R, int N, int dv, const float *S0, float *S_out, float *y, void *ws,
                          unsigned int *status, cudaStream_t s);

}  // namespace opam
