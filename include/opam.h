/*
 * opam.h -- C ABI of libopam: outer-product associative-memory layers on one
 * NVIDIA B300 (sm_103a).
 *
 * A layer keeps a fixed-size state written with outer products k (x) v and
 * read with a query, using q (k (x) v) = <q, k> v (gist.science 2605.22884
 * "Tensor Cache", Methodology 1, read mechanism; molayo1419.me "DeltaNet-family
 * linear attention variants", opening identity).  Three write rules are
 * exported:
 *   - Tensor Cache: exact softmax over a ring of the W most recent tokens; a
 *     token evicted from the ring is written A <- lambda A + eta k v^T and read
 *     as m_t = q_t A; y_t = y_local,t + sigmoid(g) m_t  (tc_layer_forward,
 *     tc_decode_step; tc_window_forward is the ring alone);
 *   - DeltaNet delta rule e_t = beta_t (v_t - S_{t-1} k_t), S_t = S_{t-1} +
 *     e_t k_t^T, o_t = S_t q_t  (delta_rule_forward, delta_decode_step);
 *   - BDH-style additive linear attention over wide, sparse, non-negative keys,
 *     S_t = S_{t-1} + v_t k_t^T, o_t = S_t q_t  (sparse_linattn_forward).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers unless stated otherwise, owned by the
 *     caller, 16-byte aligned, and every tensor is dense row-major
 *     ("contiguous") in the shape given.  The library allocates nothing and
 *     keeps no device state between calls: a call's device status lives in
 *     its own workspace (below).  Host-side it keeps a per-thread error
 *     string, the per-thread profiling hooks and process-wide launch counter
 *     of the instrumentation section, and per-device caches of attributes
 *     (SM count, shared-memory limits already raised); tc_layer_forward_noalloc
 *     alone adds its built-in device array.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously.  The return value reports argument
 *     errors and launch failures synchronously; nothing is enqueued when a
 *     call returns an error.  Device-side outcomes (a bounded wait that ran
 *     out, or any CUDA error) are read after the work with
 *     opam_check_device_error(workspace, stream).
 *   - Every state is stored key-major: element (a, b) of a d_k x d_v matrix at
 *     [a * d_v + b].  For Tensor Cache that is A = sum eta lambda^.. k v^T.
 *     DeltaNet and BDH write their state as S in R^{d_v x d_k} with read S q;
 *     the stored matrix is S^T, so S_{i,j} sits at [j * d_v + i].
 *   - Scratch memory ("workspace") is caller-provided device memory of at
 *     least the size the matching *_workspace_size() returns for the same
 *     arguments; its contents on entry do not matter.  Its first
 *     OPAM_STATUS_BYTES hold the call's device status, which the call zeroes
 *     in stream order before any of its kernels can set it, and which a
 *     kernel sets if one of its bounded waits runs out.  Calls that share a
 *     workspace must not overlap on the GPU.
 *   - Return value: OPAM_OK, or a negative opam_status; opam_last_error()
 *     then holds a one-line message (per calling thread).
 */
#ifndef OPAM_H
#define OPAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and y.  Scalars (lambda, eta, gate, beta) and every
 * state matrix are always float32. */
typedef enum { OPAM_F32 = 0, OPAM_BF16 = 1 } opam_dtype;

/* Bytes at the head of every workspace that hold the call's device status
 * (the first four 32-bit words; the rest is reserved).  Every
 * *_workspace_size() includes them. */
#define OPAM_STATUS_BYTES 256u

typedef enum {
    OPAM_OK = 0,
    OPAM_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, bad extent        */
    OPAM_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. d = 96)    */
    OPAM_ERR_CUDA = -3,         /* a CUDA launch or API call failed           */
    OPAM_ERR_TIMEOUT = -4,      /* a kernel's bounded wait ran out (see below) */
    OPAM_ERR_WORKSPACE = -5     /* workspace missing or smaller than required */
} opam_status;

/* ------------------------------------------------------------------------
 * Tensor Cache streaming state (Methodology 1: L1 ring buffer of the W most
 * recent tokens plus the L2 outer-product matrix A; Main contributions:
 * bounded state, O(W d + d_k d_v) per head).  All buffers caller-owned:
 *   ring_k  [B][H][W][d_k]  element type `dtype`; slot j holds the newest
 *           token position p < pos[b] with p mod W == j (zero when
 *           pos[b] <= j)
 *   ring_v  [B][H][W][d_v]  same slots
 *   A       [B][H][d_k][d_v] float32
 *   pos     [B] int64        tokens seen so far by sequence b (all heads)
 * ---------------------------------------------------------------------- */
typedef struct {
    void *ring_k;
    void *ring_v;
    float *A;
    int64_t *pos;
    int32_t B, H, W, d_k, d_v;
    int32_t dtype; /* opam_dtype */
} opam_tc_state;

/* Tensor Cache layer forward over a whole sequence from an empty state
 * ("Tensor Cache", Methodology 1 for the layer; Methodology 2 for the
 * parallel weighted-sum scan that makes the prefill equal to the per-token
 * writes, with no chunk averaging).
 *
 *   q, k      [B][H][T][d_k]   dtype
 *   v         [B][H][T][d_v]   dtype
 *   lambda, eta, gate  [H] float32 per-head decay, write rate, gate logit g
 *   softmax_scale      tau in softmax(tau q.k); <= 0 selects 1/sqrt(d_k)
 *   y         [B][H][T][d_v]   dtype, output:
 *       y_t = sum_{s=max(0,t-W+1)}^{t} softmax_s(tau q_t.k_s) v_s
 *           + sigmoid(g) sum_{s<=t-W} eta lambda^(t-W-s) <q_t,k_s> v_s
 *   state_out  NULL, or a state with matching B, H, W, d_k, d_v, dtype that
 *              receives the ring, A and pos = T so decoding can continue.
 *
 * Supported: d_k, d_v in {32, 64, 128}; 1 <= W; 1 <= T; B*H >= 1.
 * Errors: OPAM_ERR_INVALID_ARG for null or misaligned pointers or
 * non-positive extents, OPAM_ERR_UNSUPPORTED for other head sizes,
 * OPAM_ERR_WORKSPACE if workspace_bytes is below the required size. */
size_t tc_layer_forward_workspace_size(int B, int H, int T, int d_k, int d_v, int W,
                                       int dtype);
int tc_layer_forward(const void *q, const void *k, const void *v, int dtype,
                     int B, int H, int T, int d_k, int d_v, int W,
                     const float *lambda, const float *eta, const float *gate,
                     float softmax_scale, void *y, opam_tc_state *state_out,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Tensor Cache layer backward: the gradient of L = sum_t <dy_t, y_t> through
 * tc_layer_forward ("Tensor Cache", Methodology 2: the parallel weighted-sum
 * scan is what makes the layer trainable without chunk averaging; the pages
 * print no backward formulas, so the gradient is the exact derivative of
 * the forward definition above).  Same inputs as tc_layer_forward, plus
 *   dy        [B][H][T][d_v]  dtype, upstream gradient of y
 * and outputs (all written, none accumulated into):
 *   dq, dk    [B][H][T][d_k]  dtype
 *   dv        [B][H][T][d_v]  dtype
 *   dlambda, deta, dgate  [H] float32, summed over the batch.
 * Nothing from the forward call is needed: the softmax statistics and the
 * chunk states are recomputed.  Arithmetic is float32 throughout (bf16
 * inputs are widened on load).  Supported sizes and errors as
 * tc_layer_forward; workspace: tc_layer_backward_workspace_size() bytes. */
size_t tc_layer_backward_workspace_size(int B, int H, int T, int d_k, int d_v, int W,
                                        int dtype);
int tc_layer_backward(const void *q, const void *k, const void *v, int dtype,
                      int B, int H, int T, int d_k, int d_v, int W,
                      const float *lambda, const float *eta, const float *gate,
                      float softmax_scale, const void *dy, void *dq, void *dk, void *dv,
                      float *dlambda, float *deta, float *dgate, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Bytes of scratch built into the library for tc_layer_forward_noalloc. */
#define OPAM_STATIC_SCRATCH_BYTES (64u << 20)

/* tc_layer_forward without a workspace argument, for callers that cannot
 * allocate device memory.  The pages have no counterpart to this: it exists
 * for host software, not for the method.
 *
 * Who needs it: plugins living inside an application that owns all device
 * memory through its own allocator, and services that forbid allocation after
 * start-up (cudaMalloc can block, synchronise the device, or fail once the
 * pool is reserved).  Such callers can pass inputs and outputs but cannot
 * provide the scratch tc_layer_forward requires.
 *
 * Behaviour: identical arguments and results to tc_layer_forward, with the
 * scratch taken from a fixed OPAM_STATIC_SCRATCH_BYTES array inside the
 * library (present on every GPU that loads the library until the process
 * exits).  Nothing is allocated.  A problem whose
 * tc_layer_forward_workspace_size() exceeds OPAM_STATIC_SCRATCH_BYTES returns
 * OPAM_ERR_WORKSPACE with both sizes in opam_last_error().  Every call made
 * outside stream capture looks up the array's device address on the current
 * device (so a device reset, which may move the array, is picked up by the
 * next such call); a call under stream capture reuses the address found by
 * the last call on that device, so make one call on each device before any
 * capture, and again after a device reset.  All calls on a device share the
 * array: calls that overlap on the GPU (other streams, other threads) race
 * and must be serialised by the caller.  The call's device status sits at
 * the head of the array: opam_check_device_error(NULL, stream) reads it. */
int tc_layer_forward_noalloc(const void *q, const void *k, const void *v, int dtype,
                             int B, int H, int T, int d_k, int d_v, int W,
                             const float *lambda, const float *eta, const float *gate,
                             float softmax_scale, void *y, opam_tc_state *state_out,
                             void *stream);

/* The window-only variant of the Tensor Cache layer: the L1 ring alone,
 * i.e. sliding-window softmax attention without the L2 memory ("Tensor
 * Cache", Results: the layer's throughput is compared with pure
 * sliding-window attention).  For every token t
 *   y_t = softmax over keys max(0, t-W+1) .. t of (scale <q_t, k_s>) v_s,
 * which is tc_layer_forward with eta = 0.  It runs the same forward kernels
 * with their L2 part switched off and launches no state kernels, so the
 * difference in time between the two calls is the cost of the L2 memory.
 *   q, k [B][H][T][d_k] dtype;  v [B][H][T][d_v] dtype;  y [B][H][T][d_v]
 *   softmax_scale  <= 0 selects 1/sqrt(d_k)
 * No per-head scalars; the workspace holds only the status block
 * (tc_window_forward_workspace_size() bytes).  Same support and errors as
 * tc_layer_forward. */
size_t tc_window_forward_workspace_size(int B, int H, int T, int d_k, int d_v, int W,
                                        int dtype);
int tc_window_forward(const void *q, const void *k, const void *v, int dtype,
                      int B, int H, int T, int d_k, int d_v, int W,
                      float softmax_scale, void *y, void *workspace,
                      size_t workspace_bytes, void *stream);

/* One Tensor Cache decode step for a batch of independent sequences
 * ("Tensor Cache", Methodology 1: when the ring overwrites an entry the
 * displaced (k, v) is written into A; the new token is then read through the
 * ring softmax and q A).  For every sequence b and head h, with p = pos[b]:
 *   1. slot = p mod W; if p >= W: A <- lambda A + eta k_e v_e^T with
 *      (k_e, v_e) = ring[slot] (the token p - W);
 *   2. ring[slot] <- (k, v);
 *   3. y = softmax over the min(p+1, W) occupied slots + sigmoid(g) q A;
 * then pos[b] += 1.
 *   st          state (updated in place); st->B is the number of sequences
 *   q, k        [B][H][d_k] dtype (one token per sequence and head)
 *   v           [B][H][d_v] dtype
 *   lambda, eta, gate [H] float32; softmax_scale as above
 *   y           [B][H][d_v] dtype, output
 * Same support and errors as tc_layer_forward. */
size_t tc_decode_step_workspace_size(const opam_tc_state *st);
int tc_decode_step(opam_tc_state *st, const void *q, const void *k, const void *v,
                   const float *lambda, const float *eta, const float *gate,
                   float softmax_scale, void *y, void *workspace,
                   size_t workspace_bytes, void *stream);

/* DeltaNet delta-rule forward (molayo1419.me, "DeltaNet-family linear
 * attention variants", section "DeltaNet: write the prediction error instead
 * of the value"), evaluated chunk by chunk in an exact closed form of the
 * same recurrence:
 *   e_t = beta_t (v_t - S_{t-1} k_t),  S_t = S_{t-1} + e_t k_t^T,
 *   o_t = S_t q_t (read after the write).
 *   q, k   [B][H][T][d_k] dtype;  v [B][H][T][d_v] dtype
 *   beta   [B][H][T] float32 in [0, 1]
 *   chunk  tokens per chunk: 0 (default 64), 16, 32 or 64; results do not
 *          depend on it beyond rounding
 *   S0     NULL (zero state) or [B][H][d_k][d_v] float32 key-major start state
 *   S_out  NULL or [B][H][d_k][d_v] float32 key-major final state (may equal S0)
 *   y      [B][H][T][d_v] dtype, output o_t
 * Supported: d_k, d_v in {32, 64, 128}; bf16 with d_k, d_v in {64, 128} and
 * chunk 64 runs on the tensor cores, every other case on the CUDA cores.
 * Errors as above. */
size_t delta_rule_forward_workspace_size(int B, int H, int T, int d_k, int d_v,
                                         int chunk, int dtype);
int delta_rule_forward(const void *q, const void *k, const void *v,
                       const float *beta, int dtype, int B, int H, int T,
                       int d_k, int d_v, int chunk, const float *S0,
                       float *S_out, void *y, void *workspace,
                       size_t workspace_bytes, void *stream);

/* DeltaNet delta-rule backward: the gradient of
 * L = sum_t <dy_t, o_t> + <dS_T, S_T> through delta_rule_forward (same page
 * and section; the pages print no backward formulas, so the gradient is the
 * exact derivative of the recurrence above, taken step by step in reverse).
 *   q, k, v, beta, dtype, B, H, T, d_k, d_v, S0  as delta_rule_forward
 *   dy     [B][H][T][d_v] dtype, upstream gradient of o
 *   dS_T   NULL (zero) or [B][H][d_k][d_v] float32 key-major gradient of the
 *          final state
 *   dq, dk [B][H][T][d_k] dtype;  dv [B][H][T][d_v] dtype;  dbeta [B][H][T]
 *          float32 (all written)
 *   dS0    NULL or [B][H][d_k][d_v] float32, receives the gradient of S0
 * Arithmetic is float32; the state is carried per token (no chunking), so
 * the time is a sequential walk of 2T steps per (batch, head).  Supported:
 * d_k, d_v in {32, 64, 128}; workspace: delta_rule_backward_workspace_size()
 * bytes.  Errors as above. */
size_t delta_rule_backward_workspace_size(int B, int H, int T, int d_k, int d_v, int dtype);
int delta_rule_backward(const void *q, const void *k, const void *v, const float *beta,
                        int dtype, int B, int H, int T, int d_k, int d_v, const float *S0,
                        const void *dy, const float *dS_T, void *dq, void *dk, void *dv,
                        float *dbeta, float *dS0, void *workspace, size_t workspace_bytes,
                        void *stream);

/* One DeltaNet decode step for a batch of independent sequences (molayo1419.me,
 * "DeltaNet-family linear attention variants", section "DeltaNet: write the
 * prediction error instead of the value"): for every sequence b and head h,
 *   e = beta (v - S k),  S <- S + e k^T,  y = S q (read after the write),
 * the same step delta_rule_forward applies to each token, taken one token at a
 * time from a stored state.
 *   S      [B][H][d_k][d_v] float32 key-major state (the layout of
 *          delta_rule_forward's S_out), read and updated in place
 *   q, k   [B][H][d_k] dtype (one token per sequence and head)
 *   v      [B][H][d_v] dtype
 *   beta   [B][H] float32 in [0, 1]
 *   y      [B][H][d_v] dtype, output
 * No workspace: the step has no bounded waits, so its only device-side
 * failures are CUDA errors, which opam_check_device_error(NULL, stream)
 * reports.  Supported: d_k, d_v in {32, 64, 128}, B*H <= 65535.  Errors
 * as above; S, q, k, v, beta and y must all be non-NULL.  The state is read
 * once and written once per call (memory bound). */
int delta_decode_step(float *S, const void *q, const void *k, const void *v,
                      const float *beta, int dtype, int B, int H, int d_k, int d_v,
                      void *y, void *stream);

/* BDH-style linear attention over wide, sparse, non-negative keys
 * (ainews.random.gg BDH memory-architecture post: keys/queries are neuron
 * activations in a very high-dimensional space, the state is the accumulated
 * connectivity and a read is propagation; mo.ai.kr "Hebbian memory MLP",
 * simple construction W = sum_i v_i k_i^T):
 *   S_t = S_{t-1} + v_t k_t^T,  o_t = S_t q_t  (read after the write).
 * q and k are passed dense (the ReLU output a model produces); their supports
 * are found inside the library.  Any real values are handled exactly; the
 * speed relies on most entries being zero.
 *   q, k   [B][H][T][N] float32
 *   v      [B][H][T][d_v] float32
 *   S0     NULL or [B][H][N][d_v] float32 key-major start state
 *   S_out  NULL or [B][H][N][d_v] float32 key-major final state (may equal S0)
 *   y      [B][H][T][d_v] float32, output
 * Supported: 1 <= N <= 49152, d_v in {32, 64, 128, 256}. Errors as above.
 * Without S0 and S_out, and with N a multiple of 128, the dense rows are
 * streamed by TMA through bounded waits: one that runs out is reported by
 * opam_check_device_error (the other paths have no such wait). */
size_t sparse_linattn_forward_workspace_size(int B, int H, int T, int N, int d_v);
int sparse_linattn_forward(const float *q, const float *k, const float *v,
                           int B, int H, int T, int N, int d_v,
                           const float *S0, float *S_out, float *y,
                           void *workspace, size_t workspace_bytes, void *stream);

/* The same BDH-style attention with the wide keys and queries generated on
 * the GPU (the BDH post: the sparse non-negative activations come from a
 * low-rank factorisation followed by ReLU thresholding):
 *   k_t = max(0, xk_t U_h - theta),   q_t = max(0, xq_t U_h - theta),
 * one U_h per head shared by queries and keys.  Each tile of x U_h is a
 * tensor-core product (bf16 operands, float32 accumulation) whose epilogue
 * keeps only the entries above theta as the row's support list, so the dense
 * N-wide q and k never exist in memory; the attention itself is then the
 * same float32 computation as sparse_linattn_forward.
 *   xq, xk [B][H][T][R] bf16 (the R-dimensional token inputs)
 *   U      [H][R][N] bf16
 *   theta  threshold (finite; about 1.645 gives 5% density for unit-variance
 *          x U_h entries)
 *   v, S0, S_out, y  as sparse_linattn_forward (float32)
 * Supported: R in {64, 128, 256}, N a multiple of 128 up to 49152, d_v in
 * {32, 64, 128, 256}.  Workspace:
 * sparse_linattn_keygen_forward_workspace_size() bytes.  Errors as above;
 * a bounded wait of the key-generation kernel that runs out is reported by
 * opam_check_device_error. */
size_t sparse_linattn_keygen_forward_workspace_size(int B, int H, int T, int R, int N, int d_v);
int sparse_linattn_keygen_forward(const void *xq, const void *xk, const void *U, float theta,
                                  const float *v, int B, int H, int T, int R, int N, int d_v,
                                  const float *S0, float *S_out, float *y, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Message for the last non-OK status returned on the calling thread. */
const char *opam_last_error(void);

/* Device-side outcome of the most recent call that used `workspace`.
 * The tensor-core kernels' pipeline waits are bounded (about one second
 * each); a wait that runs out abandons the CTA's work, leaves that call's
 * outputs undefined and sets a bit in the call's status word instead of
 * hanging the GPU.  This function synchronises `stream` only (not the
 * device), then:
 *   - returns OPAM_ERR_CUDA if the stream holds a CUDA error (for example a
 *     fault of any earlier work on it);
 *   - returns OPAM_ERR_TIMEOUT, with the kernels named in opam_last_error(),
 *     if the status at the head of `workspace` is non-zero (in a
 *     debug-bounds build, OPAM_ERR_INVALID_ARG if an index check failed);
 *   - returns OPAM_OK otherwise.
 * `workspace` is the workspace of the call in question and `stream` the
 * stream that call ran on.  With workspace NULL it checks the built-in
 * scratch of tc_layer_forward_noalloc on the current device (if a call has
 * set it up there) and otherwise only the stream.  The word is not cleared
 * here: the next call that uses the workspace zeroes it. */
int opam_check_device_error(const void *workspace, void *stream);

/* ------------------------------------------------------------------------
 * Instrumentation (no counterpart on the pages; used by benchmarks).
 *
 * opam_profile_events: on the calling thread, every later entry-point call
 * records `start` (a cudaEvent_t) on its stream immediately before launching
 * its dominant kernel and `stop` immediately after it, so the caller can time
 * that kernel alone with cudaEventElapsedTime.  The dominant kernel is the
 * fused window-softmax kernel of tc_layer_forward, the split-ring kernel of
 * tc_decode_step, the chunk preparation and the sequential state pass of
 * delta_rule_forward together (tensor-core path; the state pass alone on the
 * CUDA-core path), the one
 * kernel of delta_decode_step, and for sparse_linattn_forward the block-pair
 * kernel (no start or final state) or else the chunked read and write
 * (summed over their launches: `start` goes before the first, `stop` after
 * the last).  Pass NULL, NULL to stop.
 * The records are external, so a call captured into a CUDA graph keeps them
 * as event nodes that fire on every replay.  Events stay owned by the caller.
 * Returns OPAM_OK.
 *
 * opam_kernel_launches: number of kernels this library has launched in the
 * process so far (all threads); launches recorded into a CUDA graph count
 * once, at capture. */
int opam_profile_events(void *start, void *stop);
uint64_t opam_kernel_launches(void);

/* FP32 FMA rate probe (no counterpart on the pages; used by benchmarks to
 * measure the CUDA cores' float32 peak, the roof of the float32 paths).
 * Enqueues one kernel of `blocks` CTAs x 256 threads in which every thread
 * runs 8 independent fmaf chains for `iters` rounds and stores the chains'
 * sum to out[block * 256 + thread] (`out` holds blocks * 256 floats).
 * *flops (if not NULL) receives the launch's flop count, 2 per FMA:
 * 2 * blocks * 256 * iters * 8.  Time it with events on `stream`.
 * Returns OPAM_OK, OPAM_ERR_INVALID_ARG, or OPAM_ERR_CUDA. */
int opam_fp32_fma_probe(float *out, int blocks, int iters, double *flops, void *stream);

/* Self-test of the bounded waits (no counterpart on the pages; used by the
 * tests).  Zeroes the status word of `workspace` (at least OPAM_STATUS_BYTES
 * of device memory) and launches one warp whose lane 0 waits, through the
 * same bounded mbarrier wait the tensor-core kernels use, on a barrier that
 * completes only when `arrive` is non-zero.  With arrive = 0 the wait gives
 * up after limit_cycles clock cycles (clamped to [1e3, 1e8], well under a
 * second) and sets a status bit, so opam_check_device_error(workspace,
 * stream) returns OPAM_ERR_TIMEOUT; the context stays usable.  Returns
 * OPAM_OK, OPAM_ERR_INVALID_ARG for a NULL or misaligned workspace, or
 * OPAM_ERR_CUDA if the launch fails. */
int opam_selftest_bounded_wait(int arrive, long long limit_cycles, void *workspace,
                               void *stream);

/* Debug-bounds builds (no counterpart on the pages; used by the tests).  A
 * library compiled with -DOPAM_DEBUG_BOUNDS checks the indexes of its
 * kernels' global-memory writes (and of the BDH pair kernel's shared-memory
 * accumulator): a failed check skips the access, never traps, and sets a bit
 * that opam_check_device_error reports as OPAM_ERR_INVALID_ARG.
 * opam_debug_bounds_build returns 1 for such a build and 0 otherwise.
 * opam_selftest_bounds zeroes the status of `workspace` (at least
 * OPAM_STATUS_BYTES) and runs one warp in which thread i checks i < n: with
 * n < 32 a debug-bounds build reports the failed checks, a normal build
 * nothing.  No memory is accessed.  Returns OPAM_OK, OPAM_ERR_INVALID_ARG or
 * OPAM_ERR_CUDA. */
int opam_debug_bounds_build(void);
int opam_selftest_bounds(int n, void *workspace, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* OPAM_H */
