// libopam C ABI: argument validation, workspace sizing and launch sequencing.
// Every check runs on the host before anything is enqueued, so a rejected
// call leaves the device untouched.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "opam_internal.cuh"

namespace opam {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

int cuda_fail(cudaError_t e, const char *where) {
    if (e == cudaSuccess) return OPAM_OK;
    set_error("%s: %s", where, cudaGetErrorString(e));
    return OPAM_ERR_CUDA;
}

int set_smem_limit(const void *func, int bytes, const char *where) {
    // cudaFuncSetAttribute is a driver round trip; it is needed once per
    // kernel and device (and again only if a call needs more shared memory).
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, where);
    std::lock_guard<std::mutex> lock(mu);
    int &have = done[{func, dev}];
    if (have >= bytes) return OPAM_OK;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail(e, where);
    have = bytes;
    return OPAM_OK;
}

int device_sm_count() {
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int clear_status(void *ws, cudaStream_t s) {
    return cuda_fail(cudaMemsetAsync(status_word(ws), 0, kStatusWords * sizeof(unsigned int), s),
                     "status word clear");
}

static std::atomic<uint64_t> g_launches{0};
static thread_local cudaEvent_t g_prof_start = nullptr;
static thread_local cudaEvent_t g_prof_stop = nullptr;

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
// Under stream capture the records are external, so that the captured graph
// keeps its two event nodes; otherwise they are ordinary records.
static void prof_record(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, s);
}
void prof_begin(cudaStream_t s) {
    if (g_prof_start) prof_record(g_prof_start, s);
}
void prof_end(cudaStream_t s) {
    if (g_prof_stop) prof_record(g_prof_stop, s);
}

namespace {

constexpr int kMaxGridY = 65535;
constexpr int kSparseMaxN = 49152;   // dense copy of one query row must fit shared memory

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool head_ok(int d) { return d == 32 || d == 64 || d == 128; }

#define OPAM_CHECK_PTR(p)                                                      \
    do {                                                                       \
        if (!(p)) {                                                            \
            set_error("%s: %s is NULL", fn, #p);                               \
            return OPAM_ERR_INVALID_ARG;                                       \
        }                                                                      \
        if (!aligned16(p)) {                                                   \
            set_error("%s: %s is not 16-byte aligned", fn, #p);                \
            return OPAM_ERR_INVALID_ARG;                                       \
        }                                                                      \
    } while (0)

#define OPAM_CHECK_OPT_PTR(p)                                                  \
    do {                                                                       \
        if ((p) && !aligned16(p)) {                                            \
            set_error("%s: %s is not 16-byte aligned", fn, #p);                \
            return OPAM_ERR_INVALID_ARG;                                       \
        }                                                                      \
    } while (0)

int check_tc_dims(const char *fn, int dtype, int B, int H, int T, int dk, int dv, int W) {
    if (dtype != OPAM_F32 && dtype != OPAM_BF16) {
        set_error("%s: dtype %d is not OPAM_F32 or OPAM_BF16", fn, dtype);
        return OPAM_ERR_INVALID_ARG;
    }
    if (B < 1 || H < 1 || T < 1 || W < 1 || dk < 1 || dv < 1) {
        set_error("%s: extents must be positive (B=%d H=%d T=%d W=%d d_k=%d d_v=%d)", fn, B, H, T, W,
                  dk, dv);
        return OPAM_ERR_INVALID_ARG;
    }
    if (!head_ok(dk) || !head_ok(dv)) {
        set_error("%s: head sizes d_k=%d d_v=%d not in {32, 64, 128}", fn, dk, dv);
        return OPAM_ERR_UNSUPPORTED;
    }
    if ((long long)B * H > kMaxGridY) {
        set_error("%s: B*H=%lld above %d", fn, (long long)B * H, kMaxGridY);
        return OPAM_ERR_UNSUPPORTED;
    }
    return OPAM_OK;
}

float resolve_scale(float s, int dk) { return s > 0.f ? s : 1.0f / std::sqrt((float)dk); }

int delta_chunk(int chunk) { return chunk == 0 ? 64 : chunk; }

// Scratch of the Tensor Cache prefill on the path the call takes, after the
// status block.
size_t tc_prefill_workspace(int B, int H, int T, int dk, int dv, int W, int dtype) {
    if (tc_prefill_tcgen05_supported(dtype, dk, dv))
        return OPAM_STATUS_BYTES + tc_prefill_tcgen05_workspace(B * H, T, dk, dv);
    return OPAM_STATUS_BYTES + tc_prefill_simt_workspace(B * H, T, dk, dv, W);
}

const char *status_names(unsigned int bits) {
    static thread_local char buf[256];
    buf[0] = 0;
    const struct {
        unsigned int mask;
        const char *name;
    } parts[] = {{0x7Fu * kStatusTcPrefill, "Tensor Cache prefill "},
                 {0x1Fu * kStatusDelta, "DeltaNet tensor-core "},
                 {0x7u * kStatusTcBackward, "Tensor Cache backward tensor-core "},
                 {0x3u * kStatusSparse, "BDH lists from the dense rows "},
                 {0x7u * kStatusKeygen, "BDH key generation "},
                 {kStatusSelfTest, "bounded-wait self-test "},
                 {kStatusBounds, "(index check of a debug-bounds build) "}};
    for (const auto &p : parts)
        if (bits & p.mask) strncat(buf, p.name, sizeof buf - strlen(buf) - 1);
    return buf;
}

}  // namespace
}  // namespace opam

using namespace opam;

extern "C" {

const char *opam_last_error(void) { return g_err; }

int opam_profile_events(void *start, void *stop) {
    g_prof_start = (cudaEvent_t)start;
    g_prof_stop = (cudaEvent_t)stop;
    return OPAM_OK;
}

uint64_t opam_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int opam_selftest_bounded_wait(int arrive, long long limit_cycles, void *workspace, void *stream) {
    const char *fn = "opam_selftest_bounded_wait";
    OPAM_CHECK_PTR(workspace);
    const long long limit = std::min(std::max(limit_cycles, 1000LL), 100000000LL);
    cudaStream_t s = (cudaStream_t)stream;
    if (int rc = clear_status(workspace, s)) return rc;
    return bounded_wait_selftest(arrive != 0, limit, status_word(workspace), s);
}

int opam_selftest_bounds(int n, void *workspace, void *stream) {
    const char *fn = "opam_selftest_bounds";
    OPAM_CHECK_PTR(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    if (int rc = clear_status(workspace, s)) return rc;
    return bounds_selftest(n, status_word(workspace), s);
}

int opam_debug_bounds_build(void) {
#ifdef OPAM_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

int opam_check_device_error(const void *workspace, void *stream) {
    const char *fn = "opam_check_device_error";
    if (workspace && !aligned16(workspace)) {
        set_error("%s: workspace is not 16-byte aligned", fn);
        return OPAM_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "opam_check_device_error: work on the stream failed");
    const void *ws = workspace ? workspace : noalloc_scratch_if_ready();
    if (!ws) return OPAM_OK;
    unsigned int words[kStatusWords] = {};
    e = cudaMemcpyAsync(words, ws, sizeof words, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "opam_check_device_error: reading the status words");
    unsigned int bits = 0;
    for (unsigned int w : words) bits |= w;
    if (bits == 0) return OPAM_OK;
    if (bits & kStatusBounds) {
        set_error("%s: an index check failed in a debug-bounds build (status 0x%x, %s); that call's outputs "
                  "are not valid", fn, bits, status_names(bits));
        return OPAM_ERR_INVALID_ARG;
    }
    set_error("%s: a bounded wait ran out in the %skernels (status 0x%x); that call's outputs are not "
              "valid", fn, status_names(bits), bits);
    return OPAM_ERR_TIMEOUT;
}

size_t tc_layer_forward_workspace_size(int B, int H, int T, int d_k, int d_v, int W, int dtype) {
    const char *fn = "tc_layer_forward_workspace_size";
    if (check_tc_dims(fn, dtype, B, H, T, d_k, d_v, W) != OPAM_OK) return 0;
    return tc_prefill_workspace(B, H, T, d_k, d_v, W, dtype);
}

int tc_layer_forward(const void *q, const void *k, const void *v, int dtype, int B, int H, int T,
                     int d_k, int d_v, int W, const float *lambda, const float *eta,
                     const float *gate, float softmax_scale, void *y, opam_tc_state *state_out,
                     void *workspace, size_t workspace_bytes, void *stream) {
    const char *fn = "tc_layer_forward";
    if (int rc = check_tc_dims(fn, dtype, B, H, T, d_k, d_v, W)) return rc;
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(lambda);
    OPAM_CHECK_PTR(eta);
    OPAM_CHECK_PTR(gate);
    OPAM_CHECK_PTR(y);
    if (state_out) {
        if (state_out->B != B || state_out->H != H || state_out->W != W || state_out->d_k != d_k ||
            state_out->d_v != d_v || state_out->dtype != dtype) {
            set_error("%s: state_out shape/dtype does not match the call", fn);
            return OPAM_ERR_INVALID_ARG;
        }
        OPAM_CHECK_PTR(state_out->ring_k);
        OPAM_CHECK_PTR(state_out->ring_v);
        OPAM_CHECK_PTR(state_out->A);
        OPAM_CHECK_PTR(state_out->pos);
        if ((long long)W > kMaxGridY * 1024LL) {
            set_error("%s: W=%d too large for the ring export", fn, W);
            return OPAM_ERR_UNSUPPORTED;
        }
    }
    const size_t need = tc_prefill_workspace(B, H, T, d_k, d_v, W, dtype);
    if (!workspace || workspace_bytes < need) {
        set_error("%s: workspace %zu bytes, %zu required", fn, workspace_bytes, need);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    const float scale = resolve_scale(softmax_scale, d_k);
    float *A_final = state_out ? state_out->A : nullptr;
    // The tensor-core path zeroes the status words inside its first kernel.
    if (!tc_prefill_tcgen05_supported(dtype, d_k, d_v))
        if (int rc = clear_status(workspace, s)) return rc;
    const int rc = tc_prefill_tcgen05_supported(dtype, d_k, d_v)
                       ? tc_prefill_tcgen05(q, k, v, B, H, T, d_k, d_v, W, lambda, eta, gate, scale, y,
                                            A_final, status_body(workspace), status_word(workspace), s)
                       : tc_prefill_simt(q, k, v, dtype, B, H, T, d_k, d_v, W, lambda, eta, gate, scale,
                                         y, A_final, status_body(workspace), s);
    if (rc) return rc;
    if (state_out)
        return tc_export_ring(k, v, dtype, B, H, T, d_k, d_v, W, state_out->ring_k, state_out->ring_v,
                              state_out->pos, s);
    return OPAM_OK;
}

size_t tc_window_forward_workspace_size(int B, int H, int T, int d_k, int d_v, int W, int dtype) {
    if (check_tc_dims("tc_window_forward_workspace_size", dtype, B, H, T, d_k, d_v, W) != OPAM_OK) return 0;
    return OPAM_STATUS_BYTES;
}

int tc_window_forward(const void *q, const void *k, const void *v, int dtype, int B, int H, int T,
                      int d_k, int d_v, int W, float softmax_scale, void *y, void *workspace,
                      size_t workspace_bytes, void *stream) {
    const char *fn = "tc_window_forward";
    if (int rc = check_tc_dims(fn, dtype, B, H, T, d_k, d_v, W)) return rc;
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(y);
    if (!workspace || workspace_bytes < OPAM_STATUS_BYTES) {
        set_error("%s: workspace %zu bytes, %u required", fn, workspace_bytes, OPAM_STATUS_BYTES);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    const float scale = resolve_scale(softmax_scale, d_k);
    if (int rc = clear_status(workspace, s)) return rc;
    if (tc_prefill_tcgen05_supported(dtype, d_k, d_v))
        return tc_prefill_tcgen05(q, k, v, B, H, T, d_k, d_v, W, nullptr, nullptr, nullptr, scale, y, nullptr,
                                  nullptr, status_word(workspace), s, false);
    return tc_prefill_simt(q, k, v, dtype, B, H, T, d_k, d_v, W, nullptr, nullptr, nullptr, scale, y, nullptr,
                           nullptr, s, false);
}

size_t tc_layer_backward_workspace_size(int B, int H, int T, int d_k, int d_v, int W, int dtype) {
    if (check_tc_dims("tc_layer_backward_workspace_size", dtype, B, H, T, d_k, d_v, W) != OPAM_OK) return 0;
    return OPAM_STATUS_BYTES + tc_backward_workspace(B * H, T, d_k, d_v);
}

int tc_layer_backward(const void *q, const void *k, const void *v, int dtype, int B, int H, int T, int d_k,
                      int d_v, int W, const float *lambda, const float *eta, const float *gate,
                      float softmax_scale, const void *dy, void *dq, void *dk, void *dv, float *dlambda,
                      float *deta, float *dgate, void *workspace, size_t workspace_bytes, void *stream) {
    const char *fn = "tc_layer_backward";
    if (int rc = check_tc_dims(fn, dtype, B, H, T, d_k, d_v, W)) return rc;
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(lambda);
    OPAM_CHECK_PTR(eta);
    OPAM_CHECK_PTR(gate);
    OPAM_CHECK_PTR(dy);
    OPAM_CHECK_PTR(dq);
    OPAM_CHECK_PTR(dk);
    OPAM_CHECK_PTR(dv);
    OPAM_CHECK_PTR(dlambda);
    OPAM_CHECK_PTR(deta);
    OPAM_CHECK_PTR(dgate);
    const size_t need = OPAM_STATUS_BYTES + tc_backward_workspace(B * H, T, d_k, d_v);
    if (!workspace || workspace_bytes < need) {
        set_error("%s: workspace %zu bytes, %zu required", fn, workspace_bytes, need);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    if (int rc = clear_status(workspace, s)) return rc;
    return tc_backward(q, k, v, dtype, B, H, T, d_k, d_v, W, lambda, eta, gate,
                       resolve_scale(softmax_scale, d_k), dy, dq, dk, dv, dlambda, deta, dgate,
                       status_body(workspace), status_word(workspace), s);
}

size_t tc_decode_step_workspace_size(const opam_tc_state *st) {
    if (!st) return 0;
    if (check_tc_dims("tc_decode_step_workspace_size", st->dtype, st->B, st->H, 1, st->d_k, st->d_v,
                      st->W) != OPAM_OK)
        return 0;
    return OPAM_STATUS_BYTES + tc_decode_workspace(st->B, st->H, st->d_k, st->d_v, st->W);
}

int tc_decode_step(opam_tc_state *st, const void *q, const void *k, const void *v,
                   const float *lambda, const float *eta, const float *gate, float softmax_scale,
                   void *y, void *workspace, size_t workspace_bytes, void *stream) {
    const char *fn = "tc_decode_step";
    if (!st) {
        set_error("%s: state is NULL", fn);
        return OPAM_ERR_INVALID_ARG;
    }
    if (int rc = check_tc_dims(fn, st->dtype, st->B, st->H, 1, st->d_k, st->d_v, st->W)) return rc;
    OPAM_CHECK_PTR(st->ring_k);
    OPAM_CHECK_PTR(st->ring_v);
    OPAM_CHECK_PTR(st->A);
    OPAM_CHECK_PTR(st->pos);
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(lambda);
    OPAM_CHECK_PTR(eta);
    OPAM_CHECK_PTR(gate);
    OPAM_CHECK_PTR(y);
    const size_t need = OPAM_STATUS_BYTES + tc_decode_workspace(st->B, st->H, st->d_k, st->d_v, st->W);
    if (!workspace || workspace_bytes < need) {
        set_error("%s: workspace %zu bytes, %zu required", fn, workspace_bytes, need);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    // The decode kernels have no bounded waits; the last of them zeroes the
    // status word, so no separate clear is enqueued on this hot path.
    return tc_decode(st, q, k, v, lambda, eta, gate, resolve_scale(softmax_scale, st->d_k), y,
                     status_body(workspace), status_word(workspace), (cudaStream_t)stream);
}

size_t delta_rule_forward_workspace_size(int B, int H, int T, int d_k, int d_v, int chunk, int dtype) {
    const char *fn = "delta_rule_forward_workspace_size";
    if (check_tc_dims(fn, dtype, B, H, T, d_k, d_v, 1) != OPAM_OK) return 0;
    const int C = delta_chunk(chunk);
    if (C != 16 && C != 32 && C != 64) return 0;
    if (delta_tcgen05_supported(dtype, d_k, d_v, C)) return OPAM_STATUS_BYTES + delta_tcgen05_workspace(B * H, T, d_k);
    return OPAM_STATUS_BYTES + delta_simt_workspace(B * H, T, d_k, d_v, C);
}

int delta_rule_forward(const void *q, const void *k, const void *v, const float *beta, int dtype,
                       int B, int H, int T, int d_k, int d_v, int chunk, const float *S0,
                       float *S_out, void *y, void *workspace, size_t workspace_bytes,
                       void *stream) {
    const char *fn = "delta_rule_forward";
    if (int rc = check_tc_dims(fn, dtype, B, H, T, d_k, d_v, 1)) return rc;
    const int C = delta_chunk(chunk);
    if (C != 16 && C != 32 && C != 64) {
        set_error("%s: chunk=%d not in {0, 16, 32, 64}", fn, chunk);
        return OPAM_ERR_UNSUPPORTED;
    }
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(beta);
    OPAM_CHECK_PTR(y);
    OPAM_CHECK_OPT_PTR(S0);
    OPAM_CHECK_OPT_PTR(S_out);
    const bool tc = delta_tcgen05_supported(dtype, d_k, d_v, C);
    const size_t need = OPAM_STATUS_BYTES +
                        (tc ? delta_tcgen05_workspace(B * H, T, d_k) : delta_simt_workspace(B * H, T, d_k, d_v, C));
    if (!workspace || workspace_bytes < need) {
        set_error("%s: workspace %zu bytes, %zu required", fn, workspace_bytes, need);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    if (int rc = clear_status(workspace, s)) return rc;
    if (tc)
        return delta_tcgen05(q, k, v, beta, B, H, T, d_k, d_v, S0, S_out, y, status_body(workspace),
                             status_word(workspace), s);
    return delta_simt(q, k, v, beta, dtype, B, H, T, d_k, d_v, C, S0, S_out, y, status_body(workspace), s);
}

size_t delta_rule_backward_workspace_size(int B, int H, int T, int d_k, int d_v, int dtype) {
    if (check_tc_dims("delta_rule_backward_workspace_size", dtype, B, H, T, d_k, d_v, 1) != OPAM_OK) return 0;
    return OPAM_STATUS_BYTES + delta_backward_workspace(B * H, T, d_v);
}

int delta_rule_backward(const void *q, const void *k, const void *v, const float *beta, int dtype, int B, int H,
                        int T, int d_k, int d_v, const float *S0, const void *dy, const float *dS_T, void *dq,
                        void *dk, void *dv, float *dbeta, float *dS0, void *workspace, size_t workspace_bytes,
                        void *stream) {
    const char *fn = "delta_rule_backward";
    if (int rc = check_tc_dims(fn, dtype, B, H, T, d_k, d_v, 1)) return rc;
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(beta);
    OPAM_CHECK_PTR(dy);
    OPAM_CHECK_PTR(dq);
    OPAM_CHECK_PTR(dk);
    OPAM_CHECK_PTR(dv);
    OPAM_CHECK_PTR(dbeta);
    OPAM_CHECK_OPT_PTR(S0);
    OPAM_CHECK_OPT_PTR(dS_T);
    OPAM_CHECK_OPT_PTR(dS0);
    const size_t need = OPAM_STATUS_BYTES + delta_backward_workspace(B * H, T, d_v);
    if (!workspace || workspace_bytes < need) {
        set_error("%s: workspace %zu bytes, %zu required", fn, workspace_bytes, need);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    return delta_backward(q, k, v, beta, dtype, B, H, T, d_k, d_v, S0, dy, dS_T, dq, dk, dv, dbeta, dS0,
                          status_body(workspace), status_word(workspace), (cudaStream_t)stream);
}

int delta_decode_step(float *S, const void *q, const void *k, const void *v, const float *beta,
                      int dtype, int B, int H, int d_k, int d_v, void *y, void *stream) {
    const char *fn = "delta_decode_step";
    if (int rc = check_tc_dims(fn, dtype, B, H, 1, d_k, d_v, 1)) return rc;
    OPAM_CHECK_PTR(S);
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(beta);
    OPAM_CHECK_PTR(y);
    return delta_decode(S, q, k, v, beta, dtype, B, H, d_k, d_v, y, (cudaStream_t)stream);
}

size_t sparse_linattn_forward_workspace_size(int B, int H, int T, int N, int d_v) {
    if (B < 1 || H < 1 || T < 1 || N < 1 || N > kSparseMaxN) return 0;
    if (d_v != 32 && d_v != 64 && d_v != 128 && d_v != 256) return 0;
    // The state lives in S_out when the caller supplies it; size for the
    // worst case (no S_out) so one query serves both.
    return OPAM_STATUS_BYTES + sparse_workspace(B * H, T, N, d_v, true);
}

int sparse_linattn_forward(const float *q, const float *k, const float *v, int B, int H, int T, int N,
                           int d_v, const float *S0, float *S_out, float *y, void *workspace,
                           size_t workspace_bytes, void *stream) {
    const char *fn = "sparse_linattn_forward";
    if (B < 1 || H < 1 || T < 1 || N < 1) {
        set_error("%s: extents must be positive (B=%d H=%d T=%d N=%d)", fn, B, H, T, N);
        return OPAM_ERR_INVALID_ARG;
    }
    if (N > kSparseMaxN || (d_v != 32 && d_v != 64 && d_v != 128 && d_v != 256)) {
        set_error("%s: N=%d (max %d) or d_v=%d (32/64/128/256) unsupported", fn, N, kSparseMaxN, d_v);
        return OPAM_ERR_UNSUPPORTED;
    }
    if ((long long)B * H > kMaxGridY) {
        set_error("%s: B*H above %d", fn, kMaxGridY);
        return OPAM_ERR_UNSUPPORTED;
    }
    OPAM_CHECK_PTR(q);
    OPAM_CHECK_PTR(k);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(y);
    OPAM_CHECK_OPT_PTR(S0);
    OPAM_CHECK_OPT_PTR(S_out);
    const size_t need = OPAM_STATUS_BYTES + sparse_workspace(B * H, T, N, d_v, S_out == nullptr);
    if (!workspace || workspace_bytes < need) {
        set_error("%s: workspace %zu bytes, %zu required", fn, workspace_bytes, need);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    if (int rc = clear_status(workspace, s)) return rc;
    return sparse_forward(q, k, v, B, H, T, N, d_v, S0, S_out, y, status_body(workspace), status_word(workspace), s);
}

size_t sparse_linattn_keygen_forward_workspace_size(int B, int H, int T, int R, int N, int d_v) {
    if (!bdh_keygen_supported(R, N)) return 0;
    return sparse_linattn_forward_workspace_size(B, H, T, N, d_v);
}

int sparse_linattn_keygen_forward(const void *xq, const void *xk, const void *U, float theta, const float *v,
                                  int B, int H, int T, int R, int N, int d_v, const float *S0, float *S_out,
                                  float *y, void *workspace, size_t workspace_bytes, void *stream) {
    const char *fn = "sparse_linattn_keygen_forward";
    if (B < 1 || H < 1 || T < 1 || R < 1 || N < 1) {
        set_error("%s: extents must be positive (B=%d H=%d T=%d R=%d N=%d)", fn, B, H, T, R, N);
        return OPAM_ERR_INVALID_ARG;
    }
    if (!bdh_keygen_supported(R, N) || N > kSparseMaxN ||
        (d_v != 32 && d_v != 64 && d_v != 128 && d_v != 256)) {
        set_error("%s: R=%d (64/128/256), N=%d (a multiple of 128, at most %d) or d_v=%d (32/64/128/256) "
                  "unsupported", fn, R, N, kSparseMaxN, d_v);
        return OPAM_ERR_UNSUPPORTED;
    }
    if ((long long)B * H > kMaxGridY) {
        set_error("%s: B*H above %d", fn, kMaxGridY);
        return OPAM_ERR_UNSUPPORTED;
    }
    if (!std::isfinite(theta)) {
        set_error("%s: theta is not finite", fn);
        return OPAM_ERR_INVALID_ARG;
    }
    OPAM_CHECK_PTR(xq);
    OPAM_CHECK_PTR(xk);
    OPAM_CHECK_PTR(U);
    OPAM_CHECK_PTR(v);
    OPAM_CHECK_PTR(y);
    OPAM_CHECK_OPT_PTR(S0);
    OPAM_CHECK_OPT_PTR(S_out);
    const size_t need = OPAM_STATUS_BYTES + sparse_workspace(B * H, T, N, d_v, S_out == nullptr);
    if (!workspace || workspace_bytes < need) {
        set_error("%s: workspace %zu bytes, %zu required", fn, workspace_bytes, need);
        return OPAM_ERR_WORKSPACE;
    }
    OPAM_CHECK_PTR(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    if (int rc = clear_status(workspace, s)) return rc;
    return sparse_keygen_forward(xq, xk, U, theta, v, B, H, T, R, N, d_v, S0, S_out, y, status_body(workspace),
                                 status_word(workspace), s);
}

}  // extern "C"
