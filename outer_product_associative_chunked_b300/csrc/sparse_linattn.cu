// BDH-style additive linear attention over wide, sparse, non-negative keys.
//
// ainews.random.gg, BDH memory-architecture post: keys and queries are
// neuron activations in a very wide space (about 5% non-zero after ReLU
// thresholding), the state is the accumulated connectivity and reading it is
// propagation -- a fixed-size hash table whose few buckets a sparse key
// writes.  The write is the Hebbian outer-product sum of mo.ai.kr "Hebbian
// memory MLP" (W = sum_i v_i k_i^T), per token:
//     S_t = S_{t-1} + v_t k_t^T,   o_t = S_t q_t.
//
// Layout: the state is key-major, row j = the d_v values bucket j holds, so a
// sparse key touches whole contiguous rows.  Supports are found on the GPU:
// every dense q / k row is compacted to its ascending (index, value) list.
// Tokens are then processed in chunks of kC: with S the state before the
// chunk,
//     o_t = sum_{j in supp q_t} q_t[j] S[j,:] + sum_{s in chunk, s<=t} <k_s,q_t> v_s
// and afterwards every token of the chunk adds k_s[j] v_s into row j.
#include "opam_internal.cuh"

namespace opam {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;

__global__ void compact_rows_kernel(const float *__restrict__ x, int rows, int N,
                                    int *__restrict__ idx, float *__restrict__ val,
                                    int *__restrict__ cnt) {
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *src = x + (size_t)row * N;
    int *oi = idx + (size_t)row * N;
    float *ov = val + (size_t)row * N;
    int c = 0;
    for (int base = 0; base < N; base += 32) {
        const int j = base + lane;
        const float a = j < N ? src[j] : 0.f;
        const unsigned bal = __ballot_sync(0xffffffffu, a != 0.f);
        if (a != 0.f) {
            const int p = c + __popc(bal & ((1u << lane) - 1u));
            oi[p] = j;
            ov[p] = a;
        }
        c += __popc(bal);
    }
    if (lane == 0) cnt[row] = c;
}

template <int DV>
__global__ void __launch_bounds__(kThreads)
sparse_read_kernel(int c0, int T_, int N, const int *__restrict__ kidx,
                   const float *__restrict__ kval, const int *__restrict__ kcnt,
                   const int *__restrict__ qidx, const float *__restrict__ qval,
                   const int *__restrict__ qcnt, const float *__restrict__ v,
                   const float *__restrict__ ST, float *__restrict__ y) {
    extern __shared__ float qd[];  // [N] dense copy of q_t
    __shared__ float zs[kC];
    __shared__ float red[kThreads];
    constexpr int G = kThreads / DV;
    const int ti = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const size_t row = (size_t)bh * T_ + c0 + ti;
    for (int j = tid; j < N; j += kThreads) qd[j] = 0.f;
    __syncthreads();
    const int nq = qcnt[row];
    for (int e = tid; e < nq; e += kThreads) qd[qidx[row * N + e]] = qval[row * N + e];
    __syncthreads();
    const int col = tid % DV, g = tid / DV;
    float o = 0.f;
    const float *Sb = ST + (size_t)bh * N * DV;
    for (int e = g; e < nq; e += G) o = fmaf(qval[row * N + e], Sb[(size_t)qidx[row * N + e] * DV + col], o);
    for (int si = warp; si <= ti; si += kThreads / 32) {
        const size_t srow = (size_t)bh * T_ + c0 + si;
        const int nk = kcnt[srow];
        float z = 0.f;
        for (int e = lane; e < nk; e += 32) z = fmaf(kval[srow * N + e], qd[kidx[srow * N + e]], z);
        z = warp_sum(z);
        if (lane == 0) zs[si] = z;
    }
    __syncthreads();
    for (int si = g; si <= ti; si += G)
        o = fmaf(zs[si], v[((size_t)bh * T_ + c0 + si) * DV + col], o);
    red[tid] = o;
    __syncthreads();
    if (tid < DV) {
        float s = 0.f;
        for (int gg = 0; gg < G; ++gg) s += red[gg * DV + tid];
        y[row * DV + tid] = s;
    }
}

template <int DV>
__global__ void __launch_bounds__(kThreads)
sparse_write_kernel(int c0, int T_, int N, const int *__restrict__ kidx,
                    const float *__restrict__ kval, const int *__restrict__ kcnt,
                    const float *__restrict__ v, float *__restrict__ ST) {
    constexpr int G = kThreads / DV;
    const int bh = blockIdx.y, tid = threadIdx.x;
    const size_t row = (size_t)bh * T_ + c0 + blockIdx.x;
    const int col = tid % DV, g = tid / DV;
    const float vv = v[row * DV + col];
    float *Sb = ST + (size_t)bh * N * DV;
    const int nk = kcnt[row];
    for (int e = g; e < nk; e += G)
        atomicAdd(&Sb[(size_t)kidx[row * N + e] * DV + col], kval[row * N + e] * vv);
}

struct WsLayout {
    int *kidx, *qidx, *kcnt, *qcnt;
    float *kval, *qval, *ST;
};

WsLayout carve(void *ws, int BH, int T, int N, int dv, bool need_state) {
    const size_t ent = (size_t)BH * T * N;
    char *p = (char *)ws;
    WsLayout l;
    l.kidx = (int *)p; p += align_up(sizeof(int) * ent, 256);
    l.qidx = (int *)p; p += align_up(sizeof(int) * ent, 256);
    l.kval = (float *)p; p += align_up(sizeof(float) * ent, 256);
    l.qval = (float *)p; p += align_up(sizeof(float) * ent, 256);
    l.kcnt = (int *)p; p += align_up(sizeof(int) * (size_t)BH * T, 256);
    l.qcnt = (int *)p; p += align_up(sizeof(int) * (size_t)BH * T, 256);
    l.ST = need_state ? (float *)p : nullptr;
    (void)dv;
    return l;
}

template <int DV>
int launch(const float *q, const float *k, const float *v, int BH, int T, int N, const float *S0,
           float *S_out, float *y, void *ws, cudaStream_t s) {
    const WsLayout l = carve(ws, BH, T, N, DV, S_out == nullptr);
    float *ST = S_out ? S_out : l.ST;
    const size_t state_bytes = sizeof(float) * (size_t)BH * N * DV;
    cudaError_t e;
    if (S0 == nullptr) e = cudaMemsetAsync(ST, 0, state_bytes, s);
    else if (S0 != ST) e = cudaMemcpyAsync(ST, S0, state_bytes, cudaMemcpyDeviceToDevice, s);
    else e = cudaSuccess;
    if (e != cudaSuccess) return cuda_fail(e, "sparse state init");
    const int rows = BH * T;
    compact_rows_kernel<<<ceil_div(rows, 8), 256, 0, s>>>(k, rows, N, l.kidx, l.kval, l.kcnt);
    if (int rc = launched("compact k")) return rc;
    compact_rows_kernel<<<ceil_div(rows, 8), 256, 0, s>>>(q, rows, N, l.qidx, l.qval, l.qcnt);
    if (int rc = launched("compact q")) return rc;
    const size_t smem = sizeof(float) * (size_t)N;
    e = cudaFuncSetAttribute(sparse_read_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "sparse_read smem attribute");
    prof_begin(s);
    for (int c0 = 0; c0 < T; c0 += kC) {
        const int n = min(kC, T - c0);
        sparse_read_kernel<DV><<<dim3(n, BH), kThreads, smem, s>>>(c0, T, N, l.kidx, l.kval, l.kcnt, l.qidx,
                                                                   l.qval, l.qcnt, v, ST, y);
        if (int rc = launched("sparse_read")) return rc;
        sparse_write_kernel<DV><<<dim3(n, BH), kThreads, 0, s>>>(c0, T, N, l.kidx, l.kval, l.kcnt, v, ST);
        if (int rc = launched("sparse_write")) return rc;
    }
    prof_end(s);
    return OPAM_OK;
}

}  // namespace

size_t sparse_workspace(int BH, int T, int N, int dv, bool need_state) {
    const size_t ent = (size_t)BH * T * N;
    size_t b = 2 * align_up(sizeof(int) * ent, 256) + 2 * align_up(sizeof(float) * ent, 256) +
               2 * align_up(sizeof(int) * (size_t)BH * T, 256);
    if (need_state) b += align_up(sizeof(float) * (size_t)BH * N * dv, 256);
    return b;
}

int sparse_forward(const float *q, const float *k, const float *v, int B, int H, int T, int N, int dv,
                   const float *S0, float *S_out, float *y, void *ws, cudaStream_t s) {
    const int BH = B * H;
    switch (dv) {
        case 32: return launch<32>(q, k, v, BH, T, N, S0, S_out, y, ws, s);
        case 64: return launch<64>(q, k, v, BH, T, N, S0, S_out, y, ws, s);
        case 128: return launch<128>(q, k, v, BH, T, N, S0, S_out, y, ws, s);
        case 256: return launch<256>(q, k, v, BH, T, N, S0, S_out, y, ws, s);
    }
    set_error("d_v=%d unsupported", dv);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace opam
