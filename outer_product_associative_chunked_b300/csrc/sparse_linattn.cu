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

// One CTA per (token t of the chunk, head).  o_t = q_t S (gathered over the
// support of q_t, float4 columns, LOOK loads in flight per thread) +
// sum_{s in chunk, s <= t} <k_s, q_t> v_s (keys' supports against a dense copy
// of q_t in shared memory).
template <int DV>
__global__ void __launch_bounds__(kThreads, 3)
sparse_read_kernel(int c0, int T_, int N, const int *__restrict__ kidx,
                   const float *__restrict__ kval, const int *__restrict__ kcnt,
                   const int *__restrict__ qidx, const float *__restrict__ qval,
                   const int *__restrict__ qcnt, const float *__restrict__ v,
                   const float *__restrict__ ST, float *__restrict__ y) {
    constexpr int CG = DV / 4;           // float4 column groups
    constexpr int RGN = kThreads / CG;   // support entries processed side by side
    constexpr int LOOK = 8;              // gathers in flight per thread
    extern __shared__ float qd[];        // [N] dense copy of q_t
    __shared__ float zs[kC];
    __shared__ float4 red[kThreads];
    const int ti = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const size_t row = (size_t)bh * T_ + c0 + ti;
    for (int j = tid; j < N; j += kThreads) qd[j] = 0.f;
    __syncthreads();
    const int nq = qcnt[row];
    const int *qi = qidx + row * N;
    const float *qv = qval + row * N;
    for (int e = tid; e < nq; e += kThreads) qd[qi[e]] = qv[e];
    const int cg = tid % CG, rg = tid / CG;
    const float4 *Sb = reinterpret_cast<const float4 *>(ST + (size_t)bh * N * DV);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e0 = rg; e0 < nq; e0 += RGN * LOOK) {
        float4 x[LOOK];
        float w[LOOK];
#pragma unroll
        for (int u = 0; u < LOOK; ++u) {
            const int e = e0 + u * RGN;
            const bool ok = e < nq;
            w[u] = ok ? qv[e] : 0.f;
            x[u] = ok ? Sb[(size_t)qi[e] * CG + cg] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < LOOK; ++u) {
            o.x = fmaf(w[u], x[u].x, o.x);
            o.y = fmaf(w[u], x[u].y, o.y);
            o.z = fmaf(w[u], x[u].z, o.z);
            o.w = fmaf(w[u], x[u].w, o.w);
        }
    }
    __syncthreads();  // qd complete
    for (int si = warp; si <= ti; si += kThreads / 32) {
        const size_t srow = (size_t)bh * T_ + c0 + si;
        const int nk = kcnt[srow];
        float z = 0.f;
        for (int e = lane; e < nk; e += 32) z = fmaf(kval[srow * N + e], qd[kidx[srow * N + e]], z);
        z = warp_sum(z);
        if (lane == 0) zs[si] = z;
    }
    __syncthreads();
    const float4 *vb = reinterpret_cast<const float4 *>(v + ((size_t)bh * T_ + c0) * DV);
    for (int si = rg; si <= ti; si += RGN) {
        const float z = zs[si];
        const float4 vv = vb[(size_t)si * CG + cg];
        o.x = fmaf(z, vv.x, o.x);
        o.y = fmaf(z, vv.y, o.y);
        o.z = fmaf(z, vv.z, o.z);
        o.w = fmaf(z, vv.w, o.w);
    }
    red[tid] = o;
    __syncthreads();
    if (tid < CG) {
        float4 s = red[tid];
        for (int g = 1; g < RGN; ++g) {
            const float4 a = red[g * CG + tid];
            s.x += a.x; s.y += a.y; s.z += a.z; s.w += a.w;
        }
        reinterpret_cast<float4 *>(y + row * DV)[tid] = s;
    }
}

// One CTA per (token s of the chunk, head): S[j, :] += k_s[j] v_s for every j
// in the support of k_s, as float4 vector reductions.
template <int DV>
__global__ void __launch_bounds__(kThreads)
sparse_write_kernel(int c0, int T_, int N, const int *__restrict__ kidx,
                    const float *__restrict__ kval, const int *__restrict__ kcnt,
                    const float *__restrict__ v, float *__restrict__ ST) {
    constexpr int CG = DV / 4, RGN = kThreads / CG;
    const int bh = blockIdx.y, tid = threadIdx.x;
    const size_t row = (size_t)bh * T_ + c0 + blockIdx.x;
    const int cg = tid % CG, rg = tid / CG;
    const float4 vv = reinterpret_cast<const float4 *>(v + row * DV)[cg];
    float4 *Sb = reinterpret_cast<float4 *>(ST + (size_t)bh * N * DV);
    const int nk = kcnt[row];
    const int *ki = kidx + row * N;
    const float *kv = kval + row * N;
#pragma unroll 4
    for (int e = rg; e < nk; e += RGN) {
        const float a = kv[e];
        atomicAdd(Sb + (size_t)ki[e] * CG + cg, make_float4(a * vv.x, a * vv.y, a * vv.z, a * vv.w));
    }
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
    if (int rc_ = set_smem_limit((const void *)sparse_read_kernel<DV>, (int)smem, "sparse_read smem attribute")) return rc_;
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
