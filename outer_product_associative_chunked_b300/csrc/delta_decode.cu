// DeltaNet single-token decode for a batch of independent sequences.
//
// molayo1419.me, "DeltaNet-family linear attention variants", section
// "DeltaNet: write the prediction error instead of the value":
//     e = beta (v - S k),   S <- S + e k^T,   o = S q (read after the write).
//
// The state is stored key-major, M = S^T with M[j][i] = S_{i,j} (d_k rows of
// d_v floats), the layout delta_rule_forward exports.  Column i of M is row i
// of S, and a step touches each column on its own:
//     (S k)_i = sum_j M[j][i] k_j,      (S q)_i = sum_j M[j][i] q_j,
//     e_i = beta (v_i - (S k)_i),       M[j][i] += k_j e_i,
//     o_i = (S q)_i + e_i <k, q>        (since S_new q = S q + e <k, q>).
// So one pass reads M once and writes it once: the step is bound by HBM
// (2 d_k d_v 4 bytes per sequence and head).
//
// Grid: (d_v / CB column blocks, sequences x heads).  A CTA of 256 threads
// owns CB columns of one head: thread (r, c) holds rows r*RPT .. r*RPT+RPT-1
// of column group c (4 columns, one 16-byte vector per row) in registers
// between the read and the write.  The two column sums are reduced over the
// RS row slices through shared memory.
#include "opam_internal.cuh"

namespace opam {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float4 ld_state(const float *p) {
    float4 r;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

template <int DK, int DV>
struct DecodeGeom {
    static constexpr int CB = DV < 64 ? DV : 64;  // columns per CTA
    static constexpr int CG = CB / 4;             // 16-byte column groups per CTA
    static constexpr int RS = kThreads / CG;      // row slices
    static constexpr int RPT = DK / RS;           // rows per thread
    static_assert(RS * CG == kThreads && RPT * RS == DK, "decode geometry");
};

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
delta_decode_kernel(float *__restrict__ M, const T *__restrict__ q, const T *__restrict__ k,
                    const T *__restrict__ v, const float *__restrict__ beta, T *__restrict__ y) {
    using G = DecodeGeom<DK, DV>;
    __shared__ float ks[DK], qs[DK], kq;
    __shared__ __align__(16) float es[G::CB];
    __shared__ __align__(16) float red[2][G::RS][G::CB];
    const int tid = threadIdx.x, c = tid % G::CG, r = tid / G::CG;
    const int bh = blockIdx.y, col0 = blockIdx.x * G::CB;
    float *Mh = M + (size_t)bh * DK * DV + col0 + 4 * c;

    // The state loads go first; they do not depend on the token.
    float4 m[G::RPT];
#pragma unroll
    for (int u = 0; u < G::RPT; ++u) m[u] = ld_state(Mh + (size_t)(r * G::RPT + u) * DV);

    if (tid < DK) {
        ks[tid] = Elem<T>::load(k + (size_t)bh * DK + tid);
        qs[tid] = Elem<T>::load(q + (size_t)bh * DK + tid);
    }
    __syncthreads();
    if (tid < 32) {
        float s = 0.f;
#pragma unroll
        for (int j = tid; j < DK; j += 32) s = fmaf(ks[j], qs[j], s);
        s = warp_sum(s);
        if (tid == 0) kq = s;
    }

    float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sq = sk;
#pragma unroll
    for (int u = 0; u < G::RPT; ++u) {
        const float kj = ks[r * G::RPT + u], qj = qs[r * G::RPT + u];
        sk.x = fmaf(m[u].x, kj, sk.x); sk.y = fmaf(m[u].y, kj, sk.y);
        sk.z = fmaf(m[u].z, kj, sk.z); sk.w = fmaf(m[u].w, kj, sk.w);
        sq.x = fmaf(m[u].x, qj, sq.x); sq.y = fmaf(m[u].y, qj, sq.y);
        sq.z = fmaf(m[u].z, qj, sq.z); sq.w = fmaf(m[u].w, qj, sq.w);
    }
    *reinterpret_cast<float4 *>(&red[0][r][4 * c]) = sk;
    *reinterpret_cast<float4 *>(&red[1][r][4 * c]) = sq;
    __syncthreads();

    if (tid < G::CB) {
        const int i = tid;
        float a = 0.f, b = 0.f;
#pragma unroll 8
        for (int s = 0; s < G::RS; ++s) {
            a += red[0][s][i];
            b += red[1][s][i];
        }
        const float e = beta[bh] * (Elem<T>::load(v + (size_t)bh * DV + col0 + i) - a);
        es[i] = e;
        Elem<T>::store(y + (size_t)bh * DV + col0 + i, fmaf(e, kq, b));
    }
    __syncthreads();

    const float4 e4 = *reinterpret_cast<const float4 *>(&es[4 * c]);
#pragma unroll
    for (int u = 0; u < G::RPT; ++u) {
        const float kj = ks[r * G::RPT + u];
        float4 w = m[u];
        w.x = fmaf(kj, e4.x, w.x); w.y = fmaf(kj, e4.y, w.y);
        w.z = fmaf(kj, e4.z, w.z); w.w = fmaf(kj, e4.w, w.w);
        *reinterpret_cast<float4 *>(Mh + (size_t)(r * G::RPT + u) * DV) = w;
    }
}

template <typename T, int DK, int DV>
int launch(float *S, const void *q, const void *k, const void *v, const float *beta, int BH, void *y,
           cudaStream_t s) {
    using G = DecodeGeom<DK, DV>;
    prof_begin(s);
    delta_decode_kernel<T, DK, DV><<<dim3(DV / G::CB, BH), kThreads, 0, s>>>(
        S, (const T *)q, (const T *)k, (const T *)v, beta, (T *)y);
    const int rc = launched("delta_decode");
    prof_end(s);
    return rc;
}

template <typename T, int DK>
int dispatch_dv(float *S, const void *q, const void *k, const void *v, const float *beta, int BH, int dv,
                void *y, cudaStream_t s) {
    switch (dv) {
        case 32: return launch<T, DK, 32>(S, q, k, v, beta, BH, y, s);
        case 64: return launch<T, DK, 64>(S, q, k, v, beta, BH, y, s);
        default: return launch<T, DK, 128>(S, q, k, v, beta, BH, y, s);
    }
}

template <typename T>
int dispatch(float *S, const void *q, const void *k, const void *v, const float *beta, int BH, int dk,
             int dv, void *y, cudaStream_t s) {
    switch (dk) {
        case 32: return dispatch_dv<T, 32>(S, q, k, v, beta, BH, dv, y, s);
        case 64: return dispatch_dv<T, 64>(S, q, k, v, beta, BH, dv, y, s);
        default: return dispatch_dv<T, 128>(S, q, k, v, beta, BH, dv, y, s);
    }
}

}  // namespace

int delta_decode(float *S, const void *q, const void *k, const void *v, const float *beta, int dtype,
                 int B, int H, int dk, int dv, void *y, cudaStream_t s) {
    const int BH = B * H;
    return dtype == OPAM_BF16 ? dispatch<__nv_bfloat16>(S, q, k, v, beta, BH, dk, dv, y, s)
                              : dispatch<float>(S, q, k, v, beta, BH, dk, dv, y, s);
}

}  // namespace opam
