// DeltaNet delta rule on CUDA cores (FFMA, fp32 state).
//
// molayo1419.me, "DeltaNet-family linear attention variants", section
// "DeltaNet: write the prediction error instead of the value":
//     e_t = beta_t (v_t - S_{t-1} k_t),   S_t = S_{t-1} + e_t k_t^T,
// read o_t = S_t q_t after the write.
//
// Chunked closed form (derived from the recurrence itself).  Inside a chunk,
// with rows = tokens, S0 the state at the chunk start and
// u_i = e_i = beta_i (v_i - S0 k_i - sum_{j<i} u_j <k_j, k_i>):
//     (I + diag(beta) L) U = diag(beta) (V - K S0^T),  L = strict_lower(K K^T)
// so with T = (I + diag(beta) L)^{-1} (unit lower triangular),
//     W~ = T diag(beta) K,  U~ = T diag(beta) V,  U = U~ - W~ S0^T,
//     O  = Q S0^T + (Q K^T masked to j <= i) U,   S_end = S0 + U^T K.
// W~, U~ and the masked Q K^T depend only on the chunk's inputs, so they are
// computed for all chunks in parallel (prep kernel, a forward substitution
// per chunk); the state pass is then sequential over chunks.  Rows of S
// (columns of the key-major S^T) evolve independently, so the state pass
// splits d_v over CTAs.
#include "opam_internal.cuh"

namespace opam {
namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 32;  // value columns per state-pass CTA

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
delta_prep_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                  const float *__restrict__ beta, int T_, int C, float *__restrict__ Wt,
                  float *__restrict__ Ut, float *__restrict__ P) {
    extern __shared__ float sm[];
    float *Ks = sm;                      // [C][DK+1]
    float *Qs = Ks + C * (DK + 1);       // [C][DK+1]
    float *X = Qs + C * (DK + 1);        // [C][DK+DV]  beta-scaled K|V, solved in place
    float *L = X + C * (DK + DV);        // [C][C+1]
    float *bs = L + C * (C + 1);         // [C]
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C, n = min(C, T_ - t0);
    const size_t base = (size_t)bh * T_ + t0;                 // input rows
    const size_t wbase = (size_t)bh * gridDim.x * C + t0;     // whole-chunk padded rows
    for (int idx = tid; idx < C * DK; idx += kThreads) {
        const int r = idx / DK, a = idx - r * DK;
        Ks[r * (DK + 1) + a] = r < n ? Elem<T>::load(k + (base + r) * DK + a) : 0.f;
        Qs[r * (DK + 1) + a] = r < n ? Elem<T>::load(q + (base + r) * DK + a) : 0.f;
    }
    for (int r = tid; r < C; r += kThreads) bs[r] = r < n ? beta[base + r] : 0.f;
    __syncthreads();
    for (int idx = tid; idx < C * (DK + DV); idx += kThreads) {
        const int r = idx / (DK + DV), col = idx - r * (DK + DV);
        const float x = col < DK ? Ks[r * (DK + 1) + col]
                                 : (r < n ? Elem<T>::load(v + (base + r) * DV + (col - DK)) : 0.f);
        X[idx] = bs[r] * x;
    }
    // L = strict_lower(K K^T); P = (Q K^T) masked to j <= i.
    float *Pc = P + ((size_t)bh * gridDim.x + c) * C * C;
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int i = idx / C, j = idx - i * C;
        float kk = 0.f, qk = 0.f;
        if (j <= i) {
            for (int a = 0; a < DK; ++a) {
                kk = fmaf(Ks[i * (DK + 1) + a], Ks[j * (DK + 1) + a], kk);
                qk = fmaf(Qs[i * (DK + 1) + a], Ks[j * (DK + 1) + a], qk);
            }
        }
        L[i * (C + 1) + j] = j < i ? kk : 0.f;
        Pc[idx] = qk;
    }
    __syncthreads();
    // Forward substitution, one column per thread: X_i -= beta_i sum_{j<i} L_ij X_j.
    for (int col = tid; col < DK + DV; col += kThreads) {
        for (int i = 1; i < n; ++i) {
            float acc = 0.f;
            for (int j = 0; j < i; ++j) acc = fmaf(L[i * (C + 1) + j], X[j * (DK + DV) + col], acc);
            X[i * (DK + DV) + col] -= bs[i] * acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < C * DK; idx += kThreads) {
        const int r = idx / DK, a = idx - r * DK;
        Wt[(wbase + r) * DK + a] = X[r * (DK + DV) + a];
    }
    for (int idx = tid; idx < C * DV; idx += kThreads) {
        const int r = idx / DV, b = idx - r * DV;
        Ut[(wbase + r) * DV + b] = X[r * (DK + DV) + DK + b];
    }
}

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
delta_state_kernel(const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ Wt,
                   const float *__restrict__ Ut, const float *__restrict__ P, int T_, int C,
                   int nch, const float *S0, float *S_out,
                   T *__restrict__ y) {
    extern __shared__ float sm[];
    float *ST = sm;                        // [DK][kSlice] state columns of this CTA
    float *Ws = ST + DK * kSlice;          // [C][DK+1]
    float *Qs = Ws + C * (DK + 1);         // [C][DK+1]
    float *Ks = Qs + C * (DK + 1);         // [C][DK+1]
    float *Us = Ks + C * (DK + 1);         // [C][kSlice]
    float *Ps = Us + C * kSlice;           // [C][C+1]
    const int bh = blockIdx.x, c0 = blockIdx.y * kSlice, tid = threadIdx.x;
    for (int idx = tid; idx < DK * kSlice; idx += kThreads) {
        const int a = idx / kSlice, b = idx - a * kSlice;
        ST[idx] = S0 ? S0[((size_t)bh * DK + a) * DV + c0 + b] : 0.f;
    }
    for (int ch = 0; ch < nch; ++ch) {
        const int t0 = ch * C, n = min(C, T_ - t0);
        const size_t base = (size_t)bh * T_ + t0;            // input / output rows
        const size_t wbase = (size_t)bh * nch * C + t0;      // padded W~ / U~ rows
        __syncthreads();
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int r = idx / DK, a = idx - r * DK;
            const bool ok = r < n;
            Ws[r * (DK + 1) + a] = ok ? Wt[(wbase + r) * DK + a] : 0.f;
            Qs[r * (DK + 1) + a] = ok ? Elem<T>::load(q + (base + r) * DK + a) : 0.f;
            Ks[r * (DK + 1) + a] = ok ? Elem<T>::load(k + (base + r) * DK + a) : 0.f;
        }
        const float *Pc = P + ((size_t)bh * nch + ch) * C * C;
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int i = idx / C, j = idx - i * C;
            Ps[i * (C + 1) + j] = (i < n) ? Pc[idx] : 0.f;
        }
        __syncthreads();
        // U = U~ - W~ S0^T  (this CTA's columns)
        for (int idx = tid; idx < C * kSlice; idx += kThreads) {
            const int r = idx / kSlice, b = idx - r * kSlice;
            float acc = r < n ? Ut[(wbase + r) * DV + c0 + b] : 0.f;
            for (int a = 0; a < DK; ++a) acc = fmaf(-Ws[r * (DK + 1) + a], ST[a * kSlice + b], acc);
            Us[idx] = acc;
        }
        __syncthreads();
        // O = Q S0^T + P U
        for (int idx = tid; idx < C * kSlice; idx += kThreads) {
            const int r = idx / kSlice, b = idx - r * kSlice;
            if (r >= n) continue;
            float acc = 0.f;
            for (int a = 0; a < DK; ++a) acc = fmaf(Qs[r * (DK + 1) + a], ST[a * kSlice + b], acc);
            for (int j = 0; j <= r; ++j) acc = fmaf(Ps[r * (C + 1) + j], Us[j * kSlice + b], acc);
            Elem<T>::store(y + (base + r) * DV + c0 + b, acc);
        }
        __syncthreads();
        // S^T += K^T U
        for (int idx = tid; idx < DK * kSlice; idx += kThreads) {
            const int a = idx / kSlice, b = idx - a * kSlice;
            float acc = ST[idx];
            for (int r = 0; r < n; ++r) acc = fmaf(Ks[r * (DK + 1) + a], Us[r * kSlice + b], acc);
            ST[idx] = acc;
        }
    }
    __syncthreads();
    if (S_out)
        for (int idx = tid; idx < DK * kSlice; idx += kThreads) {
            const int a = idx / kSlice, b = idx - a * kSlice;
            S_out[((size_t)bh * DK + a) * DV + c0 + b] = ST[idx];
        }
}

struct WsLayout {
    float *Wt, *Ut, *P;
};

WsLayout carve(void *ws, int BH, int T, int dk, int dv, int C) {
    const int nch = ceil_div(T, C);
    const size_t Tp = (size_t)nch * C;
    char *p = (char *)ws;
    WsLayout l;
    l.Wt = (float *)p;
    p += align_up(sizeof(float) * BH * Tp * dk, 256);
    l.Ut = (float *)p;
    p += align_up(sizeof(float) * BH * Tp * dv, 256);
    l.P = (float *)p;
    return l;
}

template <typename T, int DK, int DV>
int launch(const void *q, const void *k, const void *v, const float *beta, int BH, int T_, int C,
           const float *S0, float *S_out, void *y, void *ws, cudaStream_t s) {
    const int nch = ceil_div(T_, C);
    const WsLayout l = carve(ws, BH, T_, DK, DV, C);
    // W~ and U~ are stored padded to whole chunks (nch*C rows per unit), so
    // the prep kernel's tail rows stay inside their own unit.
    const size_t smem1 = sizeof(float) * (2 * C * (DK + 1) + C * (DK + DV) + C * (C + 1) + C);
    auto k1 = delta_prep_kernel<T, DK, DV>;
    if (int rc_ = set_smem_limit((const void *)k1, (int)smem1, "delta_prep smem attribute")) return rc_;
    k1<<<dim3(nch, BH), kThreads, smem1, s>>>((const T *)q, (const T *)k, (const T *)v, beta, T_, C,
                                             l.Wt, l.Ut, l.P);
    if (int rc = launched("delta_prep")) return rc;
    const size_t smem2 = sizeof(float) * (DK * kSlice + 3 * C * (DK + 1) + C * kSlice + C * (C + 1));
    auto k2 = delta_state_kernel<T, DK, DV>;
    if (int rc_ = set_smem_limit((const void *)k2, (int)smem2, "delta_state smem attribute")) return rc_;
    prof_begin(s);
    k2<<<dim3(BH, DV / kSlice), kThreads, smem2, s>>>((const T *)q, (const T *)k, l.Wt, l.Ut, l.P, T_,
                                                     C, nch, S0, S_out, (T *)y);
    const int rc = launched("delta_state");
    prof_end(s);
    return rc;
}

template <typename T, int DK>
int by_dv(int dv, const void *q, const void *k, const void *v, const float *beta, int BH, int T_,
          int C, const float *S0, float *S_out, void *y, void *ws, cudaStream_t s) {
    switch (dv) {
        case 32: return launch<T, DK, 32>(q, k, v, beta, BH, T_, C, S0, S_out, y, ws, s);
        case 64: return launch<T, DK, 64>(q, k, v, beta, BH, T_, C, S0, S_out, y, ws, s);
        case 128: return launch<T, DK, 128>(q, k, v, beta, BH, T_, C, S0, S_out, y, ws, s);
    }
    set_error("d_v=%d unsupported", dv);
    return OPAM_ERR_UNSUPPORTED;
}

template <typename T>
int by_dk(int dk, int dv, const void *q, const void *k, const void *v, const float *beta, int BH,
          int T_, int C, const float *S0, float *S_out, void *y, void *ws, cudaStream_t s) {
    switch (dk) {
        case 32: return by_dv<T, 32>(dv, q, k, v, beta, BH, T_, C, S0, S_out, y, ws, s);
        case 64: return by_dv<T, 64>(dv, q, k, v, beta, BH, T_, C, S0, S_out, y, ws, s);
        case 128: return by_dv<T, 128>(dv, q, k, v, beta, BH, T_, C, S0, S_out, y, ws, s);
    }
    set_error("d_k=%d unsupported", dk);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace

size_t delta_simt_workspace(int BH, int T, int dk, int dv, int C) {
    const int nch = ceil_div(T, C);
    const size_t Tp = (size_t)nch * C;
    return align_up(sizeof(float) * BH * Tp * dk, 256) + align_up(sizeof(float) * BH * Tp * dv, 256) +
           align_up(sizeof(float) * (size_t)BH * nch * C * C, 256);
}

int delta_simt(const void *q, const void *k, const void *v, const float *beta, int dtype, int B,
               int H, int T, int dk, int dv, int C, const float *S0, float *S_out, void *y, void *ws,
               cudaStream_t s) {
    if (dtype == OPAM_BF16)
        return by_dk<__nv_bfloat16>(dk, dv, q, k, v, beta, B * H, T, C, S0, S_out, y, ws, s);
    return by_dk<float>(dk, dv, q, k, v, beta, B * H, T, C, S0, S_out, y, ws, s);
}

}  // namespace opam
