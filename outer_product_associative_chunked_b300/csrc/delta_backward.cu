// DeltaNet delta-rule backward (CUDA cores, fp32 state; bf16 or fp32 tokens).
//
// molayo1419.me, "DeltaNet-family linear attention variants", section
// "DeltaNet: write the prediction error instead of the value": the forward
// step is u_t = v_t - S_{t-1} k_t, S_t = S_{t-1} + beta_t u_t k_t^T,
// o_t = S_t q_t (S is d_v x d_k).  Given do, the gradient of
// sum_t <do_t, o_t> (+ <dS_T, S_T>) follows from undoing the steps in
// reverse, with dS the gradient with respect to S_t:
//   dq_t = S_t^T do_t;  dS += do_t q_t^T;  g = dS k_t;
//   dv_t = beta_t g;  dbeta_t = <u_t, g>;
//   dk_t = beta_t dS^T u_t - S_{t-1}^T (beta_t g);
//   dS <- dS - beta_t g k_t^T.
//
// One CTA per (batch, head); its d_v/8 warps each own 8 rows of S and of dS
// in registers, a lane holding d_k/32 columns of each row as pairs updated with
// packed f32x2 FMAs (two FMAs per instruction), so every row
// update is lane-local and every column sum over the warp's rows is too.  The
// walk is sequential, so the time is the length of one warp's chain of
// instructions per token: fewer rows per warp (more warps) shorten it.
// Row sums over the columns (S k, dS k) go through a transposing warp
// reduction: 23 shuffles leave the total of row (lane mod 8) in each lane.
// Column sums over all d_v rows (dq, dk) and dbeta are combined across the
// warps in shared memory, one barrier per token.
//
// Pass 1 runs the recurrence forward from S_0 and stores every u_t; pass 2
// walks back from S_T, recovering S_{t-1} = S_t - beta_t u_t k_t^T exactly
// from the stored u_t (no division; rounding adds up linearly over the
// sequence), so no per-token state is kept.
#include <math.h>

#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {
namespace {

using sm100::fma2;

constexpr int kRows = 8;  // rows of S per warp

// x[0..7] summed over the 32 lanes; returns the total of row (lane & 7).
__device__ __forceinline__ float transpose_reduce(float (&x)[kRows]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o >= kRows; o >>= 1)
#pragma unroll
        for (int i = 0; i < kRows; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], o);
#pragma unroll
    for (int o = kRows / 2, n = kRows; o >= 1; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
            const float send = up ? x[j] : x[j + n / 2];
            const float keep = up ? x[j + n / 2] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return x[0];
}

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(DV / kRows * 32)
delta_backward_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                      const float *__restrict__ beta, const float *__restrict__ S0, const T *__restrict__ dy,
                      const float *__restrict__ dST, int Tn, float *__restrict__ U, T *__restrict__ dq,
                      T *__restrict__ dk, T *__restrict__ dv, float *__restrict__ dbeta, float *__restrict__ dS0,
                      unsigned int *__restrict__ status) {
    constexpr int CPL = DK / 32;          // columns per lane
    constexpr int CP = (CPL + 1) / 2;     // column pairs per lane (packed f32x2 arithmetic)
    constexpr int NW = DV / kRows;        // warps
    __shared__ float red[2][NW][2 * DK + 1];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, row = w * kRows + (lane & (kRows - 1));
    const int bh = blockIdx.x;
    const size_t tk = (size_t)bh * Tn * DK, tv = (size_t)bh * Tn * DV;
    // Columns of pair p: lane + 32 (2p) and lane + 32 (2p + 1); with an odd
    // count the last pair's second half is a zero column that stays zero.
    auto col = [&](int p, int h) { return lane + 32 * (2 * p + h); };
    auto has = [&](int p, int h) { return 2 * p + h < CPL; };
    float2 S[kRows][CP], dS[kRows][CP];
    // S stored key-major: S_{i,j} at [j * DV + i]
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
        for (int p = 0; p < CP; ++p) {
            float sv[2], dv2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const size_t at = (size_t)bh * DK * DV + (size_t)col(p, h) * DV + w * kRows + i;
                sv[h] = (S0 && has(p, h)) ? S0[at] : 0.f;
                dv2[h] = (dST && has(p, h)) ? dST[at] : 0.f;
            }
            S[i][p] = make_float2(sv[0], sv[1]);
            dS[i][p] = make_float2(dv2[0], dv2[1]);
        }
    auto load_pair = [&](const T *base, int p) {
        return make_float2(Elem<T>::load(base + col(p, 0)), has(p, 1) ? Elem<T>::load(base + col(p, 1)) : 0.f);
    };
    // ---- pass 1: forward, storing u_t.  The next token's inputs are loaded
    // while the current one is processed (the walk is sequential, so a load
    // issued at the top of its own step would expose the whole latency).
    float2 kn[CP];
    float bn = 0.f, vn = 0.f;
    auto fetch1 = [&](int t) {
#pragma unroll
        for (int p = 0; p < CP; ++p) kn[p] = load_pair(k + tk + (size_t)t * DK, p);
        bn = beta[(size_t)bh * Tn + t];
        vn = Elem<T>::load(v + tv + (size_t)t * DV + row);
    };
    if (Tn > 0) fetch1(0);
    for (int t = 0; t < Tn; ++t) {
        float2 kc[CP];
        float x[kRows];
#pragma unroll
        for (int p = 0; p < CP; ++p) kc[p] = kn[p];
        const float bt = bn, vr = vn;
        if (t + 1 < Tn) fetch1(t + 1);
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < CP; ++p) s2 = fma2(S[i][p], kc[p], s2);
            x[i] = s2.x + s2.y;
        }
        const float u = vr - transpose_reduce(x);
        if (lane < kRows && OPAM_BOUNDS(tv + (size_t)t * DV + row < (size_t)gridDim.x * Tn * DV, status))
            U[tv + (size_t)t * DV + row] = u;
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const float bu = bt * __shfl_sync(0xffffffffu, u, i);
            const float2 bu2 = make_float2(bu, bu);
#pragma unroll
            for (int p = 0; p < CP; ++p) S[i][p] = fma2(bu2, kc[p], S[i][p]);
        }
    }
    // ---- pass 2: reverse (next token's inputs prefetched as in pass 1)
    float2 qn[CP];
    float dn = 0.f, un = 0.f;
    auto fetch2 = [&](int t) {
#pragma unroll
        for (int p = 0; p < CP; ++p) {
            qn[p] = load_pair(q + tk + (size_t)t * DK, p);
            kn[p] = load_pair(k + tk + (size_t)t * DK, p);
        }
        bn = beta[(size_t)bh * Tn + t];
        dn = Elem<T>::load(dy + tv + (size_t)t * DV + row);
        un = U[tv + (size_t)t * DV + row];
    };
    __syncwarp();  // this lane's u stores of pass 1 precede its reloads
    if (Tn > 0) fetch2(Tn - 1);
    for (int t = Tn - 1; t >= 0; --t) {
        float2 qc[CP], kc[CP], dqp[CP], dkp[CP];
        float x[kRows];
#pragma unroll
        for (int p = 0; p < CP; ++p) {
            qc[p] = qn[p];
            kc[p] = kn[p];
            dqp[p] = make_float2(0.f, 0.f);
            dkp[p] = make_float2(0.f, 0.f);
        }
        const float bt = bn, dor = dn, ur = un;
        if (t > 0) fetch2(t - 1);
        // dq = S_t^T do;  dS += do q^T;  g = dS k
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const float di = __shfl_sync(0xffffffffu, dor, i);
            const float2 di2 = make_float2(di, di);
            float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < CP; ++p) {
                dqp[p] = fma2(S[i][p], di2, dqp[p]);
                dS[i][p] = fma2(di2, qc[p], dS[i][p]);
                s2 = fma2(dS[i][p], kc[p], s2);
            }
            x[i] = s2.x + s2.y;
        }
        const float g = transpose_reduce(x);
        const float du = bt * g;
        if (lane < kRows && OPAM_BOUNDS(tv + (size_t)t * DV + row < (size_t)gridDim.x * Tn * DV, status))
            Elem<T>::store(dv + tv + (size_t)t * DV + row, du);
        float db = lane < kRows ? ur * g : 0.f;
        db = warp_sum(db);
        // S <- S_{t-1};  dk = beta dS^T u - S_{t-1}^T du;  dS -= du k^T
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const float ui = __shfl_sync(0xffffffffu, ur, i);
            const float dui = __shfl_sync(0xffffffffu, du, i);
            const float bu = bt * ui;
            const float2 nbu2 = make_float2(-bu, -bu), bu2 = make_float2(bu, bu), ndu2 = make_float2(-dui, -dui);
#pragma unroll
            for (int p = 0; p < CP; ++p) {
                S[i][p] = fma2(nbu2, kc[p], S[i][p]);
                dkp[p] = fma2(bu2, dS[i][p], fma2(ndu2, S[i][p], dkp[p]));
                dS[i][p] = fma2(ndu2, kc[p], dS[i][p]);
            }
        }
        float(*buf)[2 * DK + 1] = red[t & 1];
#pragma unroll
        for (int p = 0; p < CP; ++p) {
            buf[w][col(p, 0)] = dqp[p].x;
            buf[w][DK + col(p, 0)] = dkp[p].x;
            if (has(p, 1)) {
                buf[w][col(p, 1)] = dqp[p].y;
                buf[w][DK + col(p, 1)] = dkp[p].y;
            }
        }
        if (lane == 0) buf[w][2 * DK] = db;
        __syncthreads();
        for (int idx = tid; idx <= 2 * DK; idx += NW * 32) {
            float s = 0.f;
#pragma unroll
            for (int ww = 0; ww < NW; ++ww) s += buf[ww][idx];
            if (!OPAM_BOUNDS(tk + (size_t)t * DK + DK <= (size_t)gridDim.x * Tn * DK, status)) continue;
            if (idx < DK)
                Elem<T>::store(dq + tk + (size_t)t * DK + idx, s);
            else if (idx < 2 * DK)
                Elem<T>::store(dk + tk + (size_t)t * DK + idx - DK, s);
            else
                dbeta[(size_t)bh * Tn + t] = s;
        }
    }
    if (dS0) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
#pragma unroll
            for (int p = 0; p < CP; ++p) {
                dS0[(size_t)bh * DK * DV + (size_t)col(p, 0) * DV + w * kRows + i] = dS[i][p].x;
                if (has(p, 1)) dS0[(size_t)bh * DK * DV + (size_t)col(p, 1) * DV + w * kRows + i] = dS[i][p].y;
            }
    }
    // nothing here waits on a barrier: the call's status words only need zeroing
    if (bh == 0 && tid < kStatusWords) status[tid] = 0u;
}

template <typename T, int DK, int DV>
int launch(const void *q, const void *k, const void *v, const float *beta, const float *S0, const void *dy,
           const float *dST, int BH, int Tn, void *dq, void *dk, void *dv, float *dbeta, float *dS0, void *ws,
           unsigned int *status, cudaStream_t s) {
    delta_backward_kernel<T, DK, DV><<<BH, DV / kRows * 32, 0, s>>>(
        (const T *)q, (const T *)k, (const T *)v, beta, S0, (const T *)dy, dST, Tn, (float *)ws, (T *)dq,
        (T *)dk, (T *)dv, dbeta, dS0, status);
    return launched("delta_backward");
}

template <typename T, int DK>
int by_dv(int dvv, const void *q, const void *k, const void *v, const float *beta, const float *S0,
          const void *dy, const float *dST, int BH, int Tn, void *dq, void *dk, void *dv, float *dbeta,
          float *dS0, void *ws, unsigned int *status, cudaStream_t s) {
    switch (dvv) {
        case 32: return launch<T, DK, 32>(q, k, v, beta, S0, dy, dST, BH, Tn, dq, dk, dv, dbeta, dS0, ws, status, s);
        case 64: return launch<T, DK, 64>(q, k, v, beta, S0, dy, dST, BH, Tn, dq, dk, dv, dbeta, dS0, ws, status, s);
        case 128: return launch<T, DK, 128>(q, k, v, beta, S0, dy, dST, BH, Tn, dq, dk, dv, dbeta, dS0, ws, status, s);
    }
    set_error("delta_rule_backward: d_v=%d unsupported", dvv);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace

size_t delta_backward_workspace(int BH, int T, int dv) { return align_up(sizeof(float) * (size_t)BH * T * dv, 256); }

int delta_backward(const void *q, const void *k, const void *v, const float *beta, int dtype, int B, int H, int T,
                   int dkk, int dvv, const float *S0, const void *dy, const float *dST, void *dq, void *dk,
                   void *dv, float *dbeta, float *dS0, void *ws, unsigned int *status, cudaStream_t s) {
    const int BH = B * H;
    prof_begin(s);
    int rc;
    if (dtype == OPAM_BF16) {
        switch (dkk) {
            case 32: rc = by_dv<__nv_bfloat16, 32>(dvv, q, k, v, beta, S0, dy, dST, BH, T, dq, dk, dv, dbeta, dS0, ws, status, s); break;
            case 64: rc = by_dv<__nv_bfloat16, 64>(dvv, q, k, v, beta, S0, dy, dST, BH, T, dq, dk, dv, dbeta, dS0, ws, status, s); break;
            case 128: rc = by_dv<__nv_bfloat16, 128>(dvv, q, k, v, beta, S0, dy, dST, BH, T, dq, dk, dv, dbeta, dS0, ws, status, s); break;
            default: set_error("delta_rule_backward: d_k=%d unsupported", dkk); return OPAM_ERR_UNSUPPORTED;
        }
    } else {
        switch (dkk) {
            case 32: rc = by_dv<float, 32>(dvv, q, k, v, beta, S0, dy, dST, BH, T, dq, dk, dv, dbeta, dS0, ws, status, s); break;
            case 64: rc = by_dv<float, 64>(dvv, q, k, v, beta, S0, dy, dST, BH, T, dq, dk, dv, dbeta, dS0, ws, status, s); break;
            case 128: rc = by_dv<float, 128>(dvv, q, k, v, beta, S0, dy, dST, BH, T, dq, dk, dv, dbeta, dS0, ws, status, s); break;
            default: set_error("delta_rule_backward: d_k=%d unsupported", dkk); return OPAM_ERR_UNSUPPORTED;
        }
    }
    prof_end(s);
    return rc;
}

}  // namespace opam
