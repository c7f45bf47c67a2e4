// Tensor Cache layer backward (CUDA cores, fp32 arithmetic; bf16 or fp32
// inputs and gradients).
//
// "Tensor Cache: Eviction-conditioned Associative Memory for Transformers"
// (gist.science 2605.22884): the layer is y_t = y_local,t + sigmoid(g) m_t
// (Methodology 1) and the parallel weighted-sum scan is what lets it train
// (Methodology 2).  Given dy, this computes the gradient of sum_t <dy_t, y_t>
// with respect to q, k, v and the per-head lambda, eta, g.
//
// Two independent parts, as in the forward:
//
// Window softmax (token s reaches y_t iff t-W < s <= t):
//   P = softmax(scale Q K^T) on the band, y_loc = P V,
//   D_t = <dy_t, y_loc,t>,  dS = P (dy V^T - D),
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dy.
//   tcb_window_dq_kernel (per block of 64 queries) recomputes the softmax
//   statistics and y_loc (first pass over the key tiles), stores LSE and D,
//   then accumulates dQ (second pass); tcb_window_dkdv_kernel (per block of
//   64 keys) walks the query tiles that see those keys.
//
// L2 memory, with shifted keys k'_u = k_{u-W}, v'_u = v_{u-W} (the token
// evicted at step u) and dm_t = sigmoid(g) dy_t:
//   m_t = sum_{u<=t} eta lambda^(t-u) <q_t, k'_u> v'_u.
// Its gradient, in chunks of C = 64 positions (row i of a chunk, n rows),
// with A_c the state before the chunk, A'_c = dA_c/dlambda, and
// R_{c+1} = sum_{t after the chunk} lambda^(t - end) q_t dm_t^T:
//   intra-chunk (tcb_l2_intra_kernel), D_ij = eta lambda^(i-j) for j <= i:
//     dq_i  += sum_j D_ij <dm_i, v'_j> k'_j,   dk'_j += sum_i D_ij <dm_i, v'_j> q_i,
//     dv'_j += sum_i D_ij <q_i, k'_j> dm_i,    m_i   += sum_j D_ij <q_i, k'_j> v'_j,
//     deta += sum_{j<=i} lambda^(i-j) <q_i,k'_j><dm_i,v'_j>,
//     dlambda += sum_{j<=i} eta (i-j) lambda^(i-j-1) <q_i,k'_j><dm_i,v'_j>;
//   chunk states (tcb_l2_scan_kernel; forward and reverse CTAs in one grid,
//   each on a 16-column slice of d_v):
//     forward: dq_i += lambda^(i+1) A_c dm_i,  m_i += lambda^(i+1) q_i A_c,
//       dlambda += (i+1) lambda^i q_i A_c dm_i + lambda^(i+1) q_i A'_c dm_i,
//       A_{c+1}  = lambda^n A_c + sum_j eta lambda^(n-1-j) k'_j v'_j^T,
//       A'_{c+1} = n lambda^(n-1) A_c + lambda^n A'_c
//                  + sum_j eta (n-1-j) lambda^(n-2-j) k'_j v'_j^T;
//     reverse: dk'_j += eta lambda^(n-j) R_{c+1} v'_j,
//       dv'_j += eta lambda^(n-j) R_{c+1}^T k'_j,
//       deta += sum_j lambda^(n-j) k'_j^T R_{c+1} v'_j,
//       R_c = lambda^n R_{c+1} + sum_i lambda^i q_i dm_i^T.
//   dg = sigmoid'(g) sum <dy, m> = (1 - sigmoid(g)) sum <dm, m>.
// dk'_u and dv'_u belong to token u - W.  tcb_finalize_kernel adds nothing
// new: it writes the fp32 accumulators out in the element type and sums the
// per-chunk scalar partials over chunks and batch in a fixed order.
//
// Every product is a 64-row tile contraction in shared memory (mm_tile:
// 256 threads as a 16 x 16 grid, each owning a 4 x (N/16) block).
#include <math.h>

#include <type_traits>

#include "opam_internal.cuh"

namespace opam {
namespace {

constexpr int kR = 64;         // rows per tile: queries, keys, chunk positions
constexpr int kThr = 256;
constexpr int kSW = 16;        // d_v columns per scan CTA
constexpr int kLS = kR + 1;    // padded stride of a 64 x 64 score tile

// acc[i][j] += sum_k A(m_i, k) B(k, n_j) with m_i = ty + 16 i, n_j = tx + 16 j;
// A(m, k) = A[m * am + k * ak], B(k, n) = B[k * bk + n * bn] (shared memory).
// AV / BV: A (B) is contiguous along k (ak = 1, bk = 1) with 16-byte aligned
// rows (am, bn and the base a multiple of 4 floats), and K a multiple of 4:
// four k steps of it come in one 16-byte load.  The FMAs run in the same
// order either way, so the results are identical.
template <int TM, int TN, bool AV = false, bool BV = false>
__device__ __forceinline__ void mm_tile(float (&acc)[TM][TN], const float *A, int am, int ak, const float *B,
                                        int bk, int bn, int K) {
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    if constexpr (AV || BV) {
#pragma unroll 2
        for (int k0 = 0; k0 < K; k0 += 4) {
            float a[TM][4], b[TN][4];
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                if constexpr (AV) {
                    const float4 x = *reinterpret_cast<const float4 *>(A + (ty + 16 * i) * am + k0);
                    a[i][0] = x.x; a[i][1] = x.y; a[i][2] = x.z; a[i][3] = x.w;
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) a[i][kk] = A[(ty + 16 * i) * am + (k0 + kk) * ak];
                }
            }
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                if constexpr (BV) {
                    const float4 x = *reinterpret_cast<const float4 *>(B + k0 + (tx + 16 * j) * bn);
                    b[j][0] = x.x; b[j][1] = x.y; b[j][2] = x.z; b[j][3] = x.w;
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) b[j][kk] = B[(k0 + kk) * bk + (tx + 16 * j) * bn];
                }
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i][kk], b[j][kk], acc[i][j]);
        }
    } else {
#pragma unroll 4
        for (int k = 0; k < K; ++k) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = A[(ty + 16 * i) * am + k * ak];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = B[k * bk + (tx + 16 * j) * bn];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
}

// Two single-column products that share A, in one pass over it:
// acc0[i] += sum_k A(m_i, k) B0(k, tx), acc1[i] += sum_k A(m_i, k) B1(k, tx)
// (the same order of operations per accumulator as two mm_tile<TM, 1> calls).
template <int TM, bool AV = false>
__device__ __forceinline__ void mm_tile_2(float (&acc0)[TM][1], float (&acc1)[TM][1], const float *A, int am, int ak,
                                          const float *B0, const float *B1, int bk, int bn, int K) {
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    if constexpr (AV) {  // A contiguous along k, as for mm_tile
#pragma unroll 2
        for (int k0 = 0; k0 < K; k0 += 4) {
            float a[TM][4];
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float4 x = *reinterpret_cast<const float4 *>(A + (ty + 16 * i) * am + k0);
                a[i][0] = x.x; a[i][1] = x.y; a[i][2] = x.z; a[i][3] = x.w;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float b0 = B0[(k0 + kk) * bk + tx * bn], b1 = B1[(k0 + kk) * bk + tx * bn];
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    acc0[i][0] = fmaf(a[i][kk], b0, acc0[i][0]);
                    acc1[i][0] = fmaf(a[i][kk], b1, acc1[i][0]);
                }
            }
        }
    } else {
#pragma unroll 4
        for (int k = 0; k < K; ++k) {
            float a[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = A[(ty + 16 * i) * am + k * ak];
            const float b0 = B0[k * bk + tx * bn], b1 = B1[k * bk + tx * bn];
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                acc0[i][0] = fmaf(a[i], b0, acc0[i][0]);
                acc1[i][0] = fmaf(a[i], b1, acc1[i][0]);
            }
        }
    }
}

// Single-column products whose A is contiguous along m (A(m, k) = A[m + k ak],
// ak a multiple of 4, 16-byte aligned base): thread ty owns rows
// mrow4(i) = 64 (i / 4) + 4 ty + i % 4, four of them per 16-byte load.
__device__ __forceinline__ int mrow4(int i) { return 64 * (i >> 2) + 4 * (threadIdx.x >> 4) + (i & 3); }

template <int TM>
__device__ __forceinline__ void mm_tile_m4(float (&acc)[TM][1], const float *A, int ak, const float *B, int bk,
                                           int bn, int K) {
    static_assert(TM % 4 == 0, "rows in groups of four");
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        float a[TM];
#pragma unroll
        for (int g = 0; g < TM / 4; ++g) {
            const float4 x = *reinterpret_cast<const float4 *>(A + 64 * g + 4 * ty + k * ak);
            a[4 * g] = x.x; a[4 * g + 1] = x.y; a[4 * g + 2] = x.z; a[4 * g + 3] = x.w;
        }
        const float b = B[k * bk + tx * bn];
#pragma unroll
        for (int i = 0; i < TM; ++i) acc[i][0] = fmaf(a[i], b, acc[i][0]);
    }
}

// The same with two B operands sharing A (as mm_tile_2).
template <int TM>
__device__ __forceinline__ void mm_tile_2_m4(float (&acc0)[TM][1], float (&acc1)[TM][1], const float *A, int ak,
                                             const float *B0, const float *B1, int bk, int bn, int K) {
    static_assert(TM % 4 == 0, "rows in groups of four");
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        float a[TM];
#pragma unroll
        for (int g = 0; g < TM / 4; ++g) {
            const float4 x = *reinterpret_cast<const float4 *>(A + 64 * g + 4 * ty + k * ak);
            a[4 * g] = x.x; a[4 * g + 1] = x.y; a[4 * g + 2] = x.z; a[4 * g + 3] = x.w;
        }
        const float b0 = B0[k * bk + tx * bn], b1 = B1[k * bk + tx * bn];
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            acc0[i][0] = fmaf(a[i], b0, acc0[i][0]);
            acc1[i][0] = fmaf(a[i], b1, acc1[i][0]);
        }
    }
}

template <int TM, int TN>
__device__ __forceinline__ void zero(float (&acc)[TM][TN]) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
}

// Rows r0 .. r0+63 of a [rows][d] tensor into shared [64][lds] as fp32,
// columns c0 .. c0+WC-1, times `mul`; rows outside [lo, hi) read as zero.
// Global reads are 16-byte vectors (8 bf16 or 4 fp32); d, c0 and WC are
// multiples of the vector length, and the tensors are 16-byte aligned.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void load(const float *p, float (&x)[4]) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&x)[8]) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

template <typename T, int WC>
__device__ __forceinline__ void load_rows(float *s, int lds, const T *g, int d, int r0, int lo, int hi, int c0,
                                          float mul = 1.f) {
    constexpr int V = Vec16<T>::N, VPR = WC / V;
    static_assert(WC % V == 0, "row width must be a whole number of vectors");
    for (int idx = threadIdx.x; idx < kR * VPR; idx += kThr) {
        const int r = idx / VPR, cv = (idx % VPR) * V, gr = r0 + r;
        float x[V];
        if (gr >= lo && gr < hi) {
            Vec16<T>::load(g + (size_t)gr * d + c0 + cv, x);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) x[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < V; ++e) s[r * lds + cv + e] = x[e] * mul;
    }
}

// The same tile in two steps, so that the global loads of the next tile can
// be in flight while the current one is used: fetch() issues the 16-byte
// loads into registers, commit() widens them into shared memory.
template <typename T, int WC>
struct TileFetch {
    static constexpr int V = Vec16<T>::N, VPR = WC / V, NV = (kR * VPR + kThr - 1) / kThr;
    uint4 raw[NV];
    __device__ __forceinline__ void fetch(const T *g, int d, int r0, int lo, int hi, int c0) {
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int idx = threadIdx.x + kThr * u;
            const int r = idx / VPR, cv = (idx % VPR) * V, gr = r0 + r;
            raw[u] = (idx < kR * VPR && gr >= lo && gr < hi)
                         ? *reinterpret_cast<const uint4 *>(g + (size_t)gr * d + c0 + cv)
                         : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __device__ __forceinline__ void commit(float *s, int lds, float mul = 1.f) const {
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int idx = threadIdx.x + kThr * u;
            if (idx >= kR * VPR) continue;
            const int r = idx / VPR, cv = (idx % VPR) * V;
            float x[V];
            if constexpr (V == 8) {
                const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[2 * i] = __uint_as_float(w[i] << 16);
                    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                }
            } else {
                x[0] = __uint_as_float(raw[u].x);
                x[1] = __uint_as_float(raw[u].y);
                x[2] = __uint_as_float(raw[u].z);
                x[3] = __uint_as_float(raw[u].w);
            }
#pragma unroll
            for (int e = 0; e < V; ++e) s[r * lds + cv + e] = x[e] * mul;
        }
    }
};

__device__ __forceinline__ float block_sum(float x, float *red) {
    x = warp_sum(x);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = x;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0)
        for (int i = 0; i < kThr / 32; ++i) s += red[i];
    return s;  // valid in thread 0
}

// ------------------------------------------------------------------ window: dQ
template <int DK, int DV>
struct WinCfg {
    static constexpr int LQ = DK + 1, LV = DV + 1;
    static constexpr int FLOATS = 2 * kR * LQ + 2 * kR * LV + kR * kLS + 4 * kR;
    static constexpr size_t SMEM = sizeof(float) * FLOATS;
};

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr)
tcb_window_dq_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                     const T *__restrict__ dy, int Tn, int W, float scale, float *__restrict__ lse_g,
                     float *__restrict__ D_g, int lstride, float *__restrict__ dQacc,
                     unsigned int *__restrict__ status) {
    using C = WinCfg<DK, DV>;
    constexpr int LQ = C::LQ, LV = C::LV, TNV = DV / 16, TNK = DK / 16;
    extern __shared__ float sm[];
    float *Qs = sm, *dYs = Qs + kR * LQ, *Ks = dYs + kR * LV, *Vs = Ks + kR * LQ, *Ps = Vs + kR * LV;
    float *rf = Ps + kR * kLS, *rm = rf + kR, *rl = rm + kR, *rD = rl + kR;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int bh = blockIdx.y, q0 = blockIdx.x * kR;
    const T *qh = q + (size_t)bh * Tn * DK, *kh = k + (size_t)bh * Tn * DK;
    const T *vh = v + (size_t)bh * Tn * DV, *dyh = dy + (size_t)bh * Tn * DV;
    load_rows<T, DK>(Qs, LQ, qh, DK, q0, 0, Tn, 0);
    load_rows<T, DV>(dYs, LV, dyh, DV, q0, 0, Tn, 0);
    if (tid < kR) {
        rm[tid] = kNegBig;
        rl[tid] = 0.f;
    }
    const int s_lo = max(0, q0 - W + 1), s_hi = min(Tn - 1, q0 + kR - 1);
    const int kt0 = s_lo / kR, kt1 = s_hi / kR;
    float O[4][TNV];
    zero(O);
    auto band = [&](int t, int s) { return s <= t && s > t - W && t < Tn; };
    // pass 1: softmax statistics and y_loc
    for (int kt = kt0; kt <= kt1; ++kt) {
        const int k0 = kt * kR;
        __syncthreads();
        load_rows<T, DK>(Ks, LQ, kh, DK, k0, 0, Tn, 0);
        load_rows<T, DV>(Vs, LV, vh, DV, k0, 0, Tn, 0);
        __syncthreads();
        float S[4][4];
        zero(S);
        mm_tile<4, 4>(S, Qs, LQ, 1, Ks, 1, LQ, DK);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = ty + 16 * i, c = tx + 16 * j;
                Ps[r * kLS + c] = band(q0 + r, k0 + c) ? S[i][j] * scale : kNegBig;
            }
        __syncthreads();
        {   // four threads per row
            const int r = tid >> 2, part = tid & 3;
            float mx = kNegBig;
            for (int c = part * 16; c < part * 16 + 16; ++c) mx = fmaxf(mx, Ps[r * kLS + c]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mold = rm[r], mnew = fmaxf(mold, mx);
            float sum = 0.f;
            for (int c = part * 16; c < part * 16 + 16; ++c) {
                const float sv = Ps[r * kLS + c];
                const float p = sv <= 0.5f * kNegBig ? 0.f : __expf(sv - mnew);
                Ps[r * kLS + c] = p;
                sum += p;
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            __syncwarp();
            if (part == 0) {
                const float alpha = __expf(mold - mnew);
                rl[r] = rl[r] * alpha + sum;
                rm[r] = mnew;
                rf[r] = alpha;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = rf[ty + 16 * i];
#pragma unroll
            for (int j = 0; j < TNV; ++j) O[i][j] *= a;
        }
        mm_tile<4, TNV>(O, Ps, kLS, 1, Vs, LV, 1, kR);
    }
    // LSE and D = <dy, y_loc> per row
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty + 16 * i;
        const float l = rl[r];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < TNV; ++j) d = fmaf(dYs[r * LV + tx + 16 * j], O[i][j] * inv, d);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        d += __shfl_xor_sync(0xffffffffu, d, 8);
        if (tx == 0) {
            const float ls = l > 0.f ? rm[r] + __logf(l) : 0.f;
            rD[r] = d;
            rf[r] = ls;
            const size_t at = (size_t)bh * lstride + q0 + r;
            if (q0 + r < Tn && OPAM_BOUNDS(at < (size_t)gridDim.y * lstride, status)) {
                lse_g[at] = ls;
                D_g[at] = d;
            }
        }
    }
    // pass 2: dQ
    float dQ[4][TNK];
    zero(dQ);
    for (int kt = kt0; kt <= kt1; ++kt) {
        const int k0 = kt * kR;
        __syncthreads();
        load_rows<T, DK>(Ks, LQ, kh, DK, k0, 0, Tn, 0);
        load_rows<T, DV>(Vs, LV, vh, DV, k0, 0, Tn, 0);
        __syncthreads();
        float S[4][4], dP[4][4];
        zero(S);
        zero(dP);
        mm_tile<4, 4>(S, Qs, LQ, 1, Ks, 1, LQ, DK);
        mm_tile<4, 4>(dP, dYs, LV, 1, Vs, 1, LV, DV);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = ty + 16 * i, c = tx + 16 * j;
                const float p = __expf(band(q0 + r, k0 + c) ? S[i][j] * scale - rf[r] : -INFINITY);  // one path per warp
                Ps[r * kLS + c] = p * (dP[i][j] - rD[r]);
            }
        __syncthreads();
        mm_tile<4, TNK>(dQ, Ps, kLS, 1, Ks, LQ, 1, kR);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = q0 + ty + 16 * i;
        if (t >= Tn) continue;
#pragma unroll
        for (int j = 0; j < TNK; ++j) {
            const size_t at = ((size_t)bh * Tn + t) * DK + tx + 16 * j;
            if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DK, status)) dQacc[at] = scale * dQ[i][j];
        }
    }
}

// ------------------------------------------------------------------ window: dK, dV
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr)
tcb_window_dkdv_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       const T *__restrict__ dy, int Tn, int W, float scale, const float *__restrict__ lse_g,
                       const float *__restrict__ D_g, int lstride, float *__restrict__ dKacc,
                       float *__restrict__ dVacc, unsigned int *__restrict__ status) {
    using C = WinCfg<DK, DV>;
    constexpr int LQ = C::LQ, LV = C::LV, TNV = DV / 16, TNK = DK / 16;
    extern __shared__ float sm[];
    float *Ks = sm, *Vs = Ks + kR * LQ, *Qs = Vs + kR * LV, *dYs = Qs + kR * LQ, *Ps = dYs + kR * LV;
    float *rL = Ps + kR * kLS, *rD = rL + kR;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int bh = blockIdx.y, k0 = blockIdx.x * kR;
    const T *qh = q + (size_t)bh * Tn * DK, *kh = k + (size_t)bh * Tn * DK;
    const T *vh = v + (size_t)bh * Tn * DV, *dyh = dy + (size_t)bh * Tn * DV;
    load_rows<T, DK>(Ks, LQ, kh, DK, k0, 0, Tn, 0);
    load_rows<T, DV>(Vs, LV, vh, DV, k0, 0, Tn, 0);
    const int t_hi = min(Tn - 1, k0 + kR - 1 + W - 1);
    const int qt0 = k0 / kR, qt1 = t_hi / kR;
    float dK[4][TNK], dV[4][TNV];
    zero(dK);
    zero(dV);
    for (int qt = qt0; qt <= qt1; ++qt) {
        const int t0 = qt * kR;
        __syncthreads();
        load_rows<T, DK>(Qs, LQ, qh, DK, t0, 0, Tn, 0);
        load_rows<T, DV>(dYs, LV, dyh, DV, t0, 0, Tn, 0);
        if (tid < kR) {
            const bool ok = t0 + tid < Tn;
            rL[tid] = ok ? lse_g[(size_t)bh * lstride + t0 + tid] : 0.f;
            rD[tid] = ok ? D_g[(size_t)bh * lstride + t0 + tid] : 0.f;
        }
        __syncthreads();
        // rows = keys (m), columns = queries (n)
        float St[4][4], dPt[4][4], Pt[4][4];
        zero(St);
        zero(dPt);
        mm_tile<4, 4>(St, Ks, LQ, 1, Qs, 1, LQ, DK);
        mm_tile<4, 4>(dPt, Vs, LV, 1, dYs, 1, LV, DV);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int s = k0 + ty + 16 * i, t = t0 + tx + 16 * j;
                const bool ok = s <= t && s > t - W && t < Tn && s < Tn;
                Pt[i][j] = __expf(ok ? St[i][j] * scale - rL[tx + 16 * j] : -INFINITY);
                Ps[(ty + 16 * i) * kLS + tx + 16 * j] = Pt[i][j];
            }
        __syncthreads();
        mm_tile<4, TNV>(dV, Ps, kLS, 1, dYs, LV, 1, kR);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                Ps[(ty + 16 * i) * kLS + tx + 16 * j] = Pt[i][j] * (dPt[i][j] - rD[tx + 16 * j]);
        __syncthreads();
        mm_tile<4, TNK>(dK, Ps, kLS, 1, Qs, LQ, 1, kR);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int s = k0 + ty + 16 * i;
        if (s >= Tn) continue;
#pragma unroll
        for (int j = 0; j < TNK; ++j) {
            const size_t at = ((size_t)bh * Tn + s) * DK + tx + 16 * j;
            if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DK, status)) dKacc[at] = scale * dK[i][j];
        }
#pragma unroll
        for (int j = 0; j < TNV; ++j) {
            const size_t at = ((size_t)bh * Tn + s) * DV + tx + 16 * j;
            if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DV, status)) dVacc[at] = dV[i][j];
        }
    }
}

// ------------------------------------------------------------------ L2: intra-chunk
template <int DK, int DV>
struct IntraCfg {
    // row strides padded to a multiple of 4 floats: 16-byte aligned rows for
    // the k-vectorised products
    static constexpr int LQ = DK + 4, LV = DV + 4;
    static_assert(LQ % 4 == 0 && LV % 4 == 0 && DK % 4 == 0 && DV % 4 == 0, "16-byte aligned rows");
    static constexpr int FLOATS = 2 * kR * LQ + 2 * kR * LV + kR * kLS + 2 * (kR + 1) + 32;
    static constexpr size_t SMEM = sizeof(float) * FLOATS;
};

// Per-head lambda powers: pw[d] = lambda^d, dpw[d] = d lambda^(d-1) (0 at d = 0).
__device__ __forceinline__ void power_tables(float *pw, float *dpw, float lm) {
    for (int d = threadIdx.x; d <= kR; d += blockDim.x) {
        pw[d] = powf(lm, (float)d);
        dpw[d] = d == 0 ? 0.f : (float)d * powf(lm, (float)(d - 1));
    }
}

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr)
tcb_l2_intra_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    const T *__restrict__ dy, int Tn, int W, int H, const float *__restrict__ lam,
                    const float *__restrict__ eta, const float *__restrict__ gate, float *__restrict__ dQacc,
                    float *__restrict__ dKacc, float *__restrict__ dVacc, float *__restrict__ part,
                    unsigned int *__restrict__ status) {
    using C = IntraCfg<DK, DV>;
    constexpr int LQ = C::LQ, LV = C::LV, TNV = DV / 16, TNK = DK / 16;
    extern __shared__ float sm[];
    float *Qs = sm, *Kp = Qs + kR * LQ, *dMs = Kp + kR * LQ, *Vp = dMs + kR * LV, *Es = Vp + kR * LV;
    float *pw = Es + kR * kLS, *dpw = pw + kR + 1, *red = dpw + kR + 1;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int c = blockIdx.x, bh = blockIdx.y, h = bh % H, u0 = c * kR;
    const float lm = lam[h], et = eta[h], sg = logistic(gate[h]);
    const T *qh = q + (size_t)bh * Tn * DK, *kh = k + (size_t)bh * Tn * DK;
    const T *vh = v + (size_t)bh * Tn * DV, *dyh = dy + (size_t)bh * Tn * DV;
    // positions u = u0 + r < Tn; the evicted token is u - W (valid when >= 0)
    load_rows<T, DK>(Qs, LQ, qh, DK, u0, 0, Tn, 0);
    load_rows<T, DV>(dMs, LV, dyh, DV, u0, 0, Tn, 0, sg);
    load_rows<T, DK>(Kp, LQ, kh, DK, u0 - W, 0, Tn - W, 0);
    load_rows<T, DV>(Vp, LV, vh, DV, u0 - W, 0, Tn - W, 0);
    power_tables(pw, dpw, lm);
    __syncthreads();
    float S1[4][4], S2[4][4];
    zero(S1);
    zero(S2);
    mm_tile<4, 4, true, true>(S1, Qs, LQ, 1, Kp, 1, LQ, DK);
    mm_tile<4, 4, true, true>(S2, dMs, LV, 1, Vp, 1, LV, DV);
    float g_eta = 0.f, g_lam = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = ty + 16 * i, cc = tx + 16 * j;
            const bool lower = cc <= r;
            const float s12 = S1[i][j] * S2[i][j];
            if (lower) {
                g_eta = fmaf(pw[r - cc], s12, g_eta);
                g_lam = fmaf(et * dpw[r - cc], s12, g_lam);
            }
            const float d = lower ? et * pw[r - cc] : 0.f;
            S1[i][j] *= d;   // E1 = D * (Q K'^T)
            S2[i][j] *= d;   // E2 = D * (dM V'^T)
            Es[r * kLS + cc] = S2[i][j];
        }
    __syncthreads();
    {   // dq += E2 K' (rows u),  dk' += E2^T Q (rows u - W)
        float a[4][TNK], b[4][TNK];
        zero(a);
        zero(b);
        mm_tile<4, TNK>(a, Es, kLS, 1, Kp, LQ, 1, kR);
        mm_tile<4, TNK>(b, Es, 1, kLS, Qs, LQ, 1, kR);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty + 16 * i, u = u0 + r;
            if (u >= Tn) continue;
#pragma unroll
            for (int j = 0; j < TNK; ++j) {
                const size_t at = ((size_t)bh * Tn + u) * DK + tx + 16 * j;
                if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DK, status)) dQacc[at] += a[i][j];
            }
            if (u - W >= 0)
#pragma unroll
                for (int j = 0; j < TNK; ++j) {
                    const size_t at = ((size_t)bh * Tn + u - W) * DK + tx + 16 * j;
                    if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DK, status)) dKacc[at] += b[i][j];
                }
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) Es[(ty + 16 * i) * kLS + tx + 16 * j] = S1[i][j];
    __syncthreads();
    float sdm = 0.f;
    {   // dv' += E1^T dM (rows u - W),  m += E1 V' (for dg)
        float a[4][TNV], b[4][TNV];
        zero(a);
        zero(b);
        mm_tile<4, TNV>(a, Es, 1, kLS, dMs, LV, 1, kR);
        mm_tile<4, TNV>(b, Es, kLS, 1, Vp, LV, 1, kR);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty + 16 * i, u = u0 + r;
#pragma unroll
            for (int j = 0; j < TNV; ++j) sdm = fmaf(dMs[r * LV + tx + 16 * j], b[i][j], sdm);
            if (u >= Tn || u - W < 0) continue;
#pragma unroll
            for (int j = 0; j < TNV; ++j) {
                const size_t at = ((size_t)bh * Tn + u - W) * DV + tx + 16 * j;
                if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DV, status)) dVacc[at] += a[i][j];
            }
        }
    }
    const float s0 = block_sum(g_lam, red);
    const float s1 = block_sum(g_eta, red);
    const float s2 = block_sum(sdm, red);
    if (tid == 0) {
        float *p = part + ((size_t)bh * gridDim.x + c) * 4;
        p[0] = s0;
        p[1] = s1;
        p[2] = s2;
        p[3] = 0.f;
    }
}

// ------------------------------------------------------------------ L2: chunk-state scans
template <int DK>
struct ScanCfg {
    // row strides padded to a multiple of 4 floats: 16-byte aligned rows for
    // the k-vectorised products
    static constexpr int LQ = DK + 4, LW = kSW + 4;
    static_assert(LQ % 4 == 0 && LW % 4 == 0 && DK % 4 == 0 && kSW % 4 == 0, "16-byte aligned rows");
    static constexpr int FLOATS = 2 * kR * LQ + 4 * kR * LW + 2 * DK * LW + 2 * (kR + 1) + 32;
    static constexpr size_t SMEM = sizeof(float) * FLOATS;
};

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr)
tcb_l2_scan_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   const T *__restrict__ dy, int Tn, int W, int H, const float *__restrict__ lam,
                   const float *__restrict__ eta, const float *__restrict__ gate, float *__restrict__ dQacc,
                   float *__restrict__ dKacc, float *__restrict__ dVacc, float *__restrict__ part_f,
                   float *__restrict__ part_r, unsigned int *__restrict__ status) {
    using C = ScanCfg<DK>;
    constexpr int LQ = C::LQ, LW = C::LW, TNK = DK / 16, TMK = DK / 16;
    constexpr bool M4 = TMK % 4 == 0;  // state rows four per 16-byte load (d_k >= 64)
    constexpr int NSL = DV / kSW;
    extern __shared__ float sm[];
    float *Qs = sm, *Kp = Qs + kR * LQ, *dMs = Kp + kR * LQ, *Vp = dMs + kR * LW, *Vw = Vp + kR * LW,
          *Vw2 = Vw + kR * LW, *St = Vw2 + kR * LW, *St2 = St + DK * LW, *pw = St2 + DK * LW, *dpw = pw + kR + 1,
          *red = dpw + kR + 1;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int sl = blockIdx.x, bh = blockIdx.y, h = bh % H, b0 = sl * kSW;
    const bool reverse = blockIdx.z == 1;
    const float lm = lam[h], et = eta[h], sg = logistic(gate[h]);
    const T *qh = q + (size_t)bh * Tn * DK, *kh = k + (size_t)bh * Tn * DK;
    const T *vh = v + (size_t)bh * Tn * DV, *dyh = dy + (size_t)bh * Tn * DV;
    const int nch = (Tn + kR - 1) / kR;
    power_tables(pw, dpw, lm);
    for (int i = tid; i < 2 * DK * LW; i += kThr) St[i] = 0.f;  // St, St2 contiguous
    float g0 = 0.f, g1 = 0.f;
    // the next chunk's tiles are fetched into registers while this one is used
    TileFetch<T, DK> fq, fk;
    TileFetch<T, kSW> fm, fv;
    auto fetch = [&](int step) {
        const int c = reverse ? nch - 1 - step : step, u0 = c * kR;
        fq.fetch(qh, DK, u0, 0, Tn, 0);
        fm.fetch(dyh, DV, u0, 0, Tn, b0);
        fk.fetch(kh, DK, u0 - W, 0, Tn - W, 0);
        fv.fetch(vh, DV, u0 - W, 0, Tn - W, b0);
    };
    fetch(0);
    for (int step = 0; step < nch; ++step) {
        const int c = reverse ? nch - 1 - step : step, u0 = c * kR, n = min(kR, Tn - u0);
        __syncthreads();
        fq.commit(Qs, LQ);
        fm.commit(dMs, LW, sg);
        fk.commit(Kp, LQ);
        fv.commit(Vp, LW);
        __syncthreads();
        if (step + 1 < nch) fetch(step + 1);
        if (!reverse) {
            // X = Q A_c, X' = Q A'_c on this slice; dq += lambda^(i+1) dM A_c^T
            float X[4][1], Xp[4][1], dq[4][TNK];
            zero(X);
            zero(Xp);
            zero(dq);
            mm_tile_2<4, true>(X, Xp, Qs, LQ, 1, St, St2, LW, 1, DK);
            mm_tile<4, TNK, true, true>(dq, dMs, LW, 1, St, 1, LW, kSW);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = ty + 16 * i, u = u0 + r;
                const float dm = dMs[r * LW + tx];
                g1 = fmaf(pw[r + 1] * X[i][0], dm, g1);                                    // <dm, m>
                g0 = fmaf(dpw[r + 1] * X[i][0] + pw[r + 1] * Xp[i][0], dm, g0);             // dlambda
                if (u < Tn)
#pragma unroll
                    for (int j = 0; j < TNK; ++j) {
                        const size_t at = ((size_t)bh * Tn + u) * DK + tx + 16 * j;
                        if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DK, status))
                            atomicAdd(&dQacc[at], pw[r + 1] * dq[i][j]);
                    }
            }
            // weighted V' rows for the state update
            for (int idx = tid; idx < kR * kSW; idx += kThr) {
                const int j = idx / kSW, b = idx - j * kSW;
                const float x = Vp[j * LW + b];
                Vw[j * LW + b] = j < n ? et * pw[n - 1 - j] * x : 0.f;
                Vw2[j * LW + b] = j < n ? et * dpw[n - 1 - j] * x : 0.f;
            }
            __syncthreads();
            float a1[TMK][1], a2[TMK][1];
            zero(a1);
            zero(a2);
            if constexpr (M4)
                mm_tile_2_m4<TMK>(a1, a2, Kp, LQ, Vw, Vw2, LW, 1, kR);
            else
                mm_tile_2<TMK>(a1, a2, Kp, 1, LQ, Vw, Vw2, LW, 1, kR);
            const float ln = pw[n], dln = dpw[n];
#pragma unroll
            for (int i = 0; i < TMK; ++i) {
                const int a = M4 ? mrow4(i) : ty + 16 * i;
                const float A0 = St[a * LW + tx], A1 = St2[a * LW + tx];
                St[a * LW + tx] = fmaf(ln, A0, a1[i][0]);
                St2[a * LW + tx] = fmaf(dln, A0, fmaf(ln, A1, a2[i][0]));
            }
        } else {
            // dk' += eta lambda^(n-j) R V'_j (over the slice), dv' += eta lambda^(n-j) R^T k'_j
            float dk[4][TNK], dvv[4][1];
            zero(dk);
            zero(dvv);
            mm_tile<4, TNK, true, true>(dk, Vp, LW, 1, St, 1, LW, kSW);
            mm_tile<4, 1, true, false>(dvv, Kp, LQ, 1, St, LW, 1, DK);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = ty + 16 * i, u = u0 + j;
                const float f = j < n ? pw[n - j] : 0.f;
                g0 = fmaf(f * dvv[i][0], Vp[j * LW + tx], g0);                               // deta
                if (u >= Tn || u - W < 0) continue;
#pragma unroll
                for (int jj = 0; jj < TNK; ++jj) {
                    const size_t at = ((size_t)bh * Tn + u - W) * DK + tx + 16 * jj;
                    if (OPAM_BOUNDS(at < (size_t)gridDim.y * Tn * DK, status)) atomicAdd(&dKacc[at], et * f * dk[i][jj]);
                }
                const size_t av = ((size_t)bh * Tn + u - W) * DV + b0 + tx;
                if (OPAM_BOUNDS(av < (size_t)gridDim.y * Tn * DV, status)) dVacc[av] += et * f * dvv[i][0];
            }
            // R <- lambda^n R + sum_i lambda^i q_i dm_i^T
            for (int idx = tid; idx < kR * kSW; idx += kThr) {
                const int i = idx / kSW, b = idx - i * kSW;
                Vw[i * LW + b] = pw[i] * dMs[i * LW + b];
            }
            __syncthreads();
            float r1[TMK][1];
            zero(r1);
            if constexpr (M4)
                mm_tile_m4<TMK>(r1, Qs, LQ, Vw, LW, 1, kR);
            else
                mm_tile<TMK, 1>(r1, Qs, 1, LQ, Vw, LW, 1, kR);
            const float ln = pw[n];
#pragma unroll
            for (int i = 0; i < TMK; ++i) {
                const int a = M4 ? mrow4(i) : ty + 16 * i;
                St[a * LW + tx] = fmaf(ln, St[a * LW + tx], r1[i][0]);
            }
        }
    }
    const float s0 = block_sum(g0, red);
    const float s1 = block_sum(g1, red);
    if (tid == 0) {
        if (reverse) {
            part_r[(size_t)bh * NSL + sl] = s0;
        } else {
            part_f[((size_t)bh * NSL + sl) * 2 + 0] = s0;
            part_f[((size_t)bh * NSL + sl) * 2 + 1] = s1;
        }
    }
}

// ------------------------------------------------------------------ finalize
// Blocks [0, nconv): fp32 accumulators -> element type.  Blocks nconv ..
// nconv + H - 1: per-head scalars, summed over batch, chunks and slices in a
// fixed order.  Thread 0 of block 0 also zeroes the call's status words
// (nothing in this backward waits on a barrier, so nothing else sets them).
template <typename T>
__global__ void __launch_bounds__(kThr)
tcb_finalize_kernel(const float *__restrict__ dQacc, const float *__restrict__ dKacc,
                    const float *__restrict__ dVacc, size_t nqk, size_t nv, int nconv, T *__restrict__ dq,
                    T *__restrict__ dk, T *__restrict__ dv, int B, int H, int nch, int nsl,
                    const float *__restrict__ part, const float *__restrict__ part_f,
                    const float *__restrict__ part_r, const float *__restrict__ gate, float *__restrict__ dlam,
                    float *__restrict__ deta, float *__restrict__ dgate, unsigned int *__restrict__ status) {
    __shared__ float red[kThr / 32];
    if ((int)blockIdx.x < nconv) {
        const size_t stride = (size_t)nconv * blockDim.x;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nqk; i += stride) {
            Elem<T>::store(dq + i, dQacc[i]);
            Elem<T>::store(dk + i, dKacc[i]);
        }
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride)
            Elem<T>::store(dv + i, dVacc[i]);
        return;
    }
    const int h = blockIdx.x - nconv;
    float a = 0.f, e = 0.f, s = 0.f;
    for (int b = 0; b < B; ++b) {
        const int bh = b * H + h;
        for (int i = threadIdx.x; i < nch; i += blockDim.x) {
            const float *p = part + ((size_t)bh * nch + i) * 4;
            a += p[0];
            e += p[1];
            s += p[2];
        }
        for (int i = threadIdx.x; i < nsl; i += blockDim.x) {
            a += part_f[((size_t)bh * nsl + i) * 2 + 0];
            s += part_f[((size_t)bh * nsl + i) * 2 + 1];
            e += part_r[(size_t)bh * nsl + i];
        }
    }
    a = block_sum(a, red);
    e = block_sum(e, red);
    s = block_sum(s, red);
    if (threadIdx.x == 0) {
        dlam[h] = a;
        deta[h] = e;
        dgate[h] = (1.f - logistic(gate[h])) * s;
    }
}

// ------------------------------------------------------------------ host
// LSE and D rows are padded to a multiple of 128 entries, so that the
// tensor-core dK/dV kernel copies each 128-query tile of them whole.
int lse_stride(int T) { return ceil_div(T, 128) * 128; }

struct BwdWs {
    float *lse, *D, *dQ, *dK, *dV, *part, *part_f, *part_r;
};

BwdWs carve_bwd(void *ws, int BH, int T, int dk, int dv) {
    const int nch = ceil_div(T, kR), nsl = dv / kSW;
    char *p = (char *)ws;
    BwdWs w;
    auto take = [&](size_t floats) {
        float *r = (float *)p;
        p += align_up(floats * sizeof(float), 256);
        return r;
    };
    const size_t ls = (size_t)BH * lse_stride(T);
    w.lse = take(ls);
    w.D = take(ls);
    w.dQ = take((size_t)BH * T * dk);
    w.dK = take((size_t)BH * T * dk);
    w.dV = take((size_t)BH * T * dv);
    w.part = take((size_t)BH * nch * 4);
    w.part_f = take((size_t)BH * nsl * 2);
    w.part_r = take((size_t)BH * nsl);
    return w;
}

template <typename T, int DK, int DV>
int run_bwd(const void *q, const void *k, const void *v, int B, int H, int Tn, int W, const float *lam,
            const float *eta, const float *gate, float scale, const void *dy, void *dq, void *dk, void *dv,
            float *dlam, float *deta, float *dgate, void *ws, unsigned int *status, cudaStream_t s) {
    const int BH = B * H, nch = ceil_div(Tn, kR), nsl = DV / kSW;
    const BwdWs w = carve_bwd(ws, BH, Tn, DK, DV);
    const T *Q = (const T *)q, *K = (const T *)k, *V = (const T *)v, *dY = (const T *)dy;
    int rc;
    const bool tc = tcb_window_dkdv_tcgen05_supported(std::is_same<T, __nv_bfloat16>::value ? OPAM_BF16 : OPAM_F32,
                                                      DK, DV);
    prof_begin(s);
    if (tc) {
        if ((rc = tcb_window_dq_tcgen05(Q, K, V, dY, BH, Tn, W, scale, w.lse, w.D, lse_stride(Tn), w.dQ, status,
                                        s)))
            return rc;
    } else {
        auto kern = tcb_window_dq_kernel<T, DK, DV>;
        const int smem = (int)WinCfg<DK, DV>::SMEM;
        if ((rc = set_smem_limit((const void *)kern, smem, "tcb_window_dq smem attribute"))) return rc;
        kern<<<dim3(nch, BH), kThr, smem, s>>>(Q, K, V, dY, Tn, W, scale, w.lse, w.D, lse_stride(Tn), w.dQ,
                                               status);
        if ((rc = launched("tcb_window_dq"))) return rc;
    }
    if (tc) {
        if ((rc = tcb_window_dkdv_tcgen05(Q, K, V, dY, BH, Tn, W, scale, w.lse, w.D, lse_stride(Tn), w.dK, w.dV,
                                          status, s)))
            return rc;
    } else {
        auto kern = tcb_window_dkdv_kernel<T, DK, DV>;
        const int smem = (int)WinCfg<DK, DV>::SMEM;
        if ((rc = set_smem_limit((const void *)kern, smem, "tcb_window_dkdv smem attribute"))) return rc;
        kern<<<dim3(nch, BH), kThr, smem, s>>>(Q, K, V, dY, Tn, W, scale, w.lse, w.D, lse_stride(Tn), w.dK, w.dV,
                                               status);
        if ((rc = launched("tcb_window_dkdv"))) return rc;
    }
    {
        auto kern = tcb_l2_intra_kernel<T, DK, DV>;
        const int smem = (int)IntraCfg<DK, DV>::SMEM;
        if ((rc = set_smem_limit((const void *)kern, smem, "tcb_l2_intra smem attribute"))) return rc;
        kern<<<dim3(nch, BH), kThr, smem, s>>>(Q, K, V, dY, Tn, W, H, lam, eta, gate, w.dQ, w.dK, w.dV, w.part,
                                               status);
        if ((rc = launched("tcb_l2_intra"))) return rc;
    }
    {
        auto kern = tcb_l2_scan_kernel<T, DK, DV>;
        const int smem = (int)ScanCfg<DK>::SMEM;
        if ((rc = set_smem_limit((const void *)kern, smem, "tcb_l2_scan smem attribute"))) return rc;
        kern<<<dim3(nsl, BH, 2), kThr, smem, s>>>(Q, K, V, dY, Tn, W, H, lam, eta, gate, w.dQ, w.dK, w.dV,
                                                  w.part_f, w.part_r, status);
        if ((rc = launched("tcb_l2_scan"))) return rc;
    }
    {
        const size_t nqk = (size_t)BH * Tn * DK, nv = (size_t)BH * Tn * DV;
        const int nconv = (int)std::min<size_t>(4 * 148, (nqk + kThr - 1) / kThr);
        tcb_finalize_kernel<T><<<nconv + H, kThr, 0, s>>>(w.dQ, w.dK, w.dV, nqk, nv, nconv, (T *)dq, (T *)dk,
                                                         (T *)dv, B, H, nch, nsl, w.part, w.part_f, w.part_r,
                                                         gate, dlam, deta, dgate, status);
        rc = launched("tcb_finalize");
        prof_end(s);
        return rc;
    }
}

template <typename T, int DK>
int bwd_dv(int dvv, const void *q, const void *k, const void *v, int B, int H, int Tn, int W, const float *lam,
           const float *eta, const float *gate, float scale, const void *dy, void *dq, void *dk, void *dv,
           float *dlam, float *deta, float *dgate, void *ws, unsigned int *status, cudaStream_t s) {
    switch (dvv) {
        case 32: return run_bwd<T, DK, 32>(q, k, v, B, H, Tn, W, lam, eta, gate, scale, dy, dq, dk, dv, dlam, deta, dgate, ws, status, s);
        case 64: return run_bwd<T, DK, 64>(q, k, v, B, H, Tn, W, lam, eta, gate, scale, dy, dq, dk, dv, dlam, deta, dgate, ws, status, s);
        case 128: return run_bwd<T, DK, 128>(q, k, v, B, H, Tn, W, lam, eta, gate, scale, dy, dq, dk, dv, dlam, deta, dgate, ws, status, s);
    }
    set_error("tc_layer_backward: d_v=%d unsupported", dvv);
    return OPAM_ERR_UNSUPPORTED;
}

template <typename T>
int bwd_dk(int dkk, int dvv, const void *q, const void *k, const void *v, int B, int H, int Tn, int W,
           const float *lam, const float *eta, const float *gate, float scale, const void *dy, void *dq, void *dk,
           void *dv, float *dlam, float *deta, float *dgate, void *ws, unsigned int *status, cudaStream_t s) {
    switch (dkk) {
        case 32: return bwd_dv<T, 32>(dvv, q, k, v, B, H, Tn, W, lam, eta, gate, scale, dy, dq, dk, dv, dlam, deta, dgate, ws, status, s);
        case 64: return bwd_dv<T, 64>(dvv, q, k, v, B, H, Tn, W, lam, eta, gate, scale, dy, dq, dk, dv, dlam, deta, dgate, ws, status, s);
        case 128: return bwd_dv<T, 128>(dvv, q, k, v, B, H, Tn, W, lam, eta, gate, scale, dy, dq, dk, dv, dlam, deta, dgate, ws, status, s);
    }
    set_error("tc_layer_backward: d_k=%d unsupported", dkk);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace

size_t tc_backward_workspace(int BH, int T, int dk, int dv) {
    const int nch = ceil_div(T, kR), nsl = dv / kSW;
    auto f = [](size_t floats) { return align_up(floats * sizeof(float), 256); };
    return 2 * f((size_t)BH * lse_stride(T)) + 2 * f((size_t)BH * T * dk) + f((size_t)BH * T * dv) + f((size_t)BH * nch * 4) +
           f((size_t)BH * nsl * 2) + f((size_t)BH * nsl);
}

int tc_backward(const void *q, const void *k, const void *v, int dtype, int B, int H, int T, int dk, int dv, int W,
                const float *lam, const float *eta, const float *gate, float scale, const void *dy, void *dq,
                void *dkk, void *dvv, float *dlam, float *deta, float *dgate, void *ws, unsigned int *status,
                cudaStream_t s) {
    if (dtype == OPAM_BF16)
        return bwd_dk<__nv_bfloat16>(dk, dv, q, k, v, B, H, T, W, lam, eta, gate, scale, dy, dq, dkk, dvv, dlam,
                                     deta, dgate, ws, status, s);
    return bwd_dk<float>(dk, dv, q, k, v, B, H, T, W, lam, eta, gate, scale, dy, dq, dkk, dvv, dlam, deta, dgate,
                         ws, status, s);
}

}  // namespace opam
