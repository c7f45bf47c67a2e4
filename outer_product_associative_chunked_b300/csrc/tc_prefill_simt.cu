// Tensor Cache layer prefill on CUDA cores (FFMA, fp32 accumulation).
//
// "Tensor Cache: Eviction-conditioned Associative Memory for Transformers"
// (gist.science 2605.22884).  Methodology 1 defines the layer: softmax over
// the W most recent tokens, eviction write A <- lambda A + eta k v^T, read
// m_t = q_t A, fuse y = y_local + sigmoid(g) m.  Methodology 2 asks for a
// parallel weighted-sum scan equal to the per-token writes.  Unrolled, token
// s is written at step s + W, so
//     m_t = sum_{s <= t-W} eta lambda^(t-W-s) <q_t, k_s> v_s.
//
// Chunking.  Queries are cut into chunks of C = 64 positions.  Query chunk j
// ([jC, jC+C)) is paired with the "shifted" key chunk [jC-W, jC-W+C): exactly
// the tokens evicted during the chunk's steps.  With A_j the state before the
// chunk (all tokens s < jC-W) and query row i:
//     m_{jC+i} = lambda^(i+1) q A_j + sum_{l<=i} eta lambda^(i-l) <q, k'_l> v'_l
//     A_{j+1}  = lambda^n A_j + sum_{l<n} eta lambda^(n-1-l) k'_l v'_l^T
// (n = rows in the chunk).  The shifted key chunk is also the first tile of
// the chunk's softmax window, so one pass over the keys [jC-W, jC+C) serves
// both: key l of that first tile feeds the L2 term when l <= i and the
// softmax when l > i.
//
// Kernels: (1) per-chunk increments dA_j, (2) a sequential scan over chunks
// that turns them into A_j in place, (3) the fused window softmax + L2 read +
// gate.  The window-only variant (l2 = false) runs kernel 3 alone with its L2
// part off.  This path serves the fp32 inputs and every head size; the bf16
// tensor-core path lives in tc_prefill_tcgen05.cu.
#include "opam_internal.cuh"

namespace opam {
namespace {

constexpr int kC = 64;  // chunk length = key tile length (tokens)

template <typename T>
__global__ void __launch_bounds__(256)
tc_chunk_delta_kernel(const T *__restrict__ k, const T *__restrict__ v, int T_, int dk, int dv,
                      int W, int H, const float *__restrict__ lam,
                      const float *__restrict__ eta, float *__restrict__ buf, int nch) {
    extern __shared__ float sm[];
    float *ks = sm;             // [kC][dk], pre-scaled by eta lambda^(n-1-l)
    float *vs = sm + kC * dk;   // [kC][dv]
    const int j = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int n = min(kC, T_ - j * kC);
    const float lm = lam[h], et = eta[h];
    for (int idx = threadIdx.x; idx < kC * dk; idx += blockDim.x) {
        const int l = idx / dk, a = idx - l * dk;
        const int p = j * kC - W + l;
        float x = 0.f;
        if (l < n && p >= 0)
            x = Elem<T>::load(k + ((size_t)bh * T_ + p) * dk + a) * (et * powf(lm, (float)(n - 1 - l)));
        ks[idx] = x;
    }
    for (int idx = threadIdx.x; idx < kC * dv; idx += blockDim.x) {
        const int l = idx / dv, b = idx - l * dv;
        const int p = j * kC - W + l;
        vs[idx] = (l < n && p >= 0) ? Elem<T>::load(v + ((size_t)bh * T_ + p) * dv + b) : 0.f;
    }
    __syncthreads();
    float *out = buf + ((size_t)bh * (nch + 1) + j) * (size_t)(dk * dv);
    for (int e = threadIdx.x; e < dk * dv; e += blockDim.x) {
        const int a = e / dv, b = e - a * dv;
        float acc = 0.f;
        for (int l = 0; l < n; ++l) acc = fmaf(ks[l * dk + a], vs[l * dv + b], acc);
        out[e] = acc;
    }
}

// buf[bh][j] holds dA_j on entry and A_j (state before chunk j) on exit;
// buf[bh][nch] receives the final state.
__global__ void tc_chunk_scan_kernel(float *__restrict__ buf, int nch, int T_, int dkdv, int H,
                                     const float *__restrict__ lam, float *__restrict__ A_final) {
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= dkdv) return;
    const float lm = lam[bh % H];
    const float lamC = powf(lm, (float)kC);
    float *base = buf + (size_t)bh * (nch + 1) * dkdv + e;
    float A = 0.f;
    for (int j = 0; j < nch; ++j) {
        const float d = base[(size_t)j * dkdv];
        base[(size_t)j * dkdv] = A;
        const int n = min(kC, T_ - j * kC);
        A = fmaf(n == kC ? lamC : powf(lm, (float)n), A, d);
    }
    base[(size_t)nch * dkdv] = A;
    if (A_final) A_final[(size_t)bh * dkdv + e] = A;
}

template <int DK, int DV>
struct FwdSmem {
    static constexpr int kQ = kC * (DK + 1);
    static constexpr int kK = kC * (DK + 1);
    static constexpr int kV = kC * DV;
    static constexpr int kS = kC * (kC + 1);
    static constexpr int kRegion = kK + kV + 2 * kS;  // reused for A_j at the end
    static_assert(kRegion >= DK * DV, "A_j must fit the key/value region");
    static constexpr int kFloats = kQ + kRegion + 3 * kC;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(256)
tc_fwd_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   int T_, int W, int H, const float *__restrict__ lam,
                   const float *__restrict__ eta, const float *__restrict__ gate, float scale,
                   const float *__restrict__ Abuf, int nch, int l2, T *__restrict__ y) {
    // l2 == 0: window only (no L2 weights, no state read, no gate term).
    using SM = FwdSmem<DK, DV>;
    extern __shared__ float sm[];
    float *Qs = sm;                       // [kC][DK+1]
    float *Ks = Qs + SM::kQ;              // [kC][DK+1]
    float *Vs = Ks + SM::kK;              // [kC][DV]
    float *Ss = Vs + SM::kV;              // [kC][kC+1] scores, then softmax weights
    float *P2 = Ss + SM::kS;              // [kC][kC+1] L2 weights of the first tile
    float *ms = P2 + SM::kS;              // running max per row
    float *ls = ms + kC;                  // running sum per row
    float *al = ls + kC;                  // rescale factor of the current tile
    float *As = Ks;                       // A_j, after the key loop

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int t0 = j * kC;
    const int nq = min(kC, T_ - t0);
    const float lm = l2 ? lam[h] : 0.f, et = l2 ? eta[h] : 0.f;
    const size_t qbase = (size_t)bh * T_;

    for (int idx = tid; idx < kC * DK; idx += 256) {
        const int r = idx / DK, a = idx - r * DK;
        Qs[r * (DK + 1) + a] = r < nq ? Elem<T>::load(q + (qbase + t0 + r) * DK + a) : 0.f;
    }
    if (tid < kC) { ms[tid] = kNegBig; ls[tid] = 0.f; }

    // PV-phase ownership: one query row, every 4th output column.
    const int prow = tid >> 2, part = tid & 3;
    constexpr int NC = DV / 4;
    float O[NC], O2[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) { O[c] = 0.f; O2[c] = 0.f; }
    // Score-phase ownership: 4 query rows x 4 keys.
    const int tr = tid >> 4, tcol = tid & 15;

    const int kstart = t0 - W, kend = t0 + nq;
    for (int kt = kstart; kt < kend; kt += kC) {
        const bool first = l2 && (kt == kstart);  // the L2 part lives in the first tile
        if (kt + kC <= 0) continue;  // whole tile before position 0
        __syncthreads();
        for (int idx = tid; idx < kC * DK; idx += 256) {
            const int l = idx / DK, a = idx - l * DK;
            const int p = kt + l;
            Ks[l * (DK + 1) + a] = (p >= 0 && p < kend) ? Elem<T>::load(k + (qbase + p) * DK + a) : 0.f;
        }
        for (int idx = tid; idx < kC * DV; idx += 256) {
            const int l = idx / DV, b = idx - l * DV;
            const int p = kt + l;
            Vs[idx] = (p >= 0 && p < kend) ? Elem<T>::load(v + (qbase + p) * DV + b) : 0.f;
        }
        __syncthreads();
        {   // raw scores q.k
            float acc[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 4
            for (int a = 0; a < DK; ++a) {
                float qa[4], ka[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) qa[r] = Qs[(tr * 4 + r) * (DK + 1) + a];
#pragma unroll
                for (int c = 0; c < 4; ++c) ka[c] = Ks[(tcol * 4 + c) * (DK + 1) + a];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(qa[r], ka[c], acc[r][c]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) Ss[(tr * 4 + r) * (kC + 1) + tcol * 4 + c] = acc[r][c];
        }
        __syncthreads();
        // Row pass: masks, online softmax, L2 weights of the first tile.
        for (int rr = 0; rr < kC / 8; ++rr) {
            const int i = warp * (kC / 8) + rr;
            const int t = t0 + i;
            float raw[2], lg[2];
            bool soft[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int l = lane + 32 * u;
                const int p = kt + l;
                raw[u] = Ss[i * (kC + 1) + l];
                soft[u] = (i < nq) && (p >= 0) && (p <= t) && (p > t - W);
                lg[u] = soft[u] ? raw[u] * scale : kNegBig;
            }
            const float mold = ms[i];
            const float mnew = fmaxf(mold, warp_max(fmaxf(lg[0], lg[1])));
            float pe[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) pe[u] = soft[u] ? expf(lg[u] - mnew) : 0.f;
            const float rs = warp_sum(pe[0] + pe[1]);
            const float alpha = expf(mold - mnew);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int l = lane + 32 * u;
                Ss[i * (kC + 1) + l] = pe[u];
                if (first) {
                    const int p = kt + l;
                    const bool l2 = (i < nq) && (p >= 0) && (l <= i);
                    P2[i * (kC + 1) + l] = l2 ? et * powf(lm, (float)(i - l)) * raw[u] : 0.f;
                }
            }
            if (lane == 0) { ms[i] = mnew; ls[i] = alpha * ls[i] + rs; al[i] = alpha; }
        }
        __syncthreads();
        {   // O <- alpha O + P V ; O2 += P2 V (first tile)
            const float a = al[prow];
#pragma unroll
            for (int c = 0; c < NC; ++c) O[c] *= a;
            for (int l = 0; l < kC; ++l) {
                const float p = Ss[prow * (kC + 1) + l];
#pragma unroll
                for (int c = 0; c < NC; ++c) O[c] = fmaf(p, Vs[l * DV + part + 4 * c], O[c]);
            }
            if (first) {
                for (int l = 0; l < kC; ++l) {
                    const float p = P2[prow * (kC + 1) + l];
#pragma unroll
                    for (int c = 0; c < NC; ++c) O2[c] = fmaf(p, Vs[l * DV + part + 4 * c], O2[c]);
                }
            }
        }
    }
    __syncthreads();
    // Carried-state read lambda^(i+1) q A_j and the gated fuse.
    if (l2) {
        const float *Aj = Abuf + ((size_t)bh * (nch + 1) + j) * (size_t)(DK * DV);
        for (int idx = tid; idx < DK * DV; idx += 256) As[idx] = Aj[idx];
    }
    __syncthreads();
    if (prow < nq) {
        float m2[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) m2[c] = 0.f;
        if (l2) {
            for (int a = 0; a < DK; ++a) {
                const float qa = Qs[prow * (DK + 1) + a];
#pragma unroll
                for (int c = 0; c < NC; ++c) m2[c] = fmaf(qa, As[a * DV + part + 4 * c], m2[c]);
            }
        }
        const float inv_l = 1.0f / ls[prow];
        const float decay = l2 ? powf(lm, (float)(prow + 1)) : 0.f;
        const float sg = l2 ? 1.0f / (1.0f + expf(-gate[h])) : 0.f;
        T *yr = y + (qbase + t0 + prow) * DV;
#pragma unroll
        for (int c = 0; c < NC; ++c)
            Elem<T>::store(yr + part + 4 * c, O[c] * inv_l + sg * fmaf(decay, m2[c], O2[c]));
    }
}

template <typename T>
__global__ void tc_export_ring_kernel(const T *__restrict__ k, const T *__restrict__ v, int T_,
                                      int dk, int dv, int W, T *__restrict__ rk,
                                      T *__restrict__ rv) {
    const int slot = blockIdx.x, bh = blockIdx.y;
    const long long t = (T_ > slot) ? slot + (long long)((T_ - 1 - slot) / W) * W : -1;
    T *dk_ = rk + ((size_t)bh * W + slot) * dk;
    T *dv_ = rv + ((size_t)bh * W + slot) * dv;
    for (int e = threadIdx.x; e < dk; e += blockDim.x)
        dk_[e] = t >= 0 ? k[((size_t)bh * T_ + t) * dk + e] : T(0.f);
    for (int e = threadIdx.x; e < dv; e += blockDim.x)
        dv_[e] = t >= 0 ? v[((size_t)bh * T_ + t) * dv + e] : T(0.f);
}

__global__ void set_pos_kernel(int64_t *pos, int B, int64_t value) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) pos[b] = value;
}

template <typename T, int DK, int DV>
int launch_fwd(const void *q, const void *k, const void *v, int BH, int T_, int W, int H,
               const float *lam, const float *eta, const float *gate, float scale,
               const float *Abuf, int nch, int l2, void *y, cudaStream_t s) {
    auto kern = tc_fwd_simt_kernel<T, DK, DV>;
    const size_t smem = FwdSmem<DK, DV>::kBytes;
    if (int rc_ = set_smem_limit((const void *)kern, (int)smem, "tc_fwd_simt smem attribute")) return rc_;
    prof_begin(s);
    kern<<<dim3(nch, BH), 256, smem, s>>>((const T *)q, (const T *)k, (const T *)v, T_, W, H, lam,
                                          eta, gate, scale, Abuf, nch, l2, (T *)y);
    const int rc = launched("tc_fwd_simt");
    prof_end(s);
    return rc;
}

template <typename T, int DK>
int dispatch_dv(int dv, const void *q, const void *k, const void *v, int BH, int T_, int W,
                int H, const float *lam, const float *eta, const float *gate, float scale,
                const float *Abuf, int nch, int l2, void *y, cudaStream_t s) {
    switch (dv) {
        case 32: return launch_fwd<T, DK, 32>(q, k, v, BH, T_, W, H, lam, eta, gate, scale, Abuf, nch, l2, y, s);
        case 64: return launch_fwd<T, DK, 64>(q, k, v, BH, T_, W, H, lam, eta, gate, scale, Abuf, nch, l2, y, s);
        case 128: return launch_fwd<T, DK, 128>(q, k, v, BH, T_, W, H, lam, eta, gate, scale, Abuf, nch, l2, y, s);
    }
    set_error("d_v=%d unsupported", dv);
    return OPAM_ERR_UNSUPPORTED;
}

template <typename T>
int run(const void *q, const void *k, const void *v, int B, int H, int T_, int dk, int dv, int W,
        const float *lam, const float *eta, const float *gate, float scale, void *y,
        float *A_final, void *ws, cudaStream_t s, int l2) {
    const int BH = B * H, nch = ceil_div(T_, kC);
    float *buf = (float *)ws;
    if (l2) {
        const size_t smem = sizeof(float) * kC * (dk + dv);
        if (int rc_ = set_smem_limit((const void *)tc_chunk_delta_kernel<T>, (int)smem, "tc_chunk_delta smem attribute")) return rc_;
        tc_chunk_delta_kernel<T><<<dim3(nch, BH), 256, smem, s>>>((const T *)k, (const T *)v, T_, dk,
                                                                  dv, W, H, lam, eta, buf, nch);
        if (int rc = launched("tc_chunk_delta")) return rc;
    }
    if (l2) {
        tc_chunk_scan_kernel<<<dim3(ceil_div(dk * dv, 256), BH), 256, 0, s>>>(buf, nch, T_, dk * dv, H,
                                                                              lam, A_final);
        if (int rc = launched("tc_chunk_scan")) return rc;
    }
    switch (dk) {
        case 32: return dispatch_dv<T, 32>(dv, q, k, v, BH, T_, W, H, lam, eta, gate, scale, buf, nch, l2, y, s);
        case 64: return dispatch_dv<T, 64>(dv, q, k, v, BH, T_, W, H, lam, eta, gate, scale, buf, nch, l2, y, s);
        case 128: return dispatch_dv<T, 128>(dv, q, k, v, BH, T_, W, H, lam, eta, gate, scale, buf, nch, l2, y, s);
    }
    set_error("d_k=%d unsupported", dk);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace

size_t tc_prefill_simt_workspace(int BH, int T, int dk, int dv, int W) {
    (void)W;
    const int nch = ceil_div(T, kC);
    return align_up(sizeof(float) * (size_t)BH * (nch + 1) * dk * dv, 256);
}

int tc_prefill_simt(const void *q, const void *k, const void *v, int dtype, int B, int H, int T,
                    int dk, int dv, int W, const float *lam, const float *eta, const float *gate,
                    float scale, void *y, float *A_final, void *ws, cudaStream_t s, bool l2) {
    if (dtype == OPAM_BF16)
        return run<__nv_bfloat16>(q, k, v, B, H, T, dk, dv, W, lam, eta, gate, scale, y, A_final, ws, s, l2);
    return run<float>(q, k, v, B, H, T, dk, dv, W, lam, eta, gate, scale, y, A_final, ws, s, l2);
}

int tc_export_ring(const void *k, const void *v, int dtype, int B, int H, int T, int dk, int dv,
                   int W, void *ring_k, void *ring_v, int64_t *pos, cudaStream_t s) {
    const dim3 grid(W, B * H);
    if (dtype == OPAM_BF16)
        tc_export_ring_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(
            (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, T, dk, dv, W,
            (__nv_bfloat16 *)ring_k, (__nv_bfloat16 *)ring_v);
    else
        tc_export_ring_kernel<float><<<grid, 128, 0, s>>>((const float *)k, (const float *)v, T, dk,
                                                          dv, W, (float *)ring_k, (float *)ring_v);
    if (int rc = launched("tc_export_ring")) return rc;
    set_pos_kernel<<<ceil_div(B, 128), 128, 0, s>>>(pos, B, (int64_t)T);
    return launched("set_pos");
}

}  // namespace opam
