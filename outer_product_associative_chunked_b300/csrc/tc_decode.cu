// Tensor Cache single-token decode for a batch of independent sequences.
//
// "Tensor Cache: Eviction-conditioned Associative Memory for Transformers"
// (gist.science 2605.22884), Methodology 1: the L1 ring holds the W most
// recent tokens; when the ring overwrites an entry the displaced (k, v) is
// written A <- lambda A + eta k v^T; the new token reads the ring with exact
// softmax and the compressed past as q A; y = y_local + sigmoid(g) q A.
//
// Work per (sequence, head) is one pass over the ring (2 W d elements) and
// one read-modify-write of A (d_k d_v floats): memory bound.  The ring is
// split over `nsplit` CTAs per (sequence, head); each CTA also owns a slice
// of A's rows, so A is streamed exactly once.  Every stream is read with
// coalesced 16-byte loads that bypass L1 (each byte is used once).  Kernel 1 writes per-split
// partials (softmax max / sum / weighted values, and the partial q A of its
// rows); kernel 2 merges them flash-decoding style, applies the gate and
// stores the new token into its ring slot (after every reader of the evicted
// entry has finished); kernel 3 advances pos.  Kernels 2 and 3 are launched
// as programmatic dependents and wait for their predecessor before reading.
#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxKeysPerSplit = 8192;

struct DecodeGeom {
    int nsplit, keys_per_split;
};

DecodeGeom geom(int W) {
    int ns = ceil_div(W, 256);
    if (ns > 64) ns = 64;
    if (ns < ceil_div(W, kMaxKeysPerSplit)) ns = ceil_div(W, kMaxKeysPerSplit);
    return {ns, ceil_div(W, ns)};
}

// 16-byte vector of T: EPV elements.
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int EPV = 4;
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int EPV = 8;
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Per (sequence, head, split): the A rows of this split (eviction write and
// the partial q A), then the softmax over this split's ring slots.
// Ring rows are read as 16-byte vectors, LPK lanes per key row (a warp load
// covers KPW consecutive rows), with q held in registers; scores go to
// shared memory, then P V reads the value rows the same way.
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
tc_decode_partial_kernel(const T *__restrict__ ring_k, const T *__restrict__ ring_v,
                         float *__restrict__ A, const int64_t *__restrict__ pos,
                         const T *__restrict__ q, const T *__restrict__ k,
                         const T *__restrict__ v, int H, int W, int keys_per_split,
                         const float *__restrict__ lam, const float *__restrict__ eta,
                         float scale, float *__restrict__ part_m, float *__restrict__ part_o,
                         float *__restrict__ part_ml) {
    constexpr int EPV = Vec<T>::EPV;
    constexpr int LPK = DK / EPV, KPW = 32 / LPK;  // lanes per key row, rows per warp load
    constexpr int LPV = DV / EPV, VPW = 32 / LPV;
    constexpr int LPA = DV / 4, RPW = 32 / LPA;    // A rows: float4 per lane
    constexpr int NW = kThreads / 32;
    constexpr int U = 4;                           // loads in flight per lane
    extern __shared__ float sm[];
    float *qs = sm;              // [DK]
    float *kes = qs + DK;        // [DK] evicted key
    float *ves = kes + DK;       // [DV] evicted value
    float *red = ves + DV;       // [NW][DV] cross-warp reduction
    float *wred = red + NW * DV; // [2 * NW]
    float *sc = wred + 2 * NW;   // [keys_per_split] scores, then weights

    const int sh = blockIdx.x, sp = blockIdx.y, nsplit = gridDim.y;
    const int b = sh / H, h = sh - b * H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t p = pos[b];
    const int slot = (int)(p % W);
    const bool evict = p >= W;
    const size_t ring_row = (size_t)sh * W;

    for (int a = tid; a < DK; a += kThreads) {
        qs[a] = Elem<T>::load(q + (size_t)sh * DK + a);
        kes[a] = evict ? Elem<T>::load(ring_k + (ring_row + slot) * DK + a) : 0.f;
    }
    for (int c = tid; c < DV; c += kThreads)
        ves[c] = evict ? Elem<T>::load(ring_v + (ring_row + slot) * DV + c) : 0.f;
    __syncthreads();

    // ---- A rows of this split: eviction write, then partial q A.
    {
        const int rows = (DK + nsplit - 1) / nsplit;
        const int r0 = sp * rows, r1 = min(DK, r0 + rows);
        const float lm = lam[h], et = eta[h];
        const int c4 = (lane % LPA) * 4;
        float *Ab = A + (size_t)sh * DK * DV;
        float pm[4] = {0.f, 0.f, 0.f, 0.f};
        for (int a = r0 + warp * RPW + lane / LPA; a < r1; a += NW * RPW) {
            float4 x = *reinterpret_cast<const float4 *>(Ab + (size_t)a * DV + c4);
            if (evict) {
                const float ek = et * kes[a];
                x.x = fmaf(lm, x.x, ek * ves[c4]);
                x.y = fmaf(lm, x.y, ek * ves[c4 + 1]);
                x.z = fmaf(lm, x.z, ek * ves[c4 + 2]);
                x.w = fmaf(lm, x.w, ek * ves[c4 + 3]);
                *reinterpret_cast<float4 *>(Ab + (size_t)a * DV + c4) = x;
            }
            const float qa = qs[a];
            pm[0] = fmaf(qa, x.x, pm[0]);
            pm[1] = fmaf(qa, x.y, pm[1]);
            pm[2] = fmaf(qa, x.z, pm[2]);
            pm[3] = fmaf(qa, x.w, pm[3]);
        }
#pragma unroll
        for (int o = LPA; o < 32; o <<= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) pm[i] += __shfl_xor_sync(0xffffffffu, pm[i], o);
        if (lane < LPA)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp * DV + c4 + i] = pm[i];
        __syncthreads();
        for (int c = tid; c < DV; c += kThreads) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += red[w * DV + c];
            part_m[((size_t)sh * nsplit + sp) * DV + c] = s;
        }
        __syncthreads();
    }

    // ---- scores of this split's occupied slots (the new token sits at `slot`).
    const int occ = (p + 1 < (int64_t)W) ? (int)(p + 1) : W;
    const int s0 = sp * keys_per_split, s1 = min(occ, s0 + keys_per_split);
    const int nk = max(0, s1 - s0);
    {
        const int ks = lane / LPK, kc = (lane % LPK) * EPV;
        float qv[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) qv[e] = qs[kc + e];
        for (int g0 = warp; g0 * KPW < nk; g0 += NW * U) {
            uint4 raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int key = (g0 + NW * u) * KPW + ks, idx = s0 + key;
                const T *src = (idx == slot) ? k + (size_t)sh * DK : ring_k + (ring_row + idx) * DK;
                raw[u] = key < nk ? ldg_stream(src + kc) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float f[EPV];
                Vec<T>::unpack(raw[u], f);
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < EPV; ++e) d = fmaf(qv[e], f[e], d);
#pragma unroll
                for (int o = LPK / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                const int key = (g0 + NW * u) * KPW + ks;
                if (lane % LPK == 0 && key < nk) sc[key] = d * scale;
            }
        }
    }
    __syncthreads();
    float mx = kNegBig;
    for (int i = tid; i < nk; i += kThreads) mx = fmaxf(mx, sc[i]);
    mx = warp_max(mx);
    if (lane == 0) wred[warp] = mx;
    __syncthreads();
    mx = kNegBig;
#pragma unroll
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, wred[w]);
    float ssum = 0.f;
    for (int i = tid; i < nk; i += kThreads) {
        const float e = __expf(sc[i] - mx);
        sc[i] = e;
        ssum += e;
    }
    ssum = warp_sum(ssum);
    if (lane == 0) wred[NW + warp] = ssum;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s += wred[NW + w];
        part_ml[((size_t)sh * nsplit + sp) * 2 + 0] = mx;
        part_ml[((size_t)sh * nsplit + sp) * 2 + 1] = s;
    }

    // ---- P V over this split's slots.
    {
        const int vs = lane / LPV, vc = (lane % LPV) * EPV;
        float acc[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
        for (int g0 = warp; g0 * VPW < nk; g0 += NW * U) {
            uint4 raw[U];
            float pw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int key = (g0 + NW * u) * VPW + vs, idx = s0 + key;
                const T *src = (idx == slot) ? v + (size_t)sh * DV : ring_v + (ring_row + idx) * DV;
                const bool ok = key < nk;
                raw[u] = ok ? ldg_stream(src + vc) : make_uint4(0u, 0u, 0u, 0u);
                pw[u] = ok ? sc[key] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float f[EPV];
                Vec<T>::unpack(raw[u], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) acc[e] = fmaf(pw[u], f[e], acc[e]);
            }
        }
#pragma unroll
        for (int o = LPV; o < 32; o <<= 1)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
        __syncthreads();  // red reused
        if (lane < LPV)
#pragma unroll
            for (int e = 0; e < EPV; ++e) red[warp * DV + vc + e] = acc[e];
        __syncthreads();
        for (int c = tid; c < DV; c += kThreads) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += red[w * DV + c];
            part_o[((size_t)sh * nsplit + sp) * DV + c] = s;
        }
    }
}

template <typename T, int DK, int DV>
__global__ void tc_decode_combine_kernel(T *__restrict__ ring_k, T *__restrict__ ring_v,
                                         const int64_t *__restrict__ pos,
                                         const T *__restrict__ k, const T *__restrict__ v,
                                         int H, int W, int nsplit,
                                         const float *__restrict__ gate,
                                         const float *__restrict__ part_m,
                                         const float *__restrict__ part_o,
                                         const float *__restrict__ part_ml, T *__restrict__ y) {
    // Launched as a programmatic dependent of the partial kernel: wait for its
    // partials (and for its reads of the evicted ring slot) before anything else.
    sm100::pdl_wait_primary();
    const int sh = blockIdx.x, b = sh / H, h = sh - b * H;
    const int tid = threadIdx.x;
    const float *ml = part_ml + (size_t)sh * nsplit * 2;
    float M = kNegBig;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[2 * s]);
    if (tid < DV) {
        float L = 0.f, o = 0.f, m = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float f = expf(ml[2 * s] - M);
            L = fmaf(ml[2 * s + 1], f, L);
            o = fmaf(part_o[((size_t)sh * nsplit + s) * DV + tid], f, o);
            m += part_m[((size_t)sh * nsplit + s) * DV + tid];
        }
        const float sg = 1.0f / (1.0f + expf(-gate[h]));
        Elem<T>::store(y + (size_t)sh * DV + tid, o / L + sg * m);
    }
    const int slot = (int)(pos[b] % W);
    for (int a = tid; a < DK; a += blockDim.x)
        ring_k[((size_t)sh * W + slot) * DK + a] = k[(size_t)sh * DK + a];
    for (int c = tid; c < DV; c += blockDim.x)
        ring_v[((size_t)sh * W + slot) * DV + c] = v[(size_t)sh * DV + c];
}

// Also zeroes the call's status words: no kernel of the decode step has a
// bounded wait, so nothing else writes it and the word reads clean after the
// step.
__global__ void advance_pos_kernel(int64_t *pos, int B, unsigned int *status) {
    sm100::pdl_wait_primary();  // every reader of pos in this step has finished
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) pos[b] += 1;
    if (b < kStatusWords) status[b] = 0u;
}

struct Parts {
    float *m, *o, *ml;
};

Parts carve(void *ws, int SH, int nsplit, int dv) {
    char *p = (char *)ws;
    Parts r;
    r.m = (float *)p;
    p += align_up(sizeof(float) * (size_t)SH * nsplit * dv, 256);
    r.o = (float *)p;
    p += align_up(sizeof(float) * (size_t)SH * nsplit * dv, 256);
    r.ml = (float *)p;
    return r;
}

template <typename T, int DK, int DV>
int launch(const opam_tc_state *st, const void *q, const void *k, const void *v, const float *lam,
           const float *eta, const float *gate, float scale, void *y, void *ws, unsigned int *status,
           cudaStream_t s) {
    const int SH = st->B * st->H;
    const DecodeGeom g = geom(st->W);
    const Parts pr = carve(ws, SH, g.nsplit, DV);
    const size_t smem = sizeof(float) * (DK + DK + DV + (kThreads / 32) * DV + 2 * (kThreads / 32) + g.keys_per_split);
    auto k1 = tc_decode_partial_kernel<T, DK, DV>;
    if (int rc_ = set_smem_limit((const void *)k1, (int)smem, "tc_decode smem attribute")) return rc_;
    prof_begin(s);
    k1<<<dim3(SH, g.nsplit), kThreads, smem, s>>>(
        (const T *)st->ring_k, (const T *)st->ring_v, st->A, st->pos, (const T *)q, (const T *)k,
        (const T *)v, st->H, st->W, g.keys_per_split, lam, eta, scale, pr.m, pr.o, pr.ml);
    if (int rc = launched("tc_decode_partial")) return rc;
    prof_end(s);
    // The combine and pos kernels are programmatic dependents: each is set up
    // while its predecessor finishes and waits (griddepcontrol) before reading.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(SH);
    cfg.blockDim = dim3(128);
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc_decode_combine_kernel<T, DK, DV>, (T *)st->ring_k,
                                       (T *)st->ring_v, (const int64_t *)st->pos, (const T *)k, (const T *)v,
                                       st->H, st->W, g.nsplit, gate, (const float *)pr.m, (const float *)pr.o,
                                       (const float *)pr.ml, (T *)y);
    if (e != cudaSuccess) return cuda_fail(e, "tc_decode_combine launch");
    if (int rc = launched("tc_decode_combine")) return rc;
    cfg.gridDim = dim3(ceil_div(st->B, 128));
    e = cudaLaunchKernelEx(&cfg, advance_pos_kernel, st->pos, st->B, status);
    if (e != cudaSuccess) return cuda_fail(e, "advance_pos launch");
    return launched("advance_pos");
}

template <typename T, int DK>
int by_dv(const opam_tc_state *st, const void *q, const void *k, const void *v, const float *lam,
          const float *eta, const float *gate, float scale, void *y, void *ws, unsigned int *status,
          cudaStream_t s) {
    switch (st->d_v) {
        case 32: return launch<T, DK, 32>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
        case 64: return launch<T, DK, 64>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
        case 128: return launch<T, DK, 128>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
    }
    set_error("d_v=%d unsupported", st->d_v);
    return OPAM_ERR_UNSUPPORTED;
}

template <typename T>
int by_dk(const opam_tc_state *st, const void *q, const void *k, const void *v, const float *lam,
          const float *eta, const float *gate, float scale, void *y, void *ws, unsigned int *status,
          cudaStream_t s) {
    switch (st->d_k) {
        case 32: return by_dv<T, 32>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
        case 64: return by_dv<T, 64>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
        case 128: return by_dv<T, 128>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
    }
    set_error("d_k=%d unsupported", st->d_k);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace

size_t tc_decode_workspace(int S, int H, int dk, int dv, int W) {
    (void)dk;
    const DecodeGeom g = geom(W);
    const size_t SH = (size_t)S * H;
    return 2 * align_up(sizeof(float) * SH * g.nsplit * dv, 256) +
           align_up(sizeof(float) * SH * g.nsplit * 2, 256);
}

int tc_decode(const opam_tc_state *st, const void *q, const void *k, const void *v,
              const float *lam, const float *eta, const float *gate, float scale, void *y,
              void *ws, unsigned int *status, cudaStream_t s) {
    if (st->dtype == OPAM_BF16)
        return by_dk<__nv_bfloat16>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
    return by_dk<float>(st, q, k, v, lam, eta, gate, scale, y, ws, status, s);
}

}  // namespace opam
