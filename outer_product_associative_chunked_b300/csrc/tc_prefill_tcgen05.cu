// Tensor Cache layer prefill on the tensor cores (bf16 inputs, fp32 state and
// accumulation): tcgen05.mma with TMEM accumulators, operands staged by TMA.
//
// "Tensor Cache: Eviction-conditioned Associative Memory for Transformers"
// (gist.science 2605.22884).  Methodology 1: softmax over the W most recent
// tokens (the ring), eviction write A <- lambda A + eta k v^T, read
// m_t = q_t A, fuse y_t = y_local,t + sigmoid(g) m_t.  Methodology 2: a
// parallel weighted-sum scan equal to the per-token writes.  Token s is
// written at step s + W, so m_t = sum_{s <= t-W} eta lambda^(t-W-s) <q_t,k_s> v_s.
//
// Blocks of C = 128 positions.  Query block j covers [jC, jC+C); the tokens
// evicted during its steps are the shifted chunk [jC-W, jC-W+C).  With A_j the
// state before the block (every token s < jC-W) and row i of the block:
//   m_{jC+i} = lambda^(i+1) q A_j + sum_{l<=i} eta lambda^(i-l) <q, k'_l> v'_l
//   A_{j+1}  = lambda^n A_j + dA_j,  dA_j = sum_{l<n} eta lambda^(n-1-l) k'_l v'_l^T
// The shifted chunk is exactly the first key tile of the block's window
// (keys [jC-W, jC+C) in tiles of 128), so one Q K^T product serves both the
// L2 term (key l <= row i) and the softmax (l > i).
//
// Three kernels:
//   tc_l2_delta_kernel  dA_j = K'^T diag(w) V' per (head, chunk) on tcgen05;
//   tc_l2_scan_kernel   A_j from the dA_j (a first-order linear recurrence per
//                       element), written as bf16 for the next kernel, and the
//                       final fp32 state;
//   tc_fwd_kernel       per (head, query block): flash-style online softmax
//                       over the window tiles (S = Q K^T and O += P V on
//                       tcgen05), the L2 term P2 V' and q A_j, and the gate.
//
// tc_fwd_kernel warp roles (192 threads): warps 0-3 own one query row per
// thread (softmax, P, epilogue); warp 4 issues TMA loads; warp 5 issues the
// MMAs and owns the TMEM allocation.  TMEM columns: S double buffer [0,256),
// O [256, 256+DV), O2 (the L2 term) [256+DV, 256+2DV); q A_j lands in the S
// buffer that is free after the last tile.  Every wait is bounded; a wait that
// runs out records a status bit (tc_prefill_tcgen05_status) and the CTA winds
// down without hanging.
#include <math.h>

#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

constexpr int kBlk = 128;          // query rows per CTA = keys per tile = chunk length
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.0f;   // lazy-rescale threshold (log2 units)

__device__ unsigned int g_status = 0;
enum : unsigned int {
    kStDeltaWait = 1u,
    kStFwdProducer = 2u,
    kStFwdMma = 4u,
    kStFwdSoftmax = 8u,
};

// --------------------------------------------------------------------- dA_j
// One CTA per (chunk j, head).  A = K'^T is read MN-major from the K' tile
// (tokens x d_k); M is fixed at 128, so for d_k = 64 the two 64-wide M blocks
// alias the same data (lanes 64..127 hold a copy and are ignored).
template <int DK, int DV>
__global__ void __launch_bounds__(128)
tc_l2_delta_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                   int T, int W, int H, const float *__restrict__ lam,
                   const float *__restrict__ eta, int nch, float *__restrict__ dA) {
    constexpr uint32_t KBYTES = kBlk * DK * 2, VBYTES = kBlk * DV * 2;
    constexpr uint32_t TCOLS = DV < 32 ? 32 : DV;
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    unsigned char *Ks = sm, *Vs = sm + KBYTES;
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tbase;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int j = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int kt = j * kBlk - W;
    const int n = min(kBlk, T - j * kBlk);
    float *out = dA + ((size_t)bh * nch + j) * (size_t)(DK * DV);
    if (kt + n <= 0) {  // nothing evicted during this chunk
        for (int e = tid; e < DK * DV / 4; e += 128)
            reinterpret_cast<float4 *>(out)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    if (warp == 0) tmem_alloc(&tbase, TCOLS);
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    if (tid == 0) {
        mbar_expect_tx(&bars[0], KBYTES + VBYTES);
#pragma unroll
        for (int b = 0; b < DK / 64; ++b) tma_load_3d(Ks + b * 16384, &mk, &bars[0], 64 * b, kt, bh);
#pragma unroll
        for (int b = 0; b < DV / 64; ++b) tma_load_3d(Vs + b * 16384, &mv, &bars[0], 64 * b, kt, bh);
    }
    bool ok = mbar_wait(&bars[0], 0);
    // Row l of V' times w_l = eta lambda^(n-1-l) (zero for rows outside the
    // chunk or before position 0); a row keeps its 16-byte chunks in place.
    {
        const int l = tid;
        const float w = (l < n && kt + l >= 0) ? eta[h] * powf(lam[h], (float)(n - 1 - l)) : 0.f;
#pragma unroll
        for (int b = 0; b < DV / 64; ++b) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t a = smem_u32(Vs) + b * 16384 + l * 128 + c * 16;
                uint32_t x[4];
                ld_shared_v4(a, x[0], x[1], x[2], x[3]);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    __nv_bfloat162 hv = *reinterpret_cast<__nv_bfloat162 *>(&x[u]);
                    float2 f = __bfloat1622float2(hv);
                    x[u] = pack_bf16(f.x * w, f.y * w);
                }
                st_shared_v4(a, x[0], x[1], x[2], x[3]);
            }
        }
        fence_async_smem();
    }
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, DV, true, true);
        const uint32_t ka = smem_u32(Ks), va = smem_u32(Vs);
#pragma unroll
        for (int k = 0; k < kBlk / 16; ++k)
            mma_ss(tm, sdesc_sw128(ka + k * 2048, DK == 128 ? 16384 : 0, 1024),
                   sdesc_sw128(va + k * 2048, 16384, 1024), idesc, k > 0 ? 1u : 0u);
        mma_commit(&bars[1]);
    }
    ok = __syncthreads_and(ok);
    if (ok) ok = mbar_wait(&bars[1], 0);
    __syncwarp();
    tc_fence_after();
    if (!ok) {
        if (tid == 0) atomicOr(&g_status, kStDeltaWait);
    } else if (warp < DK / 32) {
        const int a = tid;  // row of dA = key coordinate
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += 32) {
            float v[32];
            tmem_ld32(tm + ((uint32_t)(warp * 32) << 16) + c0, v);
            tmem_wait_ld();
            float4 *dst = reinterpret_cast<float4 *>(out + (size_t)a * DV + c0);
#pragma unroll
            for (int u = 0; u < 8; ++u) dst[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, TCOLS);
}

// --------------------------------------------------------------------- scan
// A_0 = 0, A_{j+1} = lambda^{n_j} A_j + dA_j.  Each thread owns 4 adjacent
// elements of one head's d_k x d_v state; Abf[bh][j] receives A_j (bf16) and
// A_final the state after the last chunk (fp32).
__global__ void __launch_bounds__(128)
tc_l2_scan_kernel(const float *__restrict__ dA, int nch, int T, int dkdv, int H,
                  const float *__restrict__ lam, __nv_bfloat16 *__restrict__ Abf,
                  float *__restrict__ A_final) {
    const int bh = blockIdx.y;
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (e >= dkdv) return;
    const float lm = lam[bh % H];
    const float lamC = powf(lm, (float)kBlk);
    const float *src = dA + (size_t)bh * nch * dkdv + e;
    __nv_bfloat16 *dst = Abf + (size_t)bh * nch * dkdv + e;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    int j = 0;
    for (; j + 8 <= nch; j += 8) {
        float4 d[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) d[u] = *reinterpret_cast<const float4 *>(src + (size_t)(j + u) * dkdv);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            uint2 o;
            o.x = pack_bf16(A.x, A.y);
            o.y = pack_bf16(A.z, A.w);
            *reinterpret_cast<uint2 *>(dst + (size_t)(j + u) * dkdv) = o;
            const int n = min(kBlk, T - (j + u) * kBlk);
            const float f = n == kBlk ? lamC : powf(lm, (float)n);
            A.x = fmaf(f, A.x, d[u].x);
            A.y = fmaf(f, A.y, d[u].y);
            A.z = fmaf(f, A.z, d[u].z);
            A.w = fmaf(f, A.w, d[u].w);
        }
    }
    for (; j < nch; ++j) {
        const float4 d = *reinterpret_cast<const float4 *>(src + (size_t)j * dkdv);
        uint2 o;
        o.x = pack_bf16(A.x, A.y);
        o.y = pack_bf16(A.z, A.w);
        *reinterpret_cast<uint2 *>(dst + (size_t)j * dkdv) = o;
        const int n = min(kBlk, T - j * kBlk);
        const float f = n == kBlk ? lamC : powf(lm, (float)n);
        A.x = fmaf(f, A.x, d.x);
        A.y = fmaf(f, A.y, d.y);
        A.z = fmaf(f, A.z, d.z);
        A.w = fmaf(f, A.w, d.w);
    }
    if (A_final) *reinterpret_cast<float4 *>(A_final + (size_t)bh * dkdv + e) = A;
}

// --------------------------------------------------------------------- fused forward
template <int DK, int DV>
struct Fwd {
    static constexpr uint32_t QBYTES = kBlk * DK * 2;
    static constexpr uint32_t KBYTES = kBlk * DK * 2;  // also holds A_j (DK x DV bf16)
    static constexpr uint32_t VBYTES = kBlk * DV * 2;
    static constexpr uint32_t PBYTES = kBlk * kBlk * 2;
    static constexpr uint32_t kBudget = 226 * 1024;
    static constexpr int kStagesFit = (int)((kBudget - 1024 - QBYTES - 2 * PBYTES) / (KBYTES + VBYTES));
    static constexpr int NST = kStagesFit > 4 ? 4 : kStagesFit;
    static_assert(NST >= 2, "need two K/V stages");
    static constexpr uint32_t OFF_K = QBYTES;
    static constexpr uint32_t OFF_P = QBYTES + NST * (KBYTES + VBYTES);
    static constexpr uint32_t SMEM = OFF_P + 2 * PBYTES + 1024;  // +1024: alignment slack
    static constexpr uint32_t COL_O = 256, COL_O2 = 256 + DV;
    static_assert(256 + 2 * DV <= 512, "TMEM columns");
    static constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t ID_PV = idesc_bf16_f32(128, DV, false, true);
};

struct FwdBars {
    uint64_t q_full;
    uint64_t k_full[4], v_full[4], kv_empty[4];
    uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
    uint64_t o_done, drain;
    uint32_t tbase;
    float pw[kBlk];  // eta lambda^d, d = 0..127
};

template <int DK, int DV>
__global__ void __launch_bounds__(192, 1)
tc_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap ma,
              int T, int W, int H, int nch, const float *__restrict__ lam,
              const float *__restrict__ eta, const float *__restrict__ gate, float scale,
              __nv_bfloat16 *__restrict__ y) {
    using C = Fwd<DK, DV>;
    constexpr int NST = C::NST;
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    __shared__ FwdBars B;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int jq = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int t0 = jq * kBlk;
    const int kt0 = t0 - W;  // first key of tile 0 (the shifted chunk)
    const int nt_total = (W + kBlk - 1) / kBlk + 1;
    const int j_first = (-kt0 - (kBlk - 1) > 0) ? (-kt0) / kBlk : 0;
    const int ntiles = nt_total - j_first;
    const bool has_l2 = (j_first == 0);

    if (warp == 5) tmem_alloc(&B.tbase, 512);
    if (tid == 0) {
        mbar_init(&B.q_full, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(&B.k_full[s], 1);
            mbar_init(&B.v_full[s], 1);
            mbar_init(&B.kv_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&B.s_full[s], 1);
            mbar_init(&B.s_empty[s], 4);
            mbar_init(&B.p_full[s], 4);
            mbar_init(&B.p_empty[s], 1);
        }
        mbar_init(&B.o_done, 1);
        mbar_init(&B.drain, 1);
        mbar_fence_init();
    }
    if (tid < kBlk) B.pw[tid] = eta[h] * powf(lam[h], (float)tid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;
    const uint32_t sQ = smem_u32(sm);
    const uint32_t sK0 = sQ + C::OFF_K;
    const uint32_t sP0 = sQ + C::OFF_P;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            tma_prefetch_desc(&mq);
            tma_prefetch_desc(&mk);
            tma_prefetch_desc(&mv);
            mbar_expect_tx(&B.q_full, C::QBYTES);
#pragma unroll
            for (int b = 0; b < DK / 64; ++b) tma_load_3d(sm + b * 16384, &mq, &B.q_full, 64 * b, t0, bh);
            int issued = 0;
            for (int n = 0; n <= ntiles && ok; ++n) {
                const int s = n % NST;
                if (n >= NST) ok = mbar_wait(&B.kv_empty[s], ((n / NST) - 1) & 1);
                if (!ok) break;
                unsigned char *kd = sm + C::OFF_K + s * (C::KBYTES + C::VBYTES);
                if (n < ntiles) {
                    const int kt = kt0 + kBlk * (j_first + n);
                    mbar_expect_tx(&B.k_full[s], C::KBYTES);
#pragma unroll
                    for (int b = 0; b < DK / 64; ++b) tma_load_3d(kd + b * 16384, &mk, &B.k_full[s], 64 * b, kt, bh);
                    mbar_expect_tx(&B.v_full[s], C::VBYTES);
#pragma unroll
                    for (int b = 0; b < DV / 64; ++b)
                        tma_load_3d(kd + C::KBYTES + b * 16384, &mv, &B.v_full[s], 64 * b, kt, bh);
                } else {  // the carried state A_j (bf16, d_k rows x d_v) into the K slot
                    mbar_expect_tx(&B.k_full[s], DK * DV * 2);
#pragma unroll
                    for (int b = 0; b < DV / 64; ++b)
                        tma_load_3d(kd + b * (DK * 128), &ma, &B.k_full[s], 64 * b, 0, bh * nch + jq);
                }
                ++issued;
            }
            if (!ok) atomicOr(&g_status, kStFwdProducer);
            // Drain: the newest load of each stage has landed before the CTA exits.
            bool dok = mbar_wait(&B.q_full, 0);
            for (int n = max(0, issued - NST); n < issued && dok; ++n) {
                const int s = n % NST;
                dok = mbar_wait(&B.k_full[s], (n / NST) & 1);
                if (dok && n < ntiles) dok = mbar_wait(&B.v_full[s], (n / NST) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(&B.q_full, 0);
            uint32_t use = 0;  // P-slot uses so far
            auto kdesc = [&](int s, int k) {
                return sdesc_sw128(sK0 + s * (C::KBYTES + C::VBYTES) + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
            };
            auto qdesc = [&](int k) { return sdesc_sw128(sQ + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); };
            auto vdesc = [&](int s, int k) {
                return sdesc_sw128(sK0 + s * (C::KBYTES + C::VBYTES) + C::KBYTES + k * 2048, 16384, 1024);
            };
            auto pdesc = [&](int slot, int k) {
                return sdesc_sw128(sP0 + slot * C::PBYTES + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
            };
            // O += P V (and O2 = P2 V' for tile 0) for processed tile n.
            auto pv = [&](int n) -> bool {
                const int s = n % NST;
                if (!mbar_wait(&B.v_full[s], (n / NST) & 1)) return false;
                const int uses = (n == 0 && has_l2) ? 2 : 1;
                for (int u = 0; u < uses; ++u) {
                    const int slot = use & 1;
                    if (!mbar_wait(&B.p_full[slot], (use >> 1) & 1)) return false;
                    tc_fence_after();
                    const bool l2 = (uses == 2 && u == 0);
                    const uint32_t dcol = l2 ? C::COL_O2 : C::COL_O;
#pragma unroll
                    for (int k = 0; k < kBlk / 16; ++k)
                        mma_ss(tm + dcol, pdesc(slot, k), vdesc(s, k), C::ID_PV,
                               (l2 ? k > 0 : (n > 0 || k > 0)) ? 1u : 0u);
                    mma_commit(&B.p_empty[slot]);
                    ++use;
                }
                mma_commit(&B.kv_empty[s]);
                return true;
            };
            for (int n = 0; n < ntiles && ok; ++n) {
                const int s = n % NST, sb = n & 1;
                ok = mbar_wait(&B.k_full[s], (n / NST) & 1);
                if (ok && n >= 2) ok = mbar_wait(&B.s_empty[sb], ((n - 2) >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < DK / 16; ++k)
                    mma_ss(tm + sb * 128, qdesc(k), kdesc(s, k), C::ID_S, k > 0 ? 1u : 0u);
                mma_commit(&B.s_full[sb]);
                if (n >= 1) ok = pv(n - 1);
            }
            if (ok) ok = pv(ntiles - 1);
            if (ok) {  // q A_j into the S buffer that follows the last tile
                const int n = ntiles, s = n % NST, sb = n & 1;
                ok = mbar_wait(&B.k_full[s], (n / NST) & 1);
                if (ok && n >= 2) ok = mbar_wait(&B.s_empty[sb], ((n - 2) >> 1) & 1);
                if (ok) {
                    tc_fence_after();
                    const uint32_t aslot = sK0 + s * (C::KBYTES + C::VBYTES);
#pragma unroll
                    for (int k = 0; k < DK / 16; ++k)
                        mma_ss(tm + sb * 128, qdesc(k), sdesc_sw128(aslot + k * 2048, DK * 128, 1024),
                               C::ID_PV, k > 0 ? 1u : 0u);
                    mma_commit(&B.o_done);
                }
            }
            if (!ok) atomicOr(&g_status, kStFwdMma);
            // Every MMA issued by this thread has completed before TMEM is freed.
            mma_commit(&B.drain);
            mbar_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax / epilogue (row r)
        const int r = tid;
        const int t = t0 + r;
        const uint32_t lrow = (uint32_t)(warp * 32) << 16;
        const float sc = scale * kLog2e;
        float m = kNegBig, l = 0.f;
        uint32_t use = 0;
        int last_o_use = -1;
        bool ok = true;
        auto wait_slot = [&](uint32_t u) -> bool {  // slot of use u is free again
            return u < 2 || mbar_wait(&B.p_empty[u & 1], ((u - 2) >> 1) & 1);
        };
        // Row r of a P slot: 16 chunks of 8 bf16 in the 128-byte-swizzle K-major layout.
        auto store8 = [&](uint32_t slot, int c, const float *p) {
            st_shared_v4(sP0 + slot * C::PBYTES + (c >> 3) * 16384 + sw128_off(r, c & 7),
                         pack_bf16(p[0], p[1]), pack_bf16(p[2], p[3]), pack_bf16(p[4], p[5]),
                         pack_bf16(p[6], p[7]));
        };
        for (int n = 0; n < ntiles && ok; ++n) {
            const int j = j_first + n;
            const int kt = kt0 + kBlk * j;
            const int sb = n & 1;
            ok = mbar_wait(&B.s_full[sb], (n >> 1) & 1);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            float s[kBlk];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[32];
                tmem_ld32(tm + lrow + sb * 128 + c * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = v[i];
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.s_empty[sb]);

            if (j == 0) {  // L2 part of the shifted chunk: keys l <= r at positions >= 0
                const int lo = max(0, -kt);
                ok = __all_sync(0xffffffffu, wait_slot(use));
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float p2[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 8 * c + e;
                        p2[e] = (i >= lo && i <= r) ? B.pw[(r - i) & (kBlk - 1)] * s[i] : 0.f;
                    }
                    store8(use & 1, c, p2);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.p_full[use & 1]);
                ++use;
            }
            // Softmax part: keys max(0, t-W+1) <= p <= t.
            const bool interior = (j >= 1) && (kt >= 0) && (kt <= t0 - (kBlk - 1));
            float mx = -INFINITY;
            if (interior) {
#pragma unroll
                for (int i = 0; i < kBlk; ++i) mx = fmaxf(mx, s[i]);
            } else {
                const int lo = max(0, t - W + 1) - kt, hi = t - kt;
#pragma unroll
                for (int i = 0; i < kBlk; ++i) {
                    s[i] = (i >= lo && i <= hi) ? s[i] : -INFINITY;
                    mx = fmaxf(mx, s[i]);
                }
            }
            mx *= sc;
            const bool grow = mx > m + kRescale;
            const bool rescale_o = grow && l > 0.f;
            if (__any_sync(0xffffffffu, rescale_o)) {
                // O must hold every earlier P V product before it is rescaled.
                const uint32_t u = (uint32_t)last_o_use;
                ok = __all_sync(0xffffffffu, mbar_wait(&B.p_empty[u & 1], (u >> 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const float f = rescale_o ? ex2(m - mx) : 1.f;
#pragma unroll
                for (int c0 = 0; c0 < DV; c0 += 32) {
                    float v[32];
                    tmem_ld32(tm + lrow + C::COL_O + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= f;
                    tmem_st32(tm + lrow + C::COL_O + c0, v);
                }
                tmem_wait_st();
            }
            if (grow) {
                l *= ex2(m - mx);
                m = mx;
            }
            float rs = 0.f;
#pragma unroll
            for (int i = 0; i < kBlk; ++i) {
                s[i] = ex2(fmaf(s[i], sc, -m));
                rs += s[i];
            }
            l += rs;
            ok = __all_sync(0xffffffffu, wait_slot(use));
            if (!ok) break;
#pragma unroll
            for (int c = 0; c < 16; ++c) store8(use & 1, c, &s[8 * c]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.p_full[use & 1]);
            last_o_use = (int)use;
            ++use;
        }
        // ------------------------------------------------ epilogue
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&B.o_done, 0));
        if (ok) {
            tc_fence_after();
            const uint32_t col_qa = (uint32_t)(ntiles & 1) * 128;
            const float sg = 1.0f / (1.0f + expf(-gate[h]));
            const float decay = powf(lam[h], (float)(r + 1));
            const float inv_l = l > 0.f ? 1.0f / l : 0.f;
            __nv_bfloat16 *yr = y + ((size_t)bh * T + t) * DV;
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
                float o[32], qa[32], o2[32];
                tmem_ld32(tm + lrow + C::COL_O + c0, o);
                tmem_ld32(tm + lrow + col_qa + c0, qa);
                if (has_l2) tmem_ld32(tm + lrow + C::COL_O2 + c0, o2);
                tmem_wait_ld();
                if (t < T) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a0 = fmaf(decay, qa[2 * i], has_l2 ? o2[2 * i] : 0.f);
                        float a1 = fmaf(decay, qa[2 * i + 1], has_l2 ? o2[2 * i + 1] : 0.f);
                        pk[i] = pack_bf16(fmaf(o[2 * i], inv_l, sg * a0), fmaf(o[2 * i + 1], inv_l, sg * a1));
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(yr + c0);
#pragma unroll
                    for (int u = 0; u < 4; ++u) dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                }
            }
        }
        if (!ok && lane == 0) atomicOr(&g_status, kStFwdSoftmax);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) tmem_dealloc(tm, 512);
}

template <int DK, int DV>
int run(const void *q, const void *k, const void *v, int B_, int H, int T, int W, const float *lam,
        const float *eta, const float *gate, float scale, void *y, float *A_final, void *ws,
        cudaStream_t st) {
    const int BH = B_ * H, nch = ceil_div(T, kBlk);
    float *dA = (float *)ws;
    __nv_bfloat16 *Abf = (__nv_bfloat16 *)((char *)ws + align_up(sizeof(float) * (size_t)BH * nch * DK * DV, 1024));
    CUtensorMap mq, mk, mv, mk_d, mv_d, ma;
    int rc;
    if ((rc = make_tmap_bf16_3d(&mq, q, DK, T, BH, kBlk))) return rc;
    if ((rc = make_tmap_bf16_3d(&mk, k, DK, T, BH, kBlk))) return rc;
    if ((rc = make_tmap_bf16_3d(&mv, v, DV, T, BH, kBlk))) return rc;
    if ((rc = make_tmap_bf16_3d(&ma, Abf, DV, DK, (uint64_t)BH * nch, DK))) return rc;
    mk_d = mk;
    mv_d = mv;
    {
        const int smem = kBlk * (DK + DV) * 2 + 1024;
        auto kern = tc_l2_delta_kernel<DK, DV>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "tc_l2_delta smem attribute");
        kern<<<dim3(nch, BH), 128, smem, st>>>(mk_d, mv_d, T, W, H, lam, eta, nch, dA);
        if ((rc = launched("tc_l2_delta"))) return rc;
    }
    {
        const int per = DK * DV / 4;
        tc_l2_scan_kernel<<<dim3(ceil_div(per, 128), BH), 128, 0, st>>>(dA, nch, T, DK * DV, H, lam, Abf,
                                                                       A_final);
        if ((rc = launched("tc_l2_scan"))) return rc;
    }
    {
        using Cfg = Fwd<DK, DV>;
        auto kern = tc_fwd_kernel<DK, DV>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
        if (e != cudaSuccess) return cuda_fail(e, "tc_fwd smem attribute");
        prof_begin(st);
        kern<<<dim3(nch, BH), 192, Cfg::SMEM, st>>>(mq, mk, mv, ma, T, W, H, nch, lam, eta, gate, scale,
                                                    (__nv_bfloat16 *)y);
        rc = launched("tc_fwd");
        prof_end(st);
        return rc;
    }
}

}  // namespace

bool tc_prefill_tcgen05_supported(int dtype, int dk, int dv) {
    return dtype == OPAM_BF16 && (dk == 64 || dk == 128) && (dv == 64 || dv == 128);
}

size_t tc_prefill_tcgen05_workspace(int BH, int T, int dk, int dv) {
    const size_t nch = (size_t)ceil_div(T, kBlk);
    return align_up(sizeof(float) * BH * nch * dk * dv, 1024) + align_up(2 * BH * nch * dk * dv, 1024);
}

int tc_prefill_tcgen05(const void *q, const void *k, const void *v, int B, int H, int T, int dk,
                       int dv, int W, const float *lam, const float *eta, const float *gate,
                       float scale, void *y, float *A_final, void *ws, cudaStream_t s) {
    if (dk == 64 && dv == 64) return run<64, 64>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, s);
    if (dk == 64 && dv == 128) return run<64, 128>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, s);
    if (dk == 128 && dv == 64) return run<128, 64>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, s);
    if (dk == 128 && dv == 128) return run<128, 128>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, s);
    set_error("tensor-core prefill: d_k=%d d_v=%d unsupported", dk, dv);
    return OPAM_ERR_UNSUPPORTED;
}

unsigned int tc_prefill_tcgen05_status(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (clear && v) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_status, &z, sizeof z);
    }
    return v;
}

}  // namespace opam
