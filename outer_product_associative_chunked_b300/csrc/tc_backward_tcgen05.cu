// Tensor Cache layer backward, window part of dK and dV on the tensor cores
// (bf16 q, k, v and dy; fp32 statistics and accumulators).
//
// "Tensor Cache: Eviction-conditioned Associative Memory for Transformers"
// (gist.science 2605.22884), Methodology 1: the window softmax
// y_loc = P V with P = softmax(scale Q K^T) on the band t - W < s <= t.  Its
// gradient with respect to the keys and values, for key s:
//   dV_s = sum_t P_ts dy_t,
//   dK_s = scale sum_t dS_ts q_t,   dS_ts = P_ts (<dy_t, v_s> - D_t),
// with P_ts = exp(scale <q_t, k_s> - LSE_t) and D_t = <dy_t, y_loc,t> from
// the window dQ pass (tcb_window_dq_kernel), which also writes LSE_t.
//
// One CTA per (128 keys, head) walks the query tiles of 128 that see those
// keys, in transposed form so that the keys are the MMA rows:
//   S^T  = K Q^T and dP^T = V dY^T  (tcgen05, A and B from shared memory),
//   P^T  = exp(scale S^T - LSE) on the band, dS^T = P^T (dP^T - D)
//          (eight warps, written to TMEM as packed bf16),
//   dV  += P^T dY and dK += dS^T Q  (tcgen05, A from TMEM).
// TMEM (512 columns): S^T [0,128), dP^T [128,256), dV [256,320), dK [320,384),
// P^T [384,448), dS^T [448,512).  Q, dY and the tile's LSE and D come in two
// slots, so the next tile's loads overlap this one's work.
//
// Roles (288 threads): warps 0-7 the elementwise part (warp w: key rows
// 32 (w % 4) .. +31, its TMEM lane quarter; queries 64 (w / 4) .. +63 of each
// tile); warp 8 loads by TMA, issues the MMAs and owns the TMEM allocation.
// Every wait is bounded; one that runs out sets a status bit and the CTA
// winds down without writing.
#include <math.h>

#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

constexpr int kBT = 128;  // keys per CTA, queries per tile
constexpr float kLog2e = 1.4426950408889634f;

enum : unsigned int {
    kStBwdLoad = kStatusTcBackward << 0,
    kStBwdMma = kStatusTcBackward << 1,
    kStBwdElem = kStatusTcBackward << 2,
};

struct DkdvCfg {
    static constexpr uint32_t TILE = kBT * 64 * 2;          // 128 rows x 64 bf16, 128-byte swizzle
    static constexpr uint32_t OFF_K = 0, OFF_V = TILE;
    static constexpr uint32_t OFF_SLOT = 2 * TILE;
    static constexpr uint32_t SLOT = 2 * TILE + 2 * kBT * 4;  // Q, dY, LSE, D
    static constexpr uint32_t S_Q = 0, S_DY = TILE, S_LSE = 2 * TILE, S_D = 2 * TILE + kBT * 4;
    static constexpr uint32_t OFF_BARS = OFF_SLOT + 2 * SLOT;
    static_assert(SLOT % 1024 == 0, "slots keep the 1024-byte alignment of the swizzled tiles");
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 320, COL_P = 384, COL_DS = 448;
    static constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, false, false);  // K-major A and B
    static constexpr uint32_t ID_G = idesc_bf16_f32(128, 64, false, true);    // A from TMEM, B MN-major
};

struct DkdvBars {
    uint64_t kv_full, q_full[2], q_empty[2];
    uint64_t s_full;   // S^T and dP^T of the tile are in TMEM
    uint64_t pd_full;  // the eight warps have read S^T, dP^T and written P^T, dS^T
    uint64_t pd_free;  // dV and dK of the tile have completed (P^T, dS^T may be overwritten)
    uint64_t o_done, drain;
    uint32_t tbase;
};

__global__ void __launch_bounds__(288, 1)
tcb_window_dkdv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                          const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdy,
                          const float *__restrict__ lse_g, const float *__restrict__ D_g, int lstride, int Tn,
                          int W, float scale, float *__restrict__ dKacc, float *__restrict__ dVacc,
                          unsigned int *__restrict__ status) {
    using C = DkdvCfg;
    extern __shared__ __align__(1024) unsigned char sm[];
    DkdvBars &B = *reinterpret_cast<DkdvBars *>(sm + C::OFF_BARS);
    if ((smem_u32(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStBwdLoad);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kb = blockIdx.x, bh = blockIdx.y, k0 = kb * kBT;
    const int t_hi = min(Tn - 1, k0 + kBT - 1 + W - 1);
    const int nq = t_hi / kBT - kb + 1;  // query tiles kb .. t_hi / 128
    const uint32_t s0 = smem_u32(sm);
    auto slot = [&](int i) { return C::OFF_SLOT + (uint32_t)(i & 1) * C::SLOT; };

    if (warp == 8) tmem_alloc(&B.tbase, 512);
    if (tid == 0) {
        mbar_init(&B.kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&B.q_full[s], 1);
            mbar_init(&B.q_empty[s], 1);
        }
        mbar_init(&B.s_full, 1);
        mbar_init(&B.pd_full, 8);
        mbar_init(&B.pd_free, 1);
        mbar_init(&B.o_done, 1);
        mbar_init(&B.drain, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;

    if (warp == 8) {
        // ------------------------------------------------ loads and MMAs (one thread)
        if (lane == 0) {
            bool ok = true;
            tma_prefetch_desc(&mq);
            tma_prefetch_desc(&mk);
            tma_prefetch_desc(&mv);
            tma_prefetch_desc(&mdy);
            mbar_expect_tx(&B.kv_full, 2 * C::TILE);
            tma_load_3d(sm + C::OFF_K, &mk, &B.kv_full, 0, k0, bh);
            tma_load_3d(sm + C::OFF_V, &mv, &B.kv_full, 0, k0, bh);
            // Query tile i into slot i & 1, once the MMAs of tile i - 2 have read it.
            // LSE and D rows are padded to lstride (a multiple of 128), so each
            // tile's 512 bytes are in bounds and 16-byte aligned.
            int issued = 0;  // query tiles whose loads have been issued
            auto load_q = [&](int i) -> bool {
                const int s = i & 1;
                if (i >= 2 && !mbar_wait(&B.q_empty[s], ((i >> 1) - 1) & 1)) return false;
                ++issued;
                const int t0 = (kb + i) * kBT;
                unsigned char *d = sm + slot(i);
                mbar_expect_tx(&B.q_full[s], 2 * C::TILE + 2 * kBT * 4);
                tma_load_3d(d + C::S_Q, &mq, &B.q_full[s], 0, t0, bh);
                tma_load_3d(d + C::S_DY, &mdy, &B.q_full[s], 0, t0, bh);
                bulk_load(d + C::S_LSE, lse_g + (size_t)bh * lstride + t0, kBT * 4, &B.q_full[s]);
                bulk_load(d + C::S_D, D_g + (size_t)bh * lstride + t0, kBT * 4, &B.q_full[s]);
                return true;
            };
            ok = load_q(0);
            if (ok && nq > 1) ok = load_q(1);
            if (ok) ok = mbar_wait(&B.kv_full, 0);
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t k_lo = sdesc_lo(s0 + C::OFF_K, 16), v_lo = sdesc_lo(s0 + C::OFF_V, 16);
            for (int i = 0; i <= nq && ok; ++i) {
                if (i >= 1) {
                    // dV += P^T dY, dK += dS^T Q for tile i - 1 (A from TMEM, B MN-major)
                    const int p = i - 1;
                    ok = mbar_wait(&B.pd_full, p & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t qb = sdesc_lo(s0 + slot(p) + C::S_Q, 16384);
                    const uint32_t yb = sdesc_lo(s0 + slot(p) + C::S_DY, 16384);
#pragma unroll
                    for (int k = 0; k < kBT / 16; ++k)
                        mma_ts_h(tm + C::COL_DV, tm + C::COL_P + 8 * k, yb + k * (2048 >> 4), HI, C::ID_G,
                                 (p > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                    for (int k = 0; k < kBT / 16; ++k)
                        mma_ts_h(tm + C::COL_DK, tm + C::COL_DS + 8 * k, qb + k * (2048 >> 4), HI, C::ID_G,
                                 (p > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&B.pd_free);
                    mma_commit(&B.q_empty[p & 1]);
                }
                if (i < nq) {
                    // S^T = K Q^T and dP^T = V dY^T of tile i (K-major, 64-wide contraction)
                    ok = mbar_wait(&B.q_full[i & 1], (i >> 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t q_lo = sdesc_lo(s0 + slot(i) + C::S_Q, 16);
                    const uint32_t y_lo = sdesc_lo(s0 + slot(i) + C::S_DY, 16);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss_h(tm + C::COL_S, k_lo + 2 * k, HI, q_lo + 2 * k, HI, C::ID_S, k > 0 ? 1u : 0u);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss_h(tm + C::COL_DP, v_lo + 2 * k, HI, y_lo + 2 * k, HI, C::ID_S, k > 0 ? 1u : 0u);
                    mma_commit(&B.s_full);
                }
                // tile i + 1 reuses the slot of tile i - 1, free once its dV and dK are done
                if (i >= 1 && i + 1 < nq) ok = load_q(i + 1);
            }
            if (ok) mma_commit(&B.o_done);
            if (!ok) atomicOr(status, kStBwdMma);
            // Every MMA issued here has completed before TMEM is freed; every
            // load issued has landed before the CTA's shared memory is released.
            mma_commit(&B.drain);
            mbar_wait(&B.drain, 0);
            mbar_wait(&B.kv_full, 0);
            for (int j = issued >= 2 ? issued - 2 : 0; j < issued; ++j) mbar_wait(&B.q_full[j & 1], (j >> 1) & 1);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ elementwise: P^T and dS^T
        const int q4 = warp & 3, half = warp >> 2;
        const int r = q4 * 32 + lane, s_key = k0 + r;
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        const float sl2 = scale * kLog2e;
        bool ok = true;
        for (int i = 0; i < nq && ok; ++i) {
            const int t0 = (kb + i) * kBT;
            ok = __all_sync(0xffffffffu, mbar_wait(&B.q_full[i & 1], (i >> 1) & 1));
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&B.s_full, i & 1));
            // P^T and dS^T of the previous tile are read by its dV and dK MMAs
            if (ok && i >= 1) ok = __all_sync(0xffffffffu, mbar_wait(&B.pd_free, (i - 1) & 1));
            if (!ok) break;
            tc_fence_after();
            const float *lse = reinterpret_cast<const float *>(sm + slot(i) + C::S_LSE);
            const float *Dt = reinterpret_cast<const float *>(sm + slot(i) + C::S_D);
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const int qb = half * 64 + 32 * g;  // queries qb .. qb + 31 of the tile
                float sv[32], dp[32];
                tmem_ld32(tm + lrow + C::COL_S + qb, sv);
                tmem_ld32(tm + lrow + C::COL_DP + qb, dp);
                tmem_wait_ld();
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int t = t0 + qb + e + u;
                        const bool band = s_key <= t && s_key > t - W && t < Tn && s_key < Tn;
                        // the statistics are read for every lane (the rows past T
                        // hold arbitrary values); the band selects what is used
                        const float L = lse[qb + e + u], Dv = Dt[qb + e + u];
                        const float p = ex2(band ? fmaf(sv[e + u], sl2, -L * kLog2e) : -INFINITY);
                        pv[u] = p;
                        dv[u] = band ? p * (dp[e + u] - Dv) : 0.f;
                    }
                    pk[e >> 1] = pack_bf16(pv[0], pv[1]);
                    dk[e >> 1] = pack_bf16(dv[0], dv[1]);
                }
                tmem_st16(tm + lrow + C::COL_P + qb / 2, pk);
                tmem_st16(tm + lrow + C::COL_DS + qb / 2, dk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.pd_full);
        }
        // ------------------------------------------------ epilogue: rows of dK and dV
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&B.o_done, 0));
        if (ok) {
            tc_fence_after();
            float a[32], b[32];
            tmem_ld32(tm + lrow + C::COL_DV + 32 * half, a);
            tmem_ld32(tm + lrow + C::COL_DK + 32 * half, b);
            tmem_wait_ld();
            if (s_key < Tn) {
                float4 *dv4 = reinterpret_cast<float4 *>(dVacc + ((size_t)bh * Tn + s_key) * 64 + 32 * half);
                float4 *dk4 = reinterpret_cast<float4 *>(dKacc + ((size_t)bh * Tn + s_key) * 64 + 32 * half);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    dv4[u] = make_float4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
                    dk4[u] = make_float4(scale * b[4 * u], scale * b[4 * u + 1], scale * b[4 * u + 2],
                                         scale * b[4 * u + 3]);
                }
            }
        }
        if (!ok && lane == 0) atomicOr(status, kStBwdElem);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) tmem_dealloc(tm, 512);
}

}  // namespace

bool tcb_window_dkdv_tcgen05_supported(int dtype, int dk, int dv) {
    return dtype == OPAM_BF16 && dk == 64 && dv == 64;
}

int tcb_window_dkdv_tcgen05(const void *q, const void *k, const void *v, const void *dy, int BH, int Tn, int W,
                            float scale, const float *lse, const float *D, int lstride, float *dK, float *dV,
                            unsigned int *status, cudaStream_t st) {
    if ((reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(D)) & 15u) {
        set_error("tc_layer_backward: workspace must be 16-byte aligned");
        return OPAM_ERR_INVALID_ARG;
    }
    CUtensorMap mq, mk, mv, mdy;
    int rc;
    if ((rc = make_tmap_bf16_3d(&mq, q, 64, Tn, BH, kBT))) return rc;
    if ((rc = make_tmap_bf16_3d(&mk, k, 64, Tn, BH, kBT))) return rc;
    if ((rc = make_tmap_bf16_3d(&mv, v, 64, Tn, BH, kBT))) return rc;
    if ((rc = make_tmap_bf16_3d(&mdy, dy, 64, Tn, BH, kBT))) return rc;
    const int smem = (int)(DkdvCfg::OFF_BARS + sizeof(DkdvBars));
    if ((rc = set_smem_limit((const void *)tcb_window_dkdv_tc_kernel, smem, "tcb_window_dkdv_tc smem attribute")))
        return rc;
    tcb_window_dkdv_tc_kernel<<<dim3(ceil_div(Tn, kBT), BH), 288, smem, st>>>(
        mq, mk, mv, mdy, lse, D, lstride, Tn, W, scale, dK, dV, status);
    return launched("tcb_window_dkdv_tc");
}

}  // namespace opam
