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

// ------------------------------------------------------------------ window dQ, LSE and D
// One CTA per (128 queries, head) walks the key tiles of its window twice.
// Pass 1 is the window softmax of the forward, with the two 64-key halves of
// each tile keeping their own maxima, sums and accumulators O0 / O1: it gives
// LSE_t and D_t = <dy_t, y_loc,t> (written for the dK/dV kernel).  Pass 2
// recomputes S = Q K^T and dP = dY V^T, forms dS = P (dP - D) as packed bf16
// in TMEM and accumulates dQ += dS K with dS as the A operand.
// TMEM: S [0,128), O0 [128,192), O1 [192,256), P [256,320), dP [320,448),
// dS [448,512); dQ takes the O0 columns once pass 1 has read them.
// 320 threads: warps 0-7 elementwise (rows 32 (w % 4) .., keys 64 (w / 4) ..
// of each tile), warp 8 MMA issue (owns TMEM), warp 9 TMA.
struct DqCfg {
    static constexpr uint32_t TILE = kBT * 64 * 2;
    static constexpr uint32_t OFF_Q = 0, OFF_DY = TILE, OFF_KV = 2 * TILE;
    static constexpr uint32_t KVSLOT = 2 * TILE;  // K then V
    static constexpr uint32_t OFF_BARS = OFF_KV + 2 * KVSLOT;
    static constexpr uint32_t COL_S = 0, COL_O0 = 128, COL_O1 = 192, COL_P = 256, COL_DP = 320, COL_DS = 448;
    static constexpr uint32_t COL_DQ = 128;
    static constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t ID_G = idesc_bf16_f32(128, 64, false, true);
};

struct DqBars {
    uint64_t q_full, kv_full[2], kv_empty[2];
    uint64_t s_full;                // S (pass 1) or S and dP (pass 2) of the tile are in TMEM
    uint64_t p_full[2], p_empty[2];  // pass 1, per key half: P written / its P V done
    uint64_t pd_full, pd_free;      // pass 2: dS written / its dQ product done
    uint64_t o1_done, o2_done, xe, xd, drain;
    uint32_t tbase;
    float xm[2][kBT], xl[2][kBT], xp[2][kBT];  // [key half][row]: maxima, sums, partial D
};

constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold of the running maximum

__global__ void __launch_bounds__(320, 1)
tcb_window_dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdy, int Tn,
                        int W, float scale, float *__restrict__ lse_g, float *__restrict__ D_g, int lstride,
                        float *__restrict__ dQacc, unsigned int *__restrict__ status) {
    using C = DqCfg;
    extern __shared__ __align__(1024) unsigned char sm[];
    DqBars &B = *reinterpret_cast<DqBars *>(sm + C::OFF_BARS);
    if ((smem_u32(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStBwdLoad);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qblk = blockIdx.x, bh = blockIdx.y, q0 = qblk * kBT;
    const int s_lo = max(0, q0 - W + 1), s_hi = min(Tn - 1, q0 + kBT - 1);
    const int kt0 = s_lo / kBT, nt = s_hi / kBT - kt0 + 1;  // key tiles of the window
    const uint32_t s0 = smem_u32(sm);
    // Tile j of the load stream: pass 1 for j < nt, pass 2 after; slot j & 1.
    auto kslot = [&](int j) { return C::OFF_KV + (uint32_t)(j & 1) * C::KVSLOT; };

    if (warp == 8) tmem_alloc(&B.tbase, 512);
    if (tid == 0) {
        mbar_init(&B.q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&B.kv_full[s], 1);
            mbar_init(&B.kv_empty[s], 1);
            mbar_init(&B.p_full[s], 4);
            mbar_init(&B.p_empty[s], 1);
        }
        mbar_init(&B.s_full, 1);
        mbar_init(&B.pd_full, 8);
        mbar_init(&B.pd_free, 1);
        mbar_init(&B.o1_done, 1);
        mbar_init(&B.o2_done, 1);
        mbar_init(&B.xe, 8);
        mbar_init(&B.xd, 8);
        mbar_init(&B.drain, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;

    if (warp == 9) {
        // ------------------------------------------------ TMA: Q, dY once, then K and V tiles twice
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            tma_prefetch_desc(&mq);
            tma_prefetch_desc(&mk);
            tma_prefetch_desc(&mv);
            tma_prefetch_desc(&mdy);
            mbar_expect_tx(&B.q_full, 2 * C::TILE);
            tma_load_3d(sm + C::OFF_Q, &mq, &B.q_full, 0, q0, bh);
            tma_load_3d(sm + C::OFF_DY, &mdy, &B.q_full, 0, q0, bh);
            for (int j = 0; j < 2 * nt && ok; ++j) {
                const int s = j & 1;
                if (j >= 2) ok = mbar_wait(&B.kv_empty[s], ((j >> 1) - 1) & 1);
                if (!ok) break;
                const int kt = (kt0 + (j < nt ? j : j - nt)) * kBT;
                mbar_expect_tx(&B.kv_full[s], 2 * C::TILE);
                tma_load_3d(sm + kslot(j), &mk, &B.kv_full[s], 0, kt, bh);
                tma_load_3d(sm + kslot(j) + C::TILE, &mv, &B.kv_full[s], 0, kt, bh);
                ++issued;
            }
            if (!ok) atomicOr(status, kStBwdLoad);
            // every load issued has landed before the CTA's shared memory is released
            mbar_wait(&B.q_full, 0);
            for (int j = issued >= 2 ? issued - 2 : 0; j < issued; ++j) mbar_wait(&B.kv_full[j & 1], (j >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == 8) {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            bool ok = mbar_wait(&B.q_full, 0);
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t q_lo = sdesc_lo(s0 + C::OFF_Q, 16), y_lo = sdesc_lo(s0 + C::OFF_DY, 16);
            // pass 1: S = Q K^T, then O_h += P_h V_h per key half
            for (int n = 0; n < nt && ok; ++n) {
                ok = mbar_wait(&B.kv_full[n & 1], (n >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_lo = sdesc_lo(s0 + kslot(n), 16);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_h(tm + C::COL_S, q_lo + 2 * k, HI, k_lo + 2 * k, HI, C::ID_S, k > 0 ? 1u : 0u);
                mma_commit(&B.s_full);
                const uint32_t v_mn = sdesc_lo(s0 + kslot(n) + C::TILE, 16384);
                for (int h = 0; h < 2 && ok; ++h) {
                    ok = mbar_wait(&B.p_full[h], n & 1);
                    if (!ok) break;
                    tc_fence_after();
                    // V rows 64 h + 16 k .. (MN-major B)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ts_h(tm + (h ? C::COL_O1 : C::COL_O0), tm + C::COL_P + 32 * h + 8 * k,
                                 v_mn + 512 * h + 128 * k, HI, C::ID_G, (n > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&B.p_empty[h]);
                }
                if (ok) mma_commit(&B.kv_empty[n & 1]);
            }
            if (ok) mma_commit(&B.o1_done);
            // pass 2: S and dP of tile i, then dQ += dS K of tile i - 1
            for (int i = 0; i <= nt && ok; ++i) {
                if (i >= 1) {
                    const int p = i - 1, j = nt + p;
                    ok = mbar_wait(&B.pd_full, p & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kb = sdesc_lo(s0 + kslot(j), 16384);  // K rows as MN-major B
#pragma unroll
                    for (int k = 0; k < kBT / 16; ++k)
                        mma_ts_h(tm + C::COL_DQ, tm + C::COL_DS + 8 * k, kb + k * (2048 >> 4), HI, C::ID_G,
                                 (p > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&B.pd_free);
                    mma_commit(&B.kv_empty[j & 1]);
                }
                if (i < nt) {
                    const int j = nt + i;
                    ok = mbar_wait(&B.kv_full[j & 1], (j >> 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t k_lo = sdesc_lo(s0 + kslot(j), 16), v_lo = sdesc_lo(s0 + kslot(j) + C::TILE, 16);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss_h(tm + C::COL_S, q_lo + 2 * k, HI, k_lo + 2 * k, HI, C::ID_S, k > 0 ? 1u : 0u);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss_h(tm + C::COL_DP, y_lo + 2 * k, HI, v_lo + 2 * k, HI, C::ID_S, k > 0 ? 1u : 0u);
                    mma_commit(&B.s_full);
                }
            }
            if (ok) mma_commit(&B.o2_done);
            if (!ok) atomicOr(status, kStBwdMma);
            mma_commit(&B.drain);
            mbar_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ elementwise
        const int q4 = warp & 3, half = warp >> 2;
        const int r = q4 * 32 + lane, t = q0 + r, c0 = 64 * half;
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        const uint32_t col_o = half ? C::COL_O1 : C::COL_O0;
        const float sc = scale * kLog2e;
        float m = kNegBig, l = 0.f;
        bool ok = true;
        auto band = [&](int key) { return key <= t && key > t - W && t < Tn; };
        // ---- pass 1: this half's running maximum and sum, P into TMEM
        for (int n = 0; n < nt && ok; ++n) {
            const int kt = (kt0 + n) * kBT + c0;  // this half's first key
            ok = __all_sync(0xffffffffu, mbar_wait(&B.s_full, n & 1));
            if (!ok) break;
            tc_fence_after();
            float sv[64];
            {
                float v[32];
                tmem_ld32(tm + lrow + C::COL_S + c0, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) sv[e] = v[e];
                tmem_ld32(tm + lrow + C::COL_S + c0 + 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) sv[32 + e] = v[e];
            }
            tmem_wait_ld();
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                sv[e] = band(kt + e) ? sv[e] * sc : -INFINITY;
                mx = fmaxf(mx, sv[e]);
            }
            const bool grow = mx > m + kRescaleLog2;
            const float fO = grow ? ex2(m - mx) : 1.f;
            if (grow) {
                l *= fO;
                m = mx;
            }
            float sum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float a = ex2(sv[e] - m), b = ex2(sv[e + 1] - m);
                sum += a + b;
                pk[e >> 1] = pack_bf16(a, b);
            }
            l += sum;
            // P and O of this half may be written once its previous P V has completed
            ok = __all_sync(0xffffffffu, n == 0 || mbar_wait(&B.p_empty[half], (n - 1) & 1));
            if (!ok) break;
            tc_fence_after();
            if (__any_sync(0xffffffffu, grow) && n > 0) {
#pragma unroll 1
                for (int cc = 0; cc < 64; cc += 32) {
                    float v[32];
                    tmem_ld32(tm + lrow + col_o + cc, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= fO;
                    tmem_st32(tm + lrow + col_o + cc, v);
                }
            }
            tmem_st16(tm + lrow + C::COL_P + 32 * half, reinterpret_cast<const uint32_t(&)[16]>(pk[0]));
            tmem_st16(tm + lrow + C::COL_P + 32 * half + 16, reinterpret_cast<const uint32_t(&)[16]>(pk[16]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.p_full[half]);
        }
        // ---- LSE and D: merge the halves' statistics, y_loc = (O0 f0 + O1 f1) / L
        float lse2 = 0.f, Dv = 0.f;  // LSE in log2 units
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&B.o1_done, 0));
        if (ok) {
            B.xm[half][r] = m;
            B.xl[half][r] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.xe);
            ok = __all_sync(0xffffffffu, mbar_wait(&B.xe, 0));
        }
        if (ok) {
            tc_fence_after();
            const float mo = B.xm[half ^ 1][r], lo = B.xl[half ^ 1][r];
            const float M = fmaxf(m, mo);
            const float fm = ex2(m - M), fo = ex2(mo - M);
            const float L = l * fm + lo * fo;
            lse2 = L > 0.f ? M + __log2f(L) : 0.f;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const float w0 = (half ? fo : fm) * inv, w1 = (half ? fm : fo) * inv;
            float o0[32], o1[32];
            tmem_ld32(tm + lrow + C::COL_O0 + 32 * half, o0);
            tmem_ld32(tm + lrow + C::COL_O1 + 32 * half, o1);
            tmem_wait_ld();
            float dpart = 0.f;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {  // dY row r, columns 32 half + 8 ch .. (swizzled 16-byte chunks)
                uint32_t x[4];
                ld_shared_v4(s0 + C::OFF_DY + sw128_off(r, 4 * half + ch), x[0], x[1], x[2], x[3]);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 dy2 = unpack_bf16(x[u]);
                    const int e = 8 * ch + 2 * u;
                    dpart = fmaf(fmaf(o0[e], w0, o1[e] * w1), dy2.x, dpart);
                    dpart = fmaf(fmaf(o0[e + 1], w0, o1[e + 1] * w1), dy2.y, dpart);
                }
            }
            B.xp[half][r] = dpart;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.xd);
            ok = __all_sync(0xffffffffu, mbar_wait(&B.xd, 0));
            if (ok) {
                Dv = dpart + B.xp[half ^ 1][r];
                if (half == 0 && t < Tn) {
                    lse_g[(size_t)bh * lstride + t] = lse2 * 0.6931471805599453f;  // natural log
                    D_g[(size_t)bh * lstride + t] = Dv;
                }
            }
        }
        // ---- pass 2: dS = P (dP - D) into TMEM
        for (int n = 0; n < nt && ok; ++n) {
            const int kt = (kt0 + n) * kBT + c0;
            ok = __all_sync(0xffffffffu, mbar_wait(&B.s_full, (nt + n) & 1));
            if (ok && n >= 1) ok = __all_sync(0xffffffffu, mbar_wait(&B.pd_free, (n - 1) & 1));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                float sv[32], dp[32];
                tmem_ld32(tm + lrow + C::COL_S + c0 + 32 * g, sv);
                tmem_ld32(tm + lrow + C::COL_DP + c0 + 32 * g, dp);
                tmem_wait_ld();
                uint32_t dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float d2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const bool in = band(kt + 32 * g + e + u);
                        const float p = ex2(in ? fmaf(sv[e + u], sc, -lse2) : -INFINITY);
                        d2[u] = in ? p * (dp[e + u] - Dv) : 0.f;
                    }
                    dk[e >> 1] = pack_bf16(d2[0], d2[1]);
                }
                tmem_st16(tm + lrow + C::COL_DS + 32 * half + 16 * g, dk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.pd_full);
        }
        // ---- dQ rows
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&B.o2_done, 0));
        if (ok) {
            tc_fence_after();
            float a[32];
            tmem_ld32(tm + lrow + C::COL_DQ + 32 * half, a);
            tmem_wait_ld();
            if (t < Tn) {
                float4 *d4 = reinterpret_cast<float4 *>(dQacc + ((size_t)bh * Tn + t) * 64 + 32 * half);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    d4[u] = make_float4(scale * a[4 * u], scale * a[4 * u + 1], scale * a[4 * u + 2],
                                        scale * a[4 * u + 3]);
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

namespace opam {

int tcb_window_dq_tcgen05(const void *q, const void *k, const void *v, const void *dy, int BH, int Tn, int W,
                          float scale, float *lse, float *D, int lstride, float *dQ, unsigned int *status,
                          cudaStream_t st) {
    CUtensorMap mq, mk, mv, mdy;
    int rc;
    if ((rc = make_tmap_bf16_3d(&mq, q, 64, Tn, BH, kBT))) return rc;
    if ((rc = make_tmap_bf16_3d(&mk, k, 64, Tn, BH, kBT))) return rc;
    if ((rc = make_tmap_bf16_3d(&mv, v, 64, Tn, BH, kBT))) return rc;
    if ((rc = make_tmap_bf16_3d(&mdy, dy, 64, Tn, BH, kBT))) return rc;
    const int smem = (int)(DqCfg::OFF_BARS + sizeof(DqBars));
    if ((rc = set_smem_limit((const void *)tcb_window_dq_tc_kernel, smem, "tcb_window_dq_tc smem attribute")))
        return rc;
    tcb_window_dq_tc_kernel<<<dim3(ceil_div(Tn, kBT), BH), 320, smem, st>>>(mq, mk, mv, mdy, Tn, W, scale, lse, D,
                                                                            lstride, dQ, status);
    return launched("tcb_window_dq_tc");
}

}  // namespace opam
