// DeltaNet delta rule on the tensor cores (bf16 inputs, fp32 state):
// tcgen05.mma with TMEM accumulators, operands staged by TMA.
//
// molayo1419.me, "DeltaNet-family linear attention variants", section
// "DeltaNet: write the prediction error instead of the value":
//     e_t = beta_t (v_t - S_{t-1} k_t),   S_t = S_{t-1} + e_t k_t^T,
// read o_t = S_t q_t after the write.
//
// Chunked closed form (derived from the recurrence; rows = the C = 64 tokens
// of a chunk, S0 the state at the chunk start, L = strict_lower(K K^T)):
//     T = (I + diag(beta) L)^{-1},   G = T diag(beta)
//     U = G V - (G K) S0^T                       (the chunk's e_t)
//     O = Q S0^T + (Q K^T masked to j <= i) U    (its o_t)
//     S_end = S0 + U^T K.
// Everything that depends only on the chunk's own inputs -- P = masked Q K^T,
// G^T, and W^T = -(G K)^T -- is computed for all chunks in parallel by
// delta_prep_kernel; delta_chain_kernel then walks each head's chunks in
// order with the state S^T (d_v x d_k, fp32) resident in TMEM, working in
// transposed form so that the MMA M dimension is d_v = 128:
//     U^T = V^T G^T + S0 W^T,   O^T = S0 Q^T + U^T P^T,   S += U^T K.
// The bf16 copy of S0 that feeds the first two products is refreshed from
// TMEM after every chunk; the fp32 state is never rounded.
#include <math.h>

#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

constexpr int kC = 64;  // tokens per chunk

// Bits recorded in the call's status word (the head of its workspace) when a
// bounded wait runs out.
enum : unsigned int {
    kStPrepWait = kStatusDelta << 0,
    kStChainProducer = kStatusDelta << 1,
    kStChainMma = kStatusDelta << 2,
    kStChainEpi = kStatusDelta << 3,
    kStChainAlign = kStatusDelta << 4,
};

// ------------------------------------------------------------------ prep
// One CTA (128 threads) per (chunk, head).
//  1. [Q; K] (128 x d_k, stacked in shared memory) times K^T on tcgen05:
//     TMEM lanes 0..63 hold Q K^T, lanes 64..127 hold K K^T.
//  2. Lanes 0..63 write P = (Q K^T masked to j <= i) as bf16; lanes 64..127
//     write diag(beta) strict_lower(K K^T) to shared memory.
//  3. Threads 0..63 each solve one column of T = (I + diag(beta) L)^{-1} by
//     forward substitution in fp32 registers; column j of G = T diag(beta),
//     i.e. row j of G^T, goes to shared memory (bf16, 128-byte swizzle) and
//     to global memory.
//  4. W^T = -(K^T G^T) on tcgen05 (A = K^T read MN-major from the K rows;
//     for d_k = 64 both 64-wide M blocks alias the same rows; B = G^T read
//     MN-major); row a of W^T (a < d_k) goes to global memory as bf16.
template <int DK>
struct PrepCfg {
    static constexpr uint32_t QK_BYTES = (DK / 64) * 16384;  // [Q;K], 128 rows per 64-column block
    static constexpr uint32_t OFF_G = 0;                    // G^T (64 rows x 128 B) over the Q rows of
                                                            // block 0, free after the first MMA
    static constexpr uint32_t OFF_L = QK_BYTES;             // Lb fp32 [64][64]
    static constexpr uint32_t SMEM = OFF_L + 64 * 64 * 4 + 1024;
};

// Column j of T = (I + Lb)^{-1} (Lb strictly lower) by forward substitution:
// T[i][j] = -sum_{k<i} Lb[i][k] T[k][j], T[j][j] = 1.  Every column handled
// by the calling warp is >= K0, so T[k][j] = 0 for k < K0 and those terms
// are skipped.
template <int K0>
__device__ __forceinline__ void forward_column(const float *__restrict__ Lb, int j, float (&t)[kC]) {
#pragma unroll
    for (int i = 0; i < kC; ++i) t[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int i = K0 + 1; i < kC; ++i) {
        const float4 *row = reinterpret_cast<const float4 *>(Lb + i * kC);
        float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
        for (int k4 = K0; k4 < i; k4 += 4) {
            const float4 l = row[k4 >> 2];
            // Lb[i][k] = 0 for k >= i, so whole float4 groups may be used.
            a = fma2(make_float2(l.x, l.y), make_float2(t[k4], t[k4 + 1]), a);
            if (k4 + 2 < i) b = fma2(make_float2(l.z, l.w), make_float2(t[k4 + 2], t[k4 + 3]), b);
        }
        const float acc = (a.x + a.y) + (b.x + b.y);
        t[i] = (i == j) ? 1.f : -acc;
    }
}

template <int DK>
__global__ void __launch_bounds__(128)
delta_prep_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const float *__restrict__ beta, int T, int nch, __nv_bfloat16 *__restrict__ Pg,
                  __nv_bfloat16 *__restrict__ Gg, __nv_bfloat16 *__restrict__ Wg,
                  unsigned int *__restrict__ status) {
    using C = PrepCfg<DK>;
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bars[3];
    __shared__ uint32_t tbase;
    __shared__ float bs[kC];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int t0 = c * kC, n = min(kC, T - t0);
    const uint32_t s0 = smem_u32(sm);
    float *Lb = reinterpret_cast<float *>(sm + C::OFF_L);
    if (warp == 0) tmem_alloc(&tbase, 128);
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        mbar_fence_init();
    }
    if (tid < kC) bs[tid] = tid < n ? beta[(size_t)bh * T + t0 + tid] : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    if (tid == 0) {
        mbar_expect_tx(&bars[0], 2 * (DK / 64) * 8192);
#pragma unroll
        for (int b = 0; b < DK / 64; ++b) {
            tma_load_3d(sm + b * 16384, &mq, &bars[0], 64 * b, t0, bh);
            tma_load_3d(sm + b * 16384 + 8192, &mk, &bars[0], 64 * b, t0, bh);
        }
    }
    bool ok = mbar_wait(&bars[0], 0);
    if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
        for (int k = 0; k < DK / 16; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_ss(tm, sdesc_sw128(s0 + off, 16, 1024), sdesc_sw128(s0 + off + 8192, 16, 1024), id,
                   k > 0 ? 1u : 0u);
        }
        mma_commit(&bars[1]);
    }
    ok = __syncthreads_and(ok);
    if (ok) ok = mbar_wait(&bars[1], 0);
    __syncwarp();
    tc_fence_after();
    const uint32_t lrow = (uint32_t)(warp * 32) << 16;
    if (ok) {
        float v[64];
        {
            float a[32];
            tmem_ld32(tm + lrow, a);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = a[i];
            tmem_ld32(tm + lrow + 32, a);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 + i] = a[i];
        }
        tmem_wait_ld();
        if (tid < kC) {  // P row i (only rows of this chunk are ever read)
            const int i = tid;
            uint4 *dst = reinterpret_cast<uint4 *>(Pg + (((size_t)bh * nch + c) * kC + i) * kC);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 8 * u + 2 * e;
                    w[e] = pack_bf16(j <= i ? v[j] : 0.f, j + 1 <= i ? v[j + 1] : 0.f);
                }
                dst[u] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {  // beta_i * strict_lower(K K^T) row i
            const int i = tid - kC;
            const float bi = bs[i];
            float4 *lrow4 = reinterpret_cast<float4 *>(Lb + i * kC);
#pragma unroll
            for (int j = 0; j < kC; j += 4)
                lrow4[j >> 2] = make_float4(j < i ? bi * v[j] : 0.f, j + 1 < i ? bi * v[j + 1] : 0.f,
                                            j + 2 < i ? bi * v[j + 2] : 0.f, j + 3 < i ? bi * v[j + 3] : 0.f);
        }
    }
    ok = __syncthreads_and(ok);
    // Column j of T (threads 0..63), then G[:, j] = T[:, j] beta_j.
    if (ok && tid < kC) {
        const int j = tid;
        float t[kC];
        if (warp == 0)
            forward_column<0>(Lb, j, t);
        else
            forward_column<32>(Lb, j, t);
        const float bj = bs[j];
        // Row j of G^T (= column j of G) into the swizzled tile and to global memory.
        uint4 *gdst = reinterpret_cast<uint4 *>(Gg + (((size_t)bh * nch + c) * kC + j) * kC);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const uint32_t w0 = pack_bf16(t[8 * ch] * bj, t[8 * ch + 1] * bj);
            const uint32_t w1 = pack_bf16(t[8 * ch + 2] * bj, t[8 * ch + 3] * bj);
            const uint32_t w2 = pack_bf16(t[8 * ch + 4] * bj, t[8 * ch + 5] * bj);
            const uint32_t w3 = pack_bf16(t[8 * ch + 6] * bj, t[8 * ch + 7] * bj);
            st_shared_v4(s0 + C::OFF_G + sw128_off(j, ch), w0, w1, w2, w3);
            gdst[ch] = make_uint4(w0, w1, w2, w3);
        }
        fence_async_smem();
    }
    ok = __syncthreads_and(ok);
    if (ok && tid == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16_f32(128, 64, true, true);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
            mma_ss(tm + 64, sdesc_sw128(s0 + 8192 + k * 2048, DK == 128 ? 16384 : 0, 1024),
                   sdesc_sw128(s0 + C::OFF_G + k * 2048, 8192, 1024), id, k > 0 ? 1u : 0u);
        mma_commit(&bars[2]);
    }
    ok = __syncthreads_and(ok);
    if (ok) ok = mbar_wait(&bars[2], 0);
    __syncwarp();
    tc_fence_after();
    if (ok && tid < DK) {
        float v[64];
        {
            float a[32];
            tmem_ld32(tm + lrow + 64, a);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = a[i];
            tmem_ld32(tm + lrow + 96, a);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 + i] = a[i];
        }
        tmem_wait_ld();
        uint4 *dst = reinterpret_cast<uint4 *>(Wg + (((size_t)bh * nch + c) * DK + tid) * kC);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            dst[u] = make_uint4(pack_bf16(-v[8 * u], -v[8 * u + 1]), pack_bf16(-v[8 * u + 2], -v[8 * u + 3]),
                                pack_bf16(-v[8 * u + 4], -v[8 * u + 5]), pack_bf16(-v[8 * u + 6], -v[8 * u + 7]));
    }
    if (!ok && tid == 0) atomicOr(status, kStPrepWait);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 128);
}

// ------------------------------------------------------------------ chain
// One CTA per head (d_v = 128 = the MMA M dimension).  192 threads: warp 0
// TMA, warp 1 MMA, warps 2..5 epilogue (thread = state row i, its TMEM lane).
// Per chunk: MMA1 U^T = V^T G^T + S0 W^T and O^T = S0 Q^T; epilogue 1 writes
// U^T (bf16) to shared memory; MMA2 O^T += U^T P^T and S += U^T K; epilogue 2
// refreshes the bf16 S0 and writes the chunk's outputs.
template <int DK>
struct ChainCfg {
    static constexpr uint32_t QB = (DK / 64) * 8192, KB = QB, VB = 2 * 8192, PB = 8192, GB = 8192,
                              WB = DK * 128;
    static constexpr uint32_t OQ = 0, OK_ = QB, OV = OK_ + KB, OP = OV + VB, OG = OP + PB, OW = OG + GB;
    static constexpr uint32_t STAGE = OW + WB;
    static constexpr int NS = 2;
    static constexpr uint32_t OFF_S0 = NS * STAGE;            // S0 bf16, 128 rows x DK
    static constexpr uint32_t OFF_U = OFF_S0 + (DK / 64) * 16384;  // U^T bf16, 128 rows x 64; y staging
    static constexpr uint32_t OFF_BARS = OFF_U + 16384;
    static constexpr uint32_t COL_S = 0, COL_U = DK, COL_O = DK + 64;
    static constexpr uint32_t TCOLS = DK + 128 <= 256 ? 256 : 512;
};

struct ChainBars {
    uint64_t full[2], empty[2];
    uint64_t s0_ready, u_full, ut_ready, o_full, drain;
};

template <int DK>
__global__ void __launch_bounds__(192, 1)
delta_chain_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mp,
                   const __grid_constant__ CUtensorMap mg, const __grid_constant__ CUtensorMap mw, int T,
                   int nch, const float *S0, float *S_out, __nv_bfloat16 *__restrict__ y,
                   unsigned int *__restrict__ status) {
    constexpr int DV = 128;
    using C = ChainCfg<DK>;
    extern __shared__ __align__(1024) unsigned char sm[];
    ChainBars &B = *reinterpret_cast<ChainBars *>(sm + C::OFF_BARS);
    uint32_t &tbase = *reinterpret_cast<uint32_t *>(sm + C::OFF_BARS + sizeof(ChainBars));
    if ((smem_u32(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStChainAlign);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const uint32_t s0 = smem_u32(sm);
    const bool has_s0 = S0 != nullptr;
    if (warp == 1) tmem_alloc(&tbase, C::TCOLS);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&B.full[s], 1);
            mbar_init(&B.empty[s], 1);
        }
        mbar_init(&B.s0_ready, 4);
        mbar_init(&B.u_full, 1);
        mbar_init(&B.ut_ready, 4);
        mbar_init(&B.o_full, 1);
        mbar_init(&B.drain, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            for (int c = 0; c < nch && ok; ++c) {
                const int s = c & 1;
                if (c >= 2) ok = mbar_wait(&B.empty[s], ((c >> 1) - 1) & 1);
                if (!ok) break;
                unsigned char *st = sm + s * C::STAGE;
                const int t0 = c * kC, u = bh * nch + c;
                mbar_expect_tx(&B.full[s], C::STAGE);
#pragma unroll
                for (int b = 0; b < DK / 64; ++b) {
                    tma_load_3d(st + C::OQ + b * 8192, &mq, &B.full[s], 64 * b, t0, bh);
                    tma_load_3d(st + C::OK_ + b * 8192, &mk, &B.full[s], 64 * b, t0, bh);
                }
#pragma unroll
                for (int b = 0; b < 2; ++b) tma_load_3d(st + C::OV + b * 8192, &mv, &B.full[s], 64 * b, t0, bh);
                tma_load_3d(st + C::OP, &mp, &B.full[s], 0, 0, u);
                tma_load_3d(st + C::OG, &mg, &B.full[s], 0, 0, u);
                tma_load_3d(st + C::OW, &mw, &B.full[s], 0, 0, u);
                ++issued;
            }
            if (!ok) atomicOr(status, kStChainProducer);
            bool dok = true;
            for (int c = max(0, issued - 2); c < issued && dok; ++c) dok = mbar_wait(&B.full[c & 1], (c >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            const uint32_t sS0 = s0 + C::OFF_S0, sU = s0 + C::OFF_U;
            constexpr uint32_t ID_U = idesc_bf16_f32(128, 64, true, true);    // V^T G^T
            constexpr uint32_t ID_W = idesc_bf16_f32(128, 64, false, true);   // S0 W^T
            constexpr uint32_t ID_Q = idesc_bf16_f32(128, 64, false, false);  // S0 Q^T, U^T P^T
            constexpr uint32_t ID_K = idesc_bf16_f32(128, DK, false, true);   // U^T K
            // Descriptors as a fixed upper half plus a lower half (address >> 4 |
            // leading offset): each k step is one 32-bit add in the issue loop.
            constexpr uint32_t HI = sdesc_hi(1024);
            auto kmaj = [](int k) { return (uint32_t)((k >> 2) * (16384 >> 4) + (k & 3) * 2); };  // K-major, 64-col blocks of 16 KB
            const uint32_t s0k = sdesc_lo(sS0, 16), uk = sdesc_lo(sU, 16);
            for (int c = 0; c < nch && ok; ++c) {
                const int s = c & 1;
                const uint32_t st = s0 + s * C::STAGE;
                ok = mbar_wait(&B.full[s], (c >> 1) & 1);
                if (ok) ok = mbar_wait(&B.s0_ready, c & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t v_lo = sdesc_lo(st + C::OV, 8192), g_lo = sdesc_lo(st + C::OG, 8192);
                const uint32_t w_lo = sdesc_lo(st + C::OW, 16384), q_lo = sdesc_lo(st + C::OQ, 16);
                const uint32_t p_lo = sdesc_lo(st + C::OP, 16), k_lo = sdesc_lo(st + C::OK_, 8192);
                // U^T = V^T G^T (K = 64 tokens) + S0 W^T (K = d_k)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_h(tm + C::COL_U, v_lo + k * (2048 >> 4), HI, g_lo + k * (2048 >> 4), HI, ID_U,
                             k > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < DK / 16; ++k)
                    mma_ss_h(tm + C::COL_U, s0k + kmaj(k), HI, w_lo + k * (2048 >> 4), HI, ID_W, 1u);
                mma_commit(&B.u_full);
                // O^T = S0 Q^T (the Q tile's 64-column blocks are 8 KB apart)
#pragma unroll
                for (int k = 0; k < DK / 16; ++k)
                    mma_ss_h(tm + C::COL_O, s0k + kmaj(k), HI,
                             q_lo + (uint32_t)((k >> 2) * (8192 >> 4) + (k & 3) * 2), HI, ID_Q, k > 0 ? 1u : 0u);
                ok = mbar_wait(&B.ut_ready, c & 1);
                if (!ok) break;
                tc_fence_after();
                // O^T += U^T P^T ; S += U^T K
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_h(tm + C::COL_O, uk + 2 * k, HI, p_lo + 2 * k, HI, ID_Q, 1u);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_h(tm + C::COL_S, uk + 2 * k, HI, k_lo + k * (2048 >> 4), HI, ID_K,
                             (c > 0 || has_s0 || k > 0) ? 1u : 0u);
                mma_commit(&B.o_full);
                mma_commit(&B.empty[s]);
            }
            if (!ok) atomicOr(status, kStChainMma);
            mma_commit(&B.drain);
            mbar_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue: state row i
        const int q4 = warp & 3;
        const int i = q4 * 32 + lane;  // d_v index = TMEM lane
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        bool ok = true;
        // bf16 copy of a state row into the K-major S0 tile (row i).
        auto put_s0 = [&](const float *srow) {
#pragma unroll
            for (int ch = 0; ch < DK / 8; ++ch) {
                const uint32_t a = s0 + C::OFF_S0 + (ch >> 3) * 16384 + sw128_off(i, ch & 7);
                st_shared_v4(a, pack_bf16(srow[8 * ch], srow[8 * ch + 1]), pack_bf16(srow[8 * ch + 2], srow[8 * ch + 3]),
                             pack_bf16(srow[8 * ch + 4], srow[8 * ch + 5]), pack_bf16(srow[8 * ch + 6], srow[8 * ch + 7]));
            }
        };
        {   // initial state: S0 (key-major [d_k][d_v]) or zero
            float srow[DK];
#pragma unroll
            for (int j = 0; j < DK; ++j) srow[j] = has_s0 ? S0[((size_t)bh * DK + j) * DV + i] : 0.f;
            if (has_s0) {
#pragma unroll
                for (int c0 = 0; c0 < DK; c0 += 32) {
                    float v[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = srow[c0 + e];
                    tmem_st32(tm + lrow + C::COL_S + c0, v);
                }
                tmem_wait_st();
            }
            put_s0(srow);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.s0_ready);
        }
        for (int c = 0; c < nch && ok; ++c) {
            const int t0 = c * kC, n = min(kC, T - t0);
            // ---- epilogue 1: U^T row i -> bf16 K-major tile
            ok = __all_sync(0xffffffffu, mbar_wait(&B.u_full, c & 1));
            if (!ok) break;
            tc_fence_after();
            {
                float u0[32], u1[32];
                tmem_ld32(tm + lrow + C::COL_U, u0);
                tmem_ld32(tm + lrow + C::COL_U + 32, u1);
                tmem_wait_ld();
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const float *p = ch < 4 ? &u0[8 * ch] : &u1[8 * (ch - 4)];
                    st_shared_v4(s0 + C::OFF_U + sw128_off(i, ch), pack_bf16(p[0], p[1]), pack_bf16(p[2], p[3]),
                                 pack_bf16(p[4], p[5]), pack_bf16(p[6], p[7]));
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.ut_ready);
            // ---- epilogue 2: new S (bf16 copy), outputs of the chunk
            ok = __all_sync(0xffffffffu, mbar_wait(&B.o_full, c & 1));
            if (!ok) break;
            tc_fence_after();
            {
                float srow[DK];
#pragma unroll
                for (int c0 = 0; c0 < DK; c0 += 32) {
                    float v[32];
                    tmem_ld32(tm + lrow + C::COL_S + c0, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) srow[c0 + e] = v[e];
                }
                tmem_wait_ld();
                if (c + 1 < nch) {
                    put_s0(srow);
                    fence_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&B.s0_ready);
                } else if (S_out) {
#pragma unroll
                    for (int j = 0; j < DK; ++j) S_out[((size_t)bh * DK + j) * DV + i] = srow[j];
                }
            }
            {
                // O^T row i -> y[t0 + t][i], transposed through this warp's 32
                // columns of the U tile (free once MMA2 has completed).
                float o0[32], o1[32];
                tmem_ld32(tm + lrow + C::COL_O, o0);
                tmem_ld32(tm + lrow + C::COL_O + 32, o1);
                tmem_wait_ld();
                __nv_bfloat16 *ys = reinterpret_cast<__nv_bfloat16 *>(sm + C::OFF_U);  // [64][128]
#pragma unroll
                for (int t = 0; t < kC; ++t) ys[t * DV + i] = __float2bfloat16_rn(t < 32 ? o0[t] : o1[t - 32]);
                __syncwarp();
                __nv_bfloat16 *yb = y + ((size_t)bh * T + t0) * DV + q4 * 32;
#pragma unroll
                for (int e = lane; e < kC * 4; e += 32) {  // 64 rows x four 16-byte pieces
                    const int t = e >> 2, ch = e & 3;
                    if (t < n)
                        reinterpret_cast<uint4 *>(yb + (size_t)t * DV)[ch] =
                            reinterpret_cast<const uint4 *>(ys + t * DV + q4 * 32)[ch];
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) atomicOr(status, kStChainEpi);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tm, C::TCOLS);
}

struct Ws {
    __nv_bfloat16 *P, *G, *W;
};

Ws carve(void *ws, int BH, int nch, int dk) {
    char *p = (char *)ws;
    Ws w;
    w.P = (__nv_bfloat16 *)p;
    p += align_up(2 * (size_t)BH * nch * kC * kC, 1024);
    w.G = (__nv_bfloat16 *)p;
    p += align_up(2 * (size_t)BH * nch * kC * kC, 1024);
    w.W = (__nv_bfloat16 *)p;
    (void)dk;
    return w;
}

template <int DK>
int run(const void *q, const void *k, const void *v, const float *beta, int BH, int T,
        const float *S0, float *S_out, void *y, void *ws, unsigned int *status, cudaStream_t st) {
    const int nch = ceil_div(T, kC);
    const Ws w = carve(ws, BH, nch, DK);
    CUtensorMap mq, mk, mv, mp, mg, mw;
    int rc;
    if ((rc = make_tmap_bf16_3d(&mq, q, DK, T, BH, kC))) return rc;
    if ((rc = make_tmap_bf16_3d(&mk, k, DK, T, BH, kC))) return rc;
    if ((rc = make_tmap_bf16_3d(&mv, v, 128, T, BH, kC))) return rc;
    if ((rc = make_tmap_bf16_3d(&mp, w.P, kC, kC, (uint64_t)BH * nch, kC))) return rc;
    if ((rc = make_tmap_bf16_3d(&mg, w.G, kC, kC, (uint64_t)BH * nch, kC))) return rc;
    if ((rc = make_tmap_bf16_3d(&mw, w.W, kC, DK, (uint64_t)BH * nch, DK))) return rc;
    {
        auto kern = delta_prep_kernel<DK>;
        const int smem = (int)PrepCfg<DK>::SMEM;
        if (int rc_ = set_smem_limit((const void *)kern, smem, "delta_prep smem attribute")) return rc_;
        prof_begin(st);  // the profiling bracket spans both kernels of the pass
        kern<<<dim3(nch, BH), 128, smem, st>>>(mq, mk, beta, T, nch, w.P, w.G, w.W, status);
        if ((rc = launched("delta_prep"))) return rc;
    }
    {
        using Cfg = ChainCfg<DK>;
        auto kern = delta_chain_kernel<DK>;
        const int smem = (int)(Cfg::OFF_BARS + sizeof(ChainBars) + 16);
        if (int rc_ = set_smem_limit((const void *)kern, smem, "delta_chain smem attribute")) return rc_;
        kern<<<BH, 192, smem, st>>>(mq, mk, mv, mp, mg, mw, T, nch, S0, S_out, (__nv_bfloat16 *)y, status);
        rc = launched("delta_chain");
        prof_end(st);
        return rc;
    }
}

}  // namespace

bool delta_tcgen05_supported(int dtype, int dk, int dv, int chunk) {
    return dtype == OPAM_BF16 && (dk == 64 || dk == 128) && dv == 128 && chunk == kC;
}

size_t delta_tcgen05_workspace(int BH, int T, int dk) {
    const size_t nch = (size_t)ceil_div(T, kC);
    return 2 * align_up(2 * (size_t)BH * nch * kC * kC, 1024) + align_up(2 * (size_t)BH * nch * dk * kC, 1024);
}

int delta_tcgen05(const void *q, const void *k, const void *v, const float *beta, int B, int H, int T,
                  int dk, const float *S0, float *S_out, void *y, void *ws, unsigned int *status,
                  cudaStream_t s) {
    if (dk == 64) return run<64>(q, k, v, beta, B * H, T, S0, S_out, y, ws, status, s);
    if (dk == 128) return run<128>(q, k, v, beta, B * H, T, S0, S_out, y, ws, status, s);
    set_error("tensor-core delta rule: d_k=%d unsupported", dk);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace opam
