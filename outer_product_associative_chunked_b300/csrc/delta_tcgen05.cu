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
// One CTA per head walks its chunks in order with the state S^T (d_v x d_k,
// fp32) resident in TMEM, working in transposed form so that the MMA M
// dimension is d_v = 128:
//     U^T = V^T G^T + S0 W^T,   O^T = S0 Q^T + U^T P^T,   S += U^T K,
// with P = (Q K^T masked) and W^T = -(G K)^T.  Everything that depends only
// on the chunk's own inputs -- P, G^T, W^T and the state-free part V^T G^T of
// U^T -- is produced inside the same CTA by a second warpgroup, one chunk
// ahead of the state recurrence, so none of it ever leaves the chip: HBM
// sees q, k, v and beta read once and y written once.
//
// Roles (512 threads):
//   warp 0       TMA of the q and k tiles (three stages)
//   warp 1       MMA issue for the state recurrence; owns the TMEM allocation
//   warps 2, 3   MMA issue for the chunk-local products of the even / odd
//                chunks, and TMA of the next v tile (one stage)
//   warps 4..7   state epilogue: thread = state row i (its TMEM lane)
//   warps 8..11  chunk-local epilogue and triangular solve, even chunks
//   warps 12..15 the same for the odd chunks
// The bf16 copy of S0 that feeds the products is refreshed from TMEM after
// every chunk; the fp32 state is never rounded.
#include <math.h>

#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

constexpr int kC = 64;  // tokens per chunk
// Every product whose rows are the value dimension runs with M = 128.  For
// d_v = 64 both 64-row halves of M read the same v columns (the MN-major
// operand's second block aliases the first), so TMEM lanes 64..127 carry an
// exact copy of U^T, O^T and the state; only lanes below d_v read or write
// global memory.

// Bits recorded in the call's status word (the head of its workspace) when a
// bounded wait runs out.
enum : unsigned int {
    kStPrepWait = kStatusDelta << 0,
    kStChainProducer = kStatusDelta << 1,
    kStChainMma = kStatusDelta << 2,
    kStChainEpi = kStatusDelta << 3,
    kStChainAlign = kStatusDelta << 4,
};

// Named barrier `bar` over one chunk-local warpgroup (128 threads).
__device__ __forceinline__ void prep_sync(int bar) { asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory"); }

// The fp32 64 x 64 tile of the solve keeps its rows of sixteen 16-byte
// chunks XOR-swizzled by the row index, so that a warp touching one chunk
// position in 32 different rows (thread = row) spreads over all banks.
__device__ __forceinline__ int lsw4(int i, int q) { return i * kC + (((q ^ (i & 15))) << 2); }  // chunk q of row i
__device__ __forceinline__ int lsw(int i, int j) { return lsw4(i, j >> 2) + (j & 3); }
__device__ __forceinline__ float4 ld4(const float *S, int i, int q) { return *reinterpret_cast<const float4 *>(S + lsw4(i, q)); }
__device__ __forceinline__ void st4(float *S, int i, int q, float4 v) { *reinterpret_cast<float4 *>(S + lsw4(i, q)) = v; }

// ---- warp-level products for the solve: mma.sync m16n8k8 with tf32
// operands (rounded to nearest) and fp32 accumulation.  Splitting each
// operand into a tf32 head and remainder (three products instead of one)
// left the layer's output error unchanged -- it is set by the bf16 operands
// of the state products -- and cost 10% of the forward, so one product it is.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// D (a 16 x 8 tile) += A[16 x K] B[K x 8]: fa(r, k) and fb(k, n) read the
// operands (tile-local indices).  Fragment layout of m16n8k8: with
// g = lane / 4 and t = lane % 4, A holds (g, t), (g + 8, t), (g, t + 4),
// (g + 8, t + 4); B holds (t, g), (t + 4, g); D holds (g, 2t), (g, 2t + 1),
// (g + 8, 2t), (g + 8, 2t + 1).
template <int K, class FA, class FB>
__device__ __forceinline__ void warp_tile_mma(float (&d)[4], int lane, FA fa, FB fb) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        const float av[4] = {fa(g, k0 + t), fa(g + 8, k0 + t), fa(g, k0 + t + 4), fa(g + 8, k0 + t + 4)};
        const float bv[2] = {fb(k0 + t, g), fb(k0 + t + 4, g)};
        uint32_t ah[4], bh[2];
#pragma unroll
        for (int e = 0; e < 4; ++e) asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(ah[e]) : "f"(av[e]));
#pragma unroll
        for (int e = 0; e < 2; ++e) asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(bh[e]) : "f"(bv[e]));
        mma_tf32(d, ah, bh);
    }
}

// The same for two adjacent 16 x 8 tiles (output columns n and 8 + n of fb)
// that share their A fragments.
template <int K, class FA, class FB>
__device__ __forceinline__ void warp_tile_mma2(float (&d0)[4], float (&d1)[4], int lane, FA fa, FB fb) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        const float av[4] = {fa(g, k0 + t), fa(g + 8, k0 + t), fa(g, k0 + t + 4), fa(g + 8, k0 + t + 4)};
        const float bv[4] = {fb(k0 + t, g), fb(k0 + t + 4, g), fb(k0 + t, 8 + g), fb(k0 + t + 4, 8 + g)};
        uint32_t ah[4], bh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(ah[e]) : "f"(av[e]));
            asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(bh[e]) : "f"(bv[e]));
        }
        const uint32_t bh0[2] = {bh[0], bh[1]}, bh1[2] = {bh[2], bh[3]};
        mma_tf32(d0, ah, bh0);
        mma_tf32(d1, ah, bh1);
    }
}

// T = (I + Lb)^{-1} for the strictly lower 64 x 64 Lb held in shared memory
// (fp32, swizzled rows), computed in place by the 128 chunk-local threads:
// on return the tile holds the strictly lower part of T (T is unit lower
// triangular).  Blocked inverse of a unit lower-triangular matrix: with
// 16 x 16 blocks,
//   1. the four diagonal blocks D_b = (I + L_bb)^{-1}, one column per thread
//      by forward substitution, T[r][j] = -sum_{k<r} L[r][k] T[k][j];
//   2. the blocks below them at distance one inside each 32 x 32 half,
//      T_10 = -D_1 (L_10 D_0) and T_32 = -D_3 (L_32 D_2);
//   3. the lower-left 32 x 32 block T_(1,0) = -T_(1,1) (L_(1,0) T_(0,0)).
// Entries on and above the diagonal of every stored block are zero (Lb is
// strictly lower), so each product runs over the full block width with the
// stored part of the unit-diagonal factor and the identity's share is the
// accumulator's initial value.  Steps 2 and 3 run on the warps' mma.sync
// units (one 16 x 8 output tile per warp and product in step 2, two in
// step 3).  X (fp32, 5 KB, padded rows) is scratch.
__device__ __forceinline__ void unit_lower_inverse(float *__restrict__ S, float *__restrict__ X, int tid, int bar) {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    auto at = [&](int i, int j) -> float & { return S[lsw(i, j)]; };
    // ---- 1. diagonal 16 x 16 blocks: thread (b, jj) = column jj of D_b
    {
        float tc[16];
        const int b = (tid >> 4) & 3, jj = tid & 15;
        if (tid < 64) {
#pragma unroll
            for (int r = 0; r < 16; ++r) tc[r] = (r == jj) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int k4 = 0; k4 < r; k4 += 4) {
                    const float4 l = ld4(S, 16 * b + r, 4 * b + (k4 >> 2));  // L[r][k] = 0 for k >= r
                    a0 = fmaf(l.x, tc[k4], a0);
                    a1 = fmaf(l.y, tc[k4 + 1], a1);
                    a0 = fmaf(l.z, tc[k4 + 2], a0);
                    a1 = fmaf(l.w, tc[k4 + 3], a1);
                }
                if (r > jj) tc[r] = -(a0 + a1);
            }
        }
        prep_sync(bar);
        if (tid < 64) {
#pragma unroll
            for (int r = 1; r < 16; ++r)
                if (r > jj) at(16 * b + r, 16 * b + jj) = tc[r];
        }
        prep_sync(bar);
    }
    // ---- 2. warp w: block (w / 2) (rows R0.., cols C0..), output columns 8 (w % 2)..
    {
        constexpr int XS = 24;  // padded row stride of the 16 x 16 scratch blocks
        const int blk = warp >> 1, n0 = (warp & 1) * 8;
        const int R0 = blk ? 48 : 16, C0 = blk ? 32 : 0;
        float *Xb = X + blk * 16 * XS;
        float d[4] = {at(R0 + g, C0 + n0 + 2 * t), at(R0 + g, C0 + n0 + 2 * t + 1), at(R0 + g + 8, C0 + n0 + 2 * t),
                      at(R0 + g + 8, C0 + n0 + 2 * t + 1)};  // L D_lo: the identity's share
        warp_tile_mma<16>(d, lane, [&](int r, int k) { return at(R0 + r, C0 + k); },
                          [&](int k, int n) { return at(C0 + k, C0 + n0 + n); });
        Xb[g * XS + n0 + 2 * t] = d[0];
        Xb[g * XS + n0 + 2 * t + 1] = d[1];
        Xb[(g + 8) * XS + n0 + 2 * t] = d[2];
        Xb[(g + 8) * XS + n0 + 2 * t + 1] = d[3];
        prep_sync(bar);
        float e[4] = {d[0], d[1], d[2], d[3]};  // D_hi X: the identity's share is X itself
        warp_tile_mma<16>(e, lane, [&](int r, int k) { return at(R0 + r, R0 + k); },
                          [&](int k, int n) { return Xb[k * XS + n0 + n]; });
        at(R0 + g, C0 + n0 + 2 * t) = -e[0];
        at(R0 + g, C0 + n0 + 2 * t + 1) = -e[1];
        at(R0 + g + 8, C0 + n0 + 2 * t) = -e[2];
        at(R0 + g + 8, C0 + n0 + 2 * t + 1) = -e[3];
        prep_sync(bar);
    }
    // ---- 3. warp w: rows 32 + 16 (w / 2).., output columns 16 (w % 2) + {0, 8}
    {
        constexpr int XS = 40;  // padded row stride of the 32 x 32 scratch
        const int m0 = (warp >> 1) * 16, n0 = (warp & 1) * 16;
        float d[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // L T_(0,0): the identity's share
            d[h][0] = at(32 + m0 + g, n0 + 8 * h + 2 * t);
            d[h][1] = at(32 + m0 + g, n0 + 8 * h + 2 * t + 1);
            d[h][2] = at(32 + m0 + g + 8, n0 + 8 * h + 2 * t);
            d[h][3] = at(32 + m0 + g + 8, n0 + 8 * h + 2 * t + 1);
        }
        warp_tile_mma2<32>(d[0], d[1], lane, [&](int r, int k) { return at(32 + m0 + r, k); },
                           [&](int k, int n) { return at(k, n0 + n); });
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nc = n0 + 8 * h;
            X[(m0 + g) * XS + nc + 2 * t] = d[h][0];
            X[(m0 + g) * XS + nc + 2 * t + 1] = d[h][1];
            X[(m0 + g + 8) * XS + nc + 2 * t] = d[h][2];
            X[(m0 + g + 8) * XS + nc + 2 * t + 1] = d[h][3];
        }
        prep_sync(bar);
        // T_(1,1) X: the identity's share is X itself (already in d)
        warp_tile_mma2<32>(d[0], d[1], lane, [&](int r, int k) { return at(32 + m0 + r, 32 + k); },
                           [&](int k, int n) { return X[k * XS + n0 + n]; });
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nc = n0 + 8 * h;
            at(32 + m0 + g, nc + 2 * t) = -d[h][0];
            at(32 + m0 + g, nc + 2 * t + 1) = -d[h][1];
            at(32 + m0 + g + 8, nc + 2 * t) = -d[h][2];
            at(32 + m0 + g + 8, nc + 2 * t + 1) = -d[h][3];
        }
        prep_sync(bar);
    }
}

// The same barrier, also returning whether `ok` holds in all 128 threads, so
// that the four warps leave their loop together.
__device__ __forceinline__ bool prep_all(bool ok, int bar) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(bar)
        : "memory");
    return r != 0;
}

// Shared-memory plan (bytes; every tile 1024-aligned, 128-byte swizzle).
// Buffers marked (x2) belong to the chunks of one parity: chunk c uses
// buffer c & 1, and so does the warpgroup that prepares it.
//   QK stage (x3)   per 64-column block b: q rows (8 KB) then k rows (8 KB),
//                   so that [Q; K] is one 128-row K-major operand
//   V               v rows, two 64-column blocks (16 KB)
//   P (x2)          masked Q K^T, row i = query token (8 KB)
//   W^T (x2)        row a = key dimension, 64 tokens (DK * 128 B); for
//                   DK = 128 the fp32 tile of the solve lives in the buffer
//                   of the chunk being prepared until W^T overwrites it
//   G^T (x2)        row j = column j of G (8 KB); also the solve's fp32
//                   scratch until G^T is written
//   S0              bf16 state, 128 rows x DK (K-major, 64-column blocks)
//   U               U^T bf16 (128 rows x 64 tokens); also the y staging tile
//   L (x2)          fp32 [64][64] tile of the solve (DK = 64 only)
template <int DK>
struct FusedCfg {
    static constexpr uint32_t QK = (DK / 64) * 16384;
    static constexpr uint32_t WB = DK * 128;
    static constexpr uint32_t OFF_QK = 0;
    static constexpr uint32_t OFF_V = 3 * QK;
    static constexpr uint32_t OFF_P = OFF_V + 16384;
    static constexpr uint32_t OFF_W = OFF_P + 2 * 8192;
    static constexpr uint32_t OFF_G = OFF_W + 2 * WB;
    static constexpr uint32_t OFF_S0 = OFF_G + 2 * 8192;
    static constexpr uint32_t OFF_U = OFF_S0 + (DK / 64) * 16384;
    static constexpr bool L_IN_W = WB >= 64 * 64 * 4;
    static constexpr uint32_t OFF_L = OFF_U + 16384;  // DK = 64 only
    static constexpr uint32_t OFF_BARS = OFF_L + (L_IN_W ? 0 : 2 * 16384);
    // TMEM columns: state, U^T, O^T and the chunk-local products, each of the
    // last three double-buffered by chunk parity.
    static constexpr uint32_t COL_S = 0, COL_U = DK, COL_O = DK + 128, COL_P = DK + 256;
    static constexpr uint32_t TCOLS = 512;
    static_assert(COL_P + 128 <= TCOLS, "TMEM columns");
};

struct FusedBars {
    uint64_t qk_full[3], qk_empty[3];
    uint64_t v_full[2], v_empty;  // v_full per parity of the chunk whose tile it announces
    uint64_t a_full[2], g_ready[2], w_full[2], ptm_free[2];  // per warpgroup of the chunk-local pass
    uint64_t pw_ready[2], pw_empty[2];                       // per parity of the chunk
    uint64_t s0_ready, u_full, ut_ready, o_full;
    uint64_t drain[3];
    uint32_t tbase;
};

template <int DK, int DV>
__global__ void __launch_bounds__(512, 1)
delta_fused_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const float *__restrict__ beta, int T, int nch,
                   const float *S0, float *S_out, __nv_bfloat16 *__restrict__ y,
                   unsigned int *__restrict__ status) {
    using C = FusedCfg<DK>;
    extern __shared__ __align__(1024) unsigned char sm[];
    FusedBars &B = *reinterpret_cast<FusedBars *>(sm + C::OFF_BARS);
    if ((smem_u32(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStChainAlign);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const uint32_t s0 = smem_u32(sm);
    const bool has_s0 = S0 != nullptr;
    if (warp == 1) tmem_alloc(&B.tbase, C::TCOLS);
    if (tid == 0) {
        for (int s = 0; s < 3; ++s) {
            mbar_init(&B.qk_full[s], 1);
            mbar_init(&B.qk_empty[s], 1);
            mbar_init(&B.drain[s], 1);
        }
        mbar_init(&B.v_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&B.v_full[s], 1);
            mbar_init(&B.a_full[s], 1);
            mbar_init(&B.g_ready[s], 4);
            mbar_init(&B.w_full[s], 1);
            mbar_init(&B.ptm_free[s], 4);
            mbar_init(&B.pw_ready[s], 4);
            mbar_init(&B.pw_empty[s], 1);
        }
        mbar_init(&B.s0_ready, 4);
        mbar_init(&B.u_full, 1);
        mbar_init(&B.ut_ready, 4);
        mbar_init(&B.o_full, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;
    auto qk_base = [&](int c) { return (uint32_t)(C::OFF_QK + (c % 3) * C::QK); };
    auto load_v = [&](int c) {
        uint64_t *bar = &B.v_full[c & 1];
        mbar_expect_tx(bar, kC * DV * 2);
#pragma unroll
        for (int b = 0; b < DV / 64; ++b) tma_load_3d(sm + C::OFF_V + b * 8192, &mv, bar, 64 * b, c * kC, bh);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA: q and k tiles, v of chunk 0
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            if (nch > 0) load_v(0);
            for (int c = 0; c < nch && ok; ++c) {
                const int s = c % 3;
                if (c >= 3) ok = mbar_wait(&B.qk_empty[s], ((c / 3) - 1) & 1);
                if (!ok) break;
                unsigned char *st = sm + qk_base(c);
                mbar_expect_tx(&B.qk_full[s], C::QK);
#pragma unroll
                for (int b = 0; b < DK / 64; ++b) {
                    tma_load_3d(st + b * 16384, &mq, &B.qk_full[s], 64 * b, c * kC, bh);
                    tma_load_3d(st + b * 16384 + 8192, &mk, &B.qk_full[s], 64 * b, c * kC, bh);
                }
                ++issued;
            }
            if (!ok) atomicOr(status, kStChainProducer);
            // Let the loads still in flight land before the CTA exits.
            bool dok = true;
            for (int c = max(0, issued - 3); c < issued && dok; ++c) dok = mbar_wait(&B.qk_full[c % 3], (c / 3) & 1);
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------ MMA issue: chunk-local products of one parity
        // Warp 2 serves the even chunks, warp 3 the odd ones.  After the V^T G^T
        // product of chunk c has read the v tile, this thread loads v of
        // chunk c + 1 into it.
        if (lane == 0) {
            const int g = warp - 2;
            bool ok = true;
            constexpr uint32_t ID_A = idesc_bf16_f32(128, 64, false, false);  // [Q; K] K^T
            constexpr uint32_t ID_T = idesc_bf16_f32(128, 64, true, true);    // K^T G^T, V^T G^T
            // [Q; K] K^T of chunk c into the group's TMEM region: lanes 0..63
            // Q K^T, lanes 64..127 K K^T.  The region last held W^T of chunk c - 2.
            auto issue_a = [&](int c) -> bool {
                bool r = mbar_wait(&B.qk_full[c % 3], (c / 3) & 1);
                if (r && c >= 2) r = mbar_wait(&B.ptm_free[g], ((c >> 1) - 1) & 1);
                if (!r) return false;
                tc_fence_after();
                const uint32_t qk = s0 + qk_base(c);
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_ss(tm + C::COL_P + 64 * g, sdesc_sw128(qk + off, 16, 1024),
                           sdesc_sw128(qk + off + 8192, 16, 1024), ID_A, k > 0 ? 1u : 0u);
                }
                mma_commit(&B.a_full[g]);
                return true;
            };
            if (g < nch) ok = issue_a(g);
            for (int c = g; c < nch && ok; c += 2) {
                ok = mbar_wait(&B.g_ready[g], (c >> 1) & 1);
                if (ok) ok = mbar_wait(&B.v_full[g], (c >> 1) & 1);
                if (ok && c >= 2) ok = mbar_wait(&B.pw_empty[g], ((c >> 1) - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qk = s0 + qk_base(c), gt = s0 + C::OFF_G + g * 8192;
                // W^T = K^T G^T (negated in the epilogue).  A = K^T read
                // MN-major from the k rows; for d_k = 64 both 64-wide M blocks
                // alias the same rows and the upper half is ignored.
#pragma unroll
                for (int k = 0; k < kC / 16; ++k)
                    mma_ss(tm + C::COL_P + 64 * g, sdesc_sw128(qk + 8192 + k * 2048, DK == 128 ? 16384 : 0, 1024),
                           sdesc_sw128(gt + k * 2048, 8192, 1024), ID_T, k > 0 ? 1u : 0u);
                // V^T G^T: the state-free part of U^T, into the chunk's U buffer
#pragma unroll
                for (int k = 0; k < kC / 16; ++k)
                    mma_ss(tm + C::COL_U + 64 * g, sdesc_sw128(s0 + C::OFF_V + k * 2048, DV == 128 ? 8192 : 0, 1024),
                           sdesc_sw128(gt + k * 2048, 8192, 1024), ID_T, k > 0 ? 1u : 0u);
                mma_commit(&B.w_full[g]);
                mma_commit(&B.v_empty);
                ok = mbar_wait(&B.v_empty, c & 1);
                if (!ok) break;
                if (c + 1 < nch) load_v(c + 1);
                if (c + 2 < nch) ok = issue_a(c + 2);
            }
            if (!ok) atomicOr(status, kStPrepWait);
            mma_commit(&B.drain[1 + g]);
            mbar_wait(&B.drain[1 + g], 0);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue: state recurrence
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t ID_W = idesc_bf16_f32(128, 64, false, true);   // S0 W^T
            constexpr uint32_t ID_Q = idesc_bf16_f32(128, 64, false, false);  // S0 Q^T, U^T P^T
            constexpr uint32_t ID_K = idesc_bf16_f32(128, DK, false, true);   // U^T K
            // Descriptors as a fixed upper half plus a lower half (address >> 4 |
            // leading offset): each k step is one 32-bit add in the issue loop.
            constexpr uint32_t HI = sdesc_hi(1024);
            auto kmaj = [](int k) { return (uint32_t)((k >> 2) * (16384 >> 4) + (k & 3) * 2); };  // 64-col blocks 16 KB apart
            const uint32_t s0k = sdesc_lo(s0 + C::OFF_S0, 16), uk = sdesc_lo(s0 + C::OFF_U, 16);
            for (int c = 0; c < nch && ok; ++c) {
                const int pb = c & 1;
                ok = mbar_wait(&B.qk_full[c % 3], (c / 3) & 1);
                if (ok) ok = mbar_wait(&B.pw_ready[pb], (c >> 1) & 1);
                if (ok) ok = mbar_wait(&B.s0_ready, c & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qk = s0 + qk_base(c);
                const uint32_t w_lo = sdesc_lo(s0 + C::OFF_W + pb * C::WB, 8192);
                const uint32_t q_lo = sdesc_lo(qk, 16), k_lo = sdesc_lo(qk + 8192, 16384);
                const uint32_t p_lo = sdesc_lo(s0 + C::OFF_P + pb * 8192, 16);
                const uint32_t cu = C::COL_U + 64 * pb, co = C::COL_O + 64 * pb;
                // U^T += S0 W^T (K = d_k) on top of V^T G^T
#pragma unroll
                for (int k = 0; k < DK / 16; ++k)
                    mma_ss_h(tm + cu, s0k + kmaj(k), HI, w_lo + k * (2048 >> 4), HI, ID_W, 1u);
                mma_commit(&B.u_full);
                // O^T = S0 Q^T
#pragma unroll
                for (int k = 0; k < DK / 16; ++k)
                    mma_ss_h(tm + co, s0k + kmaj(k), HI, q_lo + kmaj(k), HI, ID_Q, k > 0 ? 1u : 0u);
                ok = mbar_wait(&B.ut_ready, c & 1);
                if (!ok) break;
                tc_fence_after();
                // O^T += U^T P^T ; S += U^T K
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_h(tm + co, uk + 2 * k, HI, p_lo + 2 * k, HI, ID_Q, 1u);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_h(tm + C::COL_S, uk + 2 * k, HI, k_lo + k * (2048 >> 4), HI, ID_K,
                             (c > 0 || has_s0 || k > 0) ? 1u : 0u);
                mma_commit(&B.o_full);
                mma_commit(&B.qk_empty[c % 3]);
                mma_commit(&B.pw_empty[pb]);
            }
            if (!ok) atomicOr(status, kStChainMma);
            mma_commit(&B.drain[0]);
            mbar_wait(&B.drain[0], 0);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------ state epilogue: row i
        const int q4 = warp & 3;
        const int i = q4 * 32 + lane;  // d_v index = TMEM lane
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        bool ok = true;
        // bf16 copy of 32 state columns c0..c0+31 of row i into the K-major S0 tile.
        auto put_s0 = [&](int c0, const float (&v)[32]) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int ch = c0 / 8 + e;
                st_shared_v4(s0 + C::OFF_S0 + (ch >> 3) * 16384 + sw128_off(i, ch & 7),
                             pack_bf16(v[8 * e], v[8 * e + 1]), pack_bf16(v[8 * e + 2], v[8 * e + 3]),
                             pack_bf16(v[8 * e + 4], v[8 * e + 5]), pack_bf16(v[8 * e + 6], v[8 * e + 7]));
            }
        };
        {   // initial state: S0 (key-major [d_k][d_v]) or zero
#pragma unroll 1
            for (int c0 = 0; c0 < DK; c0 += 32) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = has_s0 ? S0[((size_t)bh * DK + c0 + e) * DV + (i & (DV - 1))] : 0.f;
                if (has_s0) tmem_st32(tm + lrow + C::COL_S + c0, v);
                put_s0(c0, v);
            }
            if (has_s0) tmem_wait_st();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.s0_ready);
        }
        for (int c = 0; c < nch && ok; ++c) {
            const int t0 = c * kC, n = min(kC, T - t0), pb = c & 1;
            // ---- U^T row i -> bf16 K-major tile
            ok = __all_sync(0xffffffffu, mbar_wait(&B.u_full, c & 1));
            if (!ok) break;
            tc_fence_after();
            {
                float u0[32], u1[32];
                tmem_ld32(tm + lrow + C::COL_U + 64 * pb, u0);
                tmem_ld32(tm + lrow + C::COL_U + 64 * pb + 32, u1);
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
            // ---- new S (bf16 copy for the next chunk), outputs of this chunk
            ok = __all_sync(0xffffffffu, mbar_wait(&B.o_full, c & 1));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < DK; c0 += 64) {
                float v0[32], v1[32];
                tmem_ld32(tm + lrow + C::COL_S + c0, v0);
                tmem_ld32(tm + lrow + C::COL_S + c0 + 32, v1);
                tmem_wait_ld();
                if (c + 1 < nch) {
                    put_s0(c0, v0);
                    put_s0(c0 + 32, v1);
                } else if (S_out && i < DV) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        S_out[((size_t)bh * DK + c0 + e) * DV + i] = v0[e];
                        S_out[((size_t)bh * DK + c0 + 32 + e) * DV + i] = v1[e];
                    }
                }
            }
            if (c + 1 < nch) {
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.s0_ready);
            }
            if (q4 * 32 < DV) {
                // O^T row i -> y[t0 + t][i], transposed through this warp's own
                // 4 KB of the U tile (the rows of U^T that only this warp
                // writes, free once the products have completed).
                float o0[32], o1[32];
                tmem_ld32(tm + lrow + C::COL_O + 64 * pb, o0);
                tmem_ld32(tm + lrow + C::COL_O + 64 * pb + 32, o1);
                tmem_wait_ld();
                __nv_bfloat16 *ys = reinterpret_cast<__nv_bfloat16 *>(sm + C::OFF_U + q4 * 4096);  // [64][32]
#pragma unroll
                for (int t = 0; t < kC; ++t) ys[t * 32 + lane] = __float2bfloat16_rn(t < 32 ? o0[t] : o1[t - 32]);
                __syncwarp();
                __nv_bfloat16 *yb = y + ((size_t)bh * T + t0) * DV + q4 * 32;
#pragma unroll
                for (int e = lane; e < kC * 4; e += 32) {  // 64 rows x four 16-byte pieces
                    const int t = e >> 2, ch = e & 3;
                    if (t < n)
                        reinterpret_cast<uint4 *>(yb + (size_t)t * DV)[ch] =
                            reinterpret_cast<const uint4 *>(ys + t * 32)[ch];
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) atomicOr(status, kStChainEpi);
    } else {
        // ------------------------------------------------ chunk-local epilogue
        // Warps 8..11 prepare the even chunks, warps 12..15 the odd ones.
        const int g = (warp - 8) >> 2, bar = 2 + g;
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;  // TMEM lane
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        const int tok = row & (kC - 1);  // the token this thread's beta belongs to
        float *Lb = reinterpret_cast<float *>(sm + (C::L_IN_W ? C::OFF_W + g * C::WB : C::OFF_L + g * 16384));
        float *X = reinterpret_cast<float *>(sm + C::OFF_G + g * 8192);
        const uint32_t pt = s0 + C::OFF_P + g * 8192, gt = s0 + C::OFF_G + g * 8192, wt = s0 + C::OFF_W + g * C::WB;
        bool ok = true;
        // beta of the thread's token, one chunk ahead (its load latency is
        // then off the chunk's path)
        auto beta_of = [&](int c) { return c < nch && c * kC + tok < T ? beta[(size_t)bh * T + c * kC + tok] : 0.f; };
        float bt_next = beta_of(g);
        for (int c = g; c < nch; c += 2) {
            const float bt = bt_next;
            bt_next = beta_of(c + 2);
            ok = __all_sync(0xffffffffu, mbar_wait(&B.a_full[g], (c >> 1) & 1));
            if (ok && c >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&B.pw_empty[g], ((c >> 1) - 1) & 1));
            tc_fence_after();
            if (ok) {
                float vv[2][32];  // [Q; K] K^T row, both halves in flight at once
                tmem_ld32(tm + lrow + C::COL_P + 64 * g, vv[0]);
                tmem_ld32(tm + lrow + C::COL_P + 64 * g + 32, vv[1]);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // 32 columns at a time
                    const float(&v)[32] = vv[h];
                    if (row < kC) {  // P row i = (Q K^T)[i][j] for j <= i
                        const int i = row;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int jl = 8 * u + 2 * e, j = 32 * h + jl;
                                w[e] = pack_bf16(j <= i ? v[jl] : 0.f, j + 1 <= i ? v[jl + 1] : 0.f);
                            }
                            st_shared_v4(pt + sw128_off(i, 4 * h + u), w[0], w[1], w[2], w[3]);
                        }
                    } else {  // solve tile row i = beta_i * strict_lower(K K^T) row i
                        const int i = row - kC;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int j = 32 * h + 4 * q;
                            st4(Lb, i, 8 * h + q,
                                make_float4(j < i ? bt * v[4 * q] : 0.f, j + 1 < i ? bt * v[4 * q + 1] : 0.f,
                                            j + 2 < i ? bt * v[4 * q + 2] : 0.f, j + 3 < i ? bt * v[4 * q + 3] : 0.f));
                        }
                    }
                }
            }
            tc_fence_before();
            ok = prep_all(ok, bar);
            if (!ok) break;
            // T = (I + Lb)^{-1} in place, then row j of G^T = column j of G =
            // T[:, j] beta_j: thread (j, half) writes four 16-byte pieces.
            unit_lower_inverse(Lb, X, row, bar);
            {
                const int j = row & (kC - 1), h = row >> 6;
#pragma unroll
                for (int ch = 4 * h; ch < 4 * h + 4; ++ch) {
                    float gv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 8 * ch + e;
                        // read unconditionally (every (i, j) lies in the tile), then select:
                        // no per-lane branch around the load
                        const float lv = Lb[lsw(i, j)];
                        gv[e] = (i == j ? 1.f : (i > j ? lv : 0.f)) * bt;
                    }
                    st_shared_v4(gt + sw128_off(j, ch), pack_bf16(gv[0], gv[1]), pack_bf16(gv[2], gv[3]),
                                 pack_bf16(gv[4], gv[5]), pack_bf16(gv[6], gv[7]));
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.g_ready[g]);
            ok = __all_sync(0xffffffffu, mbar_wait(&B.w_full[g], (c >> 1) & 1));
            tc_fence_after();
            if (ok && row < DK) {  // row a of W^T = -(K^T G^T)[a]
                float aa[2][32];
                tmem_ld32(tm + lrow + C::COL_P + 64 * g, aa[0]);
                tmem_ld32(tm + lrow + C::COL_P + 64 * g + 32, aa[1]);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float(&a)[32] = aa[h];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        st_shared_v4(wt + sw128_off(row, 4 * h + u), pack_bf16(-a[8 * u], -a[8 * u + 1]),
                                     pack_bf16(-a[8 * u + 2], -a[8 * u + 3]), pack_bf16(-a[8 * u + 4], -a[8 * u + 5]),
                                     pack_bf16(-a[8 * u + 6], -a[8 * u + 7]));
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&B.pw_ready[g]);
                mbar_arrive(&B.ptm_free[g]);
            }
            ok = prep_all(ok, bar);
            if (!ok) break;
        }
        if (!ok && lane == 0) atomicOr(status, kStPrepWait);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tm, C::TCOLS);
}

template <int DK, int DV>
int run(const void *q, const void *k, const void *v, const float *beta, int BH, int T,
        const float *S0, float *S_out, void *y, unsigned int *status, cudaStream_t st) {
    const int nch = ceil_div(T, kC);
    CUtensorMap mq, mk, mv;
    int rc;
    if ((rc = make_tmap_bf16_3d(&mq, q, DK, T, BH, kC))) return rc;
    if ((rc = make_tmap_bf16_3d(&mk, k, DK, T, BH, kC))) return rc;
    if ((rc = make_tmap_bf16_3d(&mv, v, DV, T, BH, kC))) return rc;
    using Cfg = FusedCfg<DK>;
    auto kern = delta_fused_kernel<DK, DV>;
    const int smem = (int)(Cfg::OFF_BARS + sizeof(FusedBars) + 16);
    if (int rc_ = set_smem_limit((const void *)kern, smem, "delta_fused smem attribute")) return rc_;
    prof_begin(st);
    kern<<<BH, 512, smem, st>>>(mq, mk, mv, beta, T, nch, S0, S_out, (__nv_bfloat16 *)y, status);
    rc = launched("delta_fused");
    prof_end(st);
    return rc;
}

}  // namespace

bool delta_tcgen05_supported(int dtype, int dk, int dv, int chunk) {
    return dtype == OPAM_BF16 && (dk == 64 || dk == 128) && (dv == 64 || dv == 128) && chunk == kC;
}

size_t delta_tcgen05_workspace(int BH, int T, int dk) {
    (void)BH;
    (void)T;
    (void)dk;
    return 0;
}

int delta_tcgen05(const void *q, const void *k, const void *v, const float *beta, int B, int H, int T,
                  int dk, int dv, const float *S0, float *S_out, void *y, void *ws, unsigned int *status,
                  cudaStream_t s) {
    (void)ws;
    if (dk == 64 && dv == 128) return run<64, 128>(q, k, v, beta, B * H, T, S0, S_out, y, status, s);
    if (dk == 128 && dv == 128) return run<128, 128>(q, k, v, beta, B * H, T, S0, S_out, y, status, s);
    if (dk == 64 && dv == 64) return run<64, 64>(q, k, v, beta, B * H, T, S0, S_out, y, status, s);
    if (dk == 128 && dv == 64) return run<128, 64>(q, k, v, beta, B * H, T, S0, S_out, y, status, s);
    set_error("tensor-core delta rule: d_k=%d, d_v=%d unsupported", dk, dv);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace opam
