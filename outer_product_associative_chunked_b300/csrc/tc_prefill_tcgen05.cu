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
// Chunks of C = 128 positions.  Query block j covers [jC, jC+C); the tokens
// evicted during its steps are the shifted chunk [jC-W, jC-W+C).  With A_j the
// state before the block (every token s < jC-W) and row i of the block:
//   m_{jC+i} = lambda^(i+1) q A_j + sum_{l<=i} eta lambda^(i-l) <q, k'_l> v'_l
//   A_{j+1}  = lambda^n A_j + dA_j,  dA_j = sum_{l<n} eta lambda^(n-1-l) k'_l v'_l^T
// The shifted chunk is exactly the first key tile of the block's window
// (keys [jC-W, jC+C) in tiles of 128), so one Q K^T product serves both the
// L2 term (key l <= row i) and the softmax (l > i).
//
// The chunk recurrence is split into segments of L chunks so that many CTAs
// share it: within segment g (chunks [gL, gL+L)) the state is
//   A_j = A_j^loc + lambda^(C (j - gL)) A_{gL},
// where A_j^loc starts from zero at the segment.  Three kernels:
//   tc_l2_state_kernel  per (head, segment, 64 columns of d_v), chunk after
//                       chunk: dA_j = K'^T diag(w) V' on tcgen05 and the local
//                       recurrence in fp32; writes A_j^loc (bf16) and the
//                       segment's local final state (fp32);
//   tc_l2_carry_kernel  per head: the segment start states A_{gL} (bf16) and
//                       the final state after the whole sequence (fp32);
//   tc_fwd_row_kernel   (d = 64) and tc_fwd_kernel (d = 128 and mixed sizes),
//                       per (head, query block): flash-style online softmax
//                       over the window tiles (S = Q K^T and O += P V on
//                       tcgen05, P in TMEM), the L2 term of the shifted chunk
//                       (its own accumulator at d = 64; at d = 128 folded into
//                       P, scaled by the row's final softmax statistics),
//                       q (A_j^loc + lambda^(C (j - gL)) A_{gL}), and the gate;
//                       y leaves through shared memory by TMA stores.
//
// Every wait inside these kernels is bounded; a wait that runs out records a
// bit in the call's status word (the head of its workspace, read by
// opam_check_device_error) and the CTA winds down without hanging.
#include <math.h>

#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

constexpr int kBlk = 128;          // query rows per CTA = keys per tile = chunk length
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.0f;   // lazy-rescale threshold (log2 units)

// Bits recorded in the call's status word (the head of its workspace) when a
// bounded wait runs out.
enum : unsigned int {
    kStStateProducer = kStatusTcPrefill << 0,
    kStStateMma = kStatusTcPrefill << 1,
    kStStateScan = kStatusTcPrefill << 2,
    kStFwdProducer = kStatusTcPrefill << 3,
    kStFwdMma = kStatusTcPrefill << 4,
    kStFwdSoftmax = kStatusTcPrefill << 5,
    kStFwdAlign = kStatusTcPrefill << 6,
};

// Chunks per segment of the state recurrence, at most one segment per chunk.
// For d = 64 the state pass runs one CTA per SM (padded to kStateSoloSmem so
// that two never share an SM), with twice as many chunks per segment as two
// per SM would give: on the B4 H8 T4096 W512 step this measured 62.4 against
// 64.0 us.  For the larger sizes two state CTAs per SM fill the GPU.
struct Segments {
    int nch, nseg, L;
};
constexpr uint32_t kStateSoloSmem = 116 * 1024;  // above half an SM's shared memory
Segments segments(int BH, int T, int dk, int dv, int num_sms) {
    const int nch = ceil_div(T, kBlk);
    const int units = BH * (dv / 64);
    const int per_sm = (dk == 64 && dv == 64) ? 1 : 2;
    int want = (per_sm * num_sms) / units;
    if (want < 1) want = 1;
    if (want > nch) want = nch;
    const int L = ceil_div(nch, want);
    return {nch, ceil_div(nch, L), L};
}

// --------------------------------------------------------------------- chunk states
// One CTA per (64-column slice, segment, head) walks the segment's chunks:
//   dA_j = K'^T diag(w) V' on tcgen05 (A = K'^T read MN-major from the K'
//          tile; M is fixed at 128, so for d_k = 64 both 64-wide M blocks
//          alias the same rows and TMEM lanes 64..127 hold an unused copy),
//   A_j^loc -> bf16 for the forward kernel, then A^loc <- lambda^n A^loc + dA_j
//          in fp32 registers (one state row per thread).
// Warps 0-3 weight V' rows by w_l = eta lambda^(n-1-l) (thread = token row)
// and run the recurrence (thread = state row a < d_k); warp 4 loads K'/V' by
// TMA; warp 5 issues the MMAs.  Loads, weighting and MMAs of later chunks
// overlap the recurrence of the current one.
template <int DK>
struct StateCfg {
    static constexpr uint32_t KBYTES = kBlk * DK * 2;
    static constexpr uint32_t VBYTES = kBlk * 64 * 2;
    static constexpr int NS = DK == 64 ? 3 : 2;
    static constexpr uint32_t SMEM = NS * (KBYTES + VBYTES) + 1024;
};

struct StateBars {
    uint64_t kv_full[4], scaled[4], kv_empty[4], mma_done[2], tm_free[2], drain;
    uint32_t tbase;
    unsigned int st;  // this CTA's status bits
    float pw[kBlk];   // eta lambda^d
};

template <int DK, int DV>
__global__ void __launch_bounds__(192, 2)
tc_l2_state_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                   int T, int W, int H, const float *__restrict__ lam, const float *__restrict__ eta,
                   int nch, int L, __nv_bfloat16 *__restrict__ Aloc, float *__restrict__ Lfin,
                   unsigned int *__restrict__ cta_status, unsigned int *__restrict__ status) {
    using C = StateCfg<DK>;
    constexpr int NS = C::NS;
    // Status words of the call (see the launcher): this kernel is the call's
    // first, launched after all earlier work on the stream, so its first CTA
    // zeroes the words of the later kernels before any of them can start (the
    // fence completes the stores before this CTA's launch trigger).  Its own
    // bits go to a per-CTA slot written at exit, which the carry kernel folds
    // into word 0, so no word is both cleared and set by one grid.
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) {
        status[1] = 0u;
        status[2] = 0u;
        status[3] = 0u;
        __threadfence();
    }
    pdl_launch_dependents();  // the carry kernel may be scheduled; it waits for this grid
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    __shared__ StateBars B;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x, seg = blockIdx.y, bh = blockIdx.z, h = bh % H;
    const int nseg = gridDim.y;
    const int j0 = seg * L, j1 = min(nch, j0 + L), nj = j1 - j0;
    const uint32_t s0 = smem_u32(sm);
    auto stage_k = [&](int s) { return s0 + s * (C::KBYTES + C::VBYTES); };
    auto load_kv = [&](int i) {  // K' and the V' slice of local chunk i into stage i % NS
        const int s = i % NS;
        unsigned char *kd = sm + (stage_k(s) - s0);
        const int kt = (j0 + i) * kBlk - W;
        mbar_expect_tx(&B.kv_full[s], C::KBYTES + C::VBYTES);
#pragma unroll
        for (int b = 0; b < DK / 64; ++b) tma_load_3d(kd + b * 16384, &mk, &B.kv_full[s], 64 * b, kt, bh);
        tma_load_3d(kd + C::KBYTES, &mv, &B.kv_full[s], 64 * slice, kt, bh);
    };
    if (warp == 4 && lane == 0) {  // barriers, then the first loads, before the CTA-wide sync
        for (int s = 0; s < NS; ++s) {
            mbar_init(&B.kv_full[s], 1);
            mbar_init(&B.scaled[s], 4);
            mbar_init(&B.kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&B.mma_done[b], 1);
            mbar_init(&B.tm_free[b], DK / 32);
        }
        mbar_init(&B.drain, 1);
        mbar_fence_init();
        for (int i = 0; i < NS && i < nj; ++i) load_kv(i);
    }
    if (warp == 5) tmem_alloc(&B.tbase, 128);
    if (tid == 0) B.st = 0u;
    if (tid < kBlk) B.pw[tid] = eta[h] * powf(lam[h], (float)tid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;

    if (warp == 4) {
        if (lane == 0) {
            bool ok = true;
            int issued = min(NS, nj);  // issued before the CTA-wide sync
            for (int i = issued; i < nj && ok; ++i) {
                ok = mbar_wait(&B.kv_empty[i % NS], ((i / NS) - 1) & 1);
                if (!ok) break;
                load_kv(i);
                ++issued;
            }
            if (!ok) atomicOr(&B.st, kStStateProducer);
            bool dok = true;
            for (int i = max(0, issued - NS); i < issued && dok; ++i)
                dok = mbar_wait(&B.kv_full[i % NS], (i / NS) & 1);
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t idesc = idesc_bf16_f32(128, 64, true, true);
            for (int i = 0; i < nj && ok; ++i) {
                const int s = i % NS, b = i & 1;
                ok = mbar_wait(&B.scaled[s], (i / NS) & 1);
                if (ok && i >= 2) ok = mbar_wait(&B.tm_free[b], ((i - 2) >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t ka = stage_k(s), va = ka + C::KBYTES;
#pragma unroll
                for (int k = 0; k < kBlk / 16; ++k)
                    mma_ss(tm + b * 64, sdesc_sw128(ka + k * 2048, DK == 128 ? 16384 : 0, 1024),
                           sdesc_sw128(va + k * 2048, 16384, 1024), idesc, k > 0 ? 1u : 0u);
                mma_commit(&B.mma_done[b]);
                mma_commit(&B.kv_empty[s]);
            }
            if (!ok) atomicOr(&B.st, kStStateMma);
            mma_commit(&B.drain);
            mbar_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        const int r = tid;  // token row when weighting, state row when scanning
        const uint32_t lrow = (uint32_t)(warp * 32) << 16;
        const bool scan_row = r < DK;
        const float lm = lam[h];
        const float lamC = powf(lm, (float)kBlk);
        float A[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) A[i] = 0.f;
        __nv_bfloat16 *arow = Aloc + ((size_t)bh * nch * DK + r) * DV + slice * 64;
        bool ok = true;
        // A^loc <- lambda^n A^loc + dA of local chunk i (TMEM buffer i & 1).
        auto absorb = [&](int i) -> bool {
            const int b = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&B.mma_done[b], (i >> 1) & 1))) return false;
            tc_fence_after();
            float d0[32], d1[32];
            tmem_ld32(tm + lrow + b * 64, d0);
            tmem_ld32(tm + lrow + b * 64 + 32, d1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.tm_free[b]);
            const int n = min(kBlk, T - (j0 + i) * kBlk);
            const float f = n == kBlk ? lamC : powf(lm, (float)n);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                A[e] = fmaf(f, A[e], d0[e]);
                A[32 + e] = fmaf(f, A[32 + e], d1[e]);
            }
            return true;
        };
        auto emit = [&](int j) {  // A_j^loc as bf16, 128 contiguous bytes per row
            if (!OPAM_BOUNDS(j < nch && r < DK, &B.st)) return;
            uint4 *dst = reinterpret_cast<uint4 *>(arow + (size_t)j * DK * DV);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                dst[u] = make_uint4(pack_bf16(A[8 * u], A[8 * u + 1]), pack_bf16(A[8 * u + 2], A[8 * u + 3]),
                                    pack_bf16(A[8 * u + 4], A[8 * u + 5]), pack_bf16(A[8 * u + 6], A[8 * u + 7]));
        };
        for (int i = 0; i < nj && ok; ++i) {
            const int s = i % NS, j = j0 + i;
            ok = __all_sync(0xffffffffu, mbar_wait(&B.kv_full[s], (i / NS) & 1));
            if (!ok) break;
            {   // weight row r of V' in place; chunk order rotated by row (no bank conflicts)
                const int kt = j * kBlk - W, n = min(kBlk, T - j * kBlk);
                const float w = (r < n && kt + r >= 0) ? B.pw[(n - 1 - r) & (kBlk - 1)] : 0.f;
                const __nv_bfloat162 w2 = __floats2bfloat162_rn(w, w);
                const uint32_t va = stage_k(s) + C::KBYTES + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t a = va + (((c + r) & 7) << 4);
                    uint32_t x[4];
                    ld_shared_v4(a, x[0], x[1], x[2], x[3]);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        __nv_bfloat162 hv = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&x[u]), w2);
                        x[u] = *reinterpret_cast<uint32_t *>(&hv);
                    }
                    st_shared_v4(a, x[0], x[1], x[2], x[3]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.scaled[s]);
            }
            if (scan_row) {
                if (i >= 1) ok = absorb(i - 1);
                if (ok) emit(j);
            }
        }
        if (ok && scan_row) {
            ok = absorb(nj - 1);
            if (ok && OPAM_BOUNDS(seg < nseg && slice * 64 + 64 <= DV, &B.st)) {
                float4 *dst = reinterpret_cast<float4 *>(Lfin + (((size_t)bh * nseg + seg) * DK + r) * DV + slice * 64);
#pragma unroll
                for (int u = 0; u < 16; ++u) dst[u] = make_float4(A[4 * u], A[4 * u + 1], A[4 * u + 2], A[4 * u + 3]);
            }
        }
        if (!ok && lane == 0) atomicOr(&B.st, kStStateScan);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) tmem_dealloc(tm, 128);
    if (tid == 0) cta_status[((size_t)bh * gridDim.y + seg) * gridDim.x + slice] = B.st;
}

// --------------------------------------------------------------------- segment carries
// A_{0} = 0, A_{(g+1)L} = lambda^{tokens of segment g} A_{gL} + local final of g.
// Each thread owns two groups of 4 adjacent state elements of one head (the
// second blockDim.x groups after the first).  Few CTAs and at most 48
// registers a thread, so that all of them are resident as soon as they are
// launched: the forward grid, their programmatic dependent, launches only
// once every carry CTA is.
__global__ void __launch_bounds__(128, 10)
tc_l2_carry_kernel(const float *__restrict__ Lfin, int nseg, int L, int T, int dkdv, int H,
                   const float *__restrict__ lam, __nv_bfloat16 *__restrict__ Cbf,
                   float *__restrict__ A_final, const unsigned int *__restrict__ cta_status, int n_cta,
                   unsigned int *__restrict__ status) {
    pdl_launch_dependents();  // the forward kernel may start its window tiles now
    pdl_wait_primary();       // segment finals and CTA status slots of the state kernel
    if (blockIdx.x == 0 && blockIdx.y == 0) {  // word 0 of the call: the state CTAs' bits
        __shared__ unsigned int st;
        if (threadIdx.x == 0) st = 0u;
        __syncthreads();
        unsigned int bits = 0u;
        for (int i = threadIdx.x; i < n_cta; i += blockDim.x) bits |= cta_status[i];
        if (bits) atomicOr(&st, bits);
        __syncthreads();
        if (threadIdx.x == 0) status[0] = st;
    }
    const int bh = blockIdx.y;
    const int e0 = (blockIdx.x * 2 * blockDim.x + threadIdx.x) * 4, estep = 4 * blockDim.x;
    const float lm = lam[bh % H];
    const float f = powf(lm, (float)(L * kBlk));  // decay across a full segment
    const float *src = Lfin + (size_t)bh * nseg * dkdv;
    __nv_bfloat16 *dst = Cbf + (size_t)bh * nseg * dkdv;
    float4 A[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    // Segment finals are read two at a time for both groups, so that four
    // loads overlap; the recurrence itself is a chain of FMAs.
    constexpr int kBatch = 2;
    for (int g0 = 0; g0 < nseg; g0 += kBatch) {
        float4 d[2][kBatch];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = e0 + h * estep;
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                d[h][u] = (e + 4 <= dkdv && g0 + u < nseg)
                              ? *reinterpret_cast<const float4 *>(src + (size_t)(g0 + u) * dkdv + e)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int g = g0 + u;
            if (g >= nseg) break;
            // the last segment may be shorter: its decay only matters for A_final
            const float fg = (g + 1) * L * kBlk <= T ? f : powf(lm, (float)(T - g * L * kBlk));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int e = e0 + h * estep;
                if (e + 4 <= dkdv) {
                    uint2 o;
                    o.x = pack_bf16(A[h].x, A[h].y);
                    o.y = pack_bf16(A[h].z, A[h].w);
                    *reinterpret_cast<uint2 *>(dst + (size_t)g * dkdv + e) = o;
                }
                A[h].x = fmaf(fg, A[h].x, d[h][u].x);
                A[h].y = fmaf(fg, A[h].y, d[h][u].y);
                A[h].z = fmaf(fg, A[h].z, d[h][u].z);
                A[h].w = fmaf(fg, A[h].w, d[h][u].w);
            }
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = e0 + h * estep;
        if (A_final && e + 4 <= dkdv) *reinterpret_cast<float4 *>(A_final + (size_t)bh * dkdv + e) = A[h];
    }
}

// --------------------------------------------------------------------- fused forward
template <int DK, int DV>
struct Fwd {
    static constexpr uint32_t QBYTES = kBlk * DK * 2;
    static constexpr uint32_t KBYTES = kBlk * DK * 2;  // also holds A_j^loc (DK x DV bf16)
    static constexpr uint32_t VBYTES = kBlk * DV * 2;  // also holds the segment carry
    static constexpr uint32_t kBudget = 227 * 1024 - 3072;  // 3 KB kept for the barriers block
    // Three K slots and three V slots: a K slot is free once its S product
    // has completed and a V slot once its P V has, so each tile is requested
    // well before it is needed.  P lives in TMEM.
    static constexpr int NSK = 3, NSV = 3;
    static constexpr uint32_t OFF_K = QBYTES;
    static constexpr uint32_t OFF_V = OFF_K + NSK * KBYTES;
    static constexpr uint32_t OFF_BARS = OFF_V + NSV * VBYTES;
    static_assert(OFF_BARS <= kBudget, "shared-memory budget");
    // TMEM columns: S [0,128) (q A_j lands in [0,DV) after the last tile); O
    // of key half 0 / 1; P of key half 0 / 1 (64 keys as packed bf16 pairs,
    // 32 columns each), the A operand of O += P V.
    static constexpr uint32_t COL_O0 = 128, COL_O1 = 128 + DV, COL_P = 128 + 2 * DV;
    static_assert(COL_P + 64 <= 512, "TMEM columns");
    static constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t ID_PV = idesc_bf16_f32(128, DV, false, true);
};

struct FwdBars {
    uint64_t q_full;
    uint64_t k_full[4], v_full[4], k_empty[4], v_empty[4];  // the K and V halves of a stage are freed apart
    uint64_t s_full, s_empty;
    uint64_t p_full[2], p_empty[2];  // per key half
    uint64_t c_ready, xe, o_done, drain, drain_pv;  // o_done: one commit from each issuing thread
    uint64_t y_ready;                               // the eight softmax warps have staged their y rows
    uint32_t tbase;
    float pw[kBlk];      // eta lambda^d, d = 0..127
    float xm[2][kBlk];   // [key half][row] running maxima, exchanged once at the end
    float xl[2][kBlk];   // [key half][row] running sums
};

// 352 threads.  Warps 0-7 run the softmax: warp w owns rows 32 (w % 4) .. +31
// (its TMEM lane quarter) and keys 64 (w / 4) .. +63 of every tile.  The two
// key halves of a row keep separate running maxima, sums and P V accumulators
// (O0, O1) and are merged once in the epilogue, so the softmax warps never
// wait for each other inside the tile loop.  Warp 8 issues TMA loads and
// scales the segment carry; warp 9 issues the S products (and the final
// q A products) and owns the TMEM allocation; warp 10 issues the P V
// products.  With two issuing threads the next tile's S does not queue
// behind a P V that waits for the slowest softmax warp of the previous tile.
// The shifted chunk comes last: once its softmax keys are in P the two halves
// exchange their statistics, and its L2 scores are added into P scaled by
// sigmoid(g) L / f_half, so O_half f_half / L carries them with no extra
// accumulator.  y is staged in the spent Q tile and stored by TMA.  `wave`
// is the number of CTAs resident at once (one per SM): the producer warms L2
// with the first tiles of the CTA that many places later in launch order
// (0 turns that off).
template <int DK, int DV>
__global__ void __launch_bounds__(352, 1)
tc_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap ma,
              const __grid_constant__ CUtensorMap mc, const __grid_constant__ CUtensorMap my, int T, int W,
              int H, int nch, int nseg, int L, int l2, const float *__restrict__ lam,
              const float *__restrict__ eta, const float *__restrict__ gate, float scale, int wave,
              unsigned int *__restrict__ status) {
    using C = Fwd<DK, DV>;
    constexpr int NSK = C::NSK, NSV = C::NSV;
    // All shared memory is dynamic: with no static shared memory its base is
    // 1024-byte aligned, as the 128-byte-swizzle tiles require (checked).
    extern __shared__ __align__(1024) unsigned char sm[];
    FwdBars &B = *reinterpret_cast<FwdBars *>(sm + C::OFF_BARS);
    if ((smem_u32(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStFwdAlign);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int jq = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int seg = jq / L;
    const int t0 = jq * kBlk;
    const int kt0 = t0 - W;  // first key of tile 0 (the shifted chunk)
    const int nt_total = (W + kBlk - 1) / kBlk + 1;
    const int j_first = (-kt0 - (kBlk - 1) > 0) ? (-kt0) / kBlk : 0;
    const int ntiles = nt_total - j_first;
    // l2 == 0: window only (no L2 part, no state loads, no q A term).
    const bool has_l2 = l2 && (j_first == 0);
    // Key tile j covers keys kt0 + 128 j ..; with an L2 part the tiles run
    // 1, 2, .., nt-1 and the shifted chunk (j = 0) comes last, when the row's
    // softmax statistics are final, so its L2 scores can join P scaled by them.
    auto tile_j = [&](int n) { return has_l2 ? (n + 1 < ntiles ? n + 1 : 0) : j_first + n; };

    if (warp == 9) tmem_alloc(&B.tbase, 512);
    if (tid == 0) {
        mbar_init(&B.q_full, 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(&B.k_full[s], 1);
            mbar_init(&B.k_empty[s], 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(&B.v_full[s], 1);
            mbar_init(&B.v_empty[s], 1);
        }
        mbar_init(&B.s_full, 1);
        mbar_init(&B.s_empty, 8);
        for (int hh = 0; hh < 2; ++hh) {
            mbar_init(&B.p_full[hh], 4);
            mbar_init(&B.p_empty[hh], 1);
        }
        mbar_init(&B.c_ready, 1);
        mbar_init(&B.xe, 8);
        mbar_init(&B.o_done, 2);
        mbar_init(&B.drain, 1);
        mbar_init(&B.drain_pv, 1);
        mbar_init(&B.y_ready, 8);
        mbar_fence_init();
    }
    if (l2 && tid < kBlk) B.pw[tid] = eta[h] * powf(lam[h], (float)tid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;
    const uint32_t sQ = smem_u32(sm);
    const uint32_t sK0 = sQ + C::OFF_K;

    if (warp == 8) {
        // ------------------------------------------------ TMA producer
        bool ok = true;
        const int sA = ntiles % NSK, sC = ntiles % NSV;  // slots of A_j^loc (K) and of the carry (V)
        if (lane == 0) {
            tma_prefetch_desc(&mq);
            tma_prefetch_desc(&mk);
            tma_prefetch_desc(&mv);
            tma_prefetch_desc(&my);
            mbar_expect_tx(&B.q_full, C::QBYTES);
#pragma unroll
            for (int b = 0; b < DK / 64; ++b) tma_load_3d(sm + b * 16384, &mq, &B.q_full, 64 * b, t0, bh);
            // A K slot is free once the S product of its previous tile has
            // completed, a V slot once that tile's P V has.  K of tile n + 1 is
            // requested before V of tile n, so each K tile lands well ahead of
            // its S product.
            auto kslot = [&](int n) { return sm + C::OFF_K + (n % NSK) * C::KBYTES; };
            auto vslot = [&](int n) { return sm + C::OFF_V + (n % NSV) * C::VBYTES; };
            auto load_k = [&](int n) -> bool {
                const int s = n % NSK;
                if (n >= NSK && !mbar_wait(&B.k_empty[s], ((n / NSK) - 1) & 1)) return false;
                const int kt = kt0 + kBlk * tile_j(n);
                mbar_expect_tx(&B.k_full[s], C::KBYTES);
#pragma unroll
                for (int b = 0; b < DK / 64; ++b) tma_load_3d(kslot(n) + b * 16384, &mk, &B.k_full[s], 64 * b, kt, bh);
                return true;
            };
            auto load_v = [&](int n) -> bool {
                const int s = n % NSV;
                if (n >= NSV && !mbar_wait(&B.v_empty[s], ((n / NSV) - 1) & 1)) return false;
                const int kt = kt0 + kBlk * tile_j(n);
                mbar_expect_tx(&B.v_full[s], C::VBYTES);
#pragma unroll
                for (int b = 0; b < DV / 64; ++b) tma_load_3d(vslot(n) + b * 16384, &mv, &B.v_full[s], 64 * b, kt, bh);
                return true;
            };
            if (ntiles > 0) ok = load_k(0);
            {   // L2 prefetch for the CTA one wave later in launch order (grid x = query
                // block, y = head): its Q tile and first K and V tiles
                const int nl = (int)(blockIdx.y * gridDim.x + blockIdx.x) + wave;
                if (wave > 0 && nl < (int)(gridDim.x * gridDim.y)) {
                    const int njq = nl % (int)gridDim.x, nbh = nl / (int)gridDim.x;
                    const int nt0 = njq * kBlk, nkt0 = nt0 - W;
                    const int nj_first = (-nkt0 - (kBlk - 1) > 0) ? (-nkt0) / kBlk : 0;
                    const int nnt = nt_total - nj_first;
                    const bool nl2 = l2 && nj_first == 0;
#pragma unroll
                    for (int b = 0; b < DK / 64; ++b) tma_prefetch_l2_3d(&mq, 64 * b, nt0, nbh);
                    for (int n = 0; n < 2 && n < nnt; ++n) {
                        const int kt = nkt0 + kBlk * (nl2 ? (n + 1 < nnt ? n + 1 : 0) : nj_first + n);
                        if (kt < 0) continue;
                        for (int b = 0; b < DK / 64; ++b) tma_prefetch_l2_3d(&mk, 64 * b, kt, nbh);
                        if (n == 0)
                            for (int b = 0; b < DV / 64; ++b) tma_prefetch_l2_3d(&mv, 64 * b, kt, nbh);
                    }
                }
            }
            for (int n = 0; n < ntiles && ok; ++n) {
                if (n + 1 < ntiles) ok = load_k(n + 1);
                if (ok) ok = load_v(n);
            }
            if (ok && l2) {  // A_j^loc into K slot ntiles, the segment carry into V slot ntiles
                const int n = ntiles;
                if (n >= NSK) ok = mbar_wait(&B.k_empty[sA], ((n / NSK) - 1) & 1);
                if (ok && n >= NSV) ok = mbar_wait(&B.v_empty[sC], ((n / NSV) - 1) & 1);
                if (ok) {
                    mbar_expect_tx(&B.k_full[sA], 2 * DK * DV * 2);
#pragma unroll
                    for (int b = 0; b < DV / 64; ++b) {
                        tma_load_3d(kslot(n) + b * (DK * 128), &ma, &B.k_full[sA], 64 * b, 0, bh * nch + jq);
                        tma_load_3d(vslot(n) + b * (DK * 128), &mc, &B.k_full[sA], 64 * b, 0, bh * nseg + seg);
                    }
                }
            }
            if (ok && l2) ok = mbar_wait(&B.k_full[sA], (ntiles / NSK) & 1);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && l2) {
            // Carry times lambda^(C (j - gL)), in place, so q A_j^loc and the
            // carry share one accumulator.
            const float c = powf(lam[h], (float)(kBlk * (jq - seg * L)));
            const __nv_bfloat162 c2 = __floats2bfloat162_rn(c, c);
            const uint32_t base = sQ + C::OFF_V + sC * C::VBYTES;
            for (int e = lane; e < DK * DV / 8; e += 32) {
                uint32_t x[4];
                ld_shared_v4(base + e * 16, x[0], x[1], x[2], x[3]);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    __nv_bfloat162 hv = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&x[u]), c2);
                    x[u] = *reinterpret_cast<uint32_t *>(&hv);
                }
                st_shared_v4(base + e * 16, x[0], x[1], x[2], x[3]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.c_ready);
        } else if (!ok && lane == 0) {
            atomicOr(status, kStFwdProducer);
        }
        __syncwarp();
    } else if (warp == 9 || warp == 10) {
        // ------------------------------------------------ MMA issue: S (warp 9), P V (warp 10)
        if (lane == 0) {
            bool ok = mbar_wait(&B.q_full, 0);
            // Descriptors as a fixed upper half plus a lower half (address >> 4 |
            // leading offset), so each k step is one 32-bit add in the issue loop.
            constexpr uint32_t HI = sdesc_hi(1024);
            constexpr uint32_t KSTEP = C::KBYTES >> 4, VSTEP = C::VBYTES >> 4;  // one K / V slot, encoded
            const uint32_t q_lo = sdesc_lo(sQ, 16), k_lo = sdesc_lo(sK0, 16);
            const uint32_t v_lo = sdesc_lo(sQ + C::OFF_V, 16384);
            auto kofs = [](int k) { return (uint32_t)((k >> 2) * (16384 >> 4) + (k & 3) * 2); };  // K-major k step
            if (warp == 10) {
                // O_half += P_half V of tile n, P_half (128 rows x 64 keys) from TMEM.
                constexpr uint32_t ID_PVT = idesc_bf16_f32(128, DV, false, true);
                for (int n = 0; n < ntiles && ok; ++n) {
                    const int s = n % NSV;
                    ok = mbar_wait(&B.v_full[s], (n / NSV) & 1);
                    for (int hh = 0; hh < 2 && ok; ++hh) {
                        ok = mbar_wait(&B.p_full[hh], n & 1);
                        if (!ok) break;
                        tc_fence_after();
                        // V rows 64 hh + 16 k .. of slot s (MN-major B)
                        const uint32_t vb = v_lo + (uint32_t)s * VSTEP + (uint32_t)hh * (8192 >> 4);
                        const uint32_t pt = tm + C::COL_P + 32 * hh;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts_h(tm + (hh ? C::COL_O1 : C::COL_O0), pt + 8 * k, vb + k * (2048 >> 4), HI, ID_PVT,
                                     (n > 0 || k > 0) ? 1u : 0u);
                        mma_commit(&B.p_empty[hh]);
                    }
                    if (ok) mma_commit(&B.v_empty[s]);
                }
                if (ok) mma_commit(&B.o_done);
                if (!ok) atomicOr(status, kStFwdMma);
                // Every MMA issued by this thread has completed before TMEM is freed.
                mma_commit(&B.drain_pv);
                mbar_wait(&B.drain_pv, 0);
            } else {
                for (int n = 0; n < ntiles && ok; ++n) {
                    const int s = n % NSK;
                    ok = mbar_wait(&B.k_full[s], (n / NSK) & 1);
                    if (ok && n >= 1) ok = mbar_wait(&B.s_empty, (n - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kb = k_lo + (uint32_t)s * KSTEP;
#pragma unroll
                    for (int k = 0; k < DK / 16; ++k)
                        mma_ss_h(tm, q_lo + kofs(k), HI, kb + kofs(k), HI, C::ID_S, k > 0 ? 1u : 0u);
                    mma_commit(&B.s_full);
                    mma_commit(&B.k_empty[s]);
                }
                if (ok && !l2) mma_commit(&B.o_done);
                if (ok && l2) {  // q (A_j^loc + c A_{gL}) into the S columns, once the last S has been read
                    const int n = ntiles, s = n % NSK;
                    ok = mbar_wait(&B.k_full[s], (n / NSK) & 1);
                    if (ok) ok = mbar_wait(&B.c_ready, 0);
                    if (ok) ok = mbar_wait(&B.s_empty, (n - 1) & 1);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t a_lo = sdesc_lo(sK0 + s * C::KBYTES, DK * 128);
                        const uint32_t c_lo = sdesc_lo(sQ + C::OFF_V + (n % NSV) * C::VBYTES, DK * 128);
#pragma unroll
                        for (int k = 0; k < DK / 16; ++k)
                            mma_ss_h(tm, q_lo + kofs(k), HI, a_lo + k * (2048 >> 4), HI, C::ID_PV, k > 0 ? 1u : 0u);
#pragma unroll
                        for (int k = 0; k < DK / 16; ++k)
                            mma_ss_h(tm, q_lo + kofs(k), HI, c_lo + k * (2048 >> 4), HI, C::ID_PV, 1u);
                        mma_commit(&B.o_done);
                    }
                }
                if (!ok) atomicOr(status, kStFwdMma);
                // Every MMA issued by this thread has completed before TMEM is freed.
                mma_commit(&B.drain);
                mbar_wait(&B.drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax / epilogue
        const int half = warp >> 2;            // keys 64 half .. +63 of every tile
        const int r = (warp & 3) * 32 + lane;  // query row
        const int t = t0 + r;
        const int c0 = half * 64;
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t col_o = half ? C::COL_O1 : C::COL_O0;
        const uint32_t col_p = C::COL_P + 32 * half;
        const float sc = scale * kLog2e;
        const float sg = l2 ? 1.0f / (1.0f + expf(-gate[h])) : 0.f;
        float m = kNegBig, l = 0.f;
        bool ok = true;
        // The row's merged statistics: each half leaves its maximum and sum
        // in shared memory once (after its last softmax keys), then both read
        // the other's.
        auto exchange_stats = [&]() -> bool {
            B.xm[half][r] = m;
            B.xl[half][r] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.xe);
            return __all_sync(0xffffffffu, mbar_wait(&B.xe, 0));
        };
        // 32 keys (group g of this half) of row r into P as packed bf16.
        auto store_p = [&](int g, const float *p) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(p[2 * e], p[2 * e + 1]);
            tmem_st16(tm + lrow + col_p + 16 * g, pk);
        };
        const int wrow_hi = (warp & 3) * 32 + 31;
        for (int n = 0; n < ntiles && ok; ++n) {
            const int j = tile_j(n);
            const int kt = kt0 + kBlk * j;
            const bool shifted = has_l2 && j == 0;  // the last tile: its keys l <= r are the L2 part
            ok = __all_sync(0xffffffffu, mbar_wait(&B.s_full, n & 1));
            if (!ok) break;
            tc_fence_after();
            float s[64];
            {
                float v[32];
                tmem_ld32(tm + lrow + c0, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[i] = v[i];
                tmem_ld32(tm + lrow + c0 + 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[32 + i] = v[i];
            }
            tmem_wait_ld();
            if (!shifted) {  // the shifted chunk re-reads S for its L2 scores, so S is released later
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.s_empty);
            }
            // Softmax part: keys max(0, t-W+1) <= p <= t.  On edge tiles, 32-key
            // groups masked for every row of the warp skip the exponentials.
            const bool interior = (j >= 1) && (kt >= 0) && (kt <= t0 - (kBlk - 1));
            unsigned act = 0x3u;
            float pm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
            if (interior) {
#pragma unroll
                for (int i = 0; i < 64; ++i) pm[i & 7] = fmaxf(pm[i & 7], s[i]);
            } else {
                const int lo = max(0, t - W + 1) - kt - c0, hi = t - kt - c0;
                const int wlo = __reduce_min_sync(0xffffffffu, lo), whi = __reduce_max_sync(0xffffffffu, hi);
                act = 0;
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    if (32 * g <= whi && 32 * g + 31 >= wlo) {
                        act |= 1u << g;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int i = 32 * g + e;
                            s[i] = (i >= lo && i <= hi) ? s[i] : -INFINITY;
                            pm[e & 7] = fmaxf(pm[e & 7], s[i]);
                        }
                    }
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * sc;
            const bool grow = mx > m + kRescale;
            // P may be written (and O rescaled) once the previous P V of this half has completed.
            ok = __all_sync(0xffffffffu, n == 0 || mbar_wait(&B.p_empty[half], (n - 1) & 1));
            if (!ok) break;
            tc_fence_after();
            if (__any_sync(0xffffffffu, grow) && n > 0) {
                const float f = grow ? ex2(m - mx) : 1.f;
#pragma unroll 1
                for (int cc = 0; cc < DV; cc += 32) {
                    float v[32];
                    tmem_ld32(tm + lrow + col_o + cc, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= f;
                    tmem_st32(tm + lrow + col_o + cc, v);
                }
            }
            if (grow) {
                l *= ex2(m - mx);
                m = mx;
            }
            const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m, -m);
            float2 ps[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) ps[u] = make_float2(0.f, 0.f);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                if (act & (1u << g)) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int i = 32 * g + e;
                        float2 x = fma2(make_float2(s[i], s[i + 1]), sc2, nm2);
                        x.x = ex2(x.x);
                        x.y = ex2(x.y);
                        s[i] = x.x;
                        s[i + 1] = x.y;
                        ps[(e >> 1) & 3] = add2(ps[(e >> 1) & 3], x);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[32 * g + e] = 0.f;
                }
            }
            l += ((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) + ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y));
            store_p(0, &s[0]);
            store_p(1, &s[32]);
            if (shifted) {
                // The row's statistics are now final: merge them, then the L2
                // scores eta lambda^(r-l) <q_r, k'_l> of keys l <= r (where the
                // softmax P is zero) are added into P scaled by sigmoid(g) L /
                // f_half, so that O_half f_half / L carries sigmoid(g) times
                // their sum over V'.
                ok = exchange_stats();
                if (!ok) break;
                const float mo = B.xm[half ^ 1][r], lo_ = B.xl[half ^ 1][r];
                const float Mx = fmaxf(m, mo);
                const float fs = ex2(m - Mx), fo = ex2(mo - Mx);
                const float Lt = l * fs + lo_ * fo;
                const float k2 = fs > 0.f ? sg * Lt / fs : 0.f;
                const int lo2 = max(0, -kt);  // keys at positions >= 0
                tmem_wait_st();
#pragma unroll 1
                for (int g = 0; g < 2; ++g) {
                    const int gk = c0 + 32 * g;
                    if (!((gk <= wrow_hi) && (gk + 31 >= lo2))) continue;  // no L2 key for any row of the warp
                    float v[32];
                    uint32_t pk[16];
                    tmem_ld32(tm + lrow + c0 + 32 * g, v);  // S of this group again
                    tmem_ld16u(tm + lrow + col_p + 16 * g, pk);
                    tmem_wait_ld();
                    // The table is read unconditionally and the key range only
                    // selects the factor: a load under a per-lane condition made
                    // this loop about ten times slower.
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int i = gk + e;
                        const float wa = B.pw[(r - i) & (kBlk - 1)], wb = B.pw[(r - i - 1) & (kBlk - 1)];
                        const float ka = (i >= lo2 && i <= r) ? k2 : 0.f;
                        const float kb = (i + 1 >= lo2 && i + 1 <= r) ? k2 : 0.f;
                        const float a = ka * wa * v[e], b = kb * wb * v[e + 1];
                        const float2 pv = unpack_bf16(pk[e >> 1]);
                        pk[e >> 1] = pack_bf16(pv.x + a, pv.y + b);
                    }
                    tmem_st16(tm + lrow + col_p + 16 * g, pk);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.s_empty);  // S is read: the q A products may overwrite it
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.p_full[half]);
        }
        // ------------------------------------------------ epilogue (DV/2 columns per half)
        // y rows are staged from smem offset 0 (the spent Q tile, then K slot 0)
        // with the tensor map's 128-byte swizzle, 64 columns per 16 KB box, and
        // written by one TMA store per box; rows past T are clipped by the map.
        // Every MMA has completed once o_done has, so nothing reads there.
        static_assert(DV / 64 * 16384 <= C::OFF_V, "y staging fits in front of the V slots");
        if (ok && !has_l2) ok = exchange_stats();
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&B.o_done, 0));
        if (ok) {
            tc_fence_after();
            const float m0 = B.xm[0][r], m1 = B.xm[1][r];
            const float M = fmaxf(m0, m1);
            const float f0 = ex2(m0 - M), f1 = ex2(m1 - M);
            const float lsum = B.xl[0][r] * f0 + B.xl[1][r] * f1;
            const float inv_l = lsum > 0.f ? 1.0f / lsum : 0.f;
            const float w0 = f0 * inv_l, w1 = f1 * inv_l;
            const float cq = l2 ? sg * powf(lam[h], (float)(r + 1)) : 0.f;  // sigmoid(g) lambda^(i+1)
#pragma unroll 1
            for (int cc = 0; cc < DV / 2; cc += 16) {
                const int col = half * (DV / 2) + cc;
                float o0[16], o1[16], qa[16];
                tmem_ld16(tm + lrow + C::COL_O0 + col, o0);
                tmem_ld16(tm + lrow + C::COL_O1 + col, o1);
                tmem_ld16(tm + lrow + col, qa);
                tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float v2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int e = 2 * i + u;
                        v2[u] = fmaf(o0[e], w0, fmaf(o1[e], w1, l2 ? cq * qa[e] : 0.f));
                    }
                    pk[i] = pack_bf16(v2[0], v2[1]);
                }
                const uint32_t box = sQ + (uint32_t)(col / 64) * 16384u, c16 = (uint32_t)((col % 64) / 8);
                st_shared_v4(box + sw128_off(r, c16), pk[0], pk[1], pk[2], pk[3]);
                st_shared_v4(box + sw128_off(r, c16 + 1), pk[4], pk[5], pk[6], pk[7]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.y_ready);
            if (tid == 0) {
                if (mbar_wait(&B.y_ready, 0)) {
#pragma unroll
                    for (int b = 0; b < DV / 64; ++b) tma_store_3d(&my, sm + b * 16384, 64 * b, t0, bh);
                    tma_store_commit();
                    tma_store_wait_read();
                } else {
                    ok = false;
                }
            }
        }
        if (!ok && lane == 0) atomicOr(status, kStFwdSoftmax);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) tmem_dealloc(tm, 512);
}

// --------------------------------------------------------------------- fused forward, half a row per thread
// Variant for d_k = d_v = 64 sized so that two CTAs share an SM (256 TMEM
// columns, ~99 KB of shared memory): while one CTA waits on its loads, MMAs
// or prologue/epilogue, the other runs its softmax.  288 threads: warp w < 8
// owns rows 32 (w % 4) .. +31 (its TMEM lane quarter) and keys 64 (w / 4) ..
// +63 of every tile -- half a row per thread; the two halves of a row agree
// on the row maximum (and, in the shifted chunk, on the row sum) through
// shared memory.  One thread of warp 8 issues the TMA loads and the MMAs.
// TMEM: S [0,128), O [128, 128+DV), P [128+DV, 128+DV+64) -- P is written
// by the softmax threads with tcgen05.st as packed bf16 and is the A operand
// of O += P V, so it never touches shared memory.
//
// The L2 part of the block (keys l <= i of the shifted chunk, then the state)
// has its own accumulators.  The shifted chunk is processed last: its
// softmax keys (l > i) go to P as usual, and its decayed scores
// eta lambda^(i-l) <q_i, k'_l> go to P2 over the spent S columns [0,64);
// O2 = P2 V' accumulates into S columns [64,128).  After that q A_j^loc lands
// in S columns [0,DV) and q A_{gL} in the P columns, and the epilogue forms
// y = O / L + sigmoid(g) (O2 + lambda^(i+1) (q A_j^loc + c q A_{gL})).
//
// Stages: 3 K slots (the last also takes A_j^loc and A_{gL}) and 2 V slots.
// The issuing thread learns that a slot is free from the softmax side: S(n)
// has been read once its S columns are released, and P V(n-1) has completed
// once P(n) has been published (P(n) is written only after it).
template <int DK, int DV>
struct FwdRow {
    static constexpr uint32_t QBYTES = kBlk * DK * 2;
    static constexpr uint32_t KBYTES = kBlk * DK * 2;  // also holds A_j^loc
    static constexpr uint32_t VBYTES = kBlk * DV * 2;  // also holds the segment carry
    static constexpr int NSK = 3, NSV = 2;
    static constexpr uint32_t OFF_K = QBYTES;
    static constexpr uint32_t OFF_V = OFF_K + NSK * KBYTES;
    static constexpr uint32_t OFF_BARS = OFF_V + NSV * VBYTES;
    static_assert(2 * DK * DV * 2 <= KBYTES, "A_j^loc and the carry share a K slot");
    static constexpr uint32_t COL_O = 128, COL_P = 128 + DV;
    static constexpr uint32_t TCOLS = 256;
    static_assert(COL_P + kBlk / 2 <= TCOLS, "TMEM budget");
    static_assert(DV == 64, "one 32-column half of O per softmax thread");
    static constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t ID_PV = idesc_bf16_f32(128, DV, false, true);
};

struct FwdRowBars {
    uint64_t q_full, k_full[3], v_full[2];
    uint64_t s_full, s_empty, p_full, p_empty, pv2_done, o_done, y_ready, drain;
    uint64_t xchg[4];      // per lane quarter: the two halves of its rows meet here
    uint32_t tbase;
    float cA;              // A_j = A_j^loc + cA A_{gL}: lambda^(C (j - gL))
    float pwz[32 + kBlk];  // [32 + d] = eta lambda^d for d >= 0; 0 for d < 0
    float lpow[kBlk + 1];  // lambda^d
    float xbuf[2][2][kBlk];  // [exchange parity][half][row]
};

template <int DK, int DV>
__global__ void __launch_bounds__(288, 2)
tc_fwd_row_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap ma,
                  const __grid_constant__ CUtensorMap mc, const __grid_constant__ CUtensorMap my, int T, int W,
                  int H, int nch, int nseg, int L, int l2,
                  const float *__restrict__ lam, const float *__restrict__ eta,
                  const float *__restrict__ gate, float scale, __nv_bfloat16 *__restrict__ y,
              unsigned int *__restrict__ status) {
    using C = FwdRow<DK, DV>;
    constexpr int NSK = C::NSK, NSV = C::NSV;
    extern __shared__ __align__(1024) unsigned char sm[];
    FwdRowBars &B = *reinterpret_cast<FwdRowBars *>(sm + C::OFF_BARS);
    if ((smem_u32(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStFwdAlign);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Head-major grid in descending query-block order: the late blocks of
    // every head run first, and the early ones, which have no L2 part and
    // fewer key tiles, fill the last wave.
    const int jq = (int)gridDim.y - 1 - (int)blockIdx.y, bh = blockIdx.x, h = bh % H;
    const int seg = jq / L;
    const int t0 = jq * kBlk;
    const int kt0 = t0 - W;
    const int nt_total = (W + kBlk - 1) / kBlk + 1;
    const int j_first = (-kt0 - (kBlk - 1) > 0) ? (-kt0) / kBlk : 0;
    const int ntiles = nt_total - j_first;
    // l2 == 0: window only (no L2 part, no state loads, no q A term).
    const bool has_l2 = l2 && (j_first == 0);
    // Key tile j covers keys kt0 + 128 j ..; with an L2 part the tiles run
    // 1, 2, .., nt-1 and the shifted chunk (j = 0) comes last.
    auto tile_j = [&](int n) { return has_l2 ? (n + 1 < ntiles ? n + 1 : 0) : j_first + n; };

    const uint32_t sQ = smem_u32(sm);
    const uint32_t sK0 = sQ + C::OFF_K;
    const uint32_t sV0 = sQ + C::OFF_V;
    const int nkload = ntiles + (has_l2 ? 1 : 0);  // K slot loads; the last is A_j^loc + carry
    auto load_k = [&](int i) {
        unsigned char *kd = sm + C::OFF_K + (i % NSK) * C::KBYTES;
        uint64_t *bar = &B.k_full[i % NSK];
        if (i < ntiles) {
            const int kt = kt0 + kBlk * tile_j(i);
            mbar_expect_tx(bar, C::KBYTES);
#pragma unroll
            for (int b = 0; b < DK / 64; ++b) tma_load_3d(kd + b * 16384, &mk, bar, 64 * b, kt, bh);
        } else {
            // A_j^loc and the carry come from the state and carry kernels, which
            // may still be running: wait for them (only this thread, only here)
            pdl_wait_primary();
            mbar_expect_tx(bar, 2 * DK * DV * 2);
#pragma unroll
            for (int b = 0; b < DV / 64; ++b) {
                tma_load_3d(kd + b * (DK * 128), &ma, bar, 64 * b, 0, bh * nch + jq);
                tma_load_3d(kd + DK * DV * 2 + b * (DK * 128), &mc, bar, 64 * b, 0, bh * nseg + seg);
            }
        }
    };
    auto load_v = [&](int i) {
        unsigned char *vd = sm + C::OFF_V + (i % NSV) * C::VBYTES;
        uint64_t *bar = &B.v_full[i % NSV];
        mbar_expect_tx(bar, C::VBYTES);
#pragma unroll
        for (int b = 0; b < DV / 64; ++b) tma_load_3d(vd + b * 16384, &mv, bar, 64 * b, kt0 + kBlk * tile_j(i), bh);
    };
    if (warp == 8 && lane == 0) {  // barriers, then the first loads, before the CTA-wide sync
        mbar_init(&B.q_full, 1);
        for (int s = 0; s < NSK; ++s) mbar_init(&B.k_full[s], 1);
        for (int s = 0; s < NSV; ++s) mbar_init(&B.v_full[s], 1);
        mbar_init(&B.s_full, 1);
        mbar_init(&B.s_empty, 8);
        mbar_init(&B.p_full, 8);
        mbar_init(&B.p_empty, 1);
        mbar_init(&B.pv2_done, 1);
        mbar_init(&B.o_done, 1);
        mbar_init(&B.y_ready, 8);
        mbar_init(&B.drain, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&B.xchg[i], 2);
        mbar_fence_init();
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&my);
        mbar_expect_tx(&B.q_full, C::QBYTES);
#pragma unroll
        for (int b = 0; b < DK / 64; ++b) tma_load_3d(sm + b * 16384, &mq, &B.q_full, 64 * b, t0, bh);
        for (int i = 0; i < NSK && i < nkload; ++i) load_k(i);
        for (int i = 0; i < NSV && i < ntiles; ++i) load_v(i);
    }
    __syncwarp();
    if (warp == 8) tmem_alloc(&B.tbase, C::TCOLS);
    if (tid < 32) B.pwz[tid] = 0.f;
    if (l2 && tid <= kBlk) {
        const float lh = lam[h];
        const float pw = powf(lh, (float)tid);
        B.lpow[tid] = pw;
        if (tid < kBlk) B.pwz[32 + tid] = eta[h] * pw;
        if (tid == kBlk) B.cA = powf(lh, (float)(kBlk * (jq - seg * L)));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;

    if (warp == 8) {
        // ------------------------------------------------ TMA loads and MMAs (one thread)
        if (lane == 0) {
            // descriptor halves: K-major Q / K tiles (k-step +32 B), MN-major V and A tiles (k-step +2048 B)
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t q_lo = sdesc_lo(sQ, 16);
            const uint32_t k_lo = sdesc_lo(sK0, 16);
            const uint32_t v_lo = sdesc_lo(sV0, 16384);
            const uint32_t p_tm = tm + C::COL_P, o_tm = tm + C::COL_O;
            bool ok = mbar_wait(&B.q_full, 0);
            auto pv = [&](int n) -> bool {  // O += P V of tile n, P from TMEM
                if (!mbar_wait(&B.v_full[n % NSV], (n / NSV) & 1)) return false;
                if (!mbar_wait(&B.p_full, n & 1)) return false;
                // P(n) was written after P V(n-1) completed: V slot of tile n+1 is free
                if (n >= 1 && n + 1 < ntiles) load_v(n + 1);
                tc_fence_after();
                const uint32_t vb = v_lo + (uint32_t)(n % NSV) * (C::VBYTES >> 4);
#pragma unroll
                for (int k = 0; k < kBlk / 16; ++k)
                    mma_ts_h(o_tm, p_tm + 8 * k, vb + k * (2048 >> 4), HI, C::ID_PV, (n > 0 || k > 0) ? 1u : 0u);
                mma_commit(&B.p_empty);
                return true;
            };
            for (int n = 0; n < ntiles && ok; ++n) {
                ok = mbar_wait(&B.k_full[n % NSK], (n / NSK) & 1);
                if (ok && n >= 1) {
                    ok = mbar_wait(&B.s_empty, (n - 1) & 1);
                    // S(n-1) has been read, so its K slot is free
                    if (ok && n - 1 + NSK < nkload) load_k(n - 1 + NSK);
                }
                if (!ok) break;
                tc_fence_after();
                const uint32_t kb = k_lo + (uint32_t)(n % NSK) * (C::KBYTES >> 4);
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t off = (uint32_t)((k >> 2) * (16384 >> 4) + (k & 3) * 2);
                    mma_ss_h(tm, q_lo + off, HI, kb + off, HI, C::ID_S, k > 0 ? 1u : 0u);
                }
                mma_commit(&B.s_full);
                if (n >= 1) ok = pv(n - 1);
            }
            if (ok) ok = pv(ntiles - 1);
            if (ok && has_l2) {
                // O2 = P2 V' of the shifted chunk (the last tile): P2 over S columns [0,64),
                // O2 into S columns [64,128); P2 was published with the tile's P.
                const uint32_t vb = v_lo + (uint32_t)((ntiles - 1) % NSV) * (C::VBYTES >> 4);
#pragma unroll
                for (int k = 0; k < kBlk / 16; ++k)
                    mma_ts_h(tm + 64, tm + 8 * k, vb + k * (2048 >> 4), HI, C::ID_PV, k > 0 ? 1u : 0u);
                mma_commit(&B.pv2_done);
                // then q A_j^loc into S columns [0,DV) and q A_{gL} into the P columns
                const int i = ntiles;
                ok = mbar_wait(&B.k_full[i % NSK], (i / NSK) & 1);
                if (ok) ok = mbar_wait(&B.pv2_done, 0);
                if (ok) {
                    tc_fence_after();
                    const uint32_t a_lo = sdesc_lo(sK0 + (i % NSK) * C::KBYTES, DK * 128);
#pragma unroll
                    for (int k = 0; k < DK / 16; ++k) {
                        const uint32_t qo = (uint32_t)((k >> 2) * (16384 >> 4) + (k & 3) * 2);
                        mma_ss_h(tm, q_lo + qo, HI, a_lo + k * (2048 >> 4), HI, C::ID_PV, k > 0 ? 1u : 0u);
                    }
#pragma unroll
                    for (int k = 0; k < DK / 16; ++k) {
                        const uint32_t qo = (uint32_t)((k >> 2) * (16384 >> 4) + (k & 3) * 2);
                        mma_ss_h(p_tm, q_lo + qo, HI, a_lo + ((DK * DV * 2) >> 4) + k * (2048 >> 4), HI, C::ID_PV,
                                 k > 0 ? 1u : 0u);
                    }
                }
            }
            if (ok) mma_commit(&B.o_done);
            if (!ok) atomicOr(status, kStFwdMma);
            mma_commit(&B.drain);
            mbar_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax / epilogue (row r, key half hf)
        const int q4 = warp & 3, hf = warp >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        const float sc = scale * kLog2e;
        const float sig = l2 ? 1.0f / (1.0f + expf(-gate[h])) : 0.f;
        float m = kNegBig, l = 0.f;  // l: this half's share of the row sum
        uint32_t xn = 0;             // exchanges so far (both halves count alike)
        float Lrow = 0.f;  // the row's softmax sum over both halves, once known
        bool ok = true;
        // Hand x to the other half of the row and return its value (NaN if
        // the other half never arrives; ok is then cleared).
        auto exchange = [&](float x) -> float {
            const int p = xn & 1;
            B.xbuf[p][hf][r] = x;
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.xchg[q4]);
            const bool w = __all_sync(0xffffffffu, mbar_wait(&B.xchg[q4], p));
            ++xn;
            if (!w) {
                ok = false;
                return __int_as_float(0x7fffffff);
            }
            return B.xbuf[p][hf ^ 1][r];
        };
        for (int n = 0; n < ntiles && ok; ++n) {
            const int j = tile_j(n);
            const int kt = kt0 + kBlk * j;
            const bool l2 = has_l2 && j == 0;
            // softmax keys of this row in the tile: lo..hi (window t-W < pos <= t, pos >= 0)
            const int lo = max(max(0, -kt), r + 1 - kBlk * j);
            const int hi = min(kBlk - 1, r + W - kBlk * j);
            const int lo_min = __reduce_min_sync(0xffffffffu, lo), lo_max = __reduce_max_sync(0xffffffffu, lo);
            const int hi_min = __reduce_min_sync(0xffffffffu, hi), hi_max = __reduce_max_sync(0xffffffffu, hi);
            // warp-uniform class of the 32 keys of chunk g: 0 none, 1 all, 2 per-row span
            auto cls = [&](int g) -> int {
                const int a = 32 * g, b = a + 31;
                if (b < lo_min || a > hi_max || lo_min > hi_max) return 0;
                if (a >= lo_max && b <= hi_min) return 1;
                return 2;
            };
            ok = __all_sync(0xffffffffu, mbar_wait(&B.s_full, n & 1));
            if (!ok) break;
            tc_fence_after();
            float va[32], vb[32];  // keys 64 hf + 0..31 and 64 hf + 32..63
            tmem_ld32(tm + lrow + 64 * hf, va);
            tmem_ld32(tm + lrow + 64 * hf + 32, vb);
            tmem_wait_ld();
            auto release_s = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.s_empty);
            };
            if (!l2) release_s();  // the shifted chunk re-reads S after its row-sum exchange

            // row maximum over the softmax keys, shared by the two halves
            float mx = -INFINITY;
            auto chunk_max = [&](const float(&v)[32], int g) {
                const int c = cls(g);
                if (c == 1) {
                    float a0 = fmax3f(v[0], v[1], v[2]), a1 = fmax3f(v[8], v[9], v[10]);
                    float a2 = fmax3f(v[16], v[17], v[18]), a3 = fmax3f(v[24], v[25], v[26]);
#pragma unroll
                    for (int e = 3; e < 8; e += 2) {
                        const int e1 = e + 1 < 8 ? e + 1 : e;
                        a0 = fmax3f(a0, v[e], v[e1]);
                        a1 = fmax3f(a1, v[8 + e], v[8 + e1]);
                        a2 = fmax3f(a2, v[16 + e], v[16 + e1]);
                        a3 = fmax3f(a3, v[24 + e], v[24 + e1]);
                    }
                    mx = fmax3f(mx, fmaxf(a0, a1), fmaxf(a2, a3));
                } else if (c == 2) {
                    const uint32_t bits = span_bits(lo - 32 * g, hi - 32 * g);
                    float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        a0 = fmaxf(a0, ((bits >> e) & 1u) ? v[e] : -INFINITY);
                        a1 = fmaxf(a1, ((bits >> (e + 1)) & 1u) ? v[e + 1] : -INFINITY);
                    }
                    mx = fmax3f(mx, a0, a1);
                }
            };
            chunk_max(va, 2 * hf);
            chunk_max(vb, 2 * hf + 1);
            mx = fmaxf(mx, exchange(mx));
            if (!ok) break;
            const float mxs = mx * sc;
            const bool grow = mxs > m + kRescale;
            // P may be written (and O rescaled) once the previous P V has completed.
            ok = __all_sync(0xffffffffu, n == 0 || mbar_wait(&B.p_empty, (n - 1) & 1));
            if (!ok) break;
            const float fO = grow ? ex2(m - mxs) : 1.f;  // O and l rescale when the maximum grows
            const bool rescale = __any_sync(0xffffffffu, grow) && n > 0;
            if (grow) {
                l *= fO;
                m = mxs;
            }

            const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m, -m);
            float2 acc[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) acc[u] = make_float2(0.f, 0.f);
            auto tsum = [&]() {
                return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
            };
            // softmax probabilities of chunk g, packed into P
            auto chunk_soft = [&](const float(&v)[32], int g) {
                uint32_t pk[16];
                const int c = cls(g);
                if (c == 1) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float2 x = fma2(make_float2(v[e], v[e + 1]), sc2, nm2);
                        x.x = ex2(x.x);
                        x.y = ex2(x.y);
                        acc[(e >> 1) & 1] = add2(acc[(e >> 1) & 1], x);
                        pk[e >> 1] = pack_bf16(x.x, x.y);
                    }
                } else if (c == 2) {
                    const uint32_t bits = span_bits(lo - 32 * g, hi - 32 * g);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float2 x = fma2(make_float2(v[e], v[e + 1]), sc2, nm2);
                        // masked keys select -inf (2^-inf = 0): the exponential itself is
                        // unconditional, which keeps the warp on one path
                        x.x = ex2(((bits >> e) & 1u) ? x.x : -INFINITY);
                        x.y = ex2(((bits >> (e + 1)) & 1u) ? x.y : -INFINITY);
                        acc[(e >> 1) & 1] = add2(acc[(e >> 1) & 1], x);
                        pk[e >> 1] = pack_bf16(x.x, x.y);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = 0u;
                }
                tmem_st16(tm + lrow + C::COL_P + 16 * g, pk);
            };
            if (!l2) {
                chunk_soft(vb, 2 * hf + 1);
                chunk_soft(va, 2 * hf);
            } else {
                // Shifted chunk: softmax keys (l > r) go to P as usual; the decayed L2
                // scores eta lambda^(r-l) <q_r,k'_l> of keys l <= r go to P2, written over
                // this tile's S columns [0,64) (both halves have read S: the max exchange
                // came after the loads).
                auto l2_chunk = [&](const float(&v)[32], int g) {
                    if (g > q4) {  // no key l <= r in this chunk
                        chunk_soft(v, g);
                        const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                        tmem_st8(tm + lrow + 16 * g, z);
                        tmem_st8(tm + lrow + 16 * g + 8, z);
                        return;
                    }
                    const uint32_t bits = g == q4 ? span_bits(lo - 32 * g, hi - 32 * g) : 0u;
                    const float *pw = &B.pwz[32 + r - 32 * g];  // pw[-e] = eta lambda^(r-32g-e), 0 past r
#pragma unroll
                    for (int e0 = 0; e0 < 32; e0 += 16) {
                        uint32_t ps[8], p2[8];
#pragma unroll
                        for (int e = e0; e < e0 + 16; e += 2) {
                            float2 x = fma2(make_float2(v[e], v[e + 1]), sc2, nm2);
                            x.x = ex2(((bits >> e) & 1u) ? x.x : -INFINITY);
                            x.y = ex2(((bits >> (e + 1)) & 1u) ? x.y : -INFINITY);
                            acc[(e >> 1) & 1] = add2(acc[(e >> 1) & 1], x);
                            ps[(e - e0) >> 1] = pack_bf16(x.x, x.y);
                            p2[(e - e0) >> 1] = pack_bf16(v[e] * pw[-e], v[e + 1] * pw[-e - 1]);
                        }
                        tmem_st8(tm + lrow + C::COL_P + 16 * g + e0 / 2, ps);
                        tmem_st8(tm + lrow + 16 * g + e0 / 2, p2);
                    }
                };
                l2_chunk(vb, 2 * hf + 1);
                l2_chunk(va, 2 * hf);
            }
            if (rescale) {  // this half rescales O columns 32 hf .. +31 (P V(n-1) is complete)
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < 32; cc += 16) {
                    float o[16];
                    tmem_ld16(tm + lrow + C::COL_O + 32 * hf + cc, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] *= fO;
                    tmem_st16(tm + lrow + C::COL_O + 32 * hf + cc, reinterpret_cast<const uint32_t(&)[16]>(o));
                }
            }
            tmem_wait_st();
            l += tsum();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.p_full);
        }
        // ------------------------------------------------ epilogue: y = O / L + sigmoid(g) lambda^(i+1) q A_j
        if (ok) Lrow = l + exchange(l);
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&B.o_done, 0));
        if (ok) {
            tc_fence_after();
            const float inv_l = Lrow > 0.f ? 1.0f / Lrow : 0.f;
            // sigmoid(g) lambda^(i+1), and c with A_j = A_j^loc + c A_{gL}
            const float cq = has_l2 ? sig * B.lpow[r + 1] : 0.f;
            const float cA = B.cA;
            // y row r, columns 32 hf .. +31, staged in the (spent) Q tile with the
            // tensor map's 128-byte swizzle, then one TMA store per CTA
#pragma unroll 1
            for (int cc = 0; cc < 32; cc += 16) {
                float o[16], qa[16], qc[16], o2[16];
                tmem_ld16(tm + lrow + C::COL_O + 32 * hf + cc, o);
                if (has_l2) {  // m = O2 + lambda^(i+1) q (A_j^loc + c A_{gL}), times sigmoid(g)
                    tmem_ld16(tm + lrow + 32 * hf + cc, qa);
                    tmem_ld16(tm + lrow + C::COL_P + 32 * hf + cc, qc);
                    tmem_ld16(tm + lrow + 64 + 32 * hf + cc, o2);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) qa[e] = fmaf(sig, o2[e], cq * fmaf(cA, qc[e], qa[e]));
                } else {
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) qa[e] = 0.f;
                }
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    pk[i] = pack_bf16(fmaf(o[2 * i], inv_l, qa[2 * i]), fmaf(o[2 * i + 1], inv_l, qa[2 * i + 1]));
                const uint32_t c16 = (uint32_t)((32 * hf + cc) / 8);  // 16-byte chunk of the 128-byte row
                st_shared_v4(sQ + sw128_off(r, c16), pk[0], pk[1], pk[2], pk[3]);
                st_shared_v4(sQ + sw128_off(r, c16 + 1), pk[4], pk[5], pk[6], pk[7]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.y_ready);
            if (tid == 0) {
                if (mbar_wait(&B.y_ready, 0)) {
                    tma_store_3d(&my, sm, 0, t0, bh);
                    tma_store_commit();
                    tma_store_wait_read();
                } else {
                    ok = false;
                }
            }
        }
        if (!ok && lane == 0) atomicOr(status, kStFwdSoftmax);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) tmem_dealloc(tm, C::TCOLS);
}

struct Ws {
    __nv_bfloat16 *Aloc, *Cbf;
    float *Lfin;
    unsigned int *cta_status;  // one word per state CTA
};

size_t n_state_ctas(int BH, const Segments &g, int dv) { return (size_t)(dv / 64) * g.nseg * BH; }

Ws carve(void *ws, int BH, const Segments &g, int dk, int dv) {
    char *p = (char *)ws;
    Ws w;
    w.Aloc = (__nv_bfloat16 *)p;
    p += align_up(2 * (size_t)BH * g.nch * dk * dv, 1024);
    w.Cbf = (__nv_bfloat16 *)p;
    p += align_up(2 * (size_t)BH * g.nseg * dk * dv, 1024);
    w.Lfin = (float *)p;
    p += align_up(4 * (size_t)BH * g.nseg * dk * dv, 1024);
    w.cta_status = (unsigned int *)p;
    return w;
}

size_t ws_bytes(int BH, const Segments &g, int dk, int dv) {
    return align_up(2 * (size_t)BH * g.nch * dk * dv, 1024) + align_up(2 * (size_t)BH * g.nseg * dk * dv, 1024) +
           align_up(4 * (size_t)BH * g.nseg * dk * dv, 1024) + align_up(4 * n_state_ctas(BH, g, dv), 1024);
}

int num_sms() { return device_sm_count(); }

// Status words of the call (status[0..3], the head of its workspace): with the
// L2 part, word 0 receives the state CTAs' bits from the carry kernel and
// word 1 the forward kernel's, and the state kernel zeroes words 1..3 first,
// so the call needs no separate clear.  Window only (no state kernels), the
// caller zeroes the words before the launch.
template <int DK, int DV>
int run(const void *q, const void *k, const void *v, int B_, int H, int T, int W, const float *lam,
        const float *eta, const float *gate, float scale, void *y, float *A_final, void *ws,
        unsigned int *status, cudaStream_t st, bool l2) {
    const int BH = B_ * H;
    const Segments g = segments(BH, T, DK, DV, num_sms());
    if (DK == 64 && DV == 64 && g.nch > 65535) {  // query blocks are the grid's y extent
        set_error("tc_layer_forward: T=%d above %d tokens on this path", T, 65535 * kBlk);
        return OPAM_ERR_UNSUPPORTED;
    }
    CUtensorMap mq, mk, mv, ma{}, mc{};  // ma, mc stay unused (zero) without the L2 part
    int rc;
    if ((rc = make_tmap_bf16_3d(&mq, q, DK, T, BH, kBlk))) return rc;
    if ((rc = make_tmap_bf16_3d(&mk, k, DK, T, BH, kBlk))) return rc;
    if ((rc = make_tmap_bf16_3d(&mv, v, DV, T, BH, kBlk))) return rc;
    // The carry kernel and the d = 64 forward kernel are programmatic dependents:
    // each may start before its predecessor finishes and waits (griddepcontrol)
    // only where it reads that predecessor's output.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    if (l2) {
        const Ws w = carve(ws, BH, g, DK, DV);
        if ((rc = make_tmap_bf16_3d(&ma, w.Aloc, DV, DK, (uint64_t)BH * g.nch, DK))) return rc;
        if ((rc = make_tmap_bf16_3d(&mc, w.Cbf, DV, DK, (uint64_t)BH * g.nseg, DK))) return rc;
        {
            using SC = StateCfg<DK>;
            auto kern = tc_l2_state_kernel<DK, DV>;
            const uint32_t ssm = (DK == 64 && DV == 64) ? (SC::SMEM > kStateSoloSmem ? SC::SMEM : kStateSoloSmem)
                                                        : SC::SMEM;
            if (int rc_ = set_smem_limit((const void *)kern, (int)ssm, "tc_l2_state smem attribute")) return rc_;
            kern<<<dim3(DV / 64, g.nseg, BH), 192, ssm, st>>>(mk, mv, T, W, H, lam, eta, g.nch, g.L, w.Aloc,
                                                                  w.Lfin, w.cta_status, status);
            if ((rc = launched("tc_l2_state"))) return rc;
        }
        {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(ceil_div(DK * DV / 4, 2 * 128), BH);  // two groups of 4 per thread
            cfg.blockDim = dim3(128);
            cfg.stream = st;
            cfg.attrs = pdl;
            cfg.numAttrs = 1;
            cudaError_t e = cudaLaunchKernelEx(&cfg, tc_l2_carry_kernel, (const float *)w.Lfin, g.nseg, g.L, T,
                                               DK * DV, H, lam, w.Cbf, A_final, (const unsigned int *)w.cta_status,
                                               (int)n_state_ctas(BH, g, DV), status);
            if (e != cudaSuccess) return cuda_fail(e, "tc_l2_carry launch");
            if ((rc = launched("tc_l2_carry"))) return rc;
        }
    }
    if constexpr (DK == 64 && DV == 64) {
        using Cfg = FwdRow<DK, DV>;
        auto kern = tc_fwd_row_kernel<DK, DV>;
        static_assert(Cfg::OFF_BARS + sizeof(FwdRowBars) <= 228 * 1024 / 2 - 1024, "two CTAs per SM");
        const int smem = (int)(Cfg::OFF_BARS + sizeof(FwdRowBars));
        if (int rc_ = set_smem_limit((const void *)kern, smem, "tc_fwd_row smem attribute")) return rc_;
        prof_begin(st);
        CUtensorMap my;
        if ((rc = make_tmap_bf16_3d(&my, y, DV, T, BH, kBlk))) return rc;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(BH, g.nch);
        cfg.blockDim = dim3(288);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = st;
        cfg.attrs = pdl;  // window only: no state kernels, so ordinary stream order
        cfg.numAttrs = l2 ? 1 : 0;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, ma, mc, my, T, W, H, g.nch, g.nseg, g.L,
                                           (int)l2, lam, eta, gate, scale, (__nv_bfloat16 *)y, status + 1);
        rc = e != cudaSuccess ? cuda_fail(e, "tc_fwd_row launch") : launched("tc_fwd_row");
        prof_end(st);
        return rc;
    } else {
        using Cfg = Fwd<DK, DV>;
        auto kern = tc_fwd_kernel<DK, DV>;
        static_assert(sizeof(FwdBars) <= 3072, "barriers block");
        const int smem = (int)(Cfg::OFF_BARS + sizeof(FwdBars));
        if (int rc_ = set_smem_limit((const void *)kern, smem, "tc_fwd smem attribute")) return rc_;
        CUtensorMap my;
        if ((rc = make_tmap_bf16_3d(&my, y, DV, T, BH, kBlk))) return rc;
        prof_begin(st);
        kern<<<dim3(g.nch, BH), 352, smem, st>>>(mq, mk, mv, ma, mc, my, T, W, H, g.nch, g.nseg, g.L, (int)l2,
                                                  lam, eta, gate, scale, num_sms(), status + 1);
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
    return ws_bytes(BH, segments(BH, T, dk, dv, num_sms()), dk, dv);
}

int tc_prefill_tcgen05(const void *q, const void *k, const void *v, int B, int H, int T, int dk,
                       int dv, int W, const float *lam, const float *eta, const float *gate,
                       float scale, void *y, float *A_final, void *ws, unsigned int *status,
                       cudaStream_t s, bool l2) {
    if (dk == 64 && dv == 64) return run<64, 64>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, status, s, l2);
    if (dk == 64 && dv == 128)
        return run<64, 128>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, status, s, l2);
    if (dk == 128 && dv == 64)
        return run<128, 64>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, status, s, l2);
    if (dk == 128 && dv == 128)
        return run<128, 128>(q, k, v, B, H, T, W, lam, eta, gate, scale, y, A_final, ws, status, s, l2);
    set_error("tensor-core prefill: d_k=%d d_v=%d unsupported", dk, dv);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace opam
