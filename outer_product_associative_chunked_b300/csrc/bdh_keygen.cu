// BDH key generation fused with support compaction (tcgen05 + TMA).
//
// ainews.random.gg, BDH memory-architecture post: the wide, sparse,
// non-negative activations of queries and keys come from a low-rank
// factorisation followed by ReLU thresholding.  For one head h and a token's
// R-dimensional input x,
//     a[n] = max(0, sum_r x[r] U_h[r][n] - theta),   n < N,
// with one U_h shared by queries and keys.  This kernel computes a tile of
// x U_h on the tensor cores and, in the epilogue, keeps only the entries
// above theta as the row's ascending (index, value) support list -- the
// input format of the sparse attention kernels -- so the dense N-wide rows
// are never written to or read from memory.
//
// One CTA per (128 tokens, batch x head, queries or keys), 320 threads:
//   warp 8 (lane 0)  TMA: the 128 x R x tile once, then U_h in column tiles of
//                    kNT = 128 (R x 128, MN-major, double-buffered);
//   warp 9 (lane 0)  tcgen05.mma with K = R into one of two TMEM accumulators
//                    (256 columns), so the epilogue of tile i overlaps the
//                    MMAs of tile i + 1;
//   warps 0-7        epilogue: warps w and w + 4 share TMEM lane quarter w and
//                    take 64 columns each; a thread first counts the entries
//                    above theta in its 64 values, the two halves exchange
//                    counts, then each writes its entries in place
//                    (coordinate lists: through a shared-memory stage).
// Two output forms:
//   row lists (ROWS): D = x U (M = tokens), thread = token row: a = acc -
//     theta; if a > 0 append (n, a) to the row's list (the per-row format the
//     recurrent attention reads);
//   coordinate lists (!ROWS): D = U^T x^T (M = coordinates, the U tile as the
//     MN-major A operand), thread = coordinate: it holds its 128 token values,
//     so after a scan of the tile's counts over the 128 threads it writes its
//     (token, value) entries in ascending token order -- the 128-token block's
//     coordinate-major lists that the pairwise attention reads, with no
//     per-row lists in between.
// Operands are bf16 with fp32 accumulation; x rows past T read as zero and
// are not written.  Every wait is bounded; a wait that runs out sets a bit in
// the call's status word and the CTA winds down.
#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {

using namespace sm100;

namespace {

constexpr int kM = 128;   // token rows per CTA
constexpr int kNT = 128;  // columns of U_h per tile
// Coordinate lists: a tile's entries (one contiguous range of the block's
// lists) are staged in shared memory as 8-byte (value, token) pairs when at
// most this many, then written out with coalesced stores.
constexpr int kStage = 3584;

enum : unsigned int {
    kStKgProducer = kStatusKeygen << 0,
    kStKgMma = kStatusKeygen << 1,
    kStKgEpi = kStatusKeygen << 2,
};

template <int R>
struct KgCfg {
    static constexpr uint32_t ABYTES = kM * R * 2;      // x tile, R/64 K-major blocks of 16 KB
    static constexpr uint32_t BBYTES = R * kNT * 2;     // U tile, two MN-major blocks of R x 64
    static constexpr uint32_t OFF_B = ABYTES;
    static constexpr uint32_t OFF_S = ABYTES + 2 * BBYTES;  // the stage: kStage (value, token) pairs
    static constexpr uint32_t SMEM = OFF_S + kStage * 8 + 1024;  // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct KgBars {
    uint64_t a_full, b_full[2], b_empty[2], acc_full[2], acc_empty[2], drain;
    uint32_t tbase;
};

// Named barrier 1 over the eight epilogue warps (256 threads); the second form
// also returns whether `ok` holds in every one of them, so that all eight
// leave their loop together.
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// Appends (x, t) at shared address sa, and advances sa, when x > 0 -- as
// predicated instructions, with no branch per value; then t += 1.
__device__ __forceinline__ void stage_put(uint32_t &sa, uint32_t &t, float x) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.gt.f32 q, %2, 0f00000000;\n\t"
        "@q st.shared.v2.b32 [%0], {%2, %1};\n\t"
        "@q add.u32 %0, %0, 8;\n\t"
        "add.u32 %1, %1, 1;\n\t}"
        : "+r"(sa), "+r"(t)
        : "f"(x)
        : "memory");
}
__device__ __forceinline__ bool epi_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 256, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

template <int R, bool ROWS>
__global__ void __launch_bounds__(320, 1)
bdh_keygen_kernel(const __grid_constant__ CUtensorMap mxk, const __grid_constant__ CUtensorMap mxq,
                  const __grid_constant__ CUtensorMap mu, int T, int H, int N, float theta,
                  int *__restrict__ kidx, float *__restrict__ kval, int *__restrict__ kcnt,
                  int *__restrict__ qidx, float *__restrict__ qval, int *__restrict__ qcnt,
                  int *__restrict__ coff, uint8_t *__restrict__ ct, float *__restrict__ cv,
                  unsigned int *__restrict__ status) {
    using C = KgCfg<R>;
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    __shared__ KgBars B;
    __shared__ int wtot[2][4];
    __shared__ int hcnt[2][2][kM];  // [tile parity][column half][TMEM lane]: entries in that half
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const bool is_q = blockIdx.z == 1;
    const CUtensorMap *mx = is_q ? &mxq : &mxk;
    const int ntile = N / kNT;
    if (warp == 9) tmem_alloc(&B.tbase, 256);
    if (tid == 0) {
        mbar_init(&B.a_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&B.b_full[s], 1);
            mbar_init(&B.b_empty[s], 1);
            mbar_init(&B.acc_full[s], 1);
            mbar_init(&B.acc_empty[s], 8);
        }
        mbar_init(&B.drain, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = B.tbase;
    const uint32_t sA = smem_u32(sm), sB = sA + C::OFF_B;

    if (warp == 8) {
        if (lane == 0) {
            bool ok = true;
            mbar_expect_tx(&B.a_full, C::ABYTES);
#pragma unroll
            for (int b = 0; b < R / 64; ++b) tma_load_3d(sm + b * 16384, mx, &B.a_full, 64 * b, blk * kM, bh);
            int issued = 0;
            for (int i = 0; i < ntile && ok; ++i) {
                const int s = i & 1;
                if (i >= 2) ok = mbar_wait(&B.b_empty[s], ((i >> 1) - 1) & 1);
                if (!ok) break;
                unsigned char *dst = sm + C::OFF_B + s * C::BBYTES;
                mbar_expect_tx(&B.b_full[s], C::BBYTES);
                tma_load_3d(dst, &mu, &B.b_full[s], i * kNT, 0, h);
                tma_load_3d(dst + C::BBYTES / 2, &mu, &B.b_full[s], i * kNT + 64, 0, h);
                ++issued;
            }
            if (!ok) atomicOr(status, kStKgProducer);
            // wait for this thread's copies still in flight before the CTA exits
            bool dok = mbar_wait(&B.a_full, 0);
            for (int i = max(0, issued - 2); i < issued && dok; ++i) dok = mbar_wait(&B.b_full[i & 1], (i >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == 9) {
        if (lane == 0) {
            // ROWS: D = x U, A = x (K-major), B = U (MN-major);
            // otherwise D = U^T x^T, A = U (MN-major), B = x (K-major).
            constexpr uint32_t idesc = ROWS ? idesc_bf16_f32(kM, kNT, false, true) : idesc_bf16_f32(kNT, kM, true, false);
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t x_lo = sdesc_lo(sA, 16);
            // K-major x: 16 k per step, four steps per 64-column block of 16 KB
            auto xofs = [](int k) { return (uint32_t)((k >> 2) * (16384 >> 4) + (k & 3) * 2); };
            bool ok = mbar_wait(&B.a_full, 0);
            for (int i = 0; i < ntile && ok; ++i) {
                const int s = i & 1;
                ok = mbar_wait(&B.b_full[s], (i >> 1) & 1);
                if (ok && i >= 2) ok = mbar_wait(&B.acc_empty[s], ((i >> 1) - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                // MN-major U: 16 contraction rows (2048 B) per step; the two
                // 64-column blocks are R rows x 128 B apart
                const uint32_t u_lo = sdesc_lo(sB + s * C::BBYTES, R * 128);
#pragma unroll
                for (int k = 0; k < R / 16; ++k) {
                    if constexpr (ROWS)
                        mma_ss_h(tm + s * kNT, x_lo + xofs(k), HI, u_lo + k * (2048 >> 4), HI, idesc, k > 0 ? 1u : 0u);
                    else
                        mma_ss_h(tm + s * kNT, u_lo + k * (2048 >> 4), HI, x_lo + xofs(k), HI, idesc, k > 0 ? 1u : 0u);
                }
                mma_commit(&B.acc_full[s]);
                mma_commit(&B.b_empty[s]);
            }
            if (!ok) atomicOr(status, kStKgMma);
            mma_commit(&B.drain);
            mbar_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        // epilogue: TMEM lane r = 32 (warp % 4) + lane, columns [64 hf, 64 hf + 64)
        // of the tile's 128.  ROWS: lane = token row, columns = coordinates;
        // otherwise lane = coordinate, columns = tokens.
        const int qd = warp & 3, hf = warp >> 2, r = qd * 32 + lane;
        const uint32_t tcol = (uint32_t)(qd * 32) << 16;
        const int nlive = min(kM, T - blk * kM);
        const bool row_live = r < nlive;
        const size_t cb = ((size_t)(is_q ? 1 : 0) * gridDim.y + bh) * gridDim.x + blk;  // list block (!ROWS)
        int *off = coff + cb * (size_t)(N + 1);
        uint8_t *et = ct + cb * (size_t)kM * N;
        float *ev = cv + cb * (size_t)kM * N;
        const size_t row = (size_t)bh * T + blk * kM + r;                               // list row (ROWS)
        int *oi = (is_q ? qidx : kidx) + row * (size_t)N;
        float *ov = (is_q ? qval : kval) + row * (size_t)N;
        const uint2 *stage = reinterpret_cast<const uint2 *>(sm + C::OFF_S);
        int base = 0;  // ROWS: entries of row r so far; otherwise entries of the block so far
        bool ok = true;
        for (int i = 0; i < ntile && ok; ++i) {
            const int s = i & 1;
            ok = epi_all(mbar_wait(&B.acc_full[s], (i >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            float a[64];
            tmem_ld32(tm + tcol + s * kNT + 64 * hf, *reinterpret_cast<float(*)[32]>(a));
            tmem_ld32(tm + tcol + s * kNT + 64 * hf + 32, *reinterpret_cast<float(*)[32]>(a + 32));
            tmem_wait_ld();
            // a value counts when it is above theta and its token is in the
            // sequence (tokens past T are dead columns)
            const bool tail = ROWS ? !row_live : nlive < kM;
            auto dead = [&](int c) { return ROWS || 64 * hf + c >= nlive; };
            if (tail) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (dead(c)) a[c] = -INFINITY;
            }
            int n = 0;
#pragma unroll
            for (int c = 0; c < 64; ++c) n += a[c] - theta > 0.f ? 1 : 0;
            hcnt[s][hf][r] = n;
            epi_barrier();
            const int lo = hcnt[s][0][r];
            int p, b0 = base, ttot = 0;  // !ROWS: the tile's range [b0, b0 + ttot)
            if constexpr (ROWS) {
                p = base + (hf ? lo : 0);
                base += lo + hcnt[s][1][r];
            } else {
                // exclusive scan of the coordinates' totals over the 128 lanes
                const int tot = lo + hcnt[s][1][r];
                int incl = tot;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += y;
                }
                if (hf == 0 && lane == 31) wtot[s][qd] = incl;
                epi_barrier();
                int start = base + incl - tot;
                for (int w = 0; w < qd; ++w) start += wtot[s][w];
                if (hf == 0 && OPAM_BOUNDS(i * kNT + r < N, status)) off[i * kNT + r] = start;
                p = start + (hf ? lo : 0);
                ttot = wtot[s][0] + wtot[s][1] + wtot[s][2] + wtot[s][3];
                base += ttot;
            }
            // The values are read from TMEM again, 32 columns at a time (fewer
            // live registers than holding all 64); the accumulator is released
            // after that, which is still well before the MMAs of tile i + 2.
            const bool staged = !ROWS && ttot <= kStage;  // the same in every epilogue thread
            uint32_t sa = smem_u32(stage + (p - b0)), tok = 64 * hf;  // staged: this thread's entries
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {
                float b[32];
                tmem_ld32(tm + tcol + s * kNT + 64 * hf + 32 * h2, b);
                tmem_wait_ld();
                if (tail) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (dead(32 * h2 + c)) b[c] = -INFINITY;
                }
                if (staged) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) stage_put(sa, tok, b[c] - theta);
                } else {
                    const int c0 = i * kNT + 64 * hf + 32 * h2;  // ROWS: first coordinate of these columns
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float x = b[c] - theta;
                        if (x > 0.f) {
                            if constexpr (ROWS) {
                                if (OPAM_BOUNDS(p < N, status)) {
                                    oi[p] = c0 + c;
                                    ov[p] = x;
                                }
                            } else {
                                if (OPAM_BOUNDS(p < kM * N, status)) {
                                    et[p] = (uint8_t)(64 * hf + 32 * h2 + c);
                                    ev[p] = x;
                                }
                            }
                            ++p;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.acc_empty[s]);
            if (staged) {
                epi_barrier();
                for (int j = tid; j < ttot; j += 256) {
                    if (OPAM_BOUNDS(b0 + j < kM * N, status)) {
                        const uint2 e = stage[j];
                        et[b0 + j] = (uint8_t)e.y;
                        ev[b0 + j] = __uint_as_float(e.x);
                    }
                }
            }
        }
        if (!ok && lane == 0) atomicOr(status, kStKgEpi);
        if (ok) {
            if constexpr (ROWS) {
                if (hf == 0 && row_live) (is_q ? qcnt : kcnt)[row] = base;
            } else {
                if (hf == 0 && r == 0) off[N] = base;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) tmem_dealloc(tm, 256);
}

}  // namespace

bool bdh_keygen_supported(int R, int N) { return (R == 64 || R == 128 || R == 256) && N % kNT == 0; }

int bdh_keygen(const void *xq, const void *xk, const void *U, float theta, int B, int H, int T, int R, int N,
               int *kidx, float *kval, int *kcnt, int *qidx, float *qval, int *qcnt, int *coff, uint8_t *ct,
               float *cv, unsigned int *status, cudaStream_t s) {
    const bool rows = coff == nullptr;
    const int BH = B * H;
    CUtensorMap mxk, mxq, mu;
    int rc;
    if ((rc = make_tmap_bf16_3d(&mxk, xk, R, T, BH, kM))) return rc;
    if ((rc = make_tmap_bf16_3d(&mxq, xq, R, T, BH, kM))) return rc;
    if ((rc = make_tmap_bf16_3d(&mu, U, N, R, H, R))) return rc;
    const dim3 grid(ceil_div(T, kM), BH, 2);
    auto go = [&](auto kern, uint32_t smem) -> int {
        if (int rc_ = set_smem_limit((const void *)kern, (int)smem, "bdh_keygen smem attribute")) return rc_;
        kern<<<grid, 320, smem, s>>>(mxk, mxq, mu, T, H, N, theta, kidx, kval, kcnt, qidx, qval, qcnt, coff, ct, cv,
                                     status);
        return launched("bdh_keygen");
    };
    switch (R) {
        case 64: return rows ? go(bdh_keygen_kernel<64, true>, KgCfg<64>::SMEM) : go(bdh_keygen_kernel<64, false>, KgCfg<64>::SMEM);
        case 128: return rows ? go(bdh_keygen_kernel<128, true>, KgCfg<128>::SMEM) : go(bdh_keygen_kernel<128, false>, KgCfg<128>::SMEM);
        case 256: return rows ? go(bdh_keygen_kernel<256, true>, KgCfg<256>::SMEM) : go(bdh_keygen_kernel<256, false>, KgCfg<256>::SMEM);
    }
    set_error("BDH key generation: R=%d not in {64, 128, 256}", R);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace opam
