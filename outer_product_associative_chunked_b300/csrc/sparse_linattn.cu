// BDH-style additive linear attention over wide, sparse, non-negative keys.
//
// ainews.random.gg, BDH memory-architecture post: keys and queries are
// neuron activations in a very wide space (about 5% non-zero after ReLU
// thresholding), the state is the accumulated connectivity and reading it is
// propagation -- a fixed-size hash table whose few buckets a sparse key
// writes.  The write is the Hebbian outer-product sum of mo.ai.kr "Hebbian
// memory MLP" (W = sum_i v_i k_i^T), per token:
//     S_t = S_{t-1} + v_t k_t^T,   o_t = S_t q_t.
//
// Layout: the state is key-major, row j = the d_v values bucket j holds, so a
// sparse key touches whole contiguous rows.  Supports are found on the GPU:
// every dense q / k row is compacted to its ascending (index, value) list.
// Tokens are then processed in chunks of kC: with S the state before the
// chunk,
//     o_t = sum_{j in supp q_t} q_t[j] S[j,:] + sum_{s in chunk, s<=t} <k_s,q_t> v_s
// and afterwards every token of the chunk adds k_s[j] v_s into row j.
//
// Without a start state and without a final state to return, the same output
// is computed in its pairwise form, which never materialises S:
//     o_t = sum_{s <= t} <q_t, k_s> v_s = sum_{s <= t} Z[t][s] v_s.
// Tokens are grouped in blocks of kTB; within a block the supports are
// transposed to coordinate-major lists (csc_build_kernel).  For a pair of
// blocks (tb >= sb), Z[tb][sb] = sum_j q_j-list x k_j-list is accumulated in
// shared memory from the lists of each coordinate j, and Z[tb][sb] V[sb] is
// added into o (pair_tile_kernel).  The state's traffic (every token gathering
// and scattering ~5% of the N rows) is replaced by one pass over the lists.
#include "opam_internal.cuh"
#include "sm100.cuh"

namespace opam {
namespace {

using namespace sm100;

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kTB = 128;  // tokens per block of the pairwise form (token index fits a byte)
constexpr size_t kStateL2Budget = (size_t)64 << 20;  // recurrent form: state bytes kept hot in L2

// One warp per row of a dense [rows][N] matrix: the ascending list of its
// non-zero entries (index, value) and their count.  When N is a multiple of
// 4 the row is read as float4 with eight loads in flight per lane (the dense
// rows are the largest input); a lane's four elements are consecutive, so
// ballots over the four components give every non-zero its position in order.
__device__ __forceinline__ float4 ldg_stream4(const float4 *p) {
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

__global__ void __launch_bounds__(256)
compact_rows_kernel(const float *__restrict__ x, int rows, int N, int *__restrict__ idx,
                    float *__restrict__ val, int *__restrict__ cnt) {
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *src = x + (size_t)row * N;
    int *oi = idx + (size_t)row * N;
    float *ov = val + (size_t)row * N;
    int c = 0;
    if ((N & 3) == 0) {
        constexpr int U = 8;
        const float4 *s4 = reinterpret_cast<const float4 *>(src);
        const int n4 = N >> 2;
        const unsigned below = (1u << lane) - 1u;
        for (int base = 0; base < n4; base += 32 * U) {
            float4 xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i4 = base + 32 * u + lane;
                xv[u] = i4 < n4 ? ldg_stream4(s4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float e[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
                unsigned m[4];
                int before = 0, total = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    m[k] = __ballot_sync(0xffffffffu, e[k] != 0.f);
                    before += __popc(m[k] & below);
                    total += __popc(m[k]);
                }
                int p = c + before;
                const int j = 4 * (base + 32 * u + lane);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (e[k] != 0.f) {
                        oi[p] = j + k;
                        ov[p] = e[k];
                        ++p;
                    }
                }
                c += total;
            }
        }
    } else {
        for (int base = 0; base < N; base += 32) {
            const int j = base + lane;
            const float a = j < N ? src[j] : 0.f;
            const unsigned bal = __ballot_sync(0xffffffffu, a != 0.f);
            if (a != 0.f) {
                const int p = c + __popc(bal & ((1u << lane) - 1u));
                oi[p] = j;
                ov[p] = a;
            }
            c += __popc(bal);
        }
    }
    if (lane == 0) cnt[row] = c;
}

// One CTA per (token t of the chunk, head).  o_t = q_t S (gathered over the
// support of q_t, float4 columns, LOOK loads in flight per thread) +
// sum_{s in chunk, s <= t} <k_s, q_t> v_s (keys' supports against a dense copy
// of q_t in shared memory).
template <int DV>
__global__ void __launch_bounds__(kThreads, 3)
sparse_read_kernel(int bh0, int c0, int T_, int N, const int *__restrict__ kidx,
                   const float *__restrict__ kval, const int *__restrict__ kcnt,
                   const int *__restrict__ qidx, const float *__restrict__ qval,
                   const int *__restrict__ qcnt, const float *__restrict__ v,
                   const float *__restrict__ ST, float *__restrict__ y) {
    constexpr int CG = DV / 4;           // float4 column groups
    constexpr int RGN = kThreads / CG;   // support entries processed side by side
    constexpr int LOOK = 8;              // gathers in flight per thread
    extern __shared__ float qd[];        // [N] dense copy of q_t
    __shared__ float zs[kC];
    __shared__ float4 red[kThreads];
    const int ti = blockIdx.x, bh = bh0 + blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const size_t row = (size_t)bh * T_ + c0 + ti;
    for (int j = tid; j < N; j += kThreads) qd[j] = 0.f;
    __syncthreads();
    const int nq = qcnt[row];
    const int *qi = qidx + row * N;
    const float *qv = qval + row * N;
    for (int e = tid; e < nq; e += kThreads) qd[qi[e]] = qv[e];
    const int cg = tid % CG, rg = tid / CG;
    const float4 *Sb = reinterpret_cast<const float4 *>(ST + (size_t)bh * N * DV);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e0 = rg; e0 < nq; e0 += RGN * LOOK) {
        float4 x[LOOK];
        float w[LOOK];
#pragma unroll
        for (int u = 0; u < LOOK; ++u) {
            const int e = e0 + u * RGN;
            const bool ok = e < nq;
            w[u] = ok ? qv[e] : 0.f;
            x[u] = ok ? Sb[(size_t)qi[e] * CG + cg] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < LOOK; ++u) {
            o.x = fmaf(w[u], x[u].x, o.x);
            o.y = fmaf(w[u], x[u].y, o.y);
            o.z = fmaf(w[u], x[u].z, o.z);
            o.w = fmaf(w[u], x[u].w, o.w);
        }
    }
    __syncthreads();  // qd complete
    for (int si = warp; si <= ti; si += kThreads / 32) {
        const size_t srow = (size_t)bh * T_ + c0 + si;
        const int nk = kcnt[srow];
        float z = 0.f;
        for (int e = lane; e < nk; e += 32) z = fmaf(kval[srow * N + e], qd[kidx[srow * N + e]], z);
        z = warp_sum(z);
        if (lane == 0) zs[si] = z;
    }
    __syncthreads();
    const float4 *vb = reinterpret_cast<const float4 *>(v + ((size_t)bh * T_ + c0) * DV);
    for (int si = rg; si <= ti; si += RGN) {
        const float z = zs[si];
        const float4 vv = vb[(size_t)si * CG + cg];
        o.x = fmaf(z, vv.x, o.x);
        o.y = fmaf(z, vv.y, o.y);
        o.z = fmaf(z, vv.z, o.z);
        o.w = fmaf(z, vv.w, o.w);
    }
    red[tid] = o;
    __syncthreads();
    if (tid < CG) {
        float4 s = red[tid];
        for (int g = 1; g < RGN; ++g) {
            const float4 a = red[g * CG + tid];
            s.x += a.x; s.y += a.y; s.z += a.z; s.w += a.w;
        }
        reinterpret_cast<float4 *>(y + row * DV)[tid] = s;
    }
}

// One CTA per (token s of the chunk, head): S[j, :] += k_s[j] v_s for every j
// in the support of k_s, as float4 vector reductions.
template <int DV>
__global__ void __launch_bounds__(kThreads)
sparse_write_kernel(int bh0, int c0, int T_, int N, const int *__restrict__ kidx,
                    const float *__restrict__ kval, const int *__restrict__ kcnt,
                    const float *__restrict__ v, float *__restrict__ ST) {
    constexpr int CG = DV / 4, RGN = kThreads / CG;
    const int bh = bh0 + blockIdx.y, tid = threadIdx.x;
    const size_t row = (size_t)bh * T_ + c0 + blockIdx.x;
    const int cg = tid % CG, rg = tid / CG;
    const float4 vv = reinterpret_cast<const float4 *>(v + row * DV)[cg];
    float4 *Sb = reinterpret_cast<float4 *>(ST + (size_t)bh * N * DV);
    const int nk = kcnt[row];
    const int *ki = kidx + row * N;
    const float *kv = kval + row * N;
#pragma unroll 4
    for (int e = rg; e < nk; e += RGN) {
        const float a = kv[e];
        atomicAdd(Sb + (size_t)ki[e] * CG + cg, make_float4(a * vv.x, a * vv.y, a * vv.z, a * vv.w));
    }
}

// ------------------------------------------------------------------ pairwise form
// One CTA per (token block, head, q or k): the block's supports as
// coordinate-major lists.  off[j] .. off[j+1] index the entries of coordinate
// j; each entry is (token within the block, value).  Counting and placement
// use shared-memory counters, so the order inside a coordinate is arbitrary.
__global__ void __launch_bounds__(512)
csc_build_kernel(int T, int N, int nb, const int *__restrict__ kidx, const float *__restrict__ kval,
                 const int *__restrict__ kcnt, const int *__restrict__ qidx, const float *__restrict__ qval,
                 const int *__restrict__ qcnt, int *__restrict__ coff, uint8_t *__restrict__ ct,
                 float *__restrict__ cv) {
    extern __shared__ int cnt[];  // [N]: counts, then placement cursors
    __shared__ int wsum[16];
    const int b = blockIdx.x, bh = blockIdx.y, which = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int *idx = which ? qidx : kidx;
    const float *val = which ? qval : kval;
    const int *rc = which ? qcnt : kcnt;
    const int t0 = b * kTB, nrows = min(kTB, T - t0);
    const size_t blk = ((size_t)which * gridDim.y + bh) * nb + b;
    int *off = coff + blk * (size_t)(N + 1);
    uint8_t *et = ct + blk * (size_t)kTB * N;
    float *ev = cv + blk * (size_t)kTB * N;
    for (int j = tid; j < N; j += 512) cnt[j] = 0;
    __syncthreads();
    for (int r = warp; r < nrows; r += 16) {
        const size_t row = (size_t)bh * T + t0 + r;
        const int n = rc[row];
        for (int e = lane; e < n; e += 32) atomicAdd(&cnt[idx[row * N + e]], 1);
    }
    __syncthreads();
    // exclusive scan of the N counts: a contiguous segment per thread
    const int seg = (N + 511) / 512, j0 = min(N, tid * seg), j1 = min(N, j0 + seg);
    int local = 0;
    for (int j = j0; j < j1; ++j) local += cnt[j];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += x;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < 16 ? wsum[lane] : 0;
#pragma unroll
        for (int d = 1; d < 16; d <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += x;
        }
        if (lane < 16) wsum[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? wsum[warp - 1] : 0);
    for (int j = j0; j < j1; ++j) {
        const int c = cnt[j];
        cnt[j] = run;
        off[j] = run;
        run += c;
    }
    if (tid == 0) off[N] = wsum[15];
    __syncthreads();
    for (int r = warp; r < nrows; r += 16) {
        const size_t row = (size_t)bh * T + t0 + r;
        const int n = rc[row];
        for (int e = lane; e < n; e += 32) {
            const int p = atomicAdd(&cnt[idx[row * N + e]], 1);
            et[p] = (uint8_t)r;
            ev[p] = val[row * N + e];
        }
    }
}

// Pairwise form straight from the dense rows: one CTA per (token block,
// head, q or k) streams the block's 128 rows through shared memory in
// 128 x 128 fp32 tiles and writes the coordinate-major lists of the block
// (the output of csc_build_kernel) without per-row lists in between.
//   warp 16 (lane 0)  TMA: the tiles, kCsStages in flight (rows past T read
//                     as zero);
//   warps 0-15        thread (row quarter rq, column c) counts the non-zeros
//                     of column c in rows [32 rq, 32 rq + 32); a scan over
//                     the tile's 128 columns places the lists, so each
//                     coordinate's entries come out in ascending token order.
// A tile's entries (one contiguous range of the block's lists) are staged in
// shared memory as (value, token) pairs when they fit, then written out with
// coalesced stores.  Every wait is bounded; one that runs out sets a bit in
// the call's status word and the CTA winds down.
constexpr int kCT = 128;        // columns per tile
constexpr int kCStage = 2048;   // staged entries per tile, at most
constexpr int kCsStages = 3;    // tiles in flight
constexpr int kCsWarps = 16;    // consumer warps: 4 row quarters x 4 column groups of 32
constexpr int kCsThreads = (kCsWarps + 1) * 32;
constexpr uint32_t kCsTileBytes = kTB * kCT * sizeof(float);
constexpr int kCsSmem = kCsStages * kCsTileBytes + kCStage * sizeof(uint2) + 128;  // + alignment slack

enum : unsigned int {
    kStCsProducer = kStatusSparse << 0,
    kStCsConsumer = kStatusSparse << 1,
};

// Named barrier 1 over the consumer warps; the second form also returns
// whether `ok` holds in all of them.
__device__ __forceinline__ void cs_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kCsWarps * 32) : "memory"); }
__device__ __forceinline__ bool cs_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "n"(kCsWarps * 32)
        : "memory");
    return r != 0;
}

// Appends (x, t) at shared address sa, and advances sa, when x != 0 (NaN
// included, as for the C comparison) -- as predicated instructions, with no
// branch per value; then t += 1.
__device__ __forceinline__ void stage_nonzero(uint32_t &sa, uint32_t &t, float x) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.neu.f32 q, %2, 0f00000000;\n\t"
        "@q st.shared.v2.b32 [%0], {%2, %1};\n\t"
        "@q add.u32 %0, %0, 8;\n\t"
        "add.u32 %1, %1, 1;\n\t}"
        : "+r"(sa), "+r"(t)
        : "f"(x)
        : "memory");
}

__global__ void __launch_bounds__(kCsThreads, 1)
dense_csc_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mq, int N, int nb,
                 int *__restrict__ coff, uint8_t *__restrict__ ct, float *__restrict__ cv,
                 unsigned int *__restrict__ status) {
    extern __shared__ unsigned char csraw[];
    float *tiles = reinterpret_cast<float *>(((uintptr_t)csraw + 127) & ~(uintptr_t)127);  // [stage][kTB][kCT]
    uint2 *stage = reinterpret_cast<uint2 *>(tiles + kCsStages * kTB * kCT);
    __shared__ uint64_t full[kCsStages], empty[kCsStages];
    __shared__ int cnt4[4][kCT];  // non-zeros of column c in row quarter q
    __shared__ int wtot[4];
    const int b = blockIdx.x, bh = blockIdx.y, which = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ntile = N / kCT;
    if (tid == 0) {
        for (int i = 0; i < kCsStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCsWarps);
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == kCsWarps) {
        if (lane == 0) {
            const CUtensorMap *m = which ? &mq : &mk;
            bool ok = true;
            int issued = 0;
            for (int i = 0; i < ntile && ok; ++i) {
                const int st = i % kCsStages;
                if (i >= kCsStages) ok = mbar_wait(&empty[st], (i / kCsStages - 1) & 1);
                if (!ok) break;
                mbar_expect_tx(&full[st], kCsTileBytes);
                tma_load_3d(tiles + st * kTB * kCT, m, &full[st], i * kCT, b * kTB, bh);
                ++issued;
            }
            if (!ok) atomicOr(status, kStCsProducer);
            // wait for this thread's copies still in flight before the CTA exits
            bool dok = true;
            for (int i = max(0, issued - kCsStages); i < issued && dok; ++i)
                dok = mbar_wait(&full[i % kCsStages], (i / kCsStages) & 1);
        }
        __syncwarp();
        return;
    }
    const int c = tid & (kCT - 1), rq = tid >> 7, wq = warp & 3;  // column, row quarter, column group
    const size_t blk = ((size_t)which * gridDim.y + bh) * nb + b;
    int *off = coff + blk * (size_t)(N + 1);
    uint8_t *et = ct + blk * (size_t)kTB * N;
    float *ev = cv + blk * (size_t)kTB * N;
    int base = 0;  // entries of the block so far
    bool ok = true;
    for (int i = 0; i < ntile && ok; ++i) {
        const int st = i % kCsStages;
        ok = cs_all(mbar_wait(&full[st], (i / kCsStages) & 1));
        if (!ok) break;
        const float *tile = tiles + st * kTB * kCT;
        // this thread's 32 values of column c stay in registers for the count and the placement
        float a[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) a[r] = tile[(32 * rq + r) * kCT + c];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // the tile is no longer read
        int n = 0;
#pragma unroll
        for (int r = 0; r < 32; ++r) n += a[r] != 0.f ? 1 : 0;
        cnt4[rq][c] = n;
        cs_barrier();
        // entries of column c in the row quarters before rq, and in all four
        int before = 0, tot = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int v = cnt4[q][c];
            before += q < rq ? v : 0;
            tot += v;
        }
        // inclusive scan of the column totals over this warp's 32 columns
        int incl = tot;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        if (rq == 0 && lane == 31) wtot[wq] = incl;
        cs_barrier();
        int start = base + incl - tot;
        for (int w = 0; w < wq; ++w) start += wtot[w];
        if (rq == 0) off[i * kCT + c] = start;
        const int ttot = wtot[0] + wtot[1] + wtot[2] + wtot[3];  // the tile's range [base, base + ttot)
        int p = start + before;
        const bool staged = ttot <= kCStage;  // the same in every consumer thread
        if (staged) {
            uint32_t sa = (uint32_t)__cvta_generic_to_shared(stage + (p - base)), tok = 32 * rq;
#pragma unroll
            for (int r = 0; r < 32; ++r) stage_nonzero(sa, tok, a[r]);
        } else {
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                if (a[r] != 0.f) {
                    if (OPAM_BOUNDS(p < kTB * N, status)) {
                        et[p] = (uint8_t)(32 * rq + r);
                        ev[p] = a[r];
                    }
                    ++p;
                }
            }
        }
        cs_barrier();
        if (staged) {
            for (int j = tid; j < ttot; j += kCsWarps * 32) {
                if (OPAM_BOUNDS(base + j < kTB * N, status)) {
                    const uint2 e = stage[j];
                    et[base + j] = (uint8_t)e.y;
                    ev[base + j] = __uint_as_float(e.x);
                }
            }
        }
        base += ttot;
    }
    if (!ok && lane == 0) atomicOr(status, kStCsConsumer);
    if (ok && tid == 0) off[N] = base;
}

// One CTA per (pair of token blocks tb >= sb, head):
//   Z[t][s] = sum_j q_t[j] k_s[j]  (s <= t on the diagonal block), accumulated
//   in shared memory.  Coordinates are taken in windows of kJW: the window's
//   list entries (contiguous in the coordinate-major arrays) are copied to
//   shared memory with coalesced loads, each query entry tagged with its
//   coordinate.  Then every thread takes query entries (t, q_t[j]) one after
//   another and walks the key list of the same coordinate j, adding
//   q_t[j] k_s[j] into Z[t][s]: with about six key entries per coordinate and
//   block, a lane does a few products per entry and no lane waits for a
//   coordinate's setup.  A window whose lists do not fit the buffers (dense
//   inputs) is read from global memory, one coordinate per warp.
//   Then o[tb] += Z V[sb]  (fp32, 64 output columns per pass, float4 atomics).
// Z[t][s] += x in shared memory with no value returned (a reduction, not an
// atomic read-modify-write that hands back the old value).
__device__ __forceinline__ void red_add_shared(float *p, float x) {
    asm volatile("red.shared.add.f32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)), "f"(x) : "memory");
}

constexpr int kJW = 256;    // coordinates per window
constexpr int kCap = 2048;  // list entries per window buffered in shared memory

constexpr int kBins = 32;   // query entries sorted by their key-list length: 1 .. 30, then >= 31

struct PairSmem {
    float Z[kTB * (kTB + 1)];
    uint2 qe[kCap], ke[kCap];  // the window's list entries: (value bits, token)
    uint32_t stag[kCap];       // sorted query entry k: its coordinate's key entries, first | count << 16
    int qo[kJW + 1], ko[kJW + 1];
    uint16_t sidx[kCap];       // sorted query entry k: its index in qe
    int bin[kBins];            // entries per key-list length, then the running start of each length
    int nsort;                 // query entries with at least one key entry
};

template <int DV>
__global__ void __launch_bounds__(256, 2)
pair_tile_kernel(int T, int N, int nb, const int *__restrict__ coff, const uint8_t *__restrict__ ct,
                 const float *__restrict__ cv, const float *__restrict__ v, float *__restrict__ y,
                 unsigned int *__restrict__ status) {
    constexpr int ZS = kTB + 1;  // padded row stride of the Z tile
    extern __shared__ unsigned char smraw[];
    PairSmem &P = *reinterpret_cast<PairSmem *>(smraw);
    float *Zs = P.Z;
    const int tile = blockIdx.x, bh = blockIdx.y, BH = gridDim.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int tb = (int)((sqrtf(8.f * (float)tile + 1.f) - 1.f) * 0.5f);
    while ((tb + 1) * (tb + 2) / 2 <= tile) ++tb;
    while (tb * (tb + 1) / 2 > tile) --tb;
    const int sb = tile - tb * (tb + 1) / 2;
    const bool diag = sb == tb;
    for (int i = tid; i < kTB * ZS; i += 256) Zs[i] = 0.f;
    const size_t bk = (size_t)bh * nb + sb, bq = ((size_t)BH + bh) * nb + tb;  // k lists: which 0, q: 1
    const int *ko = coff + bk * (size_t)(N + 1), *qo = coff + bq * (size_t)(N + 1);
    const uint8_t *kt = ct + bk * (size_t)kTB * N, *qt = ct + bq * (size_t)kTB * N;
    const float *kv = cv + bk * (size_t)kTB * N, *qv = cv + bq * (size_t)kTB * N;
    // The coordinate windows are software-pipelined: while window w's
    // products run, the next window's offsets and list entries are already
    // on their way into registers (its bounds were read one window earlier),
    // so the staging costs no exposed global-memory latency.
    constexpr int EPT = kCap / 256;  // list entries per thread and list, at most
    const int nwin = (N + kJW - 1) / kJW;
    int pqo = 0, pko = 0;                       // next window's offsets (entry tid)
    uint32_t pqt[EPT], pkt[EPT];
    float pqv[EPT], pkv[EPT];
    int nb_qb = 0, nb_qe = 0, nb_kb = 0, nb_ke = 0;  // bounds of the window after next
    auto fetch_bounds = [&](int w, int &qb_, int &qe_, int &kb_, int &ke_) {
        if (w < nwin) {
            const int ws = w * kJW, we = min(N, ws + kJW);
            qb_ = qo[ws];
            qe_ = qo[we];
            kb_ = ko[ws];
            ke_ = ko[we];
        }
    };
    auto fetch_window = [&](int w, int qb_, int qe_, int kb_, int ke_) {
        if (w >= nwin) return;
        const int ws = w * kJW, nw_ = min(kJW, N - ws);
        if (tid < nw_) {
            pqo = qo[ws + tid];
            pko = ko[ws + tid];
        }
        const int nq_ = qe_ - qb_, nk_ = ke_ - kb_;
        if (nq_ <= kCap && nk_ <= kCap) {
#pragma unroll
            for (int u = 0; u < EPT; ++u) {
                const int i = tid + 256 * u;
                if (i < nq_) {
                    pqt[u] = qt[qb_ + i];
                    pqv[u] = qv[qb_ + i];
                }
                if (i < nk_) {
                    pkt[u] = kt[kb_ + i];
                    pkv[u] = kv[kb_ + i];
                }
            }
        }
    };
    auto store_window = [&](int w, int qb_, int qe_, int kb_, int ke_) {
        const int ws = w * kJW, nw_ = min(kJW, N - ws);
        if (tid < nw_) {
            P.qo[tid] = pqo;
            P.ko[tid] = pko;
        }
        if (tid == 0) {  // the window's closing offsets are its bounds
            P.qo[nw_] = qe_;
            P.ko[nw_] = ke_;
        }
        const int nq_ = qe_ - qb_, nk_ = ke_ - kb_;
        if (nq_ <= kCap && nk_ <= kCap) {
#pragma unroll
            for (int u = 0; u < EPT; ++u) {
                const int i = tid + 256 * u;
                if (i < nq_) P.qe[i] = make_uint2(__float_as_uint(pqv[u]), pqt[u]);
                if (i < nk_) P.ke[i] = make_uint2(__float_as_uint(pkv[u]), pkt[u]);
            }
        }
    };
    int cq_b = 0, cq_e = 0, ck_b = 0, ck_e = 0;  // bounds of the window being staged / processed
    fetch_bounds(0, cq_b, cq_e, ck_b, ck_e);
    fetch_window(0, cq_b, cq_e, ck_b, ck_e);
    fetch_bounds(1, nb_qb, nb_qe, nb_kb, nb_ke);
    for (int w = 0; w < nwin; ++w) {
        const int w0 = w * kJW, nw = min(kJW, N - w0);
        __syncthreads();  // the previous window's buffers are no longer read (and Z is zeroed)
        store_window(w, cq_b, cq_e, ck_b, ck_e);
        if (tid < kBins) P.bin[tid] = 0;
        const int qb = cq_b, kb = ck_b;
        const int nq = cq_e - cq_b, nk = ck_e - ck_b;
        const bool fits = nq <= kCap && nk <= kCap;
        __syncthreads();
        // next window: its bounds are known, so its entries can be requested now
        cq_b = nb_qb; cq_e = nb_qe; ck_b = nb_kb; ck_e = nb_ke;
        fetch_window(w + 1, cq_b, cq_e, ck_b, ck_e);
        fetch_bounds(w + 2, nb_qb, nb_qe, nb_kb, nb_ke);
        if (fits) {
            // Query entries are sorted by the length of their coordinate's key
            // list (a counting sort over kBins lengths), so that the lanes of a
            // warp walk lists of one length; entries with no key entry drop out.
            for (int jl = tid; jl < nw; jl += 256) {
                const int nqj = P.qo[jl + 1] - P.qo[jl], nkj = P.ko[jl + 1] - P.ko[jl];
                if (nqj > 0 && nkj > 0) atomicAdd(&P.bin[min(nkj, kBins) - 1], nqj);
            }
            __syncthreads();
            if (warp == 0) {  // exclusive scan of the bins
                const int c = P.bin[lane];
                int incl = c;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += y;
                }
                P.bin[lane] = incl - c;
                if (lane == 31) P.nsort = incl;
            }
            __syncthreads();
            for (int jl = tid; jl < nw; jl += 256) {
                const int q0 = P.qo[jl] - qb, k0 = P.ko[jl];
                const int nqj = P.qo[jl + 1] - qb - q0, nkj = P.ko[jl + 1] - k0;
                if (nqj > 0 && nkj > 0) {
                    const int pos = atomicAdd(&P.bin[min(nkj, kBins) - 1], nqj);
                    const uint32_t tag = (uint32_t)(k0 - kb) | (uint32_t)nkj << 16;
                    for (int a = 0; a < nqj; ++a) {
                        P.sidx[pos + a] = (uint16_t)(q0 + a);
                        P.stag[pos + a] = tag;
                    }
                }
            }
            __syncthreads();
            const int ns = P.nsort;
            for (int k = tid; k < ns; k += 256) {
                const uint2 q = P.qe[P.sidx[k]];
                const uint32_t tag = P.stag[k];
                const int t = (int)q.y, b0 = (int)(tag & 0xffffu), n = (int)(tag >> 16);
                const float x = __uint_as_float(q.x);
                const int smax = diag ? t : kTB - 1;  // causal inside the diagonal block
                float *zrow = Zs + t * ZS;
                // four key entries' loads in flight before their reductions
                for (int u0 = 0; u0 < n; u0 += 4) {
                    uint2 k[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (u0 + u < n) k[u] = P.ke[b0 + u0 + u];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s_ = (int)k[u].y;
                        if (u0 + u < n && s_ <= smax && OPAM_BOUNDS(t < kTB && s_ < kTB, status))
                            red_add_shared(zrow + s_, x * __uint_as_float(k[u].x));
                    }
                }
            }
        } else {
            // one coordinate per warp; lane (a, b) = (lane / 4, lane % 4) takes
            // query entry a0 + a and key entry b0 + b of the two lists
            for (int jl = warp; jl < nw; jl += 8) {
                const int q0 = P.qo[jl], k0 = P.ko[jl];
                const int nqj = P.qo[jl + 1] - q0, nkj = P.ko[jl + 1] - k0;
                for (int a0 = 0; a0 < nqj; a0 += 8) {
                    const int a = a0 + (lane >> 2);
                    const bool qa = a < nqj;
                    const int t = qa ? qt[q0 + a] : 0;
                    const float x = qa ? qv[q0 + a] : 0.f;
                    const int smax = diag ? t : kTB - 1;
                    for (int b0 = 0; b0 < nkj; b0 += 4) {
                        const int b = b0 + (lane & 3);
                        if (qa && b < nkj) {
                            const int s = kt[k0 + b];
                            if (s <= smax && OPAM_BOUNDS(t < kTB && s < kTB, status))
                                red_add_shared(Zs + t * ZS + s, x * kv[k0 + b]);
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    const int rows = min(kTB, T - tb * kTB), cols = min(kTB, T - sb * kTB);
    constexpr int DVP = DV < 64 ? DV : 64;  // output columns per pass
    constexpr int CG = DVP / 8;             // column groups of 8
    constexpr int RPT = kTB / (256 / CG);   // rows per thread
    constexpr int C4 = DVP / 4;             // float4 per staged V row
    static_assert(sizeof(P.qe) + sizeof(P.ke) >= sizeof(float) * kTB * DVP, "V slice buffer");
    // the pass's V slice [cols rows][DVP columns] is staged in the (now free)
    // window buffers, so every thread's reads of it come from shared memory
    float4 *Vs = reinterpret_cast<float4 *>(P.qe);
    const int cg = tid % CG, rg = tid / CG;
    const float *vb = v + ((size_t)bh * T + sb * kTB) * DV;
    float *yb = y + ((size_t)bh * T + tb * kTB) * DV;
#pragma unroll 1
    for (int c0 = 0; c0 < DV; c0 += DVP) {
        if (c0 > 0) __syncthreads();  // the previous slice is no longer read
        for (int i = tid; i < cols * C4; i += 256) {
            const int r = i / C4, c = i % C4;
            Vs[i] = reinterpret_cast<const float4 *>(vb + (size_t)r * DV + c0)[c];
        }
        __syncthreads();
        float acc[RPT][8];
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
        const int col = c0 + 8 * cg;
#pragma unroll 4
        for (int s_ = 0; s_ < cols; ++s_) {
            const float4 va = Vs[s_ * C4 + 2 * cg], vc = Vs[s_ * C4 + 2 * cg + 1];
            const float vv[8] = {va.x, va.y, va.z, va.w, vc.x, vc.y, vc.z, vc.w};
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float z = Zs[(rg * RPT + i) * ZS + s_];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(z, vv[e], acc[i][e]);
            }
        }
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = rg * RPT + i;
            if (r < rows && OPAM_BOUNDS(((size_t)bh * T + tb * kTB + r) * DV + col + 8 <= (size_t)BH * T * DV,
                                        status)) {
                float4 *dst = reinterpret_cast<float4 *>(yb + (size_t)r * DV + col);
                atomicAdd(dst, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
                atomicAdd(dst + 1, make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]));
            }
        }
    }
}

struct WsLayout {
    int *kidx, *qidx, *kcnt, *qcnt;
    float *kval, *qval, *ST;
    int *coff;     // [2][BH][nb][N+1]   coordinate lists of the pairwise form
    uint8_t *ct;   // [2][BH][nb][kTB*N] token within the block
    float *cv;     // [2][BH][nb][kTB*N] value
};

size_t csr_bytes(int BH, int T, int N) {
    const size_t ent = (size_t)BH * T * N;
    return 2 * align_up(sizeof(int) * ent, 256) + 2 * align_up(sizeof(float) * ent, 256) +
           2 * align_up(sizeof(int) * (size_t)BH * T, 256);
}
size_t pair_bytes(int BH, int T, int N) {
    const size_t nbk = 2 * (size_t)BH * ceil_div(T, kTB);
    return align_up(sizeof(int) * nbk * (N + 1), 256) + align_up(nbk * kTB * N, 256) +
           align_up(sizeof(float) * nbk * kTB * N, 256);
}
size_t state_bytes(int BH, int N, int dv) { return align_up(sizeof(float) * (size_t)BH * N * dv, 256); }

// Per-row supports first; the state (recurrent form) or the coordinate lists
// (pairwise form) share the space after them.
WsLayout carve(void *ws, int BH, int T, int N) {
    const size_t ent = (size_t)BH * T * N;
    char *p = (char *)ws;
    WsLayout l;
    l.kidx = (int *)p; p += align_up(sizeof(int) * ent, 256);
    l.qidx = (int *)p; p += align_up(sizeof(int) * ent, 256);
    l.kval = (float *)p; p += align_up(sizeof(float) * ent, 256);
    l.qval = (float *)p; p += align_up(sizeof(float) * ent, 256);
    l.kcnt = (int *)p; p += align_up(sizeof(int) * (size_t)BH * T, 256);
    l.qcnt = (int *)p; p += align_up(sizeof(int) * (size_t)BH * T, 256);
    l.ST = (float *)p;
    const size_t nbk = 2 * (size_t)BH * ceil_div(T, kTB);
    l.coff = (int *)p; p += align_up(sizeof(int) * nbk * (N + 1), 256);
    l.ct = (uint8_t *)p; p += align_up(nbk * kTB * N, 256);
    l.cv = (float *)p;
    return l;
}

// Block pairs over the coordinate lists of the workspace: y = sum of Z V.
template <int DV>
int pairs(const WsLayout &l, const float *v, int BH, int T, int N, float *y, unsigned int *status, cudaStream_t s) {
    const int nb = ceil_div(T, kTB);
    cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * (size_t)BH * T * DV, s);
    if (e != cudaSuccess) return cuda_fail(e, "sparse output init");
    const size_t psmem = sizeof(PairSmem);
    if (int rc_ = set_smem_limit((const void *)pair_tile_kernel<DV>, (int)psmem, "pair_tile smem attribute"))
        return rc_;
    prof_begin(s);
    pair_tile_kernel<DV><<<dim3(nb * (nb + 1) / 2, BH), 256, psmem, s>>>(T, N, nb, l.coff, l.ct, l.cv, v, y,
                                                                          status);
    const int rc = launched("pair_tile");
    prof_end(s);
    return rc;
}

// Everything after the per-row supports are in the workspace.
template <int DV>
int attend(const WsLayout &l, const float *v, int BH, int T, int N, const float *S0, float *S_out, float *y,
           unsigned int *status, cudaStream_t s) {
    cudaError_t e;
    if (S0 == nullptr && S_out == nullptr) {
        // pairwise form: coordinate lists per token block, then block pairs
        const int nb = ceil_div(T, kTB);
        const size_t csmem = sizeof(int) * (size_t)N;
        if (int rc_ = set_smem_limit((const void *)csc_build_kernel, (int)csmem, "csc_build smem attribute"))
            return rc_;
        csc_build_kernel<<<dim3(nb, BH, 2), 512, csmem, s>>>(T, N, nb, l.kidx, l.kval, l.kcnt, l.qidx, l.qval,
                                                            l.qcnt, l.coff, l.ct, l.cv);
        if (int rc = launched("csc_build")) return rc;
        return pairs<DV>(l, v, BH, T, N, y, status, s);
    }
    // recurrent form: the state lives in S_out (or the workspace)
    float *ST = S_out ? S_out : l.ST;
    const size_t sbytes = sizeof(float) * (size_t)BH * N * DV;
    if (S0 == nullptr) e = cudaMemsetAsync(ST, 0, sbytes, s);
    else if (S0 != ST) e = cudaMemcpyAsync(ST, S0, sbytes, cudaMemcpyDeviceToDevice, s);
    else e = cudaSuccess;
    if (e != cudaSuccess) return cuda_fail(e, "sparse state init");
    const size_t smem = sizeof(float) * (size_t)N;
    if (int rc_ = set_smem_limit((const void *)sparse_read_kernel<DV>, (int)smem, "sparse_read smem attribute")) return rc_;
    // Heads are taken in groups whose states fit the L2 cache together, so the
    // row gathers and scatters of a group's chunks are served from L2.
    const size_t head_state = sizeof(float) * (size_t)N * DV;
    const int group = (int)max((size_t)1, min((size_t)BH, kStateL2Budget / head_state));
    prof_begin(s);
    for (int bh0 = 0; bh0 < BH; bh0 += group) {
        const int gh = min(group, BH - bh0);
        for (int c0 = 0; c0 < T; c0 += kC) {
            const int n = min(kC, T - c0);
            sparse_read_kernel<DV><<<dim3(n, gh), kThreads, smem, s>>>(bh0, c0, T, N, l.kidx, l.kval, l.kcnt,
                                                                       l.qidx, l.qval, l.qcnt, v, ST, y);
            if (int rc = launched("sparse_read")) return rc;
            sparse_write_kernel<DV><<<dim3(n, gh), kThreads, 0, s>>>(bh0, c0, T, N, l.kidx, l.kval, l.kcnt, v,
                                                                     ST);
            if (int rc = launched("sparse_write")) return rc;
        }
    }
    prof_end(s);
    return OPAM_OK;
}

template <int DV>
int launch(const float *q, const float *k, const float *v, int BH, int T, int N, const float *S0,
           float *S_out, float *y, void *ws, unsigned int *status, cudaStream_t s) {
    const WsLayout l = carve(ws, BH, T, N);
    const int rows = BH * T;
    if (S0 == nullptr && S_out == nullptr && N % kCT == 0) {
        // pairwise form: coordinate lists straight from the dense rows
        const int nb = ceil_div(T, kTB);
        CUtensorMap mk, mq;
        if (int rc_ = make_tmap_f32_3d(&mk, k, N, T, BH, kCT, kTB)) return rc_;
        if (int rc_ = make_tmap_f32_3d(&mq, q, N, T, BH, kCT, kTB)) return rc_;
        if (int rc_ = set_smem_limit((const void *)dense_csc_kernel, kCsSmem, "dense_csc smem attribute")) return rc_;
        dense_csc_kernel<<<dim3(nb, BH, 2), kCsThreads, kCsSmem, s>>>(mk, mq, N, nb, l.coff, l.ct, l.cv, status);
        if (int rc = launched("dense_csc")) return rc;
        return pairs<DV>(l, v, BH, T, N, y, status, s);
    }
    compact_rows_kernel<<<ceil_div(rows, 8), 256, 0, s>>>(k, rows, N, l.kidx, l.kval, l.kcnt);
    if (int rc = launched("compact k")) return rc;
    compact_rows_kernel<<<ceil_div(rows, 8), 256, 0, s>>>(q, rows, N, l.qidx, l.qval, l.qcnt);
    if (int rc = launched("compact q")) return rc;
    return attend<DV>(l, v, BH, T, N, S0, S_out, y, status, s);
}

}  // namespace

int sparse_keygen_forward(const void *xq, const void *xk, const void *U, float theta, const float *v, int B,
                          int H, int T, int R, int N, int dv, const float *S0, float *S_out, float *y, void *ws,
                          unsigned int *status, cudaStream_t s) {
    const int BH = B * H;
    const WsLayout l = carve(ws, BH, T, N);
    const bool pairwise = S0 == nullptr && S_out == nullptr;
    // pairwise form: the key generation writes the blocks' coordinate lists
    // itself; recurrent form: per-row lists
    if (int rc = bdh_keygen(xq, xk, U, theta, B, H, T, R, N, l.kidx, l.kval, l.kcnt, l.qidx, l.qval, l.qcnt,
                            pairwise ? l.coff : nullptr, l.ct, l.cv, status, s))
        return rc;
    if (pairwise) {
        switch (dv) {
            case 32: return pairs<32>(l, v, BH, T, N, y, status, s);
            case 64: return pairs<64>(l, v, BH, T, N, y, status, s);
            case 128: return pairs<128>(l, v, BH, T, N, y, status, s);
            case 256: return pairs<256>(l, v, BH, T, N, y, status, s);
        }
    }
    switch (dv) {
        case 32: return attend<32>(l, v, BH, T, N, S0, S_out, y, status, s);
        case 64: return attend<64>(l, v, BH, T, N, S0, S_out, y, status, s);
        case 128: return attend<128>(l, v, BH, T, N, S0, S_out, y, status, s);
        case 256: return attend<256>(l, v, BH, T, N, S0, S_out, y, status, s);
    }
    set_error("d_v=%d unsupported", dv);
    return OPAM_ERR_UNSUPPORTED;
}

size_t sparse_workspace(int BH, int T, int N, int dv, bool need_state) {
    // the state (recurrent form, when kept in the workspace) and the
    // coordinate lists (pairwise form) use the same space after the supports
    const size_t tail = pair_bytes(BH, T, N);
    const size_t st = need_state ? state_bytes(BH, N, dv) : 0;
    return csr_bytes(BH, T, N) + (tail > st ? tail : st);
}

int sparse_forward(const float *q, const float *k, const float *v, int B, int H, int T, int N, int dv,
                   const float *S0, float *S_out, float *y, void *ws, unsigned int *status, cudaStream_t s) {
    const int BH = B * H;
    switch (dv) {
        case 32: return launch<32>(q, k, v, BH, T, N, S0, S_out, y, ws, status, s);
        case 64: return launch<64>(q, k, v, BH, T, N, S0, S_out, y, ws, status, s);
        case 128: return launch<128>(q, k, v, BH, T, N, S0, S_out, y, ws, status, s);
        case 256: return launch<256>(q, k, v, BH, T, N, S0, S_out, y, ws, status, s);
    }
    set_error("d_v=%d unsupported", dv);
    return OPAM_ERR_UNSUPPORTED;
}

}  // namespace opam
