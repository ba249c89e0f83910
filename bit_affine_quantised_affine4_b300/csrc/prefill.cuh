// prefill.cuh -- the prefill chunk (up to 128 tokens) as grouped GEMMs on the
// tcgen05 tensor cores.
//
// A chunk runs so that one expert load serves many rows (devtrends page, section
// "Prestazioni nel mondo reale"; remio.ai page, section "L'affermazione dei 2
// GB..."); by definition its output equals that many independent decodes.
//
//   plan     (1 CTA)  from the router's choices: distinct experts U in ascending
//                     id, the tokens of each in ascending order, a row segment per
//                     expert (its token count rounded up to 16), the row of every
//                     (token, choice) pair.
//   gather   (grid)   tokens -> fp16 operand tiles, per expert segment (zero rows
//                     pad each segment), plus all tokens for the shared expert.
//   gemm 0   (grid)   gate/up: per (expert, 64 gate + 64 up rows) item,
//                     D[128 x n] = W x X^T over K = H on the tensor cores, then
//                     h = gelu_tanh(gate) * up written as the down's fp16 operand.
//   gemm 1   (grid)   down: per (expert, 128 output rows) item, D = Wd x h^T over
//                     K = I (Is for the shared expert), fp32 rows out.
//   combine  (grid)   y_t = sum_k gate_tk * routed_(t,k) + shared_t (+ x_t), in a
//                     fixed order.
//
// Inside a GEMM CTA: warp 8 prefetches the next item's weight block into L2 and
// copies each K step's eight packed weight tiles and the token tile with bulk
// copies (TMA) into a ring; warps 0-7 dequantise one weight tile each (w = s*q +
// b, exact, rounded once to fp16) into the swizzled operand layout; one thread of
// warp 9 issues the MMAs (fp16 x fp16 -> fp32 in tensor memory) and commits them
// to the stage's barrier; warps 0-7 then read the accumulator out of tensor
// memory for the epilogue (warps w and w+4 share a lane quarter and split the
// columns; two accumulators alternate so the next item's MMAs overlap it).  Columns of both operands are stored in the
// same permuted order within each run of 8 (see mma_core.cuh): a K permutation
// applied to both operands leaves the product unchanged, and it lets one 32-bit
// mask extract two codes into an fp16 pair.
#pragma once

#include "common.cuh"
#include "mma_core.cuh"
#include "sync.cuh"
#include "tile.cuh"
#include "umma.cuh"

namespace moe {

constexpr int kPfStages = 4;
constexpr int kPfDq = 8;             // dequant + epilogue warps (one weight tile each per K step)
constexpr int kPfProducer = kPfDq, kPfMmaWarp = kPfDq + 1;
constexpr int kPfThreads = (kPfDq + 2) * 32;
constexpr int kPfRawA = 5120;        // eight 576-byte tiles, padded to 1024
constexpr int kPfMaxN = 128;         // token rows of one item (an expert with more tokens would be
                                     // cut into slices of kPfMaxN rows; kPfMaxN-row slices with 8 stages
                                     // measured slower: 358 vs 305 us per chunk)
constexpr int kPfRaw = kPfRawA + kPfMaxN * 128;
constexpr int kPfTileA = 128 * 128;  // dequantised A: 128 rows x 64 fp16
constexpr int kPfTmemCols = 256;     // two fp32 accumulators of up to 128 columns

// Plan written by k_prefill_plan (ints in the workspace).
struct PfPlan {
    int *U;        // [1] distinct experts, [1] rows used
    int *uexp;     // [MOE_MAX_EXPERTS]
    int *urow;     // [MOE_MAX_EXPERTS] first row of the expert's segment
    int *ucnt;     // [MOE_MAX_EXPERTS] tokens of the expert
    int *rowtok;   // [Rmax] token of each row, -1 = padding
    int *rowpair;  // [Rmax] pair t * topk + k of each row
    int *uslc;     // [MOE_MAX_EXPERTS + 1] first kPfMaxN-token slice of each expert (prefix of
                   // ceil(ucnt / kPfMaxN)); uslc[U] = all slices
};

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

// ------------------------------------------------------------------ plan
__global__ void __launch_bounds__(256) k_prefill_plan(const int *__restrict__ idx, int T, int E, int topk,
                                                      int Rmax, PfPlan p) {
    __shared__ unsigned mask[MOE_MAX_EXPERTS][4];  // token bit masks (T <= 128)
    __shared__ int urow_s[MOE_MAX_EXPERTS + 1], uid[MOE_MAX_EXPERTS];
    const int tid = threadIdx.x;
    for (int i = tid; i < MOE_MAX_EXPERTS * 4; i += blockDim.x) (&mask[0][0])[i] = 0u;
    __syncthreads();
    const int P2 = T * topk;
    for (int q = tid; q < P2; q += blockDim.x) {
        const int t = q / topk, e = idx[q];
        atomicOr(&mask[e][t >> 5], 1u << (t & 31));
    }
    __syncthreads();
    // distinct experts in ascending id and their 16-padded row segments: warp w
    // scans experts 32w..32w+31 (ballot + shuffle scan), then adds the totals of the
    // warps before it
    __shared__ unsigned wsum[MOE_MAX_EXPERTS / 32];  // experts << 16 | rows of the warp's 32 experts
    __shared__ int wslc[MOE_MAX_EXPERTS / 32];       // kPfMaxN-token slices of the warp's experts
    __shared__ int ucnt_s[MOE_MAX_EXPERTS];
    __shared__ int U_s;
    const int warp = tid >> 5, lane = tid & 31, nw = (E + 31) >> 5;
    int cnt = 0, incl = 0, sincl = 0;
    unsigned bal = 0u;
    if (warp < nw) {
        const int e = 32 * warp + lane;
        cnt = e < E ? __popc(mask[e][0]) + __popc(mask[e][1]) + __popc(mask[e][2]) + __popc(mask[e][3]) : 0;
        bal = __ballot_sync(0xffffffffu, cnt > 0);
        incl = round16(cnt);
        sincl = (cnt + kPfMaxN - 1) / kPfMaxN;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            const int w = __shfl_up_sync(0xffffffffu, sincl, o);
            if (lane >= o) {
                incl += v;
                sincl += w;
            }
        }
        if (lane == 31) {
            wsum[warp] = ((unsigned)__popc(bal) << 16) | (unsigned)incl;
            wslc[warp] = sincl;
        }
    }
    __syncthreads();
    if (warp < nw) {
        int ub = 0, rb = 0, sb = 0;
        for (int w = 0; w < warp; w++) {
            ub += (int)(wsum[w] >> 16);
            rb += (int)(wsum[w] & 0xFFFFu);
            sb += wslc[w];
        }
        const int e = 32 * warp + lane;
        if (e < E) uid[e] = -1;
        if (cnt) {
            const int u = ub + __popc(bal & ((1u << lane) - 1u)), row = rb + incl - round16(cnt);
            uid[e] = u;
            p.uexp[u] = e;
            p.ucnt[u] = cnt;
            p.urow[u] = row;
            p.uslc[u] = sb + sincl - (cnt + kPfMaxN - 1) / kPfMaxN;
            urow_s[u] = row;
            ucnt_s[u] = cnt;
        }
        if (warp == nw - 1 && lane == 31) {
            const int U = ub + __popc(bal), rows = rb + incl;
            urow_s[U] = rows;
            p.U[0] = U;
            p.U[1] = rows;
            p.uslc[U] = sb + sincl;
            U_s = U;
        }
    }
    __syncthreads();
    for (int q = tid; q < P2; q += blockDim.x) {
        const int t = q / topk, e = idx[q], u = uid[e];
        int rank = 0;
        for (int w = 0; w < (t >> 5); w++) rank += __popc(mask[e][w]);
        rank += __popc(mask[e][t >> 5] & ((1u << (t & 31)) - 1u));
        p.rowtok[urow_s[u] + rank] = t;
        p.rowpair[urow_s[u] + rank] = q;
    }
    // padding rows of each segment, and unused rows up to Rmax
    const int U = U_s, used = urow_s[U];
    for (int r = tid; r < Rmax; r += blockDim.x) {
        if (r >= used) {
            p.rowtok[r] = -1;
            continue;
        }
        int lo = 0, hi = U - 1;  // segment holding row r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (urow_s[mid] <= r) lo = mid; else hi = mid - 1;
        }
        if (r - urow_s[lo] >= ucnt_s[lo]) p.rowtok[r] = -1;
    }
}

// ------------------------------------------------------------------ gather
// One thread per (row, K group, 16-byte chunk): 8 fp16 values of the token in
// operand order.  Rows [0, Rmax) are the experts' segments (per rowtok), rows
// [Rmax, Rmax + T16) all tokens for the shared expert.
__global__ void __launch_bounds__(256) k_prefill_gather(const float *__restrict__ x, int T, int H, int Rmax,
                                                        int T16, const int *__restrict__ rowtok,
                                                        const int *__restrict__ used, uint8_t *Br, uint8_t *Bs) {
    const int G = H / kGroup;
    const long long n = (long long)(Rmax + T16) * G * 8;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int ch = (int)(i & 7);
    const long long rk = i >> 3;
    const int kb = (int)(rk % G);
    const int row = (int)(rk / G);
    int t;
    uint8_t *dst;
    if (row < Rmax) {
        if (row >= used[1]) return;
        t = rowtok[row];
        dst = Br + ((size_t)kb * Rmax + row) * 128 + ((ch ^ (row & 7)) << 4);
    } else {
        const int r = row - Rmax;
        t = r < T ? r : -1;
        dst = Bs + ((size_t)kb * T16 + r) * 128 + ((ch ^ (r & 7)) << 4);
    }
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0) {
        // chunk ch holds columns 8ch + (0, 4, 1, 5, 2, 6, 3, 7) of the group
        const float4 *src = reinterpret_cast<const float4 *>(x + (size_t)t * H + kb * kGroup + 8 * ch);
        const float4 lo = __ldg(src), hi = __ldg(src + 1);
        __half2 h0 = __floats2half2_rn(lo.x, hi.x), h1 = __floats2half2_rn(lo.y, hi.y);
        __half2 h2 = __floats2half2_rn(lo.z, hi.z), h3 = __floats2half2_rn(lo.w, hi.w);
        v = make_uint4(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1),
                       *reinterpret_cast<uint32_t *>(&h2), *reinterpret_cast<uint32_t *>(&h3));
    }
    *reinterpret_cast<uint4 *>(dst) = v;
}

// ------------------------------------------------------------------ grouped GEMM
struct PrefillGemmArgs {
    int kind;  // 0: gate/up + GeGLU, 1: down
    int H, I, Is, T, T16, Rmax;
    const int *U;  // [0] distinct experts
    const int *uexp, *urow, *ucnt, *rowpair, *uslc;
    const uint8_t *experts;
    size_t stride;
    const uint8_t *shared;
    TileLayout Lr, Ls;
    const uint8_t *Br, *Bs;  // token operand tiles [kb][rows][128 B] (routed Rmax rows, shared T16 rows)
    uint8_t *Hr, *Hs;        // kind 0 output: h operand tiles for the down
    float *Yr, *Ys;          // kind 1 output: fp32 rows [pair][H], [t][H]
    unsigned *err;
};

// Item i of the launch: shared items first, then the routed experts in order.
struct PfItem {
    const uint8_t *a;    // first tile of the item's 8-tile-row block (K step 0)
    size_t a_row;        // bytes between the 8 tile rows
    int nkb;             // K steps (groups)
    const uint8_t *b;    // token tile rows of K step 0
    size_t b_kb;         // bytes between K steps of the token tiles
    int n, N;            // valid token rows, padded (multiple of 16), of this kPfMaxN-row slice
    int row0;            // first row of the slice (shared: token; routed: in the expert's segment)
    int mb;              // M block
    int u;               // routed expert, -1 = shared
};

// Items: [shared M block mb, slice sl] for mb < ms, sl < ceil(T / kPfMaxN); then per
// distinct expert u, [M block mb, slice sl] for mb < mr, sl < its slices.
__device__ __forceinline__ int pf_shared_slices(const PrefillGemmArgs &a) { return (a.T + kPfMaxN - 1) / kPfMaxN; }
__device__ __forceinline__ int pf_items(const PrefillGemmArgs &a) {
    const int ms = a.kind == 0 ? a.Is / 64 : a.H / 128, mr = a.kind == 0 ? a.I / 64 : a.H / 128;
    return ms * pf_shared_slices(a) + mr * a.uslc[a.U[0]];
}
__device__ __forceinline__ PfItem pf_item(const PrefillGemmArgs &a, int i) {
    PfItem it;
    const int ms = a.kind == 0 ? a.Is / 64 : a.H / 128;  // shared M blocks
    const int mr = a.kind == 0 ? a.I / 64 : a.H / 128;   // routed M blocks per expert
    const int nss = pf_shared_slices(a);
    if (i < ms * nss) {
        const int mb = i / nss, sl = i - mb * nss;
        it.u = -1;
        it.mb = mb;
        it.row0 = sl * kPfMaxN;
        it.n = min(kPfMaxN, a.T - it.row0);
        it.N = round16(it.n);
        it.b = (a.kind == 0 ? a.Bs : a.Hs) + (size_t)it.row0 * 128;
        it.b_kb = (size_t)a.T16 * 128;
        if (a.kind == 0) {
            it.a = a.shared + (size_t)kTileBytes * (8 * mb) * a.Ls.G;
            it.a_row = (size_t)kTileBytes * a.Ls.G;
            it.nkb = a.Ls.G;
        } else {
            it.a = a.shared + a.Ls.gu_bytes + (size_t)kTileBytes * (8 * mb) * a.Ls.Gi;
            it.a_row = (size_t)kTileBytes * a.Ls.Gi;
            it.nkb = a.Ls.Gi;
        }
    } else {
        // expert u: the last one with mr * uslc[u] <= j
        const int j = i - ms * nss;
        int lo = 0, hi = a.U[0] - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (mr * a.uslc[mid] <= j) lo = mid; else hi = mid - 1;
        }
        const int u = lo, ns = a.uslc[u + 1] - a.uslc[u], r = j - mr * a.uslc[u];
        const int mb = r / ns, sl = r - mb * ns;
        it.u = u;
        it.mb = mb;
        it.row0 = sl * kPfMaxN;
        it.n = min(kPfMaxN, a.ucnt[u] - it.row0);
        it.N = round16(it.n);
        it.b = (a.kind == 0 ? a.Br : a.Hr) + (size_t)(a.urow[u] + it.row0) * 128;
        it.b_kb = (size_t)a.Rmax * 128;
        const uint8_t *blob = a.experts + (size_t)a.uexp[u] * a.stride;
        if (a.kind == 0) {
            it.a = blob + (size_t)kTileBytes * (8 * mb) * a.Lr.G;
            it.a_row = (size_t)kTileBytes * a.Lr.G;
            it.nkb = a.Lr.G;
        } else {
            it.a = blob + a.Lr.gu_bytes + (size_t)kTileBytes * (8 * mb) * a.Lr.Gi;
            it.a_row = (size_t)kTileBytes * a.Lr.Gi;
            it.nkb = a.Lr.Gi;
        }
    }
    return it;
}

__device__ __forceinline__ uint4 deq_word(uint32_t w, __half2 s2, __half2 b2) {
    const uint32_t magic = 0x64006400u;  // fp16 1024 in both halves
    const __half2 k1024 = __halves2half2(__ushort_as_half((unsigned short)0x6400), __ushort_as_half((unsigned short)0x6400));
    uint32_t r[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint32_t v = ((w >> (4 * k)) & 0x000F000Fu) | magic;
        __half2 q = __hsub2(*reinterpret_cast<const __half2 *>(&v), k1024);  // exact codes
        __half2 d = __hfma2(q, s2, b2);
        r[k] = *reinterpret_cast<uint32_t *>(&d);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

struct PfSmem {
    uint64_t raw_full[kPfStages], stage_free[kPfStages], a_full[kPfStages];
    uint64_t acc_full[2], acc_empty[2];
    uint32_t tmem;
    int err;
};

__global__ void __launch_bounds__(kPfThreads, 1) k_prefill_gemm(const PrefillGemmArgs ga) {
    extern __shared__ __align__(1024) uint8_t psm_raw[];
    __shared__ PfSmem S;
    // the plan in shared memory: every item lookup reads it
    __shared__ int pl_U[2], pl_uslc[MOE_MAX_EXPERTS + 1], pl_ucnt[MOE_MAX_EXPERTS], pl_urow[MOE_MAX_EXPERTS],
        pl_uexp[MOE_MAX_EXPERTS];
    {
        const int U = ga.U[0];
        if (threadIdx.x == 0) pl_U[0] = U;
        for (int u = threadIdx.x; u <= U; u += blockDim.x) {
            pl_uslc[u] = ga.uslc[u];
            if (u < U) {
                pl_ucnt[u] = ga.ucnt[u];
                pl_urow[u] = ga.urow[u];
                pl_uexp[u] = ga.uexp[u];
            }
        }
    }
    PrefillGemmArgs a = ga;
    a.U = pl_U;
    a.uslc = pl_uslc;
    a.ucnt = pl_ucnt;
    a.urow = pl_urow;
    a.uexp = pl_uexp;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // 1024-aligned carve-up: raw stages | dequantised A stages | epilogue buffers
    uint8_t *base = psm_raw + ((1024u - (smem_addr(psm_raw) & 1023u)) & 1023u);
    uint8_t *raw = base;
    uint8_t *sA = raw + (size_t)kPfStages * kPfRaw;
    float *ebuf = reinterpret_cast<float *>(sA + (size_t)kPfStages * kPfTileA);  // [128 cols][64 rows]
    uint8_t *hst = reinterpret_cast<uint8_t *>(ebuf + 64 * kPfMaxN);          // [128 rows][128 B]
    volatile int *err = &S.err;

    if (tid == 0) {
        for (int s = 0; s < kPfStages; s++) {
            mbar_init(&S.raw_full[s], 1);
            mbar_init(&S.stage_free[s], 1);
            mbar_init(&S.a_full[s], kPfDq);
        }
        for (int j = 0; j < 2; j++) {
            mbar_init(&S.acc_full[j], 1);
            mbar_init(&S.acc_empty[j], kPfDq);
        }
        S.err = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&S.tmem, kPfTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    const int NI = pf_items(a);
    const int b = blockIdx.x, nC = gridDim.x;
    auto fail = [&]() {
        *err = 1;
        atomicExch(a.err, 1u);
    };

    if (warp == kPfProducer) {
        // ---------------- copies
        if (lane == 0) {
            int f = 0;
            int last[kPfStages];
            for (int s = 0; s < kPfStages; s++) last[s] = -1;
            for (int i = b; i < NI; i += nC) {
                const PfItem it = pf_item(a, i);
                // this item's weight block (first item only) and the next one's, into L2
                if (i == b) prefetch_l2(it.a, (unsigned)(8 * it.a_row));
                if (i + nC < NI) {
                    const PfItem nx = pf_item(a, i + nC);
                    prefetch_l2(nx.a, (unsigned)(8 * nx.a_row));
                }
                for (int kb = 0; kb < it.nkb; kb++, f++) {
                    const int s = f % kPfStages;
                    if (f >= kPfStages && !*err &&
                        !mbar_wait(&S.stage_free[s], ((f / kPfStages) - 1) & 1, err))
                        fail();
                    if (*err) continue;
                    uint8_t *dst = raw + (size_t)s * kPfRaw;
                    mbar_arrive_expect_tx(&S.raw_full[s], 8 * kTileBytes + it.N * 128);
                    for (int j = 0; j < 8; j++)
                        bulk_g2s(dst + j * kTileBytes, it.a + j * it.a_row + (size_t)kb * kTileBytes, kTileBytes,
                                 &S.raw_full[s]);
                    bulk_g2s(dst + kPfRawA, it.b + (size_t)kb * it.b_kb, it.N * 128, &S.raw_full[s]);
                    last[s] = f;
                }
            }
            // drain: the last copies of every stage have landed
            volatile int never = 0;
            for (int s = 0; s < kPfStages; s++)
                if (last[s] >= 0) mbar_wait(&S.raw_full[s], (last[s] / kPfStages) & 1, &never);
        }
        __syncwarp();
    } else if (warp == kPfMmaWarp) {
        // ---------------- MMA issue
        if (lane == 0) {
            int f = 0, n_it = 0;
            for (int i = b; i < NI; i += nC, n_it++) {
                const PfItem it = pf_item(a, i);
                const int ab = n_it & 1;
                if (n_it >= 2 && !*err && !mbar_wait(&S.acc_empty[ab], ((n_it >> 1) - 1) & 1, err)) fail();
                tc_fence_after();
                const uint32_t idesc = umma_idesc_f16(128, it.N);
                for (int kb = 0; kb < it.nkb; kb++, f++) {
                    const int s = f % kPfStages;
                    if (!*err && !mbar_wait(&S.a_full[s], (f / kPfStages) & 1, err)) fail();
                    tc_fence_after();
                    if (!*err) {
                        const uint32_t sa = smem_addr(sA + (size_t)s * kPfTileA);
                        const uint32_t sb = smem_addr(raw + (size_t)s * kPfRaw + kPfRawA);
#pragma unroll
                        for (int ks = 0; ks < 4; ks++)
                            umma_f16(tmem + ab * 128, umma_desc(sa + 32 * ks), umma_desc(sb + 32 * ks), idesc,
                                     kb > 0 || ks > 0);
                    }
                    umma_commit(&S.stage_free[s]);
                }
                umma_commit(&S.acc_full[ab]);
            }
            // every MMA issued here has finished before tensor memory is released
            if (f > 0) {
                volatile int never = 0;
                const int s = (f - 1) % kPfStages;
                mbar_wait(&S.stage_free[s], ((f - 1) / kPfStages) & 1, &never);
            }
        }
        __syncwarp();
    } else {
        // ---------------- dequantise + epilogue (warps 0-7)
        const int r = lane >> 2, c = lane & 3;
        const int quad = warp & 3, half = warp >> 2;  // tensor-memory lane quarter, column half
        int f = 0, n_it = 0;
        for (int i = b; i < NI; i += nC, n_it++) {
            const PfItem it = pf_item(a, i);
            for (int kb = 0; kb < it.nkb; kb++, f++) {
                const int s = f % kPfStages;
                if (!*err && !mbar_wait(&S.raw_full[s], (f / kPfStages) & 1, err)) fail();
                if (!*err) {
                    const uint8_t *rs = raw + (size_t)s * kPfRaw;
                    uint8_t *as = sA + (size_t)s * kPfTileA;
                    {
                        const int j = warp;
                        const uint4 q = *reinterpret_cast<const uint4 *>(rs + j * kTileBytes + 16 * lane);
                        const uint2 e = *reinterpret_cast<const uint2 *>(rs + j * kTileBytes + 512 + 8 * r);
                        const __half2 sa2 = __half2half2(__ushort_as_half((unsigned short)(e.x & 0xFFFFu)));
                        const __half2 ba2 = __half2half2(__ushort_as_half((unsigned short)(e.x >> 16)));
                        const __half2 sb2 = __half2half2(__ushort_as_half((unsigned short)(e.y & 0xFFFFu)));
                        const __half2 bb2 = __half2half2(__ushort_as_half((unsigned short)(e.y >> 16)));
                        const int ra = a.kind == 0 ? 8 * j + r : 16 * j + r;
                        const int rb = a.kind == 0 ? 64 + 8 * j + r : 16 * j + 8 + r;
                        *reinterpret_cast<uint4 *>(as + sw128_chunk(ra, 2 * c)) = deq_word(q.x, sa2, ba2);
                        *reinterpret_cast<uint4 *>(as + sw128_chunk(ra, 2 * c + 1)) = deq_word(q.y, sa2, ba2);
                        *reinterpret_cast<uint4 *>(as + sw128_chunk(rb, 2 * c)) = deq_word(q.z, sb2, bb2);
                        *reinterpret_cast<uint4 *>(as + sw128_chunk(rb, 2 * c + 1)) = deq_word(q.w, sb2, bb2);
                    }
                    fence_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.a_full[s]);
            }
            // epilogue of item i
            const int ab = n_it & 1;
            if (!*err && !mbar_wait(&S.acc_full[ab], (n_it >> 1) & 1, err)) fail();
            tc_fence_after();
            const uint32_t trow = tmem + ab * 128 + ((uint32_t)(32 * quad) << 16);
            const int row = 32 * quad + lane;  // accumulator row of this thread
            const int c_first = 16 * half;     // this warp takes every other 16-column chunk
            if (a.kind == 0) {
                // rows 0-63 gate, 64-127 up (intermediate index 64 mb + row % 64)
                if (quad >= 2 && !*err)
                    for (int c0 = c_first; c0 < it.N; c0 += 32) {
                        float v[16];
                        tmem_ld16(trow + c0, v);
#pragma unroll
                        for (int q = 0; q < 16; q++) ebuf[(c0 + q) * 64 + row - 64] = v[q];
                    }
                named_sync(1, kPfDq * 32);
                if (quad < 2 && !*err) {
                    const int pos = frag_pos(row);  // operand position of column `row` of the K step
                    for (int c0 = c_first; c0 < it.N; c0 += 32) {
                        float v[16];
                        tmem_ld16(trow + c0, v);
#pragma unroll
                        for (int q = 0; q < 16; q++) {
                            const int jt = c0 + q;
                            const float h = jt < it.n ? gelu_tanh(v[q]) * ebuf[jt * 64 + row] : 0.f;
                            *reinterpret_cast<__half *>(hst + (size_t)jt * 128 + (((pos >> 3) ^ (jt & 7)) << 4) +
                                                        (pos & 7) * 2) = __float2half_rn(h);
                        }
                    }
                }
                named_sync(1, kPfDq * 32);
                // the item's h rows: one K step (kb = mb) of the down operand
                uint8_t *dst = (it.u < 0 ? a.Hs + ((size_t)it.mb * a.T16 + it.row0) * 128
                                         : a.Hr + ((size_t)it.mb * a.Rmax + a.urow[it.u] + it.row0) * 128);
                if (!*err)
                    for (int v = tid; v < it.N * 8; v += kPfDq * 32)
                        reinterpret_cast<uint4 *>(dst)[v] = reinterpret_cast<const uint4 *>(hst)[v];
            } else if (!*err) {
                // output row 128 mb + row, token column j
                const int n = 128 * it.mb + row;
                for (int c0 = c_first; c0 < it.N; c0 += 32) {
                    float v[16];
                    tmem_ld16(trow + c0, v);
#pragma unroll
                    for (int q = 0; q < 16; q++) {
                        const int jt = c0 + q;
                        if (jt < it.n) {
                            if (it.u < 0)
                                a.Ys[(size_t)(it.row0 + jt) * a.H + n] = v[q];
                            else
                                a.Yr[(size_t)a.rowpair[a.urow[it.u] + it.row0 + jt] * a.H + n] = v[q];
                        }
                    }
                }
            }
            tc_fence_before();
            named_sync(1, kPfDq * 32);
            if (lane == 0) mbar_arrive(&S.acc_empty[ab]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kPfTmemCols);
    }
}

inline size_t prefill_gemm_smem() {
    return 1024 + (size_t)kPfStages * kPfRaw + (size_t)kPfStages * kPfTileA + 64 * kPfMaxN * 4 + kPfMaxN * 128;
}

// ------------------------------------------------------------------ combine
__global__ void __launch_bounds__(256) k_prefill_combine(const float *__restrict__ x, int T, int H, int topk,
                                                         int flags, const float *__restrict__ gate,
                                                         const float *__restrict__ Yr,
                                                         const float *__restrict__ Ys, float *__restrict__ y) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * H) return;
    const int t = (int)(i / H), n = (int)(i % H);
    float acc = 0.f;
    for (int k = 0; k < topk; k++) acc = fmaf(gate[t * topk + k], Yr[(size_t)(t * topk + k) * H + n], acc);
    acc += Ys[(size_t)t * H + n];
    if (flags & MOE_RESIDUAL) acc += x[(size_t)t * H + n];
    y[i] = acc;
}

}  // namespace moe
