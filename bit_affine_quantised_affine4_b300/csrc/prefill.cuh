// prefill.cuh -- the prefill chunk (up to 128 tokens) as grouped GEMMs on the
// tcgen05 tensor cores.
//
// A chunk runs so that one expert load serves many rows (devtrends page, section
// "Prestazioni nel mondo reale"; remio.ai page, section "L'affermazione dei 2
// GB..."); by definition its output equals that many independent decodes.
//
//   route    (grid)   router logits as a small fp32 GEMM split over K slices,
//                     then one warp per token sums the slices and ranks them.
//   plan     (1 CTA)  from the router's choices: distinct experts U in ascending
//                     id, the tokens of each in ascending order, a row segment per
//                     expert (its token count rounded up to 16), the row of every
//                     (token, choice) pair.
//   gather   (grid)   tokens -> fp16 operand tiles, per expert segment (zero rows
//                     pad each segment), plus all tokens for the shared expert.
//   gemm     (1/SM)   both grouped GEMMs in one launch, one CTA per SM:
//                     gate/up items (expert, 128 gate + 128 up rows): D[tokens x
//                     256] = X x W^T over K = H on the tensor cores, then h =
//                     gelu_tanh(gate) * up written as the down's fp16 operand;
//                     then down items (expert, 256 output rows): D = h x Wd^T
//                     over K = I (Is for the shared expert), fp32 rows out.  A
//                     down item starts once the gate/up items it reads h from
//                     have counted themselves done (bounded wait), so the CTAs
//                     that finish their gate/up share early run down work
//                     instead of idling; every CTA must be resident at once.
//   combine  (grid)   y_t = sum_k gate_tk * routed_(t,k) + shared_t (+ x_t), in a
//                     fixed order.
//
// Inside a GEMM CTA the tokens are the MMA's M (128 rows, the item's slice) and the
// weights its N (256 rows: one instruction covers twice the weight rows that an
// M = 128 weight operand would, for about 1.1x its issue time).  One thread of the
// token warp prefetches the next item's weight block into L2 and copies the token
// tiles (bulk copies, TMA) into the operand ring (kPfQK K steps per stage) as soon
// as the MMA releases a stage.  The sixteen dequantising warps load their tile row
// of the next stage straight from global memory into registers, then turn the
// current one (w = s*q + b, exact, rounded once to fp16) into the swizzled B operand
// of the stage; the stage's barrier completes with the token bytes and one arrival
// per dequantising thread.  One thread of the MMA warp issues the MMAs (fp16 x fp16
// -> fp32 in tensor memory) and commits them to the stage's release barrier.  Eight
// epilogue warps read the accumulator out of tensor memory (a lane per token, two
// warps per lane quarter splitting the columns) while the next item's K steps run
// into the other of two accumulators.  Columns of both operands are stored in the
// same permuted order within each run of 8 (see mma_core.cuh): a K permutation
// applied to both operands leaves the product unchanged, and it lets one 32-bit
// mask extract two codes into an fp16 pair.
#pragma once

#include <atomic>

#include "common.cuh"
#include "mma_core.cuh"
#include "route.cuh"
#include "sync.cuh"
#include "tile.cuh"
#include "umma.cuh"

namespace moe {

constexpr int kPfRows = 256;         // weight rows per item: the MMA's N (the tokens are its M = 128)
constexpr int kPfTR = kPfRows / 16;  // tile rows per item
constexpr int kPfQStages = 2;        // operand ring: token tiles and dequantised weights of kPfQK K steps
constexpr int kPfQK = 2;             // K steps per operand stage (one wait, one commit, one arrival each)
constexpr int kPfDq = kPfTR;         // dequantising warps (one weight tile row each per K step)
constexpr int kPfProducer = kPfDq, kPfMmaWarp = kPfProducer + 1;
constexpr int kPfEpi0 = kPfProducer + 2;  // first epilogue warp
constexpr int kPfEpi = 8;            // epilogue warps: each lane quarter of tensor memory twice
constexpr int kPfThreads = (kPfEpi0 + kPfEpi) * 32;
constexpr int kPfMaxN = 128;         // token rows of one item (the MMA's M): an expert with more tokens
                                     // is cut into slices of kPfMaxN rows, each its own item
constexpr int kPfTileA = kPfMaxN * 128;      // token tile: 128 rows x 64 fp16 (the MMA's A)
constexpr int kPfTileB = kPfRows * 128;      // dequantised weights: 256 rows x 64 fp16 (the MMA's B)
constexpr int kPfQ = kPfTileA + kPfTileB;    // one K step of an operand stage
constexpr int kPfTmemCols = 2 * kPfRows;     // two fp32 accumulators of 256 columns

// Plan written by k_prefill_plan (ints in the workspace).
constexpr int kPfDepShared = MOE_MAX_EXPERTS, kPfDepAll = MOE_MAX_EXPERTS + 1, kPfDeps = MOE_MAX_EXPERTS + 2;

struct PfPlan {
    int *U;        // [1] distinct experts, [1] rows used
    int *uexp;     // [MOE_MAX_EXPERTS]
    int *urow;     // [MOE_MAX_EXPERTS] first row of the expert's segment
    int *ucnt;     // [MOE_MAX_EXPERTS] tokens of the expert
    int *rowtok;   // [Rmax] token of each row, -1 = padding
    int *rowpair;  // [Rmax] pair t * topk + k of each row
    int *uslc;     // [MOE_MAX_EXPERTS + 1] first kPfMaxN-token slice of each expert (prefix of
                   // ceil(ucnt / kPfMaxN)); uslc[U] = all slices
    unsigned *dep; // [kPfDeps] finished gate/up epilogue warps: per distinct expert u, then the
                   // shared expert's (kPfDepShared) and all items' (kPfDepAll); zeroed by the plan
};

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

// ------------------------------------------------------------------ router (tiled)
// The chunk's router as a small fp32 GEMM on the CUDA cores.  Each dequantised
// router weight w = s*q + b (rounded once to fp32, as in the decode router) is
// formed once per CTA and reused by 32 tokens, instead of once per (token, row).
// CTA (ks, eb, tb): tokens 32 tb .. +31, experts 64 eb .. +63, columns of K slice
// ks (kRtSliceCols wide); thread (warp w, lane l) accumulates tokens tg + 8 i and
// experts 16 w + eg + 4 j (tg = l % 8, eg = l / 8, i, j < 4) over the slice in
// ascending column order.  Partial sums go to part[ks][t][e]; k_prefill_topk then
// adds them per token in slice order.
constexpr int kRtSliceCols = 128;               // K columns per slice (two groups)
constexpr int kRtTok = 32, kRtExp = 64;         // CTA tile
constexpr int kRtThreads = 128;
constexpr int kRtPitch = kRtSliceCols + 4;      // padded smem row (floats): conflict-free float4 reads

inline size_t prefill_route_smem() { return sizeof(float) * (size_t)(kRtTok + kRtExp) * kRtPitch; }
inline int prefill_route_slices(int H) { return (H + kRtSliceCols - 1) / kRtSliceCols; }

struct RouteTiledArgs {
    const uint32_t *rq;           // [E][H/4] 8-bit codes
    const __half *rs, *rb;        // [E][H/64]
    const float *bias;            // [E] or null
    const float *x;               // [T][H]
    int T, H, E, topk;
    float *part;                  // [KS][T][E] partial logits
    int32_t *idx;                 // [T][topk]
    float *gate;                  // [T][topk]
};

__global__ void __launch_bounds__(kRtThreads, 4) k_prefill_route(const RouteTiledArgs a) {
    extern __shared__ __align__(16) float rt_sm[];
    float *xs = rt_sm;                        // [kRtTok][kRtPitch]
    float *wsm = rt_sm + kRtTok * kRtPitch;   // [kRtExp][kRtPitch]
    const int ks = blockIdx.x, eb = blockIdx.y, tb = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = tb * kRtTok, e0 = eb * kRtExp, k0 = ks * kRtSliceCols;
    const int kw = min(kRtSliceCols, a.H - k0);  // 64 or 128
    const int G = a.H / kGroup, c4 = kw / 4;     // float4 columns of the slice
    // router rows of the tile, dequantised: 16 codes (one uint4) per step (zeros past E)
    const int c16 = kw / 16;
    for (int v = tid; v < kRtExp * c16; v += kRtThreads) {
        const int r = v / c16, c = v - r * c16, e = e0 + r;
        float *dst = wsm + r * kRtPitch + 16 * c;
        if (e < a.E) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(a.rq + (size_t)e * (a.H / 4) + k0 / 4) + c);
            const int g = (k0 + 16 * c) / kGroup;
            const float s = __half2float(a.rs[(size_t)e * G + g]), b = __half2float(a.rb[(size_t)e * G + g]);
            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int u = 0; u < 4; u++)
                *reinterpret_cast<float4 *>(dst + 4 * u) =
                    make_float4(fmaf(s, (float)(wd[u] & 0xFFu), b), fmaf(s, (float)((wd[u] >> 8) & 0xFFu), b),
                                fmaf(s, (float)((wd[u] >> 16) & 0xFFu), b), fmaf(s, (float)(wd[u] >> 24), b));
        } else {
#pragma unroll
            for (int u = 0; u < 4; u++) *reinterpret_cast<float4 *>(dst + 4 * u) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // the tokens (the previous kernel's output) and the partial sums' area (which the
    // previous chunk's combine reads) only after the previous kernel has finished
    pdl_wait();
    pdl_launch_dependents();
    // x rows of the tile (zeros past T)
    for (int v = tid; v < kRtTok * c4; v += kRtThreads) {
        const int r = v / c4, c = v - r * c4, t = t0 + r;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < a.T) val = __ldg(reinterpret_cast<const float4 *>(a.x + (size_t)t * a.H + k0) + c);
        *reinterpret_cast<float4 *>(xs + r * kRtPitch + 4 * c) = val;
    }
    __syncthreads();
    const int tg = lane & 7, eg = lane >> 3;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
    const float *xr = xs + tg * kRtPitch;
    const float *wr = wsm + (16 * warp + eg) * kRtPitch;
#pragma unroll 2
    for (int k = 0; k < kw; k += 4) {
        float4 xv[4], wv[4];
#pragma unroll
        for (int i = 0; i < 4; i++) xv[i] = *reinterpret_cast<const float4 *>(xr + 8 * i * kRtPitch + k);
#pragma unroll
        for (int j = 0; j < 4; j++) wv[j] = *reinterpret_cast<const float4 *>(wr + 4 * j * kRtPitch + k);
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float s = acc[i][j];
                s = fmaf(wv[j].x, xv[i].x, s);
                s = fmaf(wv[j].y, xv[i].y, s);
                s = fmaf(wv[j].z, xv[i].z, s);
                s = fmaf(wv[j].w, xv[i].w, s);
                acc[i][j] = s;
            }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int t = t0 + tg + 8 * i;
        if (t >= a.T) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int e = e0 + 16 * warp + eg + 4 * j;
            if (e < a.E) a.part[((size_t)ks * a.T + t) * a.E + e] = acc[i][j];
        }
    }
}

// One warp per token: the token's logits as the sum of the slices' partials in
// slice order plus the bias, then the router's top-k and softmax.
constexpr int kRtTopkWarps = 8;
__global__ void __launch_bounds__(kRtTopkWarps * 32) k_prefill_topk(const RouteTiledArgs a, int KS) {
    __shared__ float lg[kRtTopkWarps][MOE_MAX_EXPERTS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRtTopkWarps + warp;
    pdl_wait();
    pdl_launch_dependents();
    if (t >= a.T) return;
    constexpr int NV = MOE_MAX_EXPERTS / 32;
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) acc[i] = 0.f;
    // the loads of eleven slices (half of a 2816-wide row's) are issued before their
    // sums (added in slice order)
    constexpr int kQ = 11;
    int q = 0;
    for (; q + kQ <= KS; q += kQ) {
        float v[kQ][NV];
#pragma unroll
        for (int j = 0; j < kQ; j++) {
            const float *pr = a.part + ((size_t)(q + j) * a.T + t) * a.E;
#pragma unroll
            for (int i = 0; i < NV; i++) {
                const int e = lane + 32 * i;
                v[j][i] = e < a.E ? __ldcg(pr + e) : 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < kQ; j++)
#pragma unroll
            for (int i = 0; i < NV; i++) acc[i] += v[j][i];
    }
    for (; q < KS; q++) {
        const float *pr = a.part + ((size_t)q * a.T + t) * a.E;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int e = lane + 32 * i;
            if (e < a.E) acc[i] += __ldcg(pr + e);
        }
    }
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        if (e < a.E) lg[warp][e] = acc[i] + (a.bias ? a.bias[e] : 0.f);
    }
    __syncwarp();
    warp_topk_softmax<true>(lg[warp], a.E, a.topk, a.idx + t * a.topk, a.gate + t * a.topk, nullptr, nullptr);
}

// ------------------------------------------------------------------ plan
static_assert(MOE_MAX_PREFILL_TOKENS <= 128, "the plan's token masks hold 128 tokens");
constexpr int kPlanThreads = 1024;  // one (token, choice) pair per thread at T = 128, top-8
__global__ void __launch_bounds__(kPlanThreads) k_prefill_plan(const int *__restrict__ idx, int T, int E, int topk,
                                                               int Rmax, PfPlan p) {
    __shared__ unsigned mask[MOE_MAX_EXPERTS][4];  // token bit masks (T <= 128)
    __shared__ int urow_s[MOE_MAX_EXPERTS + 1], uid[MOE_MAX_EXPERTS];
    __shared__ int idx_s[MOE_MAX_PREFILL_TOKENS * MOE_MAX_TOPK];  // the routing, read once
    const int tid = threadIdx.x;
    for (int i = tid; i < MOE_MAX_EXPERTS * 4; i += blockDim.x) (&mask[0][0])[i] = 0u;
    pdl_wait();
    pdl_launch_dependents();
    // (the previous chunk's GEMM, which read the counters, has finished)
    for (int i = tid; i < kPfDeps; i += blockDim.x) p.dep[i] = 0u;
    __syncthreads();
    const int P2 = T * topk;
    for (int q = tid; q < P2; q += blockDim.x) {
        const int t = q / topk, e = __ldcg(idx + q);
        idx_s[q] = e;
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
        const int t = q / topk, e = idx_s[q], u = uid[e];
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
// operand order, over the rows the plan used (the experts' segments, per rowtok)
// and then the T16 rows of all tokens for the shared expert; a grid-stride loop, so
// the grid need not be sized for the most rows a chunk could use.
__global__ void __launch_bounds__(256) k_prefill_gather(const float *__restrict__ x, int T, int H, int Rmax,
                                                        int T16, const int *__restrict__ rowtok,
                                                        const int *__restrict__ used, uint8_t *Br, uint8_t *Bs) {
    const int G = H / kGroup;
    pdl_wait();
    pdl_launch_dependents();
    const long long per_row = (long long)G * 8;
    const long long n_routed = (long long)__ldcg(used + 1) * per_row, n = n_routed + (long long)T16 * per_row;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const bool routed = i < n_routed;
        const long long li = routed ? i : i - n_routed;
        const int ch = (int)(li & 7);
        const long long rk = li >> 3;
        const int kb = (int)(rk % G);
        const int row = (int)(rk / G);
        int t;
        uint8_t *dst;
        if (routed) {
            t = __ldcg(rowtok + row);
            dst = Br + ((size_t)kb * Rmax + row) * 128 + ((ch ^ (row & 7)) << 4);
        } else {
            t = row < T ? row : -1;
            dst = Bs + ((size_t)kb * T16 + row) * 128 + ((ch ^ (row & 7)) << 4);
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
}

// ------------------------------------------------------------------ grouped GEMM
struct PrefillGemmArgs {
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
    int sparts;              // kind 1: the shared down matrix in sparts K parts of at most I/64 groups
    float *Ys_more;          // kind 1: parts 1.. of the shared rows, [sparts - 1][T16][H]
    unsigned *dep;           // the plan's gate/up completion counters
    unsigned *err;
};

// Item i of one GEMM (kind): shared items first, then the routed experts in order.
// An item is one block of kPfRows weight rows (gate/up: the gate and up rows of 128
// intermediate indices, each tile row's 8 gate rows then its 8 up rows; down: 256
// output rows) times one slice of <= kPfMaxN tokens; the last block of a matrix may
// hold half as many rows.  (The launch runs the down items routed first.)
struct PfItem {
    const uint8_t *a;    // first tile (K step 0) of the item's first tile row
    size_t a_row;        // bytes between tile rows
    int nkb;             // K steps (groups)
    int ntr;             // tile rows (kPfTR, or kPfTR / 2 for a half block): the MMA's N is 16 ntr
    const uint8_t *b;    // token tile rows of K step 0
    size_t b_kb;         // bytes between K steps of the token tiles
    int n, N;            // valid token rows, padded (multiple of 16), of this kPfMaxN-row slice
    int row0;            // first row of the slice (shared: token; routed: in the expert's segment)
    int mb;              // block of kPfRows weight rows
    int u;               // routed expert, -1 = shared
    int part;            // shared down: K part
    int kind;            // 0: gate/up + GeGLU, 1: down
};

// Blocks of kPfTR tile rows in a matrix of `tr` tile rows.
__device__ __forceinline__ int pf_blocks(int tr) { return (tr + kPfTR - 1) / kPfTR; }
__device__ __forceinline__ int pf_shared_slices(const PrefillGemmArgs &a) { return (a.T + kPfMaxN - 1) / kPfMaxN; }
__device__ __forceinline__ int pf_items(const PrefillGemmArgs &a, int kind) {
    const int ms = kind == 0 ? pf_blocks(a.Ls.Ti) : pf_blocks(a.Ls.R) * a.sparts;
    const int mr = kind == 0 ? pf_blocks(a.Lr.Ti) : pf_blocks(a.Lr.R);
    return ms * pf_shared_slices(a) + mr * a.uslc[a.U[0]];
}
__device__ __forceinline__ PfItem pf_item(const PrefillGemmArgs &a, int kind, int i) {
    PfItem it;
    it.kind = kind;
    const int ms = kind == 0 ? pf_blocks(a.Ls.Ti) : pf_blocks(a.Ls.R) * a.sparts;  // shared (block, K part) items
    const int mr = kind == 0 ? pf_blocks(a.Lr.Ti) : pf_blocks(a.Lr.R);              // routed blocks per expert
    const int nss = pf_shared_slices(a);
    it.part = 0;
    if (i < ms * nss) {
        const int mp = i / nss, sl = i - mp * nss;
        const int mb = kind == 0 ? mp : mp / a.sparts;
        it.u = -1;
        it.mb = mb;
        it.part = kind == 0 ? 0 : mp - mb * a.sparts;
        it.row0 = sl * kPfMaxN;
        it.n = min(kPfMaxN, a.T - it.row0);
        it.N = round16(it.n);
        it.b = (kind == 0 ? a.Bs : a.Hs) + (size_t)it.row0 * 128;
        it.b_kb = (size_t)a.T16 * 128;
        if (kind == 0) {
            it.ntr = min(kPfTR, a.Ls.Ti - kPfTR * mb);
            it.a = a.shared + (size_t)kTileBytes * (kPfTR * mb) * a.Ls.G;
            it.a_row = (size_t)kTileBytes * a.Ls.G;
            it.nkb = a.Ls.G;
        } else {
            // K part p: groups [p Gi, min((p + 1) Gi, Gis)) of the shared down rows
            const int k0 = it.part * a.Lr.Gi;
            it.ntr = min(kPfTR, a.Ls.R - kPfTR * mb);
            it.a = a.shared + a.Ls.gu_bytes + (size_t)kTileBytes * ((size_t)(kPfTR * mb) * a.Ls.Gi + k0);
            it.a_row = (size_t)kTileBytes * a.Ls.Gi;
            it.nkb = a.sparts > 1 ? min(a.Lr.Gi, a.Ls.Gi - k0) : a.Ls.Gi;
            it.b += (size_t)k0 * it.b_kb;
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
        it.b = (kind == 0 ? a.Br : a.Hr) + (size_t)(a.urow[u] + it.row0) * 128;
        it.b_kb = (size_t)a.Rmax * 128;
        const uint8_t *blob = a.experts + (size_t)a.uexp[u] * a.stride;
        if (kind == 0) {
            it.ntr = min(kPfTR, a.Lr.Ti - kPfTR * mb);
            it.a = blob + (size_t)kTileBytes * (kPfTR * mb) * a.Lr.G;
            it.a_row = (size_t)kTileBytes * a.Lr.G;
            it.nkb = a.Lr.G;
        } else {
            it.ntr = min(kPfTR, a.Lr.R - kPfTR * mb);
            it.a = blob + a.Lr.gu_bytes + (size_t)kTileBytes * (kPfTR * mb) * a.Lr.Gi;
            it.a_row = (size_t)kTileBytes * a.Lr.Gi;
            it.nkb = a.Lr.Gi;
        }
    }
    return it;
}

// The 8 codes of a packed word (nibble k of each 16-bit half: one fp16 pair per k)
// as w = s*q + b in fp16.  A code is read in place as an exact fp16 integer: a
// nibble at bits 0-3 of a half under the exponent of 1024 is 1024 + q, one at bits
// 4-7 under the exponent of 64 is 64 + q (its bits are the mantissa's 1/16 places);
// one shift by 8 brings nibbles 2 and 3 to those places.  The subtraction is exact,
// the FMA rounds once.
__device__ __forceinline__ uint4 deq_word(uint32_t w, __half2 s2, __half2 b2) {
    const __half2 k1024 = __halves2half2(__ushort_as_half((unsigned short)0x6400), __ushort_as_half((unsigned short)0x6400));
    const __half2 k64 = __halves2half2(__ushort_as_half((unsigned short)0x5400), __ushort_as_half((unsigned short)0x5400));
    const uint32_t w8 = w >> 8;
    const uint32_t v[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x54005400u,
                           (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x54005400u};
    uint32_t r[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const __half2 q = __hsub2(*reinterpret_cast<const __half2 *>(&v[k]), (k & 1) ? k64 : k1024);  // exact codes
        __half2 d = __hfma2(q, s2, b2);
        r[k] = *reinterpret_cast<uint32_t *>(&d);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// True when the phase of `bar` with the given parity has completed (a non-blocking
// test, tried before the bounded waiting loop on the pipeline's hot paths).
__device__ __forceinline__ bool pf_done(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

struct PfSmem {
    uint64_t q_full[kPfQStages], q_free[kPfQStages];  // operand ring
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
    PrefillGemmArgs a = ga;
    a.U = pl_U;
    a.uslc = pl_uslc;
    a.ucnt = pl_ucnt;
    a.urow = pl_urow;
    a.uexp = pl_uexp;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // 1024-aligned operand stages (per K step: token tile, dequantised weights)
    uint8_t *base = psm_raw + ((1024u - (smem_addr(psm_raw) & 1023u)) & 1023u);
    uint8_t *qst = base;
    volatile int *err = &S.err;

    if (tid == 0) {
        for (int s = 0; s < kPfQStages; s++) {
            // full: the token copier's arrival with the token tiles' bytes, then one
            // arrival per dequantising thread
            mbar_init(&S.q_full[s], 1 + kPfDq * 32);
            mbar_init(&S.q_free[s], 1);
        }
        for (int j = 0; j < 2; j++) {
            mbar_init(&S.acc_full[j], 1);
            mbar_init(&S.acc_empty[j], kPfEpi);
        }
        S.err = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&S.tmem, kPfTmemCols);
    // the plan and the operands are the previous kernels' outputs
    pdl_wait();
    pdl_launch_dependents();
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    // one launch for both GEMMs: the gate/up items, then the down items; a down
    // item's token copier waits until the gate/up items it reads h from are done
    const int NI0 = pf_items(a, 0), NI = NI0 + pf_items(a, 1);
    // (the down items run routed first: the shared expert's K parts 1.. write into the
    // routed token tiles' area, so they wait for every gate/up item and go last)
    const int NS1 = pf_blocks(a.Ls.R) * a.sparts * pf_shared_slices(a), NR1 = NI - NI0 - NS1;
    auto item = [&](int i) -> PfItem {
        if (i < NI0) return pf_item(a, 0, i);
        const int j = i - NI0;
        return pf_item(a, 1, j < NR1 ? j + NS1 : j - NR1);
    };
    const int b = blockIdx.x, nC = gridDim.x;
    auto fail = [&]() {
        *err = 1;
        atomicExch(a.err, 1u);
    };

    if (warp == kPfProducer) {
        // ---------------- token copies (one thread): per operand stage, its token tiles
        // (the MMA's A), issued as soon as the MMA releases the stage
        if (lane == 0) {
            int f = 0;
            int qlast[kPfQStages];
            for (int s = 0; s < kPfQStages; s++) qlast[s] = -1;
            for (int i = b; i < NI; i += nC) {
                const PfItem it = item(i);
                // this item's weight block (first item only) and the next one's, into L2
                if (i == b) prefetch_l2(it.a, (unsigned)(it.ntr * it.a_row));
                if (i + nC < NI) {
                    const PfItem nx = item(i + nC);
                    prefetch_l2(nx.a, (unsigned)(nx.ntr * nx.a_row));
                }
                if (it.kind == 1 && !*err) {
                    // every epilogue warp of the gate/up items this item reads h from has
                    // stored it: the expert's, the shared expert's, or (K parts 1.., which
                    // write into the routed token tiles) all of them
                    const int mr0 = pf_blocks(a.Lr.Ti), ms0 = pf_blocks(a.Ls.Ti);
                    const int d = it.u >= 0 ? it.u : it.part == 0 ? kPfDepShared : kPfDepAll;
                    const unsigned want =
                        (unsigned)kPfEpi * (it.u >= 0 ? mr0 * (a.uslc[it.u + 1] - a.uslc[it.u])
                                            : it.part == 0 ? ms0 * pf_shared_slices(a) : NI0);
                    if (!spin_geq(a.dep + d, want, a.err)) fail();
                    fence_async_global();  // the h stores (generic proxy) before the bulk copies
                }
                for (int kb = 0; kb < it.nkb; kb += kPfQK, f++) {
                    const int q = f % kPfQStages;
                    if (f >= kPfQStages && !*err && !mbar_wait(&S.q_free[q], ((f / kPfQStages) - 1) & 1, err))
                        fail();
                    if (*err) continue;
                    const int nq = min(kPfQK, it.nkb - kb);
                    mbar_arrive_expect_tx(&S.q_full[q], nq * it.N * 128);
                    for (int h = 0; h < nq; h++)
                        bulk_g2s(qst + (size_t)(q * kPfQK + h) * kPfQ, it.b + (size_t)(kb + h) * it.b_kb, it.N * 128,
                                 &S.q_full[q]);
                    qlast[q] = f;
                }
            }
            // drain: the last copies of every stage have landed
            volatile int never = 0;
            for (int s = 0; s < kPfQStages; s++)
                if (qlast[s] >= 0) mbar_wait(&S.q_full[s], (qlast[s] / kPfQStages) & 1, &never);
        }
        __syncwarp();
    } else if (warp == kPfMmaWarp) {
        // ---------------- MMA issue: D[tokens][weight rows] += tokens x weights^T
        if (lane == 0) {
            int f = 0, n_it = 0;
            for (int i = b; i < NI; i += nC, n_it++) {
                const PfItem it = item(i);
                const int ab = n_it & 1;
                if (n_it >= 2 && !*err && !mbar_wait(&S.acc_empty[ab], ((n_it >> 1) - 1) & 1, err)) fail();
                tc_fence_after();
                const uint32_t idesc = umma_idesc_f16(128, 16 * it.ntr);
                for (int kb = 0; kb < it.nkb; kb += kPfQK, f++) {
                    const int q = f % kPfQStages, nq = min(kPfQK, it.nkb - kb);
                    if (!pf_done(&S.q_full[q], (f / kPfQStages) & 1) && !mbar_wait(&S.q_full[q], (f / kPfQStages) & 1, err))
                        fail();
                    tc_fence_after();
                    for (int h = 0; h < nq; h++) {
                        const uint32_t sa = smem_addr(qst + (size_t)(q * kPfQK + h) * kPfQ);
                        const uint32_t sb = sa + kPfTileA;
#pragma unroll
                        for (int ks = 0; ks < 4; ks++)
                            umma_f16(tmem + ab * kPfRows, umma_desc(sa + 32 * ks), umma_desc(sb + 32 * ks), idesc,
                                     kb + h > 0 || ks > 0);
                    }
                    umma_commit(&S.q_free[q]);
                }
                umma_commit(&S.acc_full[ab]);
            }
            // every MMA issued here has finished before tensor memory is released
            if (f > 0) {
                volatile int never = 0;
                const int q = (f - 1) % kPfQStages;
                mbar_wait(&S.q_free[q], ((f - 1) / kPfQStages) & 1, &never);
            }
        }
        __syncwarp();
    } else if (warp < kPfProducer) {
        // ---------------- dequantise: warp d takes tile row d of every K step: weight rows
        // 16 d + r and 16 d + 8 + r (gate/up: the gate and up rows of index 8 d + r, which
        // the epilogue finds 8 columns apart in one thread; the 8 rows of a store cover
        // every 128-byte row phase, so the swizzled stores are conflict-free).  The
        // packed tiles come straight from global memory (the item's block is prefetched
        // into L2 by the token copier), loaded one operand stage ahead into registers.
        const int d = warp;
        const int r = lane >> 2, c = lane & 3;
        const int ra = 16 * d + r, rb = ra + 8;
        const uint32_t oa0 = kPfTileA + sw128_chunk(ra, 2 * c), oa1 = kPfTileA + sw128_chunk(ra, 2 * c + 1);
        const uint32_t ob0 = kPfTileA + sw128_chunk(rb, 2 * c), ob1 = kPfTileA + sw128_chunk(rb, 2 * c + 1);
        // stage cursor: item i, first K step kb; the tiles of the stage in qv / e
        struct Cur {
            int i, kb, nkb;
            bool active;
            const uint8_t *row;  // this warp's tile row, K step 0
        };
        auto at_item = [&](int i) -> Cur {
            Cur u{i, 0, 0, false, nullptr};
            if (i < NI) {
                const PfItem it = item(i);
                u.nkb = it.nkb;
                u.active = d < it.ntr;
                u.row = it.a + (size_t)d * it.a_row;
            }
            return u;
        };
        auto load = [&](const Cur &u, uint4 (&qv)[kPfQK], uint2 (&e)[kPfQK]) {
            if (u.i >= NI || !u.active) return;
#pragma unroll
            for (int h = 0; h < kPfQK; h++)
                if (u.kb + h < u.nkb) {
                    const uint8_t *t = u.row + (size_t)(u.kb + h) * kTileBytes;
                    qv[h] = __ldcs(reinterpret_cast<const uint4 *>(t) + lane);
                    e[h] = __ldcs(reinterpret_cast<const uint2 *>(t + 512) + r);
                }
        };
        Cur cur = at_item(b);
        int f = 0;
        // one operand stage: load the next stage's tiles into (nqv, ne), write the
        // current ones (qv, e); the loop below alternates the two register sets
        auto step = [&](uint4 (&qv)[kPfQK], uint2 (&e)[kPfQK], uint4 (&nqv)[kPfQK], uint2 (&ne)[kPfQK]) {
            Cur nxt = cur;
            nxt.kb += kPfQK;
            if (nxt.kb >= nxt.nkb) nxt = at_item(cur.i + nC);
            load(nxt, nqv, ne);
            const int q = f % kPfQStages, nq = min(kPfQK, cur.nkb - cur.kb);
            // (the wait gives up at once when another warp raised the error word)
            if (f >= kPfQStages && !pf_done(&S.q_free[q], ((f / kPfQStages) - 1) & 1) &&
                !mbar_wait(&S.q_free[q], ((f / kPfQStages) - 1) & 1, err))
                fail();
            if (cur.active) {
#pragma unroll
                for (int h = 0; h < kPfQK; h++)
                    if (h < nq) {
                        uint8_t *slot = qst + (size_t)(q * kPfQK + h) * kPfQ;
                        const __half2 sa2 = __half2half2(__ushort_as_half((unsigned short)(e[h].x & 0xFFFFu)));
                        const __half2 ba2 = __half2half2(__ushort_as_half((unsigned short)(e[h].x >> 16)));
                        const __half2 sb2 = __half2half2(__ushort_as_half((unsigned short)(e[h].y & 0xFFFFu)));
                        const __half2 bb2 = __half2half2(__ushort_as_half((unsigned short)(e[h].y >> 16)));
                        *reinterpret_cast<uint4 *>(slot + oa0) = deq_word(qv[h].x, sa2, ba2);
                        *reinterpret_cast<uint4 *>(slot + oa1) = deq_word(qv[h].y, sa2, ba2);
                        *reinterpret_cast<uint4 *>(slot + ob0) = deq_word(qv[h].z, sb2, bb2);
                        *reinterpret_cast<uint4 *>(slot + ob1) = deq_word(qv[h].w, sb2, bb2);
                    }
                fence_async_smem();
            }
            mbar_arrive(&S.q_full[q]);  // each thread, after its own stores and fence
            cur = nxt;
            f++;
        };
        uint4 qa[kPfQK], qb[kPfQK];
        uint2 ea[kPfQK], eb[kPfQK];
        load(cur, qa, ea);
        while (cur.i < NI) {
            step(qa, ea, qb, eb);
            if (cur.i >= NI) break;
            step(qb, eb, qa, ea);
        }
    } else {
        // ---------------- epilogue (warps kPfEpi0..): tensor-memory lane = token slot,
        // column = weight row; each warp takes one lane quarter and one column half,
        // overlapping the next item's K steps
        const int quad = warp & 3, half = (warp - kPfEpi0) >> 2;
        int n_it = 0;
        for (int i = b; i < NI; i += nC, n_it++) {
            const PfItem it = item(i);
            const int ab = n_it & 1;
            if (!*err && !mbar_wait(&S.acc_full[ab], (n_it >> 1) & 1, err)) fail();
            tc_fence_after();
            const uint32_t trow = tmem + ab * kPfRows + ((uint32_t)(32 * quad) << 16);
            const int t = 32 * quad + lane;  // token slot of this thread
            const int c_beg = (kPfRows / 2) * half, c_end = min(c_beg + kPfRows / 2, 16 * it.ntr);
            if (!*err && 32 * quad < it.N) {
                if (it.kind == 0) {
                    // columns 16 j + k, 16 j + 8 + k: gate and up of intermediate index 128 mb +
                    // 8 j + k; h in the down's operand tiles, 8 indices (one 16-byte chunk) per 16
                    // columns, zero in the padding rows
                    const int row = (it.u < 0 ? 0 : a.urow[it.u]) + it.row0 + t;
                    for (int c0 = c_beg; c0 < c_end; c0 += 16) {
                        float v[16];
                        tmem_ld16(trow + c0, v);
                        if (t < it.N) {
                            float h[8];
#pragma unroll
                            for (int k = 0; k < 8; k++) h[k] = t < it.n ? gelu_tanh(v[k]) * v[k + 8] : 0.f;
                            const __half2 w0 = __floats2half2_rn(h[0], h[4]), w1 = __floats2half2_rn(h[1], h[5]);
                            const __half2 w2 = __floats2half2_rn(h[2], h[6]), w3 = __floats2half2_rn(h[3], h[7]);
                            const int idx = (kPfRows / 2) * it.mb + c0 / 2, kbh = idx / kGroup, ch = (idx % kGroup) / 8;
                            uint8_t *dst = it.u < 0 ? a.Hs + ((size_t)kbh * a.T16 + row) * 128
                                                    : a.Hr + ((size_t)kbh * a.Rmax + row) * 128;
                            *reinterpret_cast<uint4 *>(dst + ((ch ^ (row & 7)) << 4)) =
                                make_uint4(*reinterpret_cast<const uint32_t *>(&w0), *reinterpret_cast<const uint32_t *>(&w1),
                                           *reinterpret_cast<const uint32_t *>(&w2), *reinterpret_cast<const uint32_t *>(&w3));
                        }
                    }
                } else {
                    // columns: output rows kPfRows mb + c of the token's fp32 row
                    float *yrow = nullptr;
                    if (t < it.n)
                        yrow = it.u < 0 ? (it.part ? a.Ys_more + (size_t)(it.part - 1) * a.T16 * a.H : a.Ys) +
                                              (size_t)(it.row0 + t) * a.H
                                        : a.Yr + (size_t)a.rowpair[a.urow[it.u] + it.row0 + t] * a.H;
                    for (int c0 = c_beg; c0 < c_end; c0 += 16) {
                        float v[16];
                        tmem_ld16(trow + c0, v);
                        if (yrow) {
                            float4 *o = reinterpret_cast<float4 *>(yrow + kPfRows * it.mb + c0);
#pragma unroll
                            for (int k = 0; k < 4; k++) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                        }
                    }
                }
            }
            // each warp releases the accumulator once its own reads are done
            tc_fence_before();
            if (it.kind == 0) {
                // this warp's h stores, visible to the down items' bulk copies on any SM
                fence_async_global();
                __threadfence();
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&S.acc_empty[ab]);
                if (it.kind == 0) {
                    atomicAdd(a.dep + (it.u < 0 ? kPfDepShared : it.u), 1u);
                    atomicAdd(a.dep + kPfDepAll, 1u);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kPfTmemCols);
    }
}

// Launches a kernel of the chunk with programmatic dependent launch (each kernel
// waits for its predecessor with griddepcontrol.wait before it reads that one's
// output, and lets its own dependents start right after); a runtime that refuses
// the attribute gets plain launches from then on.
template <typename... KArgs, typename... Args>
inline cudaError_t pf_launch(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
    static std::atomic<int> pdl_ok{1};
    if (pdl_ok.load()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, args...);
        if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return e;
        (void)cudaGetLastError();
        pdl_ok.store(0);
    }
    fn<<<grid, block, smem, st>>>(args...);
    return cudaGetLastError();
}

inline size_t prefill_gemm_smem() {
    return 1024 + (size_t)kPfQStages * kPfQK * kPfQ;
}

// ------------------------------------------------------------------ combine
// One thread per 4 consecutive outputs (H is a multiple of 4): the same fixed order
// of additions per element as one thread per output, with 16-byte loads.
__global__ void __launch_bounds__(256) k_prefill_combine(const float *__restrict__ x, int T, int H, int topk,
                                                         int flags, const float *__restrict__ gate,
                                                         const float *__restrict__ Yr,
                                                         const float *__restrict__ Ys, int sparts,
                                                         const float *__restrict__ Ys_more, int T16,
                                                         float *__restrict__ y) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // float4 index
    const int H4 = H / 4;
    pdl_wait();
    pdl_launch_dependents();
    if (i >= (long long)T * H4) return;
    const int t = (int)(i / H4), n4 = (int)(i % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // every choice's row loaded before the sums (added in choice order)
    float4 v[MOE_MAX_TOPK];
    float g[MOE_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; k++)
        if (k < topk) {
            g[k] = __ldg(gate + t * topk + k);
            v[k] = __ldg(reinterpret_cast<const float4 *>(Yr + (size_t)(t * topk + k) * H) + n4);
        }
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; k++)
        if (k < topk)
            acc = make_float4(fmaf(g[k], v[k].x, acc.x), fmaf(g[k], v[k].y, acc.y), fmaf(g[k], v[k].z, acc.z),
                              fmaf(g[k], v[k].w, acc.w));
    for (int p = 0; p < sparts; p++) {  // the shared expert's K parts, in order
        const float *ys = p ? Ys_more + (size_t)(p - 1) * T16 * H : Ys;
        const float4 sv = __ldg(reinterpret_cast<const float4 *>(ys + (size_t)t * H) + n4);
        acc = make_float4(acc.x + sv.x, acc.y + sv.y, acc.z + sv.z, acc.w + sv.w);
    }
    if (flags & MOE_RESIDUAL) {
        const float4 xv = __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * H) + n4);
        acc = make_float4(acc.x + xv.x, acc.y + xv.y, acc.z + xv.z, acc.w + xv.w);
    }
    reinterpret_cast<float4 *>(y)[i] = acc;
}

}  // namespace moe
