// attn.cuh -- one attention block over a binary16 key/value cache: the 4-bit
// query/key/value projection with RoPE and the cache store, attention over split
// position ranges with an in-kernel combine, and the 4-bit output projection.
//
// The pages list attention, RoPE, RMSNorm and the quantised GEMV among the engine's
// own kernels, keep the key/value cache in FP16 -- a bounded ring for the 25
// sliding-window layers, a linear store for the 5 full layers -- and quantise the
// attention weights in the same 4-bit affine format as the experts ("TurboFieldfare:
// движок с открытым кодом...", main technical paragraph; "TurboFieldfare esegue Mac
// Gemma 4 26B in 2 GB...", section "Mac Gemma 4 26B entra nello spazio
// disponibile...").  The formulas are the plain readings: rotate-half RoPE at the
// token's position, softmax(scale q.k) over the attended positions, grouped
// key/value heads.
//
// Three launches per call:
//   k_attn_proj<kProjQKV>  [q;k;v] = Wqkv xn on the tensor cores (mma_core.cuh's
//       nibble-as-subnormal trick); a CTA owns 16 rows at dimension i and the 16
//       rows at i + d/2 of one head, so the rotation of each pair happens in its
//       epilogue; queries go to the workspace (rotated, times the score scale),
//       keys and values to their cache slots in binary16.
//   k_attn<D>  a CTA takes one key/value head, up to 8 (token, query head) rows and
//       one slice of the attended positions, in blocks of 64 with a running
//       maximum; its partial (max, sum, unnormalised output) goes to the
//       workspace and the last CTA of the slice set merges them in slice order.
//   k_attn_proj<kProjPlain>  y = Wo o (+ x).
// A sliding-window call with T tokens needs kv_len >= window + T - 1: then the T
// new entries, written before anything is read, overwrite no position that any of
// the T tokens attends to.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "mma_core.cuh"
#include "sync.cuh"

namespace moe {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnRows = 8;       // most (token, query head) rows of one attention tile
constexpr int kAttnMaxSlices = 256;
constexpr int kProjTokens = 8;     // token columns per projection CTA (the MMA's n)
constexpr int kProjQKV = 0, kProjPlain = 1;
// Warps of a projection CTA; they split the K groups.
template <int MODE> struct ProjCfg;
template <> struct ProjCfg<kProjQKV> { static constexpr int warps = 8; };
template <> struct ProjCfg<kProjPlain> { static constexpr int warps = 8; };
template <int MODE> constexpr int proj_threads() { return 32 * ProjCfg<MODE>::warps; }

struct ProjArgs {
    const uint32_t *q;  // weights [N][K], 4-bit affine, MLX layout
    const __half *s, *b;
    int N, K;
    const float *x;  // [T][K]
    int T;
    const float *norm_w;  // RMSNorm gain (QKV mode) or null
    float norm_eps;
    // QKV mode
    int nq, nkv, d, window, kv_len, p0;
    float scale;
    double freq[256];  // RoPE frequencies theta^(-2i/d), i < d/2 (fp64, from the host)
    float *qr;  // [T][nq][d] rotated queries times the score scale
    __half *kc, *vc;  // [nkv][kv_len][d]
    // plain mode
    float *y;            // [T][N]
    const float *resid;  // [T][N] or null
    unsigned *err;       // raised when a bounded wait gives up
};

__host__ __device__ inline int attn_slot(int p, int window, int kv_len) { return window > 0 ? p % kv_len : p; }

// Row stride (halves) of the staged fp16 tokens: K plus 16 bytes, so that the
// lanes of consecutive token columns start in different banks.
__host__ __device__ inline int proj_xs_stride(int K) { return K + 8; }

// Row stride (bytes) of the CTA's weight rows in shared memory: K/2 rounded so
// that it is 32 modulo 128, which puts the 8-byte fragment loads of a half-warp
// (4 rows x 4 lanes) in distinct banks.
__host__ __device__ inline int proj_wrow(int K) { return K / 2 + ((32 - (K / 2) % 128) + 128) % 128; }

// Row stride (bytes) of the CTA's scales and of its biases in shared memory.  When
// a row of G fp16 values is a multiple of 16 bytes (G a multiple of 8) the rows
// are copied one by one into a stride that is an odd multiple of 16 bytes, so
// that the 8 rows a fragment reads at one group sit in distinct banks; otherwise
// the 8-row blocks are copied whole and keep the stride 2G (G = 44: 88 bytes,
// already conflict-free).
__host__ __device__ inline int proj_srow(int K) {
    const int G = K / kGroup;
    return G % 8 ? 2 * G : 2 * G + ((2 * G) % 32 == 0 ? 16 : 0);
}

// Shared memory of a projection CTA: the 16 weight rows, their scales and biases,
// the staged tokens, their per-group sums and the cross-warp reduction.
template <int MODE>
inline size_t proj_smem_bytes(int K, int T) {
    const int rows = T < kProjTokens ? T : kProjTokens;
    return (size_t)16 * proj_wrow(K) + (size_t)2 * 16 * proj_srow(K) +
           sizeof(__half) * rows * proj_xs_stride(K) + sizeof(float) * rows * (K / kGroup) +
           sizeof(float) * ProjCfg<MODE>::warps * 16 * 8;
}

// One CTA computes 16 output rows for up to 8 tokens.  The rows of the MMA tile
// are rowA(g) = ra0 + g and rowB(g) = rb0 + g (g < 8).  In QKV mode a query or key
// tile takes 8 dimensions i..i+7 of one head as rowA and their RoPE partners
// i+d/2.. as rowB, so both halves of every rotated pair end in the same CTA; value
// tiles and the plain mode take 16 consecutive rows.
//
// The weights arrive by bulk copy (one per row, plus the two 8-row blocks of
// scales and of biases), issued at the start, before griddepcontrol.wait: the
// kernels of a step never write them.  The tokens (the previous kernel's output)
// are read after the wait.  The CTA lets its dependents start only after its own
// wait (the attention kernel relies on that).
// MINB: CTAs per SM the registers must allow (the QKV projection 4; the output
// projection 2, which leaves it more registers; a GEMV of more 16-row tiles than two
// waves of 2 per SM takes 4).
template <int MODE, int MINB = (MODE == kProjQKV ? 4 : 2)>
__global__ void __launch_bounds__(proj_threads<MODE>(), MINB) k_attn_proj(const ProjArgs a) {
    constexpr int kWarps = ProjCfg<MODE>::warps, kThreads = 32 * kWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    const int XS = proj_xs_stride(a.K), WR = proj_wrow(a.K), SR = proj_srow(a.K);
    const int G = a.K / kGroup;
    const int t0 = blockIdx.y * kProjTokens, Tc = min(kProjTokens, a.T - t0), Tr = min(a.T, kProjTokens);
    uint8_t *wq = smem;                                                     // [16][WR] codes, rows A then B
    uint8_t *wsb = smem + (size_t)16 * WR;                                  // [2 (s, b)][16][SR bytes]
    __half *xs = reinterpret_cast<__half *>(wsb + (size_t)2 * 16 * SR);     // [Tr][XS] staged tokens
    float *gsum = reinterpret_cast<float *>(xs + (size_t)Tr * XS);          // [Tr][G] sums of xs
    float *red = gsum + Tr * G;                                             // [warp][16][8]
    __shared__ float inv_r[kProjTokens];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gl = lane >> 2, c = lane & 3;

    int ra0, rb0, head = 0, i0 = 0;
    bool pair = false;
    if constexpr (MODE == kProjQKV) {
        const int per = a.d / 16, npair = (a.nq + a.nkv) * per;
        if ((int)blockIdx.x < npair) {
            head = blockIdx.x / per;
            i0 = 8 * (blockIdx.x % per);
            pair = true;
            ra0 = head * a.d + i0;
            rb0 = ra0 + a.d / 2;
        } else {
            ra0 = (a.nq + a.nkv) * a.d + 16 * (blockIdx.x - npair);
            rb0 = ra0 + 8;
        }
    } else {
        ra0 = 16 * blockIdx.x;
        rb0 = ra0 + 8;
    }

    // the CTA's weights: 16 code rows, then scales and biases of rows A and B
    if (warp == 0) {
        const unsigned row_bytes = (unsigned)(a.K / 2), srow = (unsigned)(G * sizeof(__half));
        if (lane == 0) {
            mbar_init(&bar, 1);
            mbar_fence_init();
            abort_flag = 0;
            mbar_arrive_expect_tx(&bar, 16 * row_bytes + 32 * srow);
        }
        __syncwarp();
        const uint8_t *qb = reinterpret_cast<const uint8_t *>(a.q);
        if (lane < 16) {
            const int row = lane < 8 ? ra0 + lane : rb0 + (lane - 8);
            bulk_g2s(wq + (size_t)lane * WR, qb + (size_t)row * row_bytes, row_bytes, &bar);
        }
        if (SR != 2 * G) {  // one copy per scale or bias row: lane = (s | b) x 16 rows
            const int r = lane & 15, row = r < 8 ? ra0 + r : rb0 + (r - 8);
            const __half *src = ((lane & 16) ? a.b : a.s) + (size_t)row * G;
            bulk_g2s(wsb + (size_t)(lane >> 4) * 16 * SR + (size_t)r * SR, src, srow, &bar);
        } else if (lane >= 16 && lane < 20) {  // the 8-row blocks: (scale | bias) x (rows A | rows B)
            const int k = lane - 16;
            const __half *src = ((k & 1) ? a.b : a.s) + (size_t)((k & 2) ? rb0 : ra0) * G;
            bulk_g2s(wsb + (size_t)(k & 1) * 16 * SR + ((k & 2) ? 8 * SR : 0), src, 8 * srow, &bar);
        }
    }
    const int g0 = warp * G / kWarps, g1 = (warp + 1) * G / kWarps;

    // rotation of the pair tile for epilogue thread (r = tid & 7, t = tid >> 3): the
    // angle p * f in fp64, reduced to [-pi, pi] before the fp32 sine and cosine
    float rc = 1.f, rs = 0.f;
    if (MODE == kProjQKV && pair && tid < 64) {
        const int r = tid & 7, t = tid >> 3;
        if (t < Tc) {
            const double ang = (double)(a.p0 + t0 + t) * a.freq[i0 + r];
            const double twopi = 6.283185307179586476925286766559, inv2pi = 0.15915494309189533576888376337251;
            sincosf((float)fma(-rint(ang * inv2pi), twopi, ang), &rs, &rc);
        }
    }
    pdl_wait();
    pdl_launch_dependents();

    // RMSNorm of the CTA's tokens (QKV mode with a gain): every warp sums its share of
    // each token's squares, then the warps' partials are added in warp order
    if (MODE == kProjQKV && a.norm_w) {
        __shared__ float ssp[kWarps][kProjTokens];
        for (int t = 0; t < Tc; t++) {
            const float4 *xr = reinterpret_cast<const float4 *>(a.x + (size_t)(t0 + t) * a.K);
            float ss = 0.f;
            for (int j = tid; j < a.K / 4; j += kThreads) {
                const float4 v = __ldg(xr + j);
                ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) ssp[warp][t] = ss;
        }
        __syncthreads();
        if (tid < Tc) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; w++) ss += ssp[w][tid];
            inv_r[tid] = rsqrtf(ss / (float)a.K + a.norm_eps);
        }
        __syncthreads();
    }
    // stage the tokens as fp16 in fragment order, 8 columns per thread and step,
    // and the sum of each group of 64 staged values (eight consecutive threads hold
    // one group: K/8 is a multiple of 8 and kThreads of 32); the loads of SU steps
    // are issued before any of them is used
    constexpr int SU = 4;
    const int nst = Tc * (a.K / 8);
    for (int u0 = 0; u0 < nst; u0 += SU * kThreads) {
        float4 lo[SU], hi[SU];
#pragma unroll
        for (int k = 0; k < SU; k++) {
            const int u = u0 + k * kThreads + tid;
            if (u < nst) {
                const int t = u / (a.K / 8), j = (u % (a.K / 8)) * 8;
                const float4 *xp = reinterpret_cast<const float4 *>(a.x + (size_t)(t0 + t) * a.K + j);
                lo[k] = __ldg(xp);
                hi[k] = __ldg(xp + 1);
            }
        }
#pragma unroll
        for (int k = 0; k < SU; k++) {
            const int u = u0 + k * kThreads + tid;
            float part = 0.f;
            if (u < nst) {
                const int t = u / (a.K / 8), j = (u % (a.K / 8)) * 8;
                float4 l4 = lo[k], h4 = hi[k];
                if (MODE == kProjQKV && a.norm_w) {
                    const float4 *wp = reinterpret_cast<const float4 *>(a.norm_w + j);
                    const float4 wl = __ldg(wp), wh = __ldg(wp + 1);
                    const float ir = inv_r[t];
                    l4 = make_float4(l4.x * wl.x * ir, l4.y * wl.y * ir, l4.z * wl.z * ir, l4.w * wl.w * ir);
                    h4 = make_float4(h4.x * wh.x * ir, h4.y * wh.y * ir, h4.z * wh.z * ir, h4.w * wh.w * ir);
                }
                // fragment order within the run of 8: (0,4, 1,5, 2,6, 3,7)
                __half2 h0 = __floats2half2_rn(l4.x, h4.x), h1 = __floats2half2_rn(l4.y, h4.y);
                __half2 h2 = __floats2half2_rn(l4.z, h4.z), h3 = __floats2half2_rn(l4.w, h4.w);
                *reinterpret_cast<uint4 *>(xs + (size_t)t * XS + j) =
                    make_uint4(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1),
                               *reinterpret_cast<uint32_t *>(&h2), *reinterpret_cast<uint32_t *>(&h3));
                const float2 f0 = __half22float2(h0), f1 = __half22float2(h1), f2 = __half22float2(h2),
                             f3 = __half22float2(h3);
                part = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
            }
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            if ((u & 7) == 0 && u < nst) gsum[(u / (a.K / 8)) * G + (u % (a.K / 8)) / 8] = part;
        }
    }
    __syncthreads();

    if (!mbar_wait(&bar, 0, &abort_flag)) {
        abort_flag = 1;
        atomicExch(a.err, 1u);
    }
    __syncthreads();
    if (abort_flag) {
        // a copy that never completed may still land: give it time (bounded)
        // before the CTA's shared memory is released; the error word tells the
        // caller that the outputs are not valid
        volatile int no_abort = 0;
        if (tid == 0) mbar_wait(&bar, 0, &no_abort, kWaitNs / 4);
        __syncthreads();
        return;
    }

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int ta = 2 * c, tb = 2 * c + 1;  // the lane's token columns
    const uint8_t *wa_row = wq + (size_t)gl * WR + 8 * c, *wb_row = wq + (size_t)(gl + 8) * WR + 8 * c;
    const __half *sA = reinterpret_cast<const __half *>(wsb + (size_t)gl * SR),
                 *sB = reinterpret_cast<const __half *>(wsb + (size_t)(gl + 8) * SR),
                 *bA = reinterpret_cast<const __half *>(wsb + (size_t)(16 + gl) * SR),
                 *bB = reinterpret_cast<const __half *>(wsb + (size_t)(24 + gl) * SR);
#pragma unroll 4
    for (int g = g0; g < g1; g++) {
        uint32_t xb[8];
        if (gl < Tc)
            load_b(xb, xs + (size_t)gl * XS + g * kGroup + 16 * c);
        else
            zero_b(xb);
        const uint2 wa = *reinterpret_cast<const uint2 *>(wa_row + 32 * g);
        const uint2 wb = *reinterpret_cast<const uint2 *>(wb_row + 32 * g);
        float dd[4] = {0.f, 0.f, 0.f, 0.f};
        mma_group_codes(dd, wa, wb, xb);
        const float sm0 = ta < Tc ? gsum[ta * G + g] : 0.f, sm1 = tb < Tc ? gsum[tb * G + g] : 0.f;
        const float sa = __half2float(sA[g]) * kTwo24, ba = __half2float(bA[g]);
        const float sb = __half2float(sB[g]) * kTwo24, bb = __half2float(bB[g]);
        acc[0] = fmaf(sa, dd[0], fmaf(ba, sm0, acc[0]));
        acc[1] = fmaf(sa, dd[1], fmaf(ba, sm1, acc[1]));
        acc[2] = fmaf(sb, dd[2], fmaf(bb, sm0, acc[2]));
        acc[3] = fmaf(sb, dd[3], fmaf(bb, sm1, acc[3]));
    }
    // accumulator slots: [0] (rowA gl, token 2c), [1] (gl, 2c+1), [2] (rowB gl, 2c), [3] (rowB gl, 2c+1)
    {
        float *rw = red + (size_t)warp * 128;
        rw[gl * 8 + 2 * c] = acc[0];
        rw[gl * 8 + 2 * c + 1] = acc[1];
        rw[(gl + 8) * 8 + 2 * c] = acc[2];
        rw[(gl + 8) * 8 + 2 * c + 1] = acc[3];
    }
    __syncthreads();
    auto total = [&](int r, int t) {  // r < 8: rowA gl = r; r >= 8: rowB gl = r - 8
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; w++) v += red[w * 128 + r * 8 + t];
        return v;
    };
    if constexpr (MODE == kProjPlain) {
        const int r = tid >> 3, t = tid & 7;  // the first 128 threads: 16 rows x 8 tokens
        if (tid < 128 && t < Tc) {
            const int row = r < 8 ? ra0 + r : rb0 + (r - 8);
            const size_t at = (size_t)(t0 + t) * a.N + row;
            float v = total(r, t);
            if (a.resid) v += a.resid[at];
            a.y[at] = v;
        }
        return;
    }
    if (pair) {
        if (tid < 64) {
            const int r = tid & 7, t = tid >> 3;
            if (t < Tc) {
                const float lo = total(r, t), hi = total(r + 8, t);
                const float nlo = lo * rc - hi * rs, nhi = hi * rc + lo * rs;
                const int i = i0 + r, p = a.p0 + t0 + t;
                if (head < a.nq) {
                    float *qrow = a.qr + ((size_t)(t0 + t) * a.nq + head) * a.d;
                    qrow[i] = nlo * a.scale;
                    qrow[i + a.d / 2] = nhi * a.scale;
                } else {
                    __half *krow = a.kc + ((size_t)(head - a.nq) * a.kv_len + attn_slot(p, a.window, a.kv_len)) * a.d;
                    krow[i] = __float2half_rn(nlo);
                    krow[i + a.d / 2] = __float2half_rn(nhi);
                }
            }
        }
    } else {
        const int r = tid >> 3, t = tid & 7;
        if (tid < 128 && t < Tc) {
            const int dim = (r < 8 ? ra0 + r : rb0 + (r - 8)) - (a.nq + a.nkv) * a.d, g = dim / a.d, i = dim % a.d;
            const int p = a.p0 + t0 + t;
            a.vc[((size_t)g * a.kv_len + attn_slot(p, a.window, a.kv_len)) * a.d + i] = __float2half_rn(total(r, t));
        }
    }
}

// ---------------------------------------------------------------- attention

constexpr int kAttnSlice = 32;       // positions per shared-memory block
constexpr int kAttnStages = 2;       // blocks of one CTA in flight at once
constexpr int kAttnMaxCluster = 16;  // CTAs (slices) merged in distributed shared memory

struct AttnArgs {
    const float *qr;  // [T][nq][D] rotated queries times the score scale
    const __half *kc, *vc;
    int nq, nkv, G, kv_len, window, p0, T;
    int S;             // slices of a tile's positions (gridDim.x), a multiple of the cluster size
    int nst;           // shared-memory blocks of a CTA in flight (1 or kAttnStages)
    float *part_o;     // [nkv][tiles][S / cluster][RT][D] unnormalised outputs of the clusters
    float2 *part_ml;   // [nkv][tiles][S / cluster][RT] (running max, sum of weights)
    unsigned *ticket;  // [nkv][tiles]
    unsigned *err;     // raised when a bounded wait gives up
    unsigned extra_tx;            // bytes the first block expects beyond its copies (0; fault injection)
    unsigned long long wait_ns;   // limit of each wait on a block barrier
    float *ao;         // [T][nq D]
    float *ao_user;    // optional copy of ao
};

__device__ __forceinline__ int attn_lo(int p, int window) { return window > 0 ? max(0, p - window + 1) : 0; }

// Shared memory of the attention CTA (dynamic part): the tile's queries, then
// kAttnStages blocks, each of key rows (padded by 16 bytes, so that 32 lanes
// reading 32 rows hit distinct banks) and value rows, binary16.
__host__ __device__ constexpr int attn_kstride(int D) { return D + 8; }  // halves
__host__ __device__ constexpr size_t attn_stage_bytes(int D) {
    return (size_t)kAttnSlice * attn_kstride(D) * sizeof(__half) + (size_t)kAttnSlice * D * sizeof(__half);
}
__host__ __device__ constexpr size_t attn_smem_bytes(int D, int RT, int nst = kAttnStages) {
    return (size_t)RT * D * sizeof(float) + nst * attn_stage_bytes(D);
}

// Issues the bulk copies of positions [c0, c1] (cache rows of one key/value head)
// into rows c0 - u0 .. of a block: one copy per key row (padded rows), one per
// contiguous run of value rows (a ring's wrap splits a run in two).  Lane `lane`
// of the calling warp issues every 32nd key row; lane 0 the value runs.
template <int D>
__device__ __forceinline__ void attn_copy_rows(const AttnArgs &a, const __half *kh, const __half *vh, __half *ks,
                                               __half *vs, int u0, int c0, int c1, uint64_t *bar, int lane) {
    constexpr unsigned kRow = D * sizeof(__half);
    for (int c = c0 + lane; c <= c1; c += 32)
        bulk_g2s(ks + (size_t)(c - u0) * attn_kstride(D), kh + (size_t)attn_slot(c, a.window, a.kv_len) * D, kRow, bar);
    if (lane == 0)
        while (c0 <= c1) {
            const int s0 = attn_slot(c0, a.window, a.kv_len);
            const int n = a.window > 0 ? min(c1 - c0 + 1, a.kv_len - s0) : c1 - c0 + 1;
            bulk_g2s(vs + (size_t)(c0 - u0) * D, vh + (size_t)s0 * D, (unsigned)n * kRow, bar);
            c0 += n;
        }
}

// RT: (token, query head) rows of a tile, 1, 2, 4 or 8 (the host picks the
// smallest power of two that holds the call's rows, at most 8).
//
// Grid (S slices, tiles, key/value heads); the slices of one tile run as thread
// block clusters of up to kAttnMaxCluster CTAs.  A CTA takes its slice's positions
// in blocks of kAttnSlice, nst blocks in flight (bulk copies on one mbarrier per
// stage), and keeps a running maximum and sum per row.  The host gives a slice
// two blocks and makes the tile's slices one cluster when that covers the tile
// (a window of up to 1024 positions); otherwise a slice has one block and its own
// cluster of one.  The cluster
// then merges its slices through distributed shared memory; when one cluster
// covers the tile (a decode token's window or context up to kAttnMaxCluster x 64
// positions) its leader writes the attention output directly, otherwise the
// cluster leaders post partials and the last of them (a ticket) merges those.
//
// Launched with programmatic dependent launch.  Before griddepcontrol.wait the
// CTA starts the bulk copies of the cached rows of earlier tokens (positions below
// this call's first): every kernel of the library signals its dependents only
// after its own wait, so the kernel that wrote those rows has completed by the
// time this one starts.  The rows of this call's own tokens and the queries are
// copied after the wait.
//
// Scores: lane p of every warp takes position p of the block, warp w the
// dimensions [w D/8, (w+1) D/8); each lane forms its partial dot products with the
// tile's queries (no shuffles), warp r then adds the eight partials of row r,
// lane by lane, and runs the online-softmax step.  Values: thread (plane, dims
// 2 slot_d, 2 slot_d + 1) over the positions of its plane.
template <int D, int RT>
__global__ void __launch_bounds__(kAttnThreads) k_attn(const AttnArgs a) {
    namespace cg = cooperative_groups;
    constexpr int PL = kAttnThreads / (D / 2);  // position planes of the value pass
    constexpr int DW = D / kAttnWarps;          // dimensions per warp in the score pass
    constexpr int KS = attn_kstride(D);
    extern __shared__ __align__(128) unsigned char dsm[];
    float *qs = reinterpret_cast<float *>(dsm);  // [RT][D]
    auto kst = [&](int st) {
        return reinterpret_cast<__half *>(dsm + (size_t)RT * D * sizeof(float) + st * attn_stage_bytes(D));
    };
    auto vst = [&](int st) { return kst(st) + (size_t)kAttnSlice * KS; };
    __shared__ float scp[kAttnWarps][RT][kAttnSlice];  // partial scores of each warp
    __shared__ float sc[RT][kAttnSlice];
    __shared__ __align__(16) float red[PL][RT][D];  // the slice's output ends in red[0]
    __shared__ float m_run[RT], l_run[RT], alpha[RT], den[RT], cm[RT];
    __shared__ float ew[RT][kAttnMaxSlices];  // merge: weight of each slice or cluster
    __shared__ float4 part4[kAttnThreads];    // merge: [nph][kAttnThreads / nph] partial sums
    __shared__ int row_p[RT], row_lo[RT];
    __shared__ __align__(8) uint64_t bar[kAttnStages];
    __shared__ int abort_flag;
    __shared__ unsigned last;
    cg::cluster_group cl = cg::this_cluster();
    const int CS = (int)cl.num_blocks(), crank = (int)cl.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, tile = blockIdx.y, h = blockIdx.z;
    const int tiles = gridDim.y, ncl = a.S / CS, cidx = s / CS;
    const int R = min(RT, a.T * a.G - tile * RT);  // live rows of this tile

    // the tile's positions [A, B] and this slice of them, in blocks of kAttnSlice
    const int t_first = tile * RT / a.G, t_last = (tile * RT + R - 1) / a.G;
    const int A = attn_lo(a.p0 + t_first, a.window), B = a.p0 + t_last;
    const int L = (B - A + a.S) / a.S;  // ceil((B - A + 1) / S)
    const int j0 = A + s * L, j1 = min(B, j0 + L - 1);
    const int nblk = j0 <= j1 ? (j1 - j0 + kAttnSlice) / kAttnSlice : 0;
    auto block_n = [&](int bk) { return min(kAttnSlice, j1 - (j0 + bk * kAttnSlice) + 1); };
    const __half *kh = a.kc + (size_t)h * a.kv_len * D;
    const __half *vh = a.vc + (size_t)h * a.kv_len * D;
    const int first = min(nblk, a.nst);  // blocks copied at the start

    if (warp == 0) {
        if (lane == 0) {
            for (int st = 0; st < kAttnStages; st++) mbar_init(&bar[st], 1);
            mbar_fence_init();
            abort_flag = 0;
            // the first blocks' rows (and, on stage 0, the queries)
            for (int bk = 0; bk < first; bk++)
                mbar_arrive_expect_tx(&bar[bk], (unsigned)(2 * block_n(bk) * D * sizeof(__half)) +
                                                    (bk == 0 ? (unsigned)(R * D * sizeof(float)) + a.extra_tx : 0u));
        }
        __syncwarp();
        for (int bk = 0; bk < first; bk++) {
            const int u0 = j0 + bk * kAttnSlice;
            attn_copy_rows<D>(a, kh, vh, kst(bk), vst(bk), u0, u0, min(u0 + block_n(bk) - 1, a.p0 - 1), &bar[bk], lane);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (warp == 0 && nblk) {
        for (int bk = 0; bk < first; bk++) {
            const int u0 = j0 + bk * kAttnSlice;
            attn_copy_rows<D>(a, kh, vh, kst(bk), vst(bk), u0, max(u0, a.p0), u0 + block_n(bk) - 1, &bar[bk], lane);
        }
        // queries: row r is token t's head h G + g
        for (int r = lane; r < R; r += 32) {
            const int rg = tile * RT + r, t = rg / a.G, g = rg % a.G;
            bulk_g2s(qs + (size_t)r * D, a.qr + ((size_t)t * a.nq + h * a.G + g) * D, D * sizeof(float), &bar[0]);
        }
    }
    if (tid < RT) {
        const int rg = tile * RT + tid;
        const int p = tid < R ? a.p0 + rg / a.G : -1;
        row_p[tid] = p;
        row_lo[tid] = tid < R ? attn_lo(p, a.window) : 0;
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
        alpha[tid] = 0.f;
    }
    __syncthreads();

    const int slot_d = tid % (D / 2), plane = tid / (D / 2);
    float acc[RT][2];
#pragma unroll
    for (int r = 0; r < RT; r++) acc[r][0] = acc[r][1] = 0.f;

    int issued = first, bk = 0;
    for (; bk < nblk; bk++) {
        const int st = bk % a.nst;
        const unsigned phase = (unsigned)(bk / a.nst) & 1u;
        const int u0 = j0 + bk * kAttnSlice, nb = block_n(bk);
        const __half *ks = kst(st), *vs = vst(st);
        if (!mbar_wait(&bar[st], phase, &abort_flag, a.wait_ns)) {
            abort_flag = 1;
            atomicExch(a.err, 1u);
        }
        __syncthreads();
        if (abort_flag) break;
        // partial scores: lane = position, warp = dimensions [warp DW, warp DW + DW)
        {
            float part[RT];
#pragma unroll
            for (int r = 0; r < RT; r++) part[r] = 0.f;
            if (lane < nb) {
                const __half *krow = ks + (size_t)lane * KS + warp * DW;
#pragma unroll
                for (int c8 = 0; c8 < DW / 8; c8++) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(krow + 8 * c8);
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                    float kf[8];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ww[i]));
                        kf[2 * i] = f.x;
                        kf[2 * i + 1] = f.y;
                    }
#pragma unroll
                    for (int r = 0; r < RT; r++) {
                        const float4 q0 = *reinterpret_cast<const float4 *>(qs + (size_t)r * D + warp * DW + 8 * c8);
                        const float4 q1 = *reinterpret_cast<const float4 *>(qs + (size_t)r * D + warp * DW + 8 * c8 + 4);
                        float v = part[r];
                        v = fmaf(q0.x, kf[0], v); v = fmaf(q0.y, kf[1], v);
                        v = fmaf(q0.z, kf[2], v); v = fmaf(q0.w, kf[3], v);
                        v = fmaf(q1.x, kf[4], v); v = fmaf(q1.y, kf[5], v);
                        v = fmaf(q1.z, kf[6], v); v = fmaf(q1.w, kf[7], v);
                        part[r] = v;
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < RT; r++) scp[warp][r][lane] = part[r];
        }
        __syncthreads();
        // row r (warp r): the score of position lane, the running maximum and weights
        if (warp < R) {
            float v = -INFINITY;
            if (lane < nb) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kAttnWarps; w++) sum += scp[w][warp][lane];
                const int j = u0 + lane;
                v = (j >= row_lo[warp] && j <= row_p[warp]) ? sum : -INFINITY;
            }
            float m = v;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float mo = m_run[warp], mn = fmaxf(mo, m);
            const float e = (lane < nb && mn != -INFINITY) ? __expf(v - mn) : 0.f;
            sc[warp][lane] = e;
            float l = e;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (lane == 0) {
                const float al = mo == -INFINITY ? 0.f : __expf(mo - mn);
                alpha[warp] = al;
                l_run[warp] = l_run[warp] * al + l;
                m_run[warp] = mn;
            }
        }
        __syncthreads();
        // values
#pragma unroll
        for (int r = 0; r < RT; r++) {
            acc[r][0] *= alpha[r];
            acc[r][1] *= alpha[r];
        }
#pragma unroll 4
        for (int jj = plane; jj < nb; jj += PL) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(vs + (size_t)jj * D + 2 * slot_d));
#pragma unroll
            for (int r = 0; r < RT; r++) {
                const float w = sc[r][jj];
                acc[r][0] = fmaf(w, v.x, acc[r][0]);
                acc[r][1] = fmaf(w, v.y, acc[r][1]);
            }
        }
        __syncthreads();  // the stage's rows and the scores are free again
        if (issued < nblk && warp == 0) {  // the next block into the freed stage
            const int u2 = j0 + issued * kAttnSlice, n2 = block_n(issued);
            if (lane == 0) mbar_arrive_expect_tx(&bar[st], (unsigned)(2 * n2 * D * sizeof(__half)));
            __syncwarp();
            attn_copy_rows<D>(a, kh, vh, kst(st), vst(st), u2, u2, u2 + n2 - 1, &bar[st], lane);
        }
        if (issued < nblk) issued++;
    }
    if (abort_flag) {
        // copies that never completed may still land: give each stage in flight time
        // (bounded) before the CTA's shared memory is released; the slice then counts
        // as empty (the error word tells the caller that the outputs are not valid)
        volatile int no_abort = 0;
        if (tid == 0)
            for (int k = bk; k < issued; k++)
                mbar_wait(&bar[k % a.nst], (unsigned)(k / a.nst) & 1u, &no_abort, a.wait_ns);
#pragma unroll
        for (int r = 0; r < RT; r++) acc[r][0] = acc[r][1] = 0.f;
        if (tid < RT) {
            m_run[tid] = -INFINITY;
            l_run[tid] = 0.f;
        }
        __syncthreads();
    }

    // the slice's output (planes summed in order) into red[0]
#pragma unroll
    for (int r = 0; r < RT; r++) {
        red[plane][r][2 * slot_d] = acc[r][0];
        red[plane][r][2 * slot_d + 1] = acc[r][1];
    }
    __syncthreads();
    if (PL > 1)
        for (int u = tid; u < RT * (D / 4); u += kAttnThreads) {
            const int r = u / (D / 4), i = (u % (D / 4)) * 4;
            float4 v = *reinterpret_cast<const float4 *>(&red[0][r][i]);
#pragma unroll
            for (int pl = 1; pl < PL; pl++) {
                const float4 w = *reinterpret_cast<const float4 *>(&red[pl][r][i]);
                v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
            }
            *reinterpret_cast<float4 *>(&red[0][r][i]) = v;
        }

    // ---- the cluster's slices merged by its leader (distributed shared memory)
    cl.sync();
    if (crank == 0) {
        if (warp < R) {  // row `warp`: the largest maximum, each slice's weight, the total
            const float mk = lane < CS ? *cl.map_shared_rank(&m_run[warp], lane) : -INFINITY;
            const float lk = lane < CS ? *cl.map_shared_rank(&l_run[warp], lane) : 0.f;
            float M = lk > 0.f ? mk : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float e = lk > 0.f ? __expf(mk - M) : 0.f;
            if (lane < CS) ew[warp][lane] = e;
            float lt = lk * e;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
            if (lane == 0) {
                cm[warp] = M;
                den[warp] = lt;
            }
        }
        __syncthreads();
        for (int u = tid; u < R * (D / 4); u += kAttnThreads) {
            const int r = u / (D / 4), i = (u % (D / 4)) * 4;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k0 = 0; k0 < CS; k0 += 4) {  // four CTAs' rows in flight at a time
                float4 v[4];
#pragma unroll
                for (int k = 0; k < 4; k++)
                    v[k] = k0 + k < CS ? *reinterpret_cast<const float4 *>(cl.map_shared_rank(&red[0][r][i], k0 + k))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const float e = k0 + k < CS ? ew[r][k0 + k] : 0.f;
                    o.x = fmaf(v[k].x, e, o.x); o.y = fmaf(v[k].y, e, o.y);
                    o.z = fmaf(v[k].z, e, o.z); o.w = fmaf(v[k].w, e, o.w);
                }
            }
            if (ncl == 1) {  // the whole tile: the attention output
                const int rg = tile * RT + r, t = rg / a.G, g = rg % a.G;
                const float inv = 1.f / den[r];
                const float4 out = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
                const size_t at = (size_t)t * a.nq * D + (size_t)(h * a.G + g) * D + i;
                *reinterpret_cast<float4 *>(a.ao + at) = out;
                if (a.ao_user) *reinterpret_cast<float4 *>(a.ao_user + at) = out;
            } else {
                const size_t pbase = (((size_t)h * tiles + tile) * ncl + cidx) * RT;
                *reinterpret_cast<float4 *>(a.part_o + (pbase + r) * D + i) = o;
            }
        }
        if (ncl > 1 && tid < R) {
            const size_t pbase = (((size_t)h * tiles + tile) * ncl + cidx) * RT;
            a.part_ml[pbase + tid] = make_float2(cm[tid], den[tid]);
        }
    }
    cl.sync();  // the leader has read every slice: the others may leave
    if (crank != 0 || ncl == 1) return;

    // ---- several clusters: the last leader of (head, tile) merges their partials
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&a.ticket[h * tiles + tile], 1u);
        last = prev == (unsigned)ncl - 1u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const size_t pb0 = ((size_t)h * tiles + tile) * ncl * RT;
    if (warp < R) {
        constexpr int PerLane = kAttnMaxSlices / 32;
        float2 ml[PerLane];
#pragma unroll
        for (int k = 0; k < PerLane; k++) {
            const int q = lane + 32 * k;
            ml[k] = q < ncl ? __ldcg(a.part_ml + pb0 + (size_t)q * RT + warp) : make_float2(-INFINITY, 0.f);
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < PerLane; k++)
            if (ml[k].y > 0.f) M = fmaxf(M, ml[k].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float l = 0.f;
#pragma unroll
        for (int k = 0; k < PerLane; k++) {
            const int q = lane + 32 * k;
            const float e = ml[k].y > 0.f ? __expf(ml[k].x - M) : 0.f;
            if (q < ncl) ew[warp][q] = e;
            l = fmaf(ml[k].y, e, l);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) den[warp] = l;
    }
    __syncthreads();
    // the weighted sum of the partials, four dimensions per item; the partials are
    // split over nph phases when there are fewer items than threads
    const int items = R * (D / 4);
    const int nph = items >= kAttnThreads ? 1 : kAttnThreads / items;
    const int per = kAttnThreads / nph;
    for (int base = 0; base < items; base += per) {
        const int it = base + tid % per, ph = tid / per;
        const bool live = it < items && ph < nph;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
            const int r = it / (D / 4), i = (it % (D / 4)) * 4;
            const float4 *src = reinterpret_cast<const float4 *>(a.part_o + (pb0 + r) * D + i);
            const size_t stride = (size_t)RT * D / 4;  // float4s from one partial to the next
            for (int q = ph; q < ncl; q += 8 * nph) {
                float4 v[8];
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const int qq = q + k * nph;
                    v[k] = qq < ncl ? __ldcg(src + (size_t)qq * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const int qq = q + k * nph;
                    const float e = qq < ncl ? ew[r][qq] : 0.f;
                    num.x = fmaf(v[k].x, e, num.x); num.y = fmaf(v[k].y, e, num.y);
                    num.z = fmaf(v[k].z, e, num.z); num.w = fmaf(v[k].w, e, num.w);
                }
            }
        }
        if (nph > 1) {
            __syncthreads();
            if (live) part4[ph * per + (it - base)] = num;
            __syncthreads();
            if (ph != 0 || !live) continue;
            for (int k = 1; k < nph; k++) {
                const float4 w = part4[k * per + (it - base)];
                num.x += w.x; num.y += w.y; num.z += w.z; num.w += w.w;
            }
        } else if (!live) {
            continue;
        }
        const int r = it / (D / 4), i = (it % (D / 4)) * 4;
        const int rg = tile * RT + r, t = rg / a.G, g = rg % a.G;
        const float inv = 1.f / den[r];
        const float4 o = make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
        const size_t at = (size_t)t * a.nq * D + (size_t)(h * a.G + g) * D + i;
        *reinterpret_cast<float4 *>(a.ao + at) = o;
        if (a.ao_user) *reinterpret_cast<float4 *>(a.ao_user + at) = o;
    }
    if (tid == 0) a.ticket[h * tiles + tile] = 0u;  // ready for the next call
}

}  // namespace moe
