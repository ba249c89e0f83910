// simple_kernels.cuh -- quantiser, standalone 4-bit GEMV, and the CUDA-core expert
// kernels (gate/up + GeGLU, down + gate-weighted combine).
#pragma once

#include "common.cuh"

namespace moe {

// ------------------------------------------------------------------ quantiser
// One thread per (row, group of 64).  Same fp32 operations, in the same order,
// as the definition in moe.h, with explicitly rounded intrinsics so that the
// compiler cannot contract them.
__global__ void k_quantise(const float *__restrict__ w, int N, int K, int bits, uint32_t *q,
                           __half *s, __half *b) {
    const int G = K / kGroup;
    long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)N * G) return;
    const int n = (int)(gid / G), g = (int)(gid % G);
    const float *v = w + (size_t)n * K + (size_t)g * kGroup;
    float mn = v[0], mx = v[0];
    for (int j = 1; j < kGroup; j++) {
        float a = v[j];
        if (a < mn) mn = a;
        if (a > mx) mx = a;
    }
    const unsigned qmax = (1u << bits) - 1u;
    float step = __fdiv_rn(__fsub_rn(mx, mn), (float)qmax);
    __half sh = __float2half_rn(step);
    __half bh = __float2half_rn(mn);
    s[(size_t)n * G + g] = sh;
    b[(size_t)n * G + g] = bh;
    const float sf = __half2float(sh), bf = __half2float(bh);
    const int per_word = 32 / bits;
    uint32_t *out = q + (size_t)n * (K * bits / 32) + (size_t)g * (kGroup / per_word);
    for (int wi = 0; wi < kGroup / per_word; wi++) {
        uint32_t word = 0;
        for (int i = 0; i < per_word; i++) {
            unsigned code = 0;
            if (sf != 0.0f) {
                float t = rintf(__fdiv_rn(__fsub_rn(v[wi * per_word + i], bf), sf));
                t = fminf(fmaxf(t, 0.0f), (float)qmax);
                code = (unsigned)t;
            }
            word |= code << (bits * i);
        }
        out[wi] = word;
    }
}

// ------------------------------------------------------------------ 4-bit dot helpers
// Eight dequantised weights of one word times eight x values.
__device__ __forceinline__ float dot8(uint32_t word, float s, float b, float4 x0, float4 x1,
                                      float acc) {
    acc = fmaf(fmaf(s, (float)((word >> 0) & 0xFu), b), x0.x, acc);
    acc = fmaf(fmaf(s, (float)((word >> 4) & 0xFu), b), x0.y, acc);
    acc = fmaf(fmaf(s, (float)((word >> 8) & 0xFu), b), x0.z, acc);
    acc = fmaf(fmaf(s, (float)((word >> 12) & 0xFu), b), x0.w, acc);
    acc = fmaf(fmaf(s, (float)((word >> 16) & 0xFu), b), x1.x, acc);
    acc = fmaf(fmaf(s, (float)((word >> 20) & 0xFu), b), x1.y, acc);
    acc = fmaf(fmaf(s, (float)((word >> 24) & 0xFu), b), x1.z, acc);
    acc = fmaf(fmaf(s, (float)((word >> 28) & 0xFu), b), x1.w, acc);
    return acc;
}

// ------------------------------------------------------------------ standalone GEMV
// One warp per output row; y[n] = sum_j w[n][j] x[j].
__global__ void __launch_bounds__(128) k_qgemv4_simple(QMat m, const float *__restrict__ x,
                                                       float *__restrict__ y) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * 4 + warp;
    if (n >= m.rows) return;
    const int wpr = m.K / 8, G = m.K / kGroup;
    const uint32_t *row = m.q + (size_t)n * wpr;
    float acc = 0.f;
    for (int w = lane; w < wpr; w += 32) {
        uint32_t word = __ldg(row + w);
        int g = w >> 3;
        float s = __half2float(m.s[(size_t)n * G + g]), b = __half2float(m.b[(size_t)n * G + g]);
        const float4 *xv = (const float4 *)(x + 8 * w);
        acc = dot8(word, s, b, __ldg(xv), __ldg(xv + 1), acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) y[n] = acc;
}

// ------------------------------------------------------------------ expert gate/up
// Item = (distinct expert u, 16 gate rows + the matching 16 up rows), or a tile
// of the shared expert.  h = gelu_tanh(gate . x) * (up . x) per token.
constexpr int kTok = 4;  // tokens per register chunk

__global__ void __launch_bounds__(128) k_expert_up_simple(LayerDev ly, const float *__restrict__ x,
                                                          int T, Ws ws) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tilesR = ly.I / 16;
    const unsigned U = __ldcg(&ws.ctrl[kU]);
    int item = blockIdx.x;
    const bool shared = item >= ws.Umax * tilesR;
    QMat m;
    int Ie, ntok, tile;
    const int *plist = nullptr;
    float *hout;
    if (!shared) {
        const int u = item / tilesR;
        tile = item % tilesR;
        if (u >= (int)U) return;
        const int e = ws.uexp[u];
        m = gu_view(ly.experts + (size_t)e * ly.stride, ly.L, ly.H, ly.I);
        Ie = ly.I;
        ntok = ws.ucount[u];
        plist = ws.ulist + (size_t)u * ws.Tmax;
        hout = ws.h;
    } else {
        tile = item - ws.Umax * tilesR;
        m = gu_view(ly.shared, ly.Ls, ly.H, ly.Is);
        Ie = ly.Is;
        ntok = T;
        hout = ws.hs;
    }
    const int wpr = ly.H / 8, G = ly.H / kGroup;
    for (int r = 0; r < 4; r++) {
        const int i = tile * 16 + warp * 4 + r;
        const uint32_t *rg = m.q + (size_t)i * wpr;
        const uint32_t *ru = m.q + (size_t)(Ie + i) * wpr;
        for (int c0 = 0; c0 < ntok; c0 += kTok) {
            float ag[kTok], au[kTok];
            const float *xp[kTok];
#pragma unroll
            for (int tt = 0; tt < kTok; tt++) {
                ag[tt] = au[tt] = 0.f;
                int c = c0 + tt < ntok ? c0 + tt : ntok - 1;
                int t = plist ? plist[c] / ly.topk : c;
                xp[tt] = x + (size_t)t * ly.H;
            }
            for (int w = lane; w < wpr; w += 32) {
                uint32_t wg = __ldg(rg + w), wu = __ldg(ru + w);
                int g = w >> 3;
                float sg = __half2float(m.s[(size_t)i * G + g]), bg = __half2float(m.b[(size_t)i * G + g]);
                float su = __half2float(m.s[(size_t)(Ie + i) * G + g]);
                float bu = __half2float(m.b[(size_t)(Ie + i) * G + g]);
#pragma unroll
                for (int tt = 0; tt < kTok; tt++) {
                    const float4 *xv = (const float4 *)(xp[tt] + 8 * w);
                    float4 x0 = __ldg(xv), x1 = __ldg(xv + 1);
                    ag[tt] = dot8(wg, sg, bg, x0, x1, ag[tt]);
                    au[tt] = dot8(wu, su, bu, x0, x1, au[tt]);
                }
            }
#pragma unroll
            for (int tt = 0; tt < kTok; tt++) {
                float a = warp_sum(ag[tt]), u = warp_sum(au[tt]);
                if (lane == 0 && c0 + tt < ntok) {
                    int c = c0 + tt;
                    int row = plist ? plist[c] : c;  // pair id (routed) or token (shared)
                    hout[(size_t)row * Ie + i] = gelu_tanh(a) * u;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ expert down + combine
// Item = (distinct expert u, 16 output rows) or (shared, 16 rows): partial[pair][n]
// = Wd_u[n] . h[pair].  The last item to finish a 16-row tile (ticket) combines
// y[t][n] = sum_k gate[t][k] partial[(t,k)][n] + partial_shared[t][n] (+ x[t][n])
// in that fixed order.
__global__ void __launch_bounds__(128) k_expert_down_simple(LayerDev ly, const float *__restrict__ x,
                                                            int T, int flags, float *__restrict__ y,
                                                            Ws ws) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = ly.H / 16;
    const unsigned U = __ldcg(&ws.ctrl[kU]);
    int item = blockIdx.x;
    const bool shared = item >= ws.Umax * tiles;
    QMat m;
    int Ke, ntok, tile;
    const int *plist = nullptr;
    const float *hin;
    const size_t shared_base = (size_t)ws.Tmax * ly.topk;
    if (!shared) {
        const int u = item / tiles;
        tile = item % tiles;
        if (u >= (int)U) return;
        const int e = ws.uexp[u];
        m = down_view(ly.experts + (size_t)e * ly.stride, ly.L, ly.H, ly.I);
        Ke = ly.I;
        ntok = ws.ucount[u];
        plist = ws.ulist + (size_t)u * ws.Tmax;
        hin = ws.h;
    } else {
        tile = item - ws.Umax * tiles;
        m = down_view(ly.shared, ly.Ls, ly.H, ly.Is);
        Ke = ly.Is;
        ntok = T;
        hin = ws.hs;
    }
    const int wpr = Ke / 8, G = Ke / kGroup;
    for (int r = 0; r < 4; r++) {
        const int n = tile * 16 + warp * 4 + r;
        const uint32_t *rw = m.q + (size_t)n * wpr;
        for (int c0 = 0; c0 < ntok; c0 += kTok) {
            float acc[kTok];
            const float *hp[kTok];
#pragma unroll
            for (int tt = 0; tt < kTok; tt++) {
                acc[tt] = 0.f;
                int c = c0 + tt < ntok ? c0 + tt : ntok - 1;
                int row = plist ? plist[c] : c;
                hp[tt] = hin + (size_t)row * Ke;
            }
            for (int w = lane; w < wpr; w += 32) {
                uint32_t word = __ldg(rw + w);
                int g = w >> 3;
                float s = __half2float(m.s[(size_t)n * G + g]), b = __half2float(m.b[(size_t)n * G + g]);
#pragma unroll
                for (int tt = 0; tt < kTok; tt++) {
                    const float4 *hv = (const float4 *)(hp[tt] + 8 * w);
                    acc[tt] = dot8(word, s, b, __ldcg(hv), __ldcg(hv + 1), acc[tt]);
                }
            }
#pragma unroll
            for (int tt = 0; tt < kTok; tt++) {
                float v = warp_sum(acc[tt]);
                if (lane == 0 && c0 + tt < ntok) {
                    int c = c0 + tt;
                    size_t prow = plist ? (size_t)plist[c] : shared_base + c;
                    ws.partial[prow * ly.H + n] = v;
                }
            }
        }
    }
    __shared__ int is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned old = atomicAdd(&ws.tile_cnt[tile], 1u);
        is_last = (old == U);  // U routed items + 1 shared item per tile
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int idx = threadIdx.x; idx < 16 * T; idx += blockDim.x) {
        const int t = idx / 16, n = tile * 16 + idx % 16;
        float acc = 0.f;
        for (int k = 0; k < ly.topk; k++)
            acc = fmaf(__ldcg(&ws.gate[t * ly.topk + k]),
                       __ldcg(&ws.partial[(size_t)(t * ly.topk + k) * ly.H + n]), acc);
        acc += __ldcg(&ws.partial[(shared_base + t) * ly.H + n]);
        if (flags & MOE_RESIDUAL) acc += x[(size_t)t * ly.H + n];
        y[(size_t)t * ly.H + n] = acc;
    }
    if (threadIdx.x == 0) ws.tile_cnt[tile] = 0u;
}

}  // namespace moe
