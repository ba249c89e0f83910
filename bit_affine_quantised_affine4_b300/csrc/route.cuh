// route.cuh -- router GEMV (8-bit affine) and top-k with softmax gates.
//
// Router: logits[t][e] = sum_j (s q + b)[e][j] x[t][j] (+ bias[e]); the 8-bit
// router and the top-8 choice per token per layer are the devtrends page's
// "Qual e il trucco principale dell'architettura" and the remio.ai page's
// "L'affermazione dei 2 GB...".  Gates (softmax over the chosen logits) and the
// tie rule (equal logits -> lower expert index) are this library's reading.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRouteWarps = 8;  // one router row per warp

// Order-preserving key of a logit for the top-k: a larger value gives a larger
// key; -0 and +0 are equal; NaN gets 1, below every number; 0 marks an entry
// that is out of range or already taken.
__device__ __forceinline__ unsigned topk_key(float v) {
    if (v != v) return 1u;
    if (v == 0.f) v = 0.f;
    const unsigned u = __float_as_uint(v);
    const unsigned k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return k > 1u ? k : 2u;
}

// Top-k of one token's E logits by one warp, then softmax over the chosen ones.
// Larger logit first, equal logits -> lower expert index.  Each round takes the
// warp maximum of the keys (__reduce_max_sync) and the lowest index holding it
// (__reduce_min_sync).  lrow: the token's logits (read through L2: other CTAs
// may have written them).  Writes idx_dst/gate_dst (any memory) and, when
// non-null, idx_out/gate_out.
__device__ void warp_topk_softmax(const float *lrow, int E, int topk, int *idx_dst, float *gate_dst,
                                  int32_t *idx_out, float *gate_out) {
    const int lane = threadIdx.x & 31;
    constexpr int NV = MOE_MAX_EXPERTS / 32;
    unsigned key[NV];
    float val[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        val[i] = e < E ? __ldcg(lrow + e) : 0.f;
        key[i] = e < E ? topk_key(val[i]) : 0u;
    }
    float sel_v[MOE_MAX_TOPK];
    int sel_i[MOE_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; k++) {
        sel_v[k] = 0.f;
        sel_i[k] = 0;
        if (k < topk) {
            unsigned best = key[0];
            int bi = lane;
#pragma unroll
            for (int i = 1; i < NV; i++)
                if (key[i] > best) {
                    best = key[i];
                    bi = lane + 32 * i;
                }
            const unsigned m = __reduce_max_sync(0xffffffffu, best);
            const int win = __reduce_min_sync(0xffffffffu, best == m ? bi : 0x7fffffff);
            float v = 0.f;
#pragma unroll
            for (int i = 0; i < NV; i++)
                if (win == lane + 32 * i) {
                    v = val[i];
                    key[i] = 0u;
                }
            sel_v[k] = __shfl_sync(0xffffffffu, v, win & 31);
            sel_i[k] = win;
        }
    }
    if (lane == 0) {
        const float m = sel_v[0];
        float ex[MOE_MAX_TOPK];
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < MOE_MAX_TOPK; k++) {
            ex[k] = k < topk ? expf(sel_v[k] - m) : 0.f;
            z += ex[k];
        }
#pragma unroll
        for (int k = 0; k < MOE_MAX_TOPK; k++) {
            if (k < topk) {
                const float g = ex[k] / z;
                idx_dst[k] = sel_i[k];
                gate_dst[k] = g;
                if (idx_out) idx_out[k] = sel_i[k];
                if (gate_out) gate_out[k] = g;
            }
        }
    }
}

// logits for router rows e (one per warp) for all T tokens; the last CTA to finish
// runs top-k + softmax for every token.
template <int TCH>
__global__ void __launch_bounds__(kRouteWarps * 32)
k_route(LayerDev ly, const float *__restrict__ x, int T, Ws ws, int32_t *idx_out, float *gate_out,
        float *logits_out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouteWarps + warp;
    const int wpr = ly.H / 4;
    const int G = ly.H / kGroup;
    if (e < ly.E) {
        const uint32_t *row = ly.rq + (size_t)e * wpr;
        for (int t0 = 0; t0 < T; t0 += TCH) {
            float acc[TCH];
#pragma unroll
            for (int i = 0; i < TCH; i++) acc[i] = 0.f;
            for (int w = lane; w < wpr; w += 32) {
                uint32_t word = __ldg(row + w);
                int g = w >> 4;
                float s = __half2float(ly.rs[(size_t)e * G + g]);
                float b = __half2float(ly.rb[(size_t)e * G + g]);
                float wv[4];
#pragma unroll
                for (int i = 0; i < 4; i++) wv[i] = fmaf(s, (float)((word >> (8 * i)) & 0xFFu), b);
#pragma unroll
                for (int tt = 0; tt < TCH; tt++) {
                    if (t0 + tt < T) {
                        float4 xv = __ldg((const float4 *)(x + (size_t)(t0 + tt) * ly.H) + w);
                        acc[tt] = fmaf(wv[0], xv.x, acc[tt]);
                        acc[tt] = fmaf(wv[1], xv.y, acc[tt]);
                        acc[tt] = fmaf(wv[2], xv.z, acc[tt]);
                        acc[tt] = fmaf(wv[3], xv.w, acc[tt]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < TCH; tt++) {
                float v = warp_sum(acc[tt]);
                if (lane == 0 && t0 + tt < T) {
                    if (ly.bias) v += ly.bias[e];
                    ws.logits[(size_t)(t0 + tt) * ly.E + e] = v;
                    if (logits_out) logits_out[(size_t)(t0 + tt) * ly.E + e] = v;
                }
            }
        }
    }
    __shared__ int is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned tk = atomicAdd(&ws.ctrl[kRouteTicket], 1u);
        is_last = (tk == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int t = warp; t < T; t += kRouteWarps)
        warp_topk_softmax(ws.logits + (size_t)t * ly.E, ly.E, ly.topk, idx_out + t * ly.topk,
                          gate_out + t * ly.topk, nullptr, nullptr);
    if (threadIdx.x == 0) ws.ctrl[kRouteTicket] = 0u;
}

}  // namespace moe
