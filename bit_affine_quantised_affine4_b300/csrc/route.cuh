// route.cuh -- router GEMV (8-bit affine), top-k with softmax gates, and the
// per-call schedule of distinct experts.
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

// Ranking used by top-k: larger value first, equal values -> lower index.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// Top-k of token t's E logits by one warp; writes idx/gate (workspace + optional
// caller outputs).
__device__ void warp_topk_softmax(const float *logits, int E, int topk, int t, int *ws_idx,
                                  float *ws_gate, int32_t *idx_out, float *gate_out) {
    const int lane = threadIdx.x & 31;
    float v[MOE_MAX_EXPERTS / 32];
    unsigned taken = 0;
#pragma unroll
    for (int i = 0; i < MOE_MAX_EXPERTS / 32; i++) {
        int e = lane + 32 * i;
        float x = e < E ? __ldcg(logits + (size_t)t * E + e) : -INFINITY;
        v[i] = (x != x) ? -INFINITY : x;  // NaN ranks last
    }
    float sel_v[MOE_MAX_TOPK];
    int sel_i[MOE_MAX_TOPK];
    for (int k = 0; k < topk; k++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < MOE_MAX_EXPERTS / 32; i++) {
            int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && ranks_before(v[i], e, bv, bi)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_before(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        sel_v[k] = bv;
        sel_i[k] = bi;
    }
    if (lane == 0) {
        float m = sel_v[0];
        float ex[MOE_MAX_TOPK];
        float z = 0.f;
        for (int k = 0; k < topk; k++) {
            ex[k] = expf(sel_v[k] - m);
            z += ex[k];
        }
        for (int k = 0; k < topk; k++) {
            float g = ex[k] / z;
            ws_idx[t * topk + k] = sel_i[k];
            ws_gate[t * topk + k] = g;
            if (idx_out) idx_out[t * topk + k] = sel_i[k];
            if (gate_out) gate_out[t * topk + k] = g;
        }
    }
}

// Distinct experts of the call in ascending id order, and for each the pairs
// p = t*topk + k that chose it, ascending (a stable counting sort).  Run by one
// CTA after all idx are written.
__device__ void build_schedule(const LayerDev &ly, int T, Ws ws) {
    __shared__ int cnt[MOE_MAX_EXPERTS];
    __shared__ int uid[MOE_MAX_EXPERTS];
    __shared__ int fill[MOE_MAX_EXPERTS];
    const int P = T * ly.topk;
    for (int e = threadIdx.x; e < ly.E; e += blockDim.x) {
        cnt[e] = 0;
        fill[e] = 0;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) atomicAdd(&cnt[ws.idx[p]], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        int U = 0;
        for (int e = 0; e < ly.E; e++) {
            if (cnt[e] > 0) {
                uid[e] = U;
                ws.uexp[U] = e;
                ws.ucount[U] = cnt[e];
                U++;
            } else {
                uid[e] = -1;
            }
        }
        ws.ctrl[kU] = (unsigned)U;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        for (int base = 0; base < P; base += 32) {
            int p = base + lane;
            int e = p < P ? ws.idx[p] : -1 - lane;
            unsigned same = __match_any_sync(0xffffffffu, e);
            int rank = __popc(same & ((1u << lane) - 1u));
            if (p < P) {
                int u = uid[e];
                ws.ulist[(size_t)u * ws.Tmax + fill[u] + rank] = p;
            }
            __syncwarp();
            if (p < P && rank == 0) fill[uid[e]] += __popc(same);
            __syncwarp();
        }
    }
}

// logits for router rows e (one per warp) for all T tokens; the last CTA to finish
// runs top-k + softmax for every token and builds the schedule.
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
        warp_topk_softmax(ws.logits, ly.E, ly.topk, t, ws.idx, ws.gate, idx_out, gate_out);
    __syncthreads();
    build_schedule(ly, T, ws);
    if (threadIdx.x == 0) ws.ctrl[kRouteTicket] = 0u;
}

}  // namespace moe
