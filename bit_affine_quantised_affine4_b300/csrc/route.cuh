// route.cuh -- router GEMV (8-bit affine) and top-k with softmax gates.
//
// Router: logits[t][e] = sum_j (s q + b)[e][j] x[t][j] (+ bias[e]); the 8-bit
// router and the top-8 choice per token per layer are the devtrends page's
// "Qual e il trucco principale dell'architettura" and the remio.ai page's
// "L'affermazione dei 2 GB...".  Gates (softmax over the chosen logits) and the
// tie rule (equal logits -> lower expert index) are this library's reading.
#pragma once

#include "common.cuh"
#include "lfu_dev.cuh"

namespace moe {


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
// Larger logit first, equal logits -> lower expert index.  Each lane holds NV
// keys (experts lane, lane + 32, ...); each round takes the warp maximum of the
// keys (__reduce_max_sync) and the lowest index holding it (__reduce_min_sync),
// and lane k keeps the k-th choice.  The gates are then computed by lanes
// 0..topk-1 together.  lrow: the token's logits (read through L2 when SMEM is
// false: other CTAs may have written them).  Writes idx_dst/gate_dst (any
// memory) and, when non-null, idx_out/gate_out.
template <bool SMEM, int NV>
__device__ void warp_topk_softmax_nv(const float *lrow, int E, int topk, int *idx_dst, float *gate_dst,
                                     int32_t *idx_out, float *gate_out) {
    const int lane = threadIdx.x & 31;
    unsigned key[NV];
    float val[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        val[i] = e < E ? (SMEM ? lrow[e] : __ldcg(lrow + e)) : 0.f;
        key[i] = e < E ? topk_key(val[i]) : 0u;
    }
    float my_v = 0.f;
    int my_i = 0;
#pragma unroll 1
    for (int k = 0; k < topk; k++) {
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
        v = __shfl_sync(0xffffffffu, v, win & 31);
        if (lane == k) {
            my_v = v;
            my_i = win;
        }
    }
    // softmax over the chosen logits (the first is the largest)
    const float m0 = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < topk ? expf(my_v - m0) : 0.f;
    const float z = warp_sum(ex);
    if (lane < topk) {
        const float g = ex / z;
        idx_dst[lane] = my_i;
        gate_dst[lane] = g;
        if (idx_out) idx_out[lane] = my_i;
        if (gate_out) gate_out[lane] = g;
    }
}

template <bool SMEM = false>
__device__ __forceinline__ void warp_topk_softmax(const float *lrow, int E, int topk, int *idx_dst, float *gate_dst,
                                                  int32_t *idx_out, float *gate_out) {
    if (E <= 128)
        warp_topk_softmax_nv<SMEM, 4>(lrow, E, topk, idx_dst, gate_dst, idx_out, gate_out);
    else
        warp_topk_softmax_nv<SMEM, MOE_MAX_EXPERTS / 32>(lrow, E, topk, idx_dst, gate_dst, idx_out, gate_out);
}

// x columns 8p..8p+7 of a token row as two float4, multiplied elementwise by the
// RMSNorm weight g when one is given (the 1 / rms factor is applied to the sums).
__device__ __forceinline__ void load_x8(const float4 *xt, const float4 *g4, int p, float4 &x0, float4 &x1) {
    x0 = __ldg(xt + 2 * p);
    x1 = __ldg(xt + 2 * p + 1);
    if (g4) {
        const float4 g0 = __ldg(g4 + 2 * p), g1 = __ldg(g4 + 2 * p + 1);
        x0 = make_float4(x0.x * g0.x, x0.y * g0.y, x0.z * g0.z, x0.w * g0.w);
        x1 = make_float4(x1.x * g1.x, x1.y * g1.y, x1.z * g1.z, x1.w * g1.w);
    }
}

// Partial router logit of row e for token t over the word pairs [p0, p1) of the
// 8-bit row (pair p holds columns 8p..8p+7), summed over the warp; x is scaled
// elementwise by g when g is non-null.
__device__ __forceinline__ float router_dot(const uint32_t *rq, const __half *rs, const __half *rb, int H,
                                            const float *x, int e, int t, int p0, int p1,
                                            const float *g = nullptr) {
    const int lane = threadIdx.x & 31, G = H / kGroup;
    const uint2 *row = reinterpret_cast<const uint2 *>(rq + (size_t)e * (H / 4));
    const float4 *xt = reinterpret_cast<const float4 *>(x + (size_t)t * H);
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    const __half *sr = rs + (size_t)e * G, *br = rb + (size_t)e * G;
    float acc = 0.f;
#pragma unroll 4
    for (int p = p0 + lane; p < p1; p += 32) {
        const uint2 w = __ldg(row + p);
        const float s = __half2float(sr[p >> 3]), bb = __half2float(br[p >> 3]);
        float4 x0, x1;
        load_x8(xt, g4, p, x0, x1);
        acc = fmaf(fmaf(s, (float)(w.x & 0xFFu), bb), x0.x, acc);
        acc = fmaf(fmaf(s, (float)((w.x >> 8) & 0xFFu), bb), x0.y, acc);
        acc = fmaf(fmaf(s, (float)((w.x >> 16) & 0xFFu), bb), x0.z, acc);
        acc = fmaf(fmaf(s, (float)(w.x >> 24), bb), x0.w, acc);
        acc = fmaf(fmaf(s, (float)(w.y & 0xFFu), bb), x1.x, acc);
        acc = fmaf(fmaf(s, (float)((w.y >> 8) & 0xFFu), bb), x1.y, acc);
        acc = fmaf(fmaf(s, (float)((w.y >> 16) & 0xFFu), bb), x1.z, acc);
        acc = fmaf(fmaf(s, (float)(w.y >> 24), bb), x1.w, acc);
    }
    return warp_sum(acc);
}

constexpr int kRouteTok = 16;  // tokens per router CTA (one warp each)
constexpr int kRouteExp = 4;   // router rows per CTA (each token vector read once for all of them)

// Router rows e0 .. e0 + NE - 1 (those < E) for token t, over the whole row:
// router_dot's arithmetic for each row, with each x element loaded once for all.
// With a RMSNorm weight g, x is scaled by g and *ss receives the token's sum of
// squares of x (the caller applies 1 / rms to the sums).
template <int NE>
__device__ __forceinline__ void router_dot_rows(const uint32_t *rq, const __half *rs, const __half *rb, int H,
                                                int E, const float *x, int e0, int t, float (&out)[NE],
                                                const float *g = nullptr, float *ss = nullptr) {
    const int lane = threadIdx.x & 31, G = H / kGroup, np = H / 8;
    const float4 *xt = reinterpret_cast<const float4 *>(x + (size_t)t * H);
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    float acc[NE];
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < NE; j++) acc[j] = 0.f;
#pragma unroll 2
    for (int p = lane; p < np; p += 32) {
        float4 x0 = __ldg(xt + 2 * p), x1 = __ldg(xt + 2 * p + 1);
        if (g4) {
            sq += x0.x * x0.x + x0.y * x0.y + x0.z * x0.z + x0.w * x0.w;
            sq += x1.x * x1.x + x1.y * x1.y + x1.z * x1.z + x1.w * x1.w;
            const float4 g0 = __ldg(g4 + 2 * p), g1 = __ldg(g4 + 2 * p + 1);
            x0 = make_float4(x0.x * g0.x, x0.y * g0.y, x0.z * g0.z, x0.w * g0.w);
            x1 = make_float4(x1.x * g1.x, x1.y * g1.y, x1.z * g1.z, x1.w * g1.w);
        }
#pragma unroll
        for (int j = 0; j < NE; j++) {
            const int e = e0 + j < E ? e0 + j : E - 1;
            const uint2 w = __ldg(reinterpret_cast<const uint2 *>(rq + (size_t)e * (H / 4)) + p);
            const float sc = __half2float(rs[(size_t)e * G + (p >> 3)]), bb = __half2float(rb[(size_t)e * G + (p >> 3)]);
            float a = acc[j];
            a = fmaf(fmaf(sc, (float)(w.x & 0xFFu), bb), x0.x, a);
            a = fmaf(fmaf(sc, (float)((w.x >> 8) & 0xFFu), bb), x0.y, a);
            a = fmaf(fmaf(sc, (float)((w.x >> 16) & 0xFFu), bb), x0.z, a);
            a = fmaf(fmaf(sc, (float)(w.x >> 24), bb), x0.w, a);
            a = fmaf(fmaf(sc, (float)(w.y & 0xFFu), bb), x1.x, a);
            a = fmaf(fmaf(sc, (float)((w.y >> 8) & 0xFFu), bb), x1.y, a);
            a = fmaf(fmaf(sc, (float)((w.y >> 16) & 0xFFu), bb), x1.z, a);
            a = fmaf(fmaf(sc, (float)(w.y >> 24), bb), x1.w, a);
            acc[j] = a;
        }
    }
#pragma unroll
    for (int j = 0; j < NE; j++) out[j] = warp_sum(acc[j]);
    if (ss) *ss = warp_sum(sq);
}

// 1 / sqrt(mean square + eps): the RMSNorm factor of a row from its sum of squares.
__device__ __forceinline__ float rms_inv(float sumsq, int H, float eps) {
    return rsqrtf(sumsq / (float)H + eps);
}

// CTA (r, g): router rows 4r..4r+3 for tokens 16g..16g+15, one warp per token
// over the whole rows.  The last CTA of token group g (a ticket per group) ranks
// the group's tokens, one warp per token; with a device-resident cache policy
// (lfu) it then runs the policy's step on the routing.  When idx_host is set (page-locked host
// memory mapped into the device's address space) the group's choices also go
// there, followed by flag_host[g] = seq once they are visible to the host.
__global__ void __launch_bounds__(kRouteTok * 32)
k_route(LayerDev ly, const float *__restrict__ x, int T, Ws ws, int32_t *idx_out, float *gate_out,
        float *logits_out, int32_t *idx_host, unsigned *flag_host, unsigned seq, DevLfu *lfu) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * kRouteExp, t = blockIdx.y * kRouteTok + warp;
    if (t < T) {
        float v[kRouteExp], ss = 0.f;
        router_dot_rows<kRouteExp>(ly.rq, ly.rs, ly.rb, ly.H, ly.E, x, e0, t, v, ly.norm_w,
                                   ly.norm_w ? &ss : nullptr);
        const float inv = ly.norm_w ? rms_inv(ss, ly.H, ly.norm_eps) : 1.f;
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < kRouteExp; j++) {
                const int e = e0 + j;
                if (e >= ly.E) break;
                const float lv = (ly.norm_w ? v[j] * inv : v[j]) + (ly.bias ? ly.bias[e] : 0.f);
                ws.logits[(size_t)t * ly.E + e] = lv;
                if (logits_out) logits_out[(size_t)t * ly.E + e] = lv;
            }
    }
    __shared__ int is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned tk = atomicAdd(&ws.ticket[blockIdx.y], 1u);
        is_last = (tk == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if (t < T)
        warp_topk_softmax(ws.logits + (size_t)t * ly.E, ly.E, ly.topk, idx_out + t * ly.topk,
                          gate_out + t * ly.topk, idx_host ? idx_host + t * ly.topk : nullptr, nullptr);
    if (threadIdx.x == 0) ws.ticket[blockIdx.y] = 0u;
    if (lfu) {
        // the cache policy's step on this call's routing (one token group: T <= 16)
        __syncthreads();
        if (threadIdx.x == 0) dev_lfu_step(lfu, idx_out, T * ly.topk);
    }
    if (idx_host) {
        __threadfence_system();
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence_system();
            *(volatile unsigned *)(flag_host + blockIdx.y) = seq;
        }
    }
}

}  // namespace moe
