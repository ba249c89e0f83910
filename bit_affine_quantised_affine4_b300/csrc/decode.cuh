// decode.cuh -- the whole MoE layer for 1..16 decode tokens in one persistent kernel.
//
// The layer (devtrends page, section "Qual e il trucco principale dell'architettura";
// remio.ai page, sections "Mac Gemma 4 26B entra nello spazio disponibile..." and
// "L'affermazione dei 2 GB..."): an 8-bit router picks 8 experts per token, the
// routed experts and an always-on shared expert run GeGLU FFNs on 4-bit affine
// weights, and the outputs are combined with the softmax gates.
//
// Work is cut into items taken from three queues in order; an item only ever waits
// for items of earlier queues or earlier positions, which running CTAs hold, so the
// schedule cannot deadlock whatever the number of resident CTAs.
//   queue 0: router items (convert a slice of the tokens to fp16 fragment order,
//            then 8 router rows; the last one runs top-k/softmax and publishes the
//            schedule), shared gate/up items (16 gate + 16 up rows), shared down
//            items (64 output rows; they prefetch their weights to L2, then wait
//            for the shared activations)
//   queue 1: routed gate/up items, (distinct expert, 16 rows) -- after routing
//   queue 2: routed down items, (distinct expert, 64 rows); they prefetch, wait for
//            their expert's activations, and the last item of each 64-row tile
//            combines y = sum_k g_k * routed_k + shared (+ x) in fixed order.
// Every wait is bounded: on expiry the kernel raises the workspace error flag and
// all CTAs drain without further work.  The last CTA to leave resets the control
// words so the workspace is ready for the next call.
#pragma once

#include "common.cuh"
#include "mma_core.cuh"
#include "route.cuh"

namespace moe {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kRouterRows = kDecWarps;  // router rows per router item
constexpr int kDownRows = 64;           // output rows per down item
constexpr long long kSpinLimit = 1ll << 22;  // polls of ~128 ns: about half a second

struct DecodeArgs {
    LayerDev ly;
    const float *x;
    int T;
    int flags;
    float *y;
    int32_t *idx_out;
    float *gate_out;
    Ws ws;
    int R;  // router items
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One thread waits until *p >= target; false if the wait gave up or another CTA did.
__device__ bool wait_geq(const unsigned *p, unsigned target, unsigned *err) {
    for (long long it = 0; it < kSpinLimit; it++) {
        if (ld_acquire(p) >= target) return true;
        if (*(volatile unsigned *)err) return false;
        __nanosleep(128);
    }
    atomicExch(err, 1u);
    return false;
}

// CTA-wide wait; returns false (for every thread) on timeout/abort.
__device__ bool cta_wait(const unsigned *p, unsigned target, unsigned *err, int *s_flag) {
    if (threadIdx.x == 0) {
        *s_flag = wait_geq(p, target, err) ? 1 : 0;
        __threadfence();
    }
    __syncthreads();
    bool ok = *s_flag != 0;
    __syncthreads();
    return ok;
}

__device__ __forceinline__ void l2_prefetch(const void *p, unsigned bytes) {
    // bulk prefetch of a 16-byte aligned range into L2
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ router item
__device__ void router_item(const DecodeArgs &a, int r, int *s_flag) {
    const LayerDev &ly = a.ly;
    const Ws &ws = a.ws;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = ly.H / kGroup;
    // 1. tokens -> fp16 fragment order, groups [g0, g1) of every token
    {
        const int g0 = r * G / a.R, g1 = (r + 1) * G / a.R;
        const int n = (g1 - g0) * a.T * 32;  // (token, group, pair of columns)
        for (int i = threadIdx.x; i < n; i += kDecThreads) {
            const int l = i & 31, tg = i >> 5;
            const int t = tg / (g1 - g0), g = g0 + tg % (g1 - g0);
            const int k = g * kGroup + 2 * l;
            const float2 v = __ldg(reinterpret_cast<const float2 *>(a.x + (size_t)t * ly.H + k));
            __half *row = ws.x16 + (size_t)t * ly.H;
            row[frag_pos(k)] = __float2half_rn(v.x);
            row[frag_pos(k + 1)] = __float2half_rn(v.y);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&ws.ctrl[kXPrep], 1u);
        }
    }
    // 2. router rows: one per warp, all tokens
    const int e = r * kRouterRows + warp;
    if (e < ly.E) {
        const int wpr = ly.H / 4;
        const uint32_t *row = ly.rq + (size_t)e * wpr;
        float acc[MOE_MAX_DECODE_TOKENS];
#pragma unroll
        for (int t = 0; t < MOE_MAX_DECODE_TOKENS; t++) acc[t] = 0.f;
        for (int w0 = 2 * lane; w0 < wpr; w0 += 64) {
            const uint2 wd = ldg_u2(row + w0);
            const int g = w0 >> 4;  // 16 words per group of 64 bytes
            const float s = __half2float(ly.rs[(size_t)e * G + g]);
            const float b = __half2float(ly.rb[(size_t)e * G + g]);
            float wv[8];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                wv[i] = fmaf(s, (float)((wd.x >> (8 * i)) & 0xFFu), b);
                wv[4 + i] = fmaf(s, (float)((wd.y >> (8 * i)) & 0xFFu), b);
            }
#pragma unroll
            for (int t = 0; t < MOE_MAX_DECODE_TOKENS; t++) {
                if (t < a.T) {
                    const float4 *xv = reinterpret_cast<const float4 *>(a.x + (size_t)t * ly.H + 4 * w0);
                    const float4 x0 = __ldg(xv), x1 = __ldg(xv + 1);
                    float v = acc[t];
                    v = fmaf(wv[0], x0.x, v); v = fmaf(wv[1], x0.y, v);
                    v = fmaf(wv[2], x0.z, v); v = fmaf(wv[3], x0.w, v);
                    v = fmaf(wv[4], x1.x, v); v = fmaf(wv[5], x1.y, v);
                    v = fmaf(wv[6], x1.z, v); v = fmaf(wv[7], x1.w, v);
                    acc[t] = v;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MOE_MAX_DECODE_TOKENS; t++) {
            if (t < a.T) {
                float v = warp_sum(acc[t]);
                if (lane == 0) ws.logits[(size_t)t * ly.E + e] = v + (ly.bias ? ly.bias[e] : 0.f);
            }
        }
    }
    // 3. the last router item ranks the experts and publishes the schedule
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        *s_flag = atomicAdd(&ws.ctrl[kRouteTicket], 1u) == (unsigned)(a.R - 1);
    }
    __syncthreads();
    const bool last = *s_flag;
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int t = warp; t < a.T; t += kDecWarps)
        warp_topk_softmax(ws.logits, ly.E, ly.topk, t, ws.idx, ws.gate, a.idx_out, a.gate_out);
    __syncthreads();
    build_schedule(ly, a.T, ws);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicExch(&ws.ctrl[kRouted], 1u);
    }
}

// ------------------------------------------------------------------ token slots
// Up to 16 token slots per item: slot j reads B row brow[j] and writes output row
// orow[j].
struct Slots {
    int n;
    int brow[MOE_MAX_DECODE_TOKENS];
    int orow[MOE_MAX_DECODE_TOKENS];
};

// ------------------------------------------------------------------ gate/up item
// 16 gate rows [i0, i0+16) and the up rows [Ie+i0, ...) of one expert matrix; the
// CTA's 8 warps split the K groups, then reduce through shared memory and apply
// GeGLU.  Output: fp16 activations in fragment order.
template <int NCH>
__device__ void gateup_item(const DecodeArgs &a, QMat m, int Ie, int i0, const Slots &sl,
                            __half *hout, unsigned *done, float *smem) {
    const LayerDev &ly = a.ly;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
    const int G = ly.H / kGroup, wpr = ly.H / 8;
    // stage scales and biases of the 32 rows: [4][16][G] halves
    __half *sb = reinterpret_cast<__half *>(smem);
    {
        const int per = 16 * G * 2 / 16;  // 16-byte chunks per (part, 16 rows)
        for (int i = threadIdx.x; i < 4 * per; i += kDecThreads) {
            const int part = i / per, ch = i % per;
            const __half *src = ((part & 1) ? m.b : m.s) + (size_t)(i0 + ((part >> 1) ? Ie : 0)) * G;
            reinterpret_cast<uint4 *>(sb + part * 16 * G)[ch] = __ldg(reinterpret_cast<const uint4 *>(src) + ch);
        }
    }
    const uint32_t *qg_a = m.q + (size_t)(i0 + gl) * wpr + 2 * c;
    const uint32_t *qg_b = qg_a + 8 * (size_t)wpr;
    const uint32_t *qu_a = qg_a + (size_t)Ie * wpr;
    const uint32_t *qu_b = qu_a + 8 * (size_t)wpr;
    const int g0 = warp * G / kDecWarps, g1 = (warp + 1) * G / kDecWarps;
    float accg[NCH][4], accu[NCH][4];
#pragma unroll
    for (int ch = 0; ch < NCH; ch++)
#pragma unroll
        for (int i = 0; i < 4; i++) accg[ch][i] = accu[ch][i] = 0.f;
    __syncthreads();
    // two groups per step, the next step's weights loaded before this step's math
    uint2 cur[2][4], nxt[2][4];
    auto load = [&](uint2 (&dst)[2][4], int g) {
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const int gg = (g + k < g1) ? g + k : g;
            dst[k][0] = ldg_u2(qg_a + gg * 8);
            dst[k][1] = ldg_u2(qg_b + gg * 8);
            dst[k][2] = ldg_u2(qu_a + gg * 8);
            dst[k][3] = ldg_u2(qu_b + gg * 8);
        }
    };
    if (g0 < g1) load(cur, g0);
    for (int g = g0; g < g1; g += 2) {
        if (g + 2 < g1) load(nxt, g + 2);
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const int gg = g + k;
            if (gg < g1) {
                const float sga = __half2float(sb[0 * 16 * G + gl * G + gg]) * kTwo24;
                const float bga = __half2float(sb[1 * 16 * G + gl * G + gg]);
                const float sgb = __half2float(sb[0 * 16 * G + (gl + 8) * G + gg]) * kTwo24;
                const float bgb = __half2float(sb[1 * 16 * G + (gl + 8) * G + gg]);
                const float sua = __half2float(sb[2 * 16 * G + gl * G + gg]) * kTwo24;
                const float bua = __half2float(sb[3 * 16 * G + gl * G + gg]);
                const float sub = __half2float(sb[2 * 16 * G + (gl + 8) * G + gg]) * kTwo24;
                const float bub = __half2float(sb[3 * 16 * G + (gl + 8) * G + gg]);
#pragma unroll
                for (int ch = 0; ch < NCH; ch++) {
                    uint32_t xb[8];
                    const int slot = ch * 8 + gl;
                    if (slot < sl.n)
                        load_b(xb, a.ws.x16 + (size_t)sl.brow[slot] * ly.H + gg * kGroup + 16 * c);
                    else
                        zero_b(xb);
                    float dsum[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_group_sums(dsum, xb);
                    float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_group_codes(dg, cur[k][0], cur[k][1], xb);
                    mma_group_codes(du, cur[k][2], cur[k][3], xb);
                    apply_affine(accg[ch], dg, dsum, sga, bga, sgb, bgb);
                    apply_affine(accu[ch], du, dsum, sua, bua, sub, bub);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 2; k++)
#pragma unroll
            for (int r = 0; r < 4; r++) cur[k][r] = nxt[k][r];
    }
    // reduce the 8 warps' partial sums: red[warp][ch][2][32 lanes][4]
    __syncthreads();  // sb no longer needed; reuse the buffer
    float *red = smem;
#pragma unroll
    for (int ch = 0; ch < NCH; ch++)
#pragma unroll
        for (int i = 0; i < 4; i++) {
            red[(((warp * NCH + ch) * 2 + 0) * 32 + lane) * 4 + i] = accg[ch][i];
            red[(((warp * NCH + ch) * 2 + 1) * 32 + lane) * 4 + i] = accu[ch][i];
        }
    __syncthreads();
    for (int v = threadIdx.x; v < NCH * 32 * 4; v += kDecThreads) {
        const int ch = v / 128, ln = (v / 4) % 32, i = v % 4;
        float gsum = 0.f, usum = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; w++) {
            gsum += red[(((w * NCH + ch) * 2 + 0) * 32 + ln) * 4 + i];
            usum += red[(((w * NCH + ch) * 2 + 1) * 32 + ln) * 4 + i];
        }
        const int row = (ln >> 2) + ((i & 2) ? 8 : 0);
        const int slot = ch * 8 + 2 * (ln & 3) + (i & 1);
        if (slot < sl.n) {
            const float hval = gelu_tanh(gsum) * usum;
            hout[(size_t)sl.orow[slot] * Ie + frag_pos(i0 + row)] = __float2half_rn(hval);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(done, 1u);
    }
}

// ------------------------------------------------------------------ down item
// 64 output rows [n0, n0+64) of one down matrix (K = Ie): warps = 4 row tiles x 2
// K halves.  Writes per-slot partial rows, then takes the tile's ticket; the last
// contributor of the tile combines y.
template <int NCH>
__device__ void down_item(const DecodeArgs &a, QMat m, int n0, const Slots &sl, const __half *hin,
                          unsigned target, float *smem, int *s_flag) {
    const LayerDev &ly = a.ly;
    const Ws &ws = a.ws;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
    const int Ke = m.K, G = Ke / kGroup, wpr = Ke / 8;
    __half *sb = reinterpret_cast<__half *>(smem);
    {
        const int per = kDownRows * G * 2 / 16;
        for (int i = threadIdx.x; i < 2 * per; i += kDecThreads) {
            const int part = i / per, ch = i % per;
            const __half *src = (part ? m.b : m.s) + (size_t)n0 * G;
            reinterpret_cast<uint4 *>(sb + part * kDownRows * G)[ch] =
                __ldg(reinterpret_cast<const uint4 *>(src) + ch);
        }
    }
    const int rt = warp & 3, kh = warp >> 2;
    const int ra = rt * 16 + gl;  // row within the 64-row tile
    const uint32_t *qa = m.q + (size_t)(n0 + ra) * wpr + 2 * c;
    const uint32_t *qb = qa + 8 * (size_t)wpr;
    const int g0 = kh * G / 2, g1 = (kh + 1) * G / 2;
    float acc[NCH][4];
#pragma unroll
    for (int ch = 0; ch < NCH; ch++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[ch][i] = 0.f;
    __syncthreads();
    uint2 cur[4][2], nxt[4][2];
    auto load = [&](uint2 (&dst)[4][2], int g) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int gg = (g + k < g1) ? g + k : g;
            dst[k][0] = ldg_u2(qa + gg * 8);
            dst[k][1] = ldg_u2(qb + gg * 8);
        }
    };
    if (g0 < g1) load(cur, g0);
    for (int g = g0; g < g1; g += 4) {
        if (g + 4 < g1) load(nxt, g + 4);
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int gg = g + k;
            if (gg < g1) {
                const float sa = __half2float(sb[ra * G + gg]) * kTwo24;
                const float ba = __half2float(sb[kDownRows * G + ra * G + gg]);
                const float sbb = __half2float(sb[(ra + 8) * G + gg]) * kTwo24;
                const float bb = __half2float(sb[kDownRows * G + (ra + 8) * G + gg]);
#pragma unroll
                for (int ch = 0; ch < NCH; ch++) {
                    uint32_t xb[8];
                    const int slot = ch * 8 + gl;
                    if (slot < sl.n)
                        load_b(xb, hin + (size_t)sl.brow[slot] * Ke + gg * kGroup + 16 * c);
                    else
                        zero_b(xb);
                    float dsum[4] = {0.f, 0.f, 0.f, 0.f}, d[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_group_sums(dsum, xb);
                    mma_group_codes(d, cur[k][0], cur[k][1], xb);
                    apply_affine(acc[ch], d, dsum, sa, ba, sbb, bb);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
            cur[k][0] = nxt[k][0];
            cur[k][1] = nxt[k][1];
        }
    }
    // reduce the two K halves; write partial rows (fp32) of every slot
    __syncthreads();
    float *red = smem;  // [2 halves][4 tiles][NCH][32][4]
#pragma unroll
    for (int ch = 0; ch < NCH; ch++)
#pragma unroll
        for (int i = 0; i < 4; i++) red[((((kh * 4 + rt) * NCH + ch) * 32) + lane) * 4 + i] = acc[ch][i];
    __syncthreads();
    for (int v = threadIdx.x; v < 4 * NCH * 128; v += kDecThreads) {
        const int t4 = v / (NCH * 128), ch = (v / 128) % NCH, ln = (v / 4) % 32, i = v % 4;
        const float val = red[((((0 * 4 + t4) * NCH + ch) * 32) + ln) * 4 + i] +
                          red[((((1 * 4 + t4) * NCH + ch) * 32) + ln) * 4 + i];
        const int row = t4 * 16 + (ln >> 2) + ((i & 2) ? 8 : 0);
        const int slot = ch * 8 + 2 * (ln & 3) + (i & 1);
        if (slot < sl.n) ws.partial[(size_t)sl.orow[slot] * ly.H + n0 + row] = val;
    }
    // ticket of this 64-row tile: U routed contributions + 1 shared
    __syncthreads();
    const int tile = n0 / kDownRows;
    if (threadIdx.x == 0) {
        __threadfence();
        *s_flag = atomicAdd(&ws.tile_cnt[tile], 1u) == target;
    }
    __syncthreads();
    const bool last = *s_flag;
    __syncthreads();
    if (!last) return;
    __threadfence();
    const size_t shared_base = (size_t)ws.Tmax * ly.topk;
    for (int v = threadIdx.x; v < kDownRows * a.T; v += kDecThreads) {
        const int t = v / kDownRows, n = n0 + v % kDownRows;
        float acc2 = 0.f;
        for (int k = 0; k < ly.topk; k++)
            acc2 = fmaf(__ldcg(&ws.gate[t * ly.topk + k]),
                        __ldcg(&ws.partial[(size_t)(t * ly.topk + k) * ly.H + n]), acc2);
        acc2 += __ldcg(&ws.partial[(shared_base + t) * ly.H + n]);
        if (a.flags & MOE_RESIDUAL) acc2 += __ldg(&a.x[(size_t)t * ly.H + n]);
        a.y[(size_t)t * ly.H + n] = acc2;
    }
    if (threadIdx.x == 0) ws.tile_cnt[tile] = 0u;
}

// ------------------------------------------------------------------ the kernel
template <int NCH>
__global__ void __launch_bounds__(kDecThreads) k_decode(DecodeArgs a) {
    extern __shared__ __align__(16) float smem[];
    __shared__ int s_item, s_flag, s_abort;
    __shared__ Slots sl;
    const LayerDev &ly = a.ly;
    const Ws &ws = a.ws;
    const int tilesS = ly.Is / 16, downS = ly.H / kDownRows, tilesR = ly.I / 16;
    const int n0 = a.R + tilesS + downS;
    if (threadIdx.x == 0) s_abort = 0;
    __syncthreads();
    unsigned U = 0;
    for (int q = 0; q < 3 && !s_abort; q++) {
        if (q == 1) {
            if (!cta_wait(&ws.ctrl[kRouted], 1u, &ws.ctrl[kErr], &s_flag)) {
                s_abort = 1;
                break;
            }
            U = __ldcg(&ws.ctrl[kU]);
        }
        const int count = q == 0 ? n0 : (q == 1 ? (int)U * tilesR : (int)U * downS);
        while (true) {
            if (threadIdx.x == 0) s_item = (int)atomicAdd(&ws.ctrl[kQueue0 + q], 1u);
            __syncthreads();
            const int it = s_item;
            __syncthreads();
            if (it >= count) break;
            if (q == 0 && it < a.R) {
                router_item(a, it, &s_flag);
            } else if (q == 0 && it < a.R + tilesS) {
                const int k = it - a.R;
                if (threadIdx.x < MOE_MAX_DECODE_TOKENS) {
                    sl.brow[threadIdx.x] = sl.orow[threadIdx.x] = threadIdx.x;
                    if (threadIdx.x == 0) sl.n = a.T;
                }
                if (!cta_wait(&ws.ctrl[kXPrep], (unsigned)a.R, &ws.ctrl[kErr], &s_flag)) {
                    s_abort = 1;
                    break;
                }
                gateup_item<NCH>(a, gu_view(ly.shared, ly.Ls, ly.H, ly.Is), ly.Is, 16 * k, sl, ws.hs16,
                                 &ws.ctrl[kSharedUp], smem);
            } else if (q == 0) {
                const int m = it - a.R - tilesS;
                QMat d = down_view(ly.shared, ly.Ls, ly.H, ly.Is);
                if (threadIdx.x == 0) {
                    const int G = d.K / kGroup;
                    l2_prefetch(d.q + (size_t)m * kDownRows * (d.K / 8), kDownRows * d.K / 2);
                    l2_prefetch(d.s + (size_t)m * kDownRows * G, kDownRows * G * 2);
                    l2_prefetch(d.b + (size_t)m * kDownRows * G, kDownRows * G * 2);
                }
                if (threadIdx.x < MOE_MAX_DECODE_TOKENS) {
                    sl.brow[threadIdx.x] = threadIdx.x;
                    sl.orow[threadIdx.x] = ws.Tmax * ly.topk + threadIdx.x;
                    if (threadIdx.x == 0) sl.n = a.T;
                }
                if (!cta_wait(&ws.ctrl[kSharedUp], (unsigned)tilesS, &ws.ctrl[kErr], &s_flag)) {
                    s_abort = 1;
                    break;
                }
                // the tile ticket target (U) is only known after routing
                if (!cta_wait(&ws.ctrl[kRouted], 1u, &ws.ctrl[kErr], &s_flag)) {
                    s_abort = 1;
                    break;
                }
                const unsigned Ucur = __ldcg(&ws.ctrl[kU]);
                down_item<NCH>(a, d, m * kDownRows, sl, ws.hs16, Ucur, smem, &s_flag);
            } else {
                const int u = q == 1 ? it / tilesR : it / downS;
                const int e = __ldcg(&ws.uexp[u]);
                const uint8_t *blob = ly.experts + (size_t)e * ly.stride;
                if (threadIdx.x < MOE_MAX_DECODE_TOKENS) {
                    const int cnt = __ldcg(&ws.ucount[u]);
                    const int p = threadIdx.x < cnt ? __ldcg(&ws.ulist[(size_t)u * ws.Tmax + threadIdx.x]) : 0;
                    sl.brow[threadIdx.x] = q == 1 ? p / ly.topk : p;
                    sl.orow[threadIdx.x] = p;
                    if (threadIdx.x == 0) sl.n = cnt;
                }
                if (q == 1) {
                    __syncthreads();
                    gateup_item<NCH>(a, gu_view(blob, ly.L, ly.H, ly.I), ly.I, 16 * (it % tilesR), sl,
                                     ws.h16, &ws.up_done[u], smem);
                } else {
                    const int m = it % downS;
                    QMat d = down_view(blob, ly.L, ly.H, ly.I);
                    if (threadIdx.x == 0) {
                        const int G = d.K / kGroup;
                        l2_prefetch(d.q + (size_t)m * kDownRows * (d.K / 8), kDownRows * d.K / 2);
                        l2_prefetch(d.s + (size_t)m * kDownRows * G, kDownRows * G * 2);
                        l2_prefetch(d.b + (size_t)m * kDownRows * G, kDownRows * G * 2);
                    }
                    if (!cta_wait(&ws.up_done[u], (unsigned)tilesR, &ws.ctrl[kErr], &s_flag)) {
                        s_abort = 1;
                        break;
                    }
                    down_item<NCH>(a, d, m * kDownRows, sl, ws.h16, U, smem, &s_flag);
                }
            }
        }
    }
    // leave; the last CTA resets the control words for the next call
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_flag = atomicAdd(&ws.ctrl[kExit], 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_flag) {
        __threadfence();
        const unsigned Umax = (unsigned)ws.Umax;
        for (unsigned i = threadIdx.x; i < Umax; i += kDecThreads) ws.up_done[i] = 0u;
        if (threadIdx.x == 0) {
            ws.ctrl[kRouteTicket] = 0u;
            ws.ctrl[kQueue0] = ws.ctrl[kQueue1] = ws.ctrl[kQueue2] = 0u;
            ws.ctrl[kXPrep] = ws.ctrl[kRouted] = ws.ctrl[kSharedUp] = 0u;
            ws.ctrl[kExit] = 0u;
        }
    }
}

// Dynamic shared memory of k_decode: the larger of the staged scales/biases and the
// reduction buffers.
inline size_t decode_smem_bytes(const moe_layer_t &l, int nch) {
    const size_t G = l.H / kGroup, Gd = (l.I > l.Is ? l.I : l.Is) / kGroup;
    size_t sb_up = 4 * 16 * G * 2, sb_down = 2 * kDownRows * Gd * 2;
    size_t red_up = (size_t)kDecWarps * nch * 2 * 32 * 4 * 4;
    size_t red_down = (size_t)2 * 4 * nch * 32 * 4 * 4;
    size_t m = sb_up;
    if (sb_down > m) m = sb_down;
    if (red_up > m) m = red_up;
    if (red_down > m) m = red_down;
    return m;
}

}  // namespace moe
