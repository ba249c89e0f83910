// common.cuh -- shared device/host definitions of libmoe (layouts, workspace, helpers).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kGroup = 64;

__host__ __device__ inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

// Byte offsets of the six parts of an expert blob of shape (H, I):
// [gate; up] rows 2I x H, then down rows H x I; each part 256-byte aligned.
struct BlobLayout {
    size_t gu_q, gu_s, gu_b, d_q, d_s, d_b, total;
};

__host__ __device__ inline BlobLayout blob_layout(int H, int I) {
    BlobLayout L;
    size_t off = 0;
    L.gu_q = off; off = up256(off + size_t(2) * I * H / 2);
    L.gu_s = off; off = up256(off + size_t(2) * I * (H / kGroup) * 2);
    L.gu_b = off; off = up256(off + size_t(2) * I * (H / kGroup) * 2);
    L.d_q = off;  off = up256(off + size_t(H) * I / 2);
    L.d_s = off;  off = up256(off + size_t(H) * (I / kGroup) * 2);
    L.d_b = off;  off = up256(off + size_t(H) * (I / kGroup) * 2);
    L.total = off;
    return L;
}

// A packed 4-bit matrix view: rows of K/8 words, fp16 scale/bias per 64 columns.
struct QMat {
    const uint32_t *q;
    const __half *s, *b;
    int rows, K;
};

__host__ __device__ inline QMat gu_view(const uint8_t *blob, const BlobLayout &L, int H, int I) {
    return QMat{(const uint32_t *)(blob + L.gu_q), (const __half *)(blob + L.gu_s),
                (const __half *)(blob + L.gu_b), 2 * I, H};
}
__host__ __device__ inline QMat down_view(const uint8_t *blob, const BlobLayout &L, int H, int I) {
    return QMat{(const uint32_t *)(blob + L.d_q), (const __half *)(blob + L.d_s),
                (const __half *)(blob + L.d_b), H, I};
}

// The layer as the kernels see it.
struct LayerDev {
    int H, E, topk, I, Is;
    const uint32_t *rq;
    const __half *rs, *rb;
    const uint8_t *experts;
    size_t stride;
    const uint8_t *shared;
    const float *bias;
    BlobLayout L, Ls;
};

// Workspace (see moe_workspace_bytes).  Control words live at the start:
enum CtrlWord {
    kErr = 0,        // a bounded wait gave up (sticky until moe_workspace_status)
    kRouteTicket,    // router items finished (the last one runs top-k)
    kU,              // number of distinct routed experts of this call
    kQueue0,         // work queue: router, shared gate/up, shared down items
    kQueue1,         // work queue: routed gate/up items
    kQueue2,         // work queue: routed down items
    kXPrep,          // router items whose slice of x is converted
    kRouted,         // 1 once idx/gate/schedule are published
    kSharedUp,       // shared gate/up items finished
    kExit,           // CTAs finished (the last one resets the control words)
    kCtrlWords = 16
};

struct Ws {
    unsigned *ctrl;
    unsigned *tile_cnt;  // [H/16] tickets of the down combine (16-row tiles)
    unsigned *up_done;   // [Umax] gate/up items finished per distinct expert
    float *logits;       // [Tmax][E]
    int *idx;            // [Tmax][topk]
    float *gate;         // [Tmax][topk]
    int *uexp;           // [Umax] expert id of distinct expert u (ascending ids)
    int *ucount;         // [Umax] tokens using u
    int *ulist;          // [Umax][Tmax] pair ids p = t*topk + k, ascending
    float *h;            // [Tmax*topk][I]  routed activations (fp32 path)
    float *hs;           // [Tmax][Is]      shared activations (fp32 path)
    float *partial;      // [Tmax*topk + Tmax][H] per-pair down outputs, then shared
    __half *x16;         // [Tmax][H]   tokens in fp16, fragment order
    float *xsum;         // [Tmax][H/64] group sums of the fp16 tokens
    __half *h16;         // [Tmax*topk][I] routed activations, fp16 fragment order
    __half *hs16;        // [Tmax][Is]     shared activations, fp16 fragment order
    int Tmax, Umax;
};

struct WsLayout {
    size_t ctrl, logits, idx, gate, uexp, ucount, ulist, h, hs, partial, x16, xsum, h16, hs16, total;
    int Tmax, Umax;
};

inline WsLayout ws_layout(const moe_layer_t &l, int Tmax) {
    WsLayout W;
    W.Tmax = Tmax;
    W.Umax = Tmax * l.topk < l.E ? Tmax * l.topk : l.E;
    size_t off = 0;
    W.ctrl = off;    off = up256(off + sizeof(unsigned) * (kCtrlWords + l.H / 16 + W.Umax));
    W.logits = off;  off = up256(off + sizeof(float) * Tmax * l.E);
    W.idx = off;     off = up256(off + sizeof(int) * Tmax * l.topk);
    W.gate = off;    off = up256(off + sizeof(float) * Tmax * l.topk);
    W.uexp = off;    off = up256(off + sizeof(int) * W.Umax);
    W.ucount = off;  off = up256(off + sizeof(int) * W.Umax);
    W.ulist = off;   off = up256(off + sizeof(int) * size_t(W.Umax) * Tmax);
    W.h = off;       off = up256(off + sizeof(float) * size_t(Tmax) * l.topk * l.I);
    W.hs = off;      off = up256(off + sizeof(float) * size_t(Tmax) * l.Is);
    W.partial = off; off = up256(off + sizeof(float) * size_t(Tmax) * (l.topk + 1) * l.H);
    W.x16 = off;     off = up256(off + sizeof(__half) * size_t(Tmax) * l.H);
    W.xsum = off;    off = up256(off + sizeof(float) * size_t(Tmax) * (l.H / kGroup));
    W.h16 = off;     off = up256(off + sizeof(__half) * size_t(Tmax) * l.topk * l.I);
    W.hs16 = off;    off = up256(off + sizeof(__half) * size_t(Tmax) * l.Is);
    W.total = off;
    return W;
}

inline Ws ws_bind(void *base, const WsLayout &W, const moe_layer_t &l) {
    uint8_t *p = (uint8_t *)base;
    Ws w;
    w.ctrl = (unsigned *)(p + W.ctrl);
    w.tile_cnt = w.ctrl + kCtrlWords;
    w.up_done = w.tile_cnt + l.H / 16;
    w.logits = (float *)(p + W.logits);
    w.idx = (int *)(p + W.idx);
    w.gate = (float *)(p + W.gate);
    w.uexp = (int *)(p + W.uexp);
    w.ucount = (int *)(p + W.ucount);
    w.ulist = (int *)(p + W.ulist);
    w.h = (float *)(p + W.h);
    w.hs = (float *)(p + W.hs);
    w.partial = (float *)(p + W.partial);
    w.x16 = (__half *)(p + W.x16);
    w.xsum = (float *)(p + W.xsum);
    w.h16 = (__half *)(p + W.h16);
    w.hs16 = (__half *)(p + W.hs16);
    w.Tmax = W.Tmax;
    w.Umax = W.Umax;
    return w;
}

// GELU, tanh form.
__device__ __forceinline__ float gelu_tanh(float z) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * z * (1.0f + tanhf(c * (z + 0.044715f * z * z * z)));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace moe
