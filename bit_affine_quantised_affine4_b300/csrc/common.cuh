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
    const float *norm_w;  // RMSNorm weight when the router reads RMSNorm(x) (else null)
    float norm_eps;
    BlobLayout L, Ls;
};

// Workspace (see moe_workspace_bytes).  Control words live at the start:
enum CtrlWord {
    kErr = 0,         // a bounded wait gave up (sticky until moe_workspace_status)
    kRouteTicket,     // standalone router: CTAs finished (the last one runs top-k)
    kRouteCnt,        // decode: router rows published (cumulative over calls)
    kGuDone,          // decode: gate/up tiles finished (cumulative over calls)
    kRouteBase,       // decode: kRouteCnt at the start of the next call (8-byte aligned pair
    kGuBase,          //   with kGuBase, the same for kGuDone); written by CTA 0 at its end
    kCtrlWords = 16
};

// Parts of the shared expert's down matrix (K = Is) cut to the routed experts'
// K = I, so that every down unit has at most I/64 groups.
__host__ __device__ inline int shared_parts(int I, int Is) { return (Is / kGroup + I / kGroup - 1) / (I / kGroup); }

struct Ws {
    unsigned *ctrl;
    unsigned *ticket;  // [H/16] tickets of the 16-row output tiles
    float *logits;     // [Tmax][E]
    int *idx;          // [Tmax][topk] routing of a separate router launch (cached decode)
    float *gate;       // [Tmax][topk]
    __half *h16;       // [Tmax*topk][I]  routed activations (compact slots)
    __half *hs16;      // [Tmax][Is]      shared activations
    float *pr;         // [Tmax*topk][H]  routed down partials
    float *ps;         // [P][Tmax][H]    shared down partials
    float *xh, *yh;    // [Tmax][H]       device copies of a host call's x and y
    int *ih;           // [Tmax][topk]    and of its routing outputs
    float *gh;         // [Tmax][topk]
    // prefill chunk (grouped GEMMs)
    int *plan;         // U, rows used, uexp[256], urow[256], ucnt[256], rowtok[Rmax], rowpair[Rmax],
                       // uslc[257], dep[258]
    uint8_t *Br, *Bs;  // token operand tiles: [H/64][Rmax][128 B], [H/64][T16][128 B]
    uint8_t *Hr, *Hs;  // h operand tiles:     [I/64][Rmax][128 B], [Is/64][T16][128 B]
    float *Yr, *Ys;    // down rows: [Tmax*topk][H], [T16][H]
    float *xn;         // [Tmax][H] RMSNorm(x) of a pre-norm prefill chunk
    int Tmax;
};

// Rows of the prefill's per-expert segments (each expert's token count rounded
// up to 16) for T tokens: at most T*topk tokens plus 15 padding rows per expert.
inline int prefill_rows(const moe_layer_t &l, int T) {
    const int p = T * l.topk, u = p < l.E ? p : l.E;
    return (p + 15 * u + 15) & ~15;
}

// The control words and the 16-row-tile tickets sit in a header of fixed size
// (enough tickets for the largest hidden size the layer calls accept), so one
// workspace can serve layers of different shapes in turn: every call leaves the
// header zeroed for the next one whatever the layer.
constexpr int kMaxHiddenLayer = 4096;
constexpr int kMaxTickets = kMaxHiddenLayer / 16;
constexpr size_t kWsHeaderBytes = (kCtrlWords + kMaxTickets) * sizeof(unsigned);

struct WsLayout {
    size_t ctrl, logits, idx, gate, h16, hs16, pr, ps, xh, yh, ih, gh, decode_total;
    size_t plan, Br, Bs, Hr, Hs, Yr, Ys, xn, total;
    int Tmax;
};

inline WsLayout ws_layout(const moe_layer_t &l, int Tmax) {
    WsLayout W;
    W.Tmax = Tmax;
    const int P = shared_parts(l.I, l.Is);
    size_t off = 0;
    W.ctrl = off;   off = up256(off + kWsHeaderBytes);
    W.logits = off; off = up256(off + sizeof(float) * Tmax * l.E);
    W.idx = off;    off = up256(off + sizeof(int) * Tmax * l.topk);
    W.gate = off;   off = up256(off + sizeof(float) * Tmax * l.topk);
    W.h16 = off;    off = up256(off + sizeof(__half) * size_t(Tmax) * l.topk * l.I);
    W.hs16 = off;   off = up256(off + sizeof(__half) * size_t(Tmax) * l.Is);
    W.pr = off;     off = up256(off + sizeof(float) * size_t(Tmax) * l.topk * l.H);
    W.ps = off;     off = up256(off + sizeof(float) * size_t(P) * Tmax * l.H);
    W.xh = off;     off = up256(off + sizeof(float) * size_t(Tmax) * l.H);
    W.yh = off;     off = up256(off + sizeof(float) * size_t(Tmax) * l.H);
    W.ih = off;     off = up256(off + sizeof(int) * size_t(Tmax) * l.topk);
    W.gh = off;     off = up256(off + sizeof(float) * size_t(Tmax) * l.topk);
    W.decode_total = off;
    const int Rmax = prefill_rows(l, Tmax), T16 = (Tmax + 15) & ~15;
    W.plan = off;   off = up256(off + sizeof(int) * (2 + 3 * MOE_MAX_EXPERTS + 2 * size_t(Rmax) + 2 * MOE_MAX_EXPERTS + 3));
    W.Br = off;     off = up256(off + size_t(l.H / kGroup) * Rmax * 128);
    W.Bs = off;     off = up256(off + size_t(l.H / kGroup) * T16 * 128);
    W.Hr = off;     off = up256(off + size_t(l.I / kGroup) * Rmax * 128);
    W.Hs = off;     off = up256(off + size_t(l.Is / kGroup) * T16 * 128);
    W.Yr = off;     off = up256(off + sizeof(float) * size_t(Tmax) * l.topk * l.H);
    W.Ys = off;     off = up256(off + sizeof(float) * size_t(T16) * l.H);
    W.xn = off;     off = up256(off + sizeof(float) * size_t(Tmax) * l.H);
    W.total = off;
    return W;
}

inline Ws ws_bind(void *base, const WsLayout &W, const moe_layer_t &l) {
    uint8_t *p = (uint8_t *)base;
    Ws w;
    w.ctrl = (unsigned *)(p + W.ctrl);
    w.ticket = w.ctrl + kCtrlWords;
    w.logits = (float *)(p + W.logits);
    w.idx = (int *)(p + W.idx);
    w.gate = (float *)(p + W.gate);
    w.h16 = (__half *)(p + W.h16);
    w.hs16 = (__half *)(p + W.hs16);
    w.pr = (float *)(p + W.pr);
    w.ps = (float *)(p + W.ps);
    w.xh = (float *)(p + W.xh);
    w.yh = (float *)(p + W.yh);
    w.ih = (int *)(p + W.ih);
    w.gh = (float *)(p + W.gh);
    w.plan = (int *)(p + W.plan);
    w.Br = p + W.Br;
    w.Bs = p + W.Bs;
    w.Hr = p + W.Hr;
    w.Hs = p + W.Hs;
    w.Yr = (float *)(p + W.Yr);
    w.Ys = (float *)(p + W.Ys);
    w.xn = (float *)(p + W.xn);
    w.Tmax = W.Tmax;
    (void)l;
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

// Consumes a pending moe_debug_inject of kind `what` (true if there was one).
bool take_injection(int what);

// y = W x for one token with the output-projection kernel of the attention block
// (16-row tiles, weights by bulk copy into shared memory): N a multiple of 16,
// K <= 8192, every operand 16-byte aligned.  Defined with that kernel.
int qgemv_rows16(const uint32_t *q, const __half *s, const __half *b, int N, int K, const float *x, float *y,
                 cudaStream_t st);

}  // namespace moe
