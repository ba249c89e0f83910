// moe_api.cu -- the C ABI of libmoe (include/moe.h): argument checks, workspace
// layout and kernel launches.  All arithmetic runs in the kernels included below.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <atomic>
#include <chrono>
#include <mutex>

#include "common.cuh"
#include "route.cuh"
#include "quantise.cuh"
#include "tile.cuh"
#include "decode.cuh"
#include "prefill.cuh"
#include "gemv.cuh"
#include "sample.cuh"
#include "lfu.h"

using namespace moe;

namespace {

cudaStream_t as_stream(void *s) { return (cudaStream_t)s; }

// Fault injection for tests of the error paths (moe_debug_inject): the next
// eligible call consumes it.
std::atomic<int> g_inject{MOE_INJECT_NONE};
constexpr unsigned long long kInjectWaitNs = 2ull * 1000 * 1000;  // 2 ms

bool take_inject(int what) {
    int v = what;
    return g_inject.compare_exchange_strong(v, MOE_INJECT_NONE);
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool layer_ok(const moe_layer_t *l) {
    if (!l) return false;
    if (l->H <= 0 || l->H % 128 || l->I <= 0 || l->I % kGroup || l->Is <= 0 || l->Is % kGroup)
        return false;
    if (l->E <= 0 || l->E > MOE_MAX_EXPERTS || l->topk <= 0 || l->topk > MOE_MAX_TOPK ||
        l->topk > l->E)
        return false;
    if (!l->r_q || !l->r_s || !l->r_b || !l->shared) return false;
    if (!aligned(l->r_q, 16) || !aligned(l->r_s, 16) || !aligned(l->r_b, 16) ||
        !aligned(l->shared, 256))
        return false;
    return true;
}

bool experts_ok(const moe_layer_t *l) {
    return l->experts && aligned(l->experts, 256) && l->expert_stride % 256 == 0 &&
           l->expert_stride >= tile_layout(l->H, l->I).total;
}

LayerDev layer_dev(const moe_layer_t *l) {
    LayerDev d;
    d.H = l->H;
    d.E = l->E;
    d.topk = l->topk;
    d.I = l->I;
    d.Is = l->Is;
    d.rq = l->r_q;
    d.rs = (const __half *)l->r_s;
    d.rb = (const __half *)l->r_b;
    d.experts = (const uint8_t *)l->experts;
    d.stride = l->expert_stride;
    d.shared = (const uint8_t *)l->shared;
    d.bias = l->logit_bias;
    d.norm_w = nullptr;
    d.norm_eps = l->norm_eps;
    d.L = blob_layout(l->H, l->I);
    d.Ls = blob_layout(l->H, l->Is);
    return d;
}

int cuda_status() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (getenv("MOE_DEBUG")) fprintf(stderr, "libmoe: CUDA error %s\n", cudaGetErrorString(e));
        return MOE_ECUDA;
    }
    return MOE_OK;
}

// The workspace layout depends on T_max; recover the largest T_max whose layout
// fits in ws_bytes (it is what the caller sized it for, or larger).  Decode uses
// only the layout's prefix (decode_total); the prefill chunk needs all of it.
// Only the header is carried from call to call, and it sits at a fixed place.
WsLayout ws_fit(const moe_layer_t *l, size_t ws_bytes, bool full) {
    // the sizes grow with T_max: a binary search over 1..MOE_MAX_PREFILL_TOKENS, and the
    // last answer is kept per thread (a decode loop binds the same workspace every call)
    struct Key {
        int H, E, topk, I, Is, full;
        size_t bytes;
        bool operator==(const Key &o) const {
            return H == o.H && E == o.E && topk == o.topk && I == o.I && Is == o.Is && full == o.full &&
                   bytes == o.bytes;
        }
    };
    static thread_local Key last_key{-1, 0, 0, 0, 0, 0, 0};
    static thread_local WsLayout last;
    const Key key{l->H, l->E, l->topk, l->I, l->Is, full ? 1 : 0, ws_bytes};
    if (key == last_key) return last;
    auto size_of = [&](int t) {
        const WsLayout w = ws_layout(*l, t);
        return full ? w.total : w.decode_total;
    };
    int lo = 1, hi = MOE_MAX_PREFILL_TOKENS;  // the answer: the largest fitting T_max, else 1
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (size_of(mid) <= ws_bytes) lo = mid; else hi = mid - 1;
    }
    last = ws_layout(*l, lo);
    last_key = key;
    return last;
}

// Binds the caller's workspace: the layout is the one for the largest T_max whose
// size fits ws_bytes (what moe_workspace_bytes was asked for, or more).
int bind_ws(const moe_layer_t *l, int T, void *d_ws, size_t ws_bytes, Ws *out, bool full = false) {
    if (!d_ws || !aligned(d_ws, 256)) return MOE_EWORKSPACE;
    WsLayout W = ws_fit(l, ws_bytes, full);
    if ((full ? W.total : W.decode_total) > ws_bytes || W.Tmax < T) return MOE_EWORKSPACE;
    *out = ws_bind(d_ws, W, *l);
    return MOE_OK;
}

int launch_route(const moe_layer_t *l, const LayerDev &ly, const float *x, int T, Ws ws,
                 int32_t *idx, float *gate, float *logits, cudaStream_t st, int32_t *idx_host = nullptr,
                 unsigned *flag_host = nullptr, unsigned seq = 0, bool prenorm = false, DevLfu *lfu = nullptr) {
    const dim3 grid((l->E + kRouteExp - 1) / kRouteExp, (T + kRouteTok - 1) / kRouteTok);
    LayerDev lr = ly;
    lr.norm_w = prenorm ? l->norm_w : nullptr;
    lr.norm_eps = l->norm_eps;
    k_route<<<grid, kRouteTok * 32, 0, st>>>(lr, x, T, ws, idx, gate, logits, idx_host, flag_host, seq, lfu);
    return cuda_status();
}

// Flags a layer call accepts; MOE_PRENORM needs the layer's RMSNorm weight.
bool flags_ok(const moe_layer_t *l, int flags) {
    if (flags & ~(MOE_RESIDUAL | MOE_PRENORM)) return false;
    if ((flags & MOE_PRENORM) && (!l->norm_w || !aligned(l->norm_w, 16) || !(l->norm_eps >= 0.f)))
        return false;
    return true;
}

int check_layer_call(const moe_layer_t *l, const float *x, int T, int Tlimit, int flags,
                     const float *y) {
    if (!layer_ok(l) || !experts_ok(l) || !x || !y || T < 1 || T > Tlimit) return MOE_EINVAL;
    if (!flags_ok(l, flags)) return MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(y, 16) || x == y) return MOE_EINVAL;
    return MOE_OK;
}

// The device's address of a page-locked host buffer mapped into its address space
// (null when p is null or not such a buffer).
template <typename T>
T *mapped_alias(T *p) {
    if (!p) return nullptr;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
    return reinterpret_cast<T *>(at.devicePointer);
}

// x staging ahead of a decode launch: the decode (programmatic dependent launch) may
// start its weight-only prologue at once and waits for this kernel before it reads x.
__global__ void __launch_bounds__(256) k_copy16(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t n) {
    pdl_launch_dependents();
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = src[i];
}

// RMSNorm, one CTA per row: y = x * w / sqrt(mean(x^2) + eps).
__global__ void __launch_bounds__(256) k_rmsnorm(const float *x, const float *__restrict__ w, float eps, int H,
                                                 float *y) {
    const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)blockIdx.x * H);
    float4 *yr = reinterpret_cast<float4 *>(y + (size_t)blockIdx.x * H);
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
    __shared__ float part[8];
    __shared__ float inv;
    float sq = 0.f;
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x) {
        const float4 v = xr[i];
        sq += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    sq = warp_sum(sq);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); i++) s += part[i];
        inv = rms_inv(s, H, eps);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x) {
        const float4 v = xr[i], g = __ldg(w4 + i);
        yr[i] = make_float4(v.x * g.x * inv, v.y * g.y * inv, v.z * g.z * inv, v.w * g.w * inv);
    }
}

struct DecodeCfg {
    int device = -1, sms = 0, smem_optin = 0;
    size_t static_smem[2][5] = {};
    bool attr_set[2][5] = {};
    int attr_smem[2][5] = {};
};

template <int NCH, int GPW>
void *decode_fn() { return (void *)k_decode<NCH, GPW>; }

void *decode_kernel(int nch, int gpw) {
    static void *const table[2][5] = {
        {decode_fn<1, 1>(), decode_fn<1, 2>(), decode_fn<1, 3>(), decode_fn<1, 4>(), decode_fn<1, 5>()},
        {decode_fn<2, 1>(), decode_fn<2, 2>(), decode_fn<2, 3>(), decode_fn<2, 4>(), decode_fn<2, 5>()}};
    return table[nch - 1][gpw - 1];
}

struct DecodePlan {
    DecodeArgs a;
    void *fn = nullptr;
    long long smem = 0;
    int nC = 0;
};

// Arguments and launch shape of the decode kernel for one call (experts from
// the layer; a cache replaces them before the launch).
int decode_plan(const moe_layer_t *l, const float *x, int T, int flags, float *y, int32_t *idx_out,
                float *gate_out, const Ws &ws, DecodePlan *plan) {
    static thread_local DecodeCfg cfg;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status();
    if (cfg.device != dev) {
        cfg = DecodeCfg();
        cfg.device = dev;
        if (cudaDeviceGetAttribute(&cfg.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&cfg.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return cuda_status();
    }
    DecodeArgs &a = plan->a;
    memset(&a, 0, sizeof(a));
    a.H = l->H; a.E = l->E; a.topk = l->topk; a.I = l->I; a.Is = l->Is;
    a.rq = l->r_q; a.rs = (const __half *)l->r_s; a.rb = (const __half *)l->r_b; a.bias = l->logit_bias;
    a.experts = (const uint8_t *)l->experts; a.stride = l->expert_stride; a.shared = (const uint8_t *)l->shared;
    a.Lr = tile_layout(l->H, l->I);
    a.Ls = tile_layout(l->H, l->Is);
    a.P = shared_parts(l->I, l->Is);
    a.x = x; a.T = T; a.flags = flags; a.y = y; a.idx_out = idx_out; a.gate_out = gate_out;
    a.ctrl = ws.ctrl; a.ticket = ws.ticket; a.logits = ws.logits; a.h16 = ws.h16; a.hs16 = ws.hs16;
    a.pr = ws.pr; a.ps = ws.ps;
    a.mode = kModeShared | kModeRouted;
    a.route_extra = 0;
    a.route_wait_ns = kWaitNs;
    a.norm_w = l->norm_w;
    a.norm_eps = l->norm_eps;
    const int nch = T > 8 ? 2 : 1;
    const int gpw = (a.Lr.G + kCW - 1) / kCW;
    if (gpw > 5 || l->H > kMaxHiddenLayer) return MOE_EINVAL;  // hidden size above 4096
    const int nC = cfg.sms;
    if ((l->E + nC - 1) / nC > kMaxRouterRows) return MOE_EINVAL;
    const int R = a.Lr.R, Gi = a.Lr.Gi;
    const int Umax = T * l->topk < l->E ? T * l->topk : l->E;
    const long long units_cta = ((long long)(a.P + Umax) * R + nC - 1) / nC;
    if (units_cta > kMaxUnitsPerCta) return MOE_EINVAL;
    const int hsm_mats = (int)((units_cta + R - 1) / R) + 1;
    a.SB = (int)(((size_t)(a.Lr.G > Gi ? a.Lr.G : Gi) * kTileBytes + 127) / 128 * 128);
    a.UPS = a.SB / (Gi * kTileBytes);
    a.hsm_mat_bytes = Gi * T * 128;
    void *fn = decode_kernel(nch, gpw);
    size_t &st = cfg.static_smem[nch - 1][gpw - 1];
    if (st == 0) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return cuda_status();
        st = fa.sharedSizeBytes + 1;  // +1: computed
    }
    const long long budget = (long long)cfg.smem_optin - (long long)(st - 1);
    // the h region also stages the T x E router logits while the routing is built
    long long hsm = (long long)hsm_mats * a.hsm_mat_bytes;
    const long long lg = ((long long)T * l->E * 4 + 127) / 128 * 128;
    if (hsm < lg) hsm = lg;
    int stages = kMaxStages;
    long long smem = 0;
    for (; stages >= 2; stages--) {
        const long long red = (long long)(stages + 2) * kCW * nch * 512;  // gate/up partial-sum slots
        smem = (long long)stages * a.SB + red + hsm + (long long)hsm_mats * Gi * 16 * 4;
        if (smem <= budget) break;
    }
    if (stages < 2) return MOE_EINVAL;
    a.stages = stages;
    a.red_off = stages * a.SB;
    a.hsm_off = a.red_off + (stages + 2) * kCW * nch * 512;
    a.hsum_off = (int)(a.hsm_off + hsm);
    if (cfg.attr_smem[nch - 1][gpw - 1] < smem) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return cuda_status();
        cfg.attr_smem[nch - 1][gpw - 1] = (int)smem;
    }
    plan->fn = fn;
    plan->smem = smem;
    plan->nC = nC;
    return MOE_OK;
}

// One CTA per SM, launched with programmatic dependent launch: when the previous
// operation on the stream is a decode kernel, this one starts on each SM as that
// kernel leaves it, and runs its prologue there (barrier set-up, weight copies and
// prefetches) before waiting for it (griddepcontrol.wait).  It is not a
// cooperative launch -- a cooperative grid starts only once the whole GPU is
// free -- but its CTAs are resident together all the same: the previous decode
// kernel signals launch_dependents at its start, so all of its CTAs are resident
// before this grid launches, and this grid's CTAs take SMs as those exit (any
// other predecessor has finished before the launch).  Every cross-CTA wait is
// bounded in any case.  If the runtime refuses programmatic dependent launch, a
// cooperative launch is used from then on.
int decode_launch(DecodePlan &plan, int mode, void *stream) {
    static std::atomic<int> pdl_ok{1};  // shared by every calling thread
    plan.a.mode = mode;
    void *args[] = {&plan.a};
    if (pdl_ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(plan.nC);
        cfg.blockDim = dim3(kDecThreads);
        cfg.dynamicSmemBytes = (size_t)plan.smem;
        cfg.stream = as_stream(stream);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelExC(&cfg, plan.fn, args);
        if (e == cudaSuccess) return MOE_OK;
        if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return cuda_status();
        (void)cudaGetLastError();
        pdl_ok.store(0);
    }
    if (cudaLaunchCooperativeKernel(plan.fn, dim3(plan.nC), dim3(kDecThreads), args, (size_t)plan.smem,
                                    as_stream(stream)) != cudaSuccess)
        return cuda_status();
    return cuda_status();
}

int run_decode(const moe_layer_t *l, const float *x, int T, int flags, float *y, int32_t *idx_out,
               float *gate_out, void *d_ws, size_t ws_bytes, void *stream) {
    Ws ws;
    int rc = bind_ws(l, T, d_ws, ws_bytes, &ws);
    if (rc) return rc;
    DecodePlan plan;
    if ((rc = decode_plan(l, x, T, flags, y, idx_out, gate_out, ws, &plan))) return rc;
    if (take_inject(MOE_INJECT_WAIT)) {
        // the routing wait expects one router row more than there are: it runs out
        plan.a.route_extra = 1;
        plan.a.route_wait_ns = kInjectWaitNs;
    }
    return decode_launch(plan, kModeShared | kModeRouted, stream);
}

// Prefill chunk: router, plan, gather, both grouped GEMMs on the tensor cores in
// one launch, combine (prefill.cuh).
int run_layer_chunk(const moe_layer_t *l, const float *x, int T, int flags, float *y,
                    int32_t *idx_out, float *gate_out, void *d_ws, size_t ws_bytes, void *stream) {
    Ws ws;
    int rc = bind_ws(l, T, d_ws, ws_bytes, &ws, true);
    if (rc) return rc;
    static thread_local int sms = 0, dev_seen = -1, smem_set = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status();
    if (dev != dev_seen) {
        dev_seen = dev;
        smem_set = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cuda_status();
    }
    if (!smem_set) {
        if (cudaFuncSetAttribute(k_prefill_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)prefill_gemm_smem()) != cudaSuccess ||
            cudaFuncSetAttribute(k_prefill_route, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)prefill_route_smem()) != cudaSuccess)
            return cuda_status();
        smem_set = 1;
    }
    cudaStream_t st = as_stream(stream);
    LayerDev ly = layer_dev(l);
    // with MOE_PRENORM the chunk runs on RMSNorm(x) (a copy in the workspace); the
    // residual below still adds the raw x
    const float *xin = x;
    if (flags & MOE_PRENORM) {
        k_rmsnorm<<<T, 256, 0, st>>>(x, l->norm_w, l->norm_eps, l->H, ws.xn);
        if ((rc = cuda_status())) return rc;
        xin = ws.xn;
    }
    // the router: tiled over (K slice, 64 experts, 32 tokens) when the slices' partial
    // sums fit in the down GEMM's fp32 output rows (unused until that GEMM runs)
    const int KS = prefill_route_slices(l->H), nEB = (l->E + kRtExp - 1) / kRtExp;
    const int nTB = (T + kRtTok - 1) / kRtTok;
    if ((size_t)KS * l->E <= (size_t)l->topk * l->H) {
        RouteTiledArgs ra;
        ra.rq = ly.rq; ra.rs = ly.rs; ra.rb = ly.rb; ra.bias = ly.bias;
        ra.x = xin; ra.T = T; ra.H = l->H; ra.E = l->E; ra.topk = l->topk;
        ra.part = ws.Yr; ra.idx = ws.idx; ra.gate = ws.gate;
        if (pf_launch(k_prefill_route, dim3(KS, nEB, nTB), dim3(kRtThreads), prefill_route_smem(), st, ra) !=
                cudaSuccess ||
            pf_launch(k_prefill_topk, dim3((T + kRtTopkWarps - 1) / kRtTopkWarps), dim3(kRtTopkWarps * 32), 0, st,
                      ra, KS) != cudaSuccess)
            return cuda_status();
    } else if ((rc = launch_route(l, ly, xin, T, ws, ws.idx, ws.gate, nullptr, st))) {
        return rc;
    }
    const int P2 = T * l->topk;
    if (idx_out && cudaMemcpyAsync(idx_out, ws.idx, sizeof(int32_t) * P2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return cuda_status();
    if (gate_out && cudaMemcpyAsync(gate_out, ws.gate, sizeof(float) * P2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return cuda_status();
    const int Rmax = prefill_rows(*l, T), T16 = (T + 15) & ~15;
    PfPlan plan;
    plan.U = ws.plan;
    plan.uexp = ws.plan + 2;
    plan.urow = plan.uexp + MOE_MAX_EXPERTS;
    plan.ucnt = plan.urow + MOE_MAX_EXPERTS;
    plan.rowtok = plan.ucnt + MOE_MAX_EXPERTS;
    plan.rowpair = plan.rowtok + Rmax;
    plan.uslc = plan.rowpair + Rmax;
    plan.dep = reinterpret_cast<unsigned *>(plan.uslc + MOE_MAX_EXPERTS + 1);
    if (pf_launch(k_prefill_plan, dim3(1), dim3(kPlanThreads), 0, st, (const int *)ws.idx, T, l->E, l->topk, Rmax, plan) !=
        cudaSuccess)
        return cuda_status();
    // (a grid-stride loop over the rows the plan used: 8 CTAs of 256 per SM)
    const long long gthreads = (long long)(Rmax + T16) * (l->H / kGroup) * 8;
    const long long gneed = (gthreads + 255) / 256;
    const unsigned gblocks = (unsigned)(gneed < 8LL * sms ? gneed : 8LL * sms);
    if (pf_launch(k_prefill_gather, dim3(gblocks), dim3(256), 0, st, xin, T, l->H, Rmax,
                  T16, (const int *)plan.rowtok, (const int *)plan.U, ws.Br, ws.Bs) != cudaSuccess)
        return cuda_status();
    PrefillGemmArgs g;
    g.H = l->H; g.I = l->I; g.Is = l->Is; g.T = T; g.T16 = T16; g.Rmax = Rmax;
    g.U = plan.U; g.uexp = plan.uexp; g.urow = plan.urow; g.ucnt = plan.ucnt; g.rowpair = plan.rowpair; g.uslc = plan.uslc;
    g.experts = (const uint8_t *)l->experts; g.stride = l->expert_stride; g.shared = (const uint8_t *)l->shared;
    g.Lr = tile_layout(l->H, l->I);
    g.Ls = tile_layout(l->H, l->Is);
    g.Br = ws.Br; g.Bs = ws.Bs; g.Hr = ws.Hr; g.Hs = ws.Hs; g.Yr = ws.Yr; g.Ys = ws.Ys;
    // the down GEMM cuts the shared expert's K = Is into parts of the routed experts'
    // K = I (equal items over the CTAs); parts 1.. go to the gate/up token tiles' area,
    // free once the gate/up GEMM has run
    const int sp = shared_parts(l->I, l->Is);
    const size_t br_bytes = (size_t)(l->H / kGroup) * Rmax * 128;
    g.sparts = (sp > 1 && (size_t)(sp - 1) * T16 * l->H * sizeof(float) <= br_bytes) ? sp : 1;
    g.Ys_more = reinterpret_cast<float *>(ws.Br);
    g.err = &ws.ctrl[kErr];
    const int sparts = g.sparts;
    g.dep = plan.dep;
    // both GEMMs in one launch of one CTA per SM (all resident: the down items wait on
    // the gate/up items' counters)
    if (pf_launch(k_prefill_gemm, dim3(sms), dim3(kPfThreads), prefill_gemm_smem(), st, g) != cudaSuccess)
        return cuda_status();
    const long long cthreads = (long long)T * (l->H / 4);
    if (pf_launch(k_prefill_combine, dim3((unsigned)((cthreads + 255) / 256)), dim3(256), 0, st, x, T, l->H,
                  l->topk, flags, (const float *)ws.gate, (const float *)ws.Yr, (const float *)ws.Ys, sparts,
                  (const float *)g.Ys_more, T16, y) != cudaSuccess)
        return cuda_status();
    return MOE_OK;
}

}  // namespace

// ------------------------------------------------------------------ LFU policy and cache
struct moe_lfu {
    moe::LfuPolicy policy;
    moe_lfu(int slots, int E) : policy(slots, E) {}
};

struct moe_cache {
    int H, E, I, slots, device;
    size_t blob, host_stride;
    const uint8_t *h_experts;
    // device-resident policy (moe_cache_set_device_policy): the state in device
    // memory and the device's address of the host blobs
    int dev_policy = 0;
    moe::DevLfu *d_lfu = nullptr;
    const uint8_t *h_experts_dev = nullptr;
    uint8_t *d_slots = nullptr;
    int32_t *h_idx = nullptr;  // page-locked, device-mapped: the step's routing (the router writes it)
    int32_t *d_idx = nullptr;  // its device address
    unsigned *h_flag = nullptr, *d_flag = nullptr;  // the router's per-call flag (after h_idx)
    unsigned seq = 0;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_copies = nullptr;
    moe::LfuPolicy policy;
    uint64_t h2d_bytes = 0;
    moe_cache(int slots_, int E_) : policy(slots_, E_) {}
};

namespace {

// The cache's policy state as the device keeps it.
moe::DevLfu dev_state_of(const moe::LfuPolicy &p, uint64_t h2d_bytes) {
    moe::DevLfu d;
    memset(&d, 0, sizeof(d));
    d.slots = p.slots();
    d.E = p.experts();
    d.step = p.steps();
    d.hits = p.hits();
    d.misses = p.misses();
    d.h2d_bytes = h2d_bytes;
    for (int s = 0; s < kDevLfuMaxSlots; s++) {
        d.expert_of[s] = s < p.slots() ? p.expert_in(s) : -1;
        d.count[s] = s < p.slots() ? p.count_of(s) : 0u;
        d.last[s] = s < p.slots() ? p.last_of(s) : 0;
    }
    for (int e = 0; e < MOE_MAX_EXPERTS; e++) d.where[e] = (short)(e < p.experts() ? p.slot_of(e) : -1);
    return d;
}

// Brings a device-resident policy's state back into the host policy (waits for
// the device first).
int cache_pull(moe_cache *c) {
    if (!c->dev_policy) return MOE_OK;
    moe::DevLfu d;
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(&d, c->d_lfu, sizeof(d), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_status();
    uint32_t cnt[kDevLfuMaxSlots];
    int64_t last[kDevLfuMaxSlots];
    for (int s = 0; s < kDevLfuMaxSlots; s++) {
        cnt[s] = d.count[s];
        last[s] = d.last[s];
    }
    c->policy.load(d.expert_of, cnt, last, d.step, d.hits, d.misses);
    c->h2d_bytes = d.h2d_bytes;
    return MOE_OK;
}

void cache_free(moe_cache *c) {
    if (!c) return;
    if (c->d_slots) cudaFree(c->d_slots);
    if (c->d_lfu) cudaFree(c->d_lfu);
    if (c->h_idx) cudaFreeHost(c->h_idx);  // h_flag lives in the same allocation
    if (c->ev_copies) cudaEventDestroy(c->ev_copies);
    if (c->side) cudaStreamDestroy(c->side);
    delete c;
}

// Decode through a cache: router launch (it writes the routing into mapped host
// memory and then a per-call flag, which the host polls), LFU step, copies of the
// missing experts on the side stream, then the shared expert (overlapping the
// copies) and the routed experts.
int run_decode_cached(const moe_layer_t *l, const float *x, int T, int flags, float *y, int32_t *idx_out,
                      float *gate_out, moe_cache *c, void *d_ws, size_t ws_bytes, void *stream) {
    if (c->H != l->H || c->E != l->E || c->I != l->I) return MOE_EINVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status();
    if (dev != c->device) return MOE_EINVAL;
    Ws ws;
    int rc = bind_ws(l, T, d_ws, ws_bytes, &ws);
    if (rc) return rc;
    cudaStream_t st = as_stream(stream);
    LayerDev ly = layer_dev(l);
    if (c->dev_policy) {
        // everything on `stream`, nothing waited for on the host: the router's ranking
        // CTA runs the policy step, the fetch kernel copies the misses from host
        // memory into their slots, the decode kernel reads the slot map on the device
        if (T * l->topk > c->slots) return MOE_ECAPACITY;
        if ((rc = launch_route(l, ly, x, T, ws, ws.idx, ws.gate, nullptr, st, nullptr, nullptr, 0,
                               flags & MOE_PRENORM, c->d_lfu)))
            return rc;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cuda_status();
        k_cache_fetch<<<2 * sms, 256, 0, st>>>(c->d_lfu, c->h_experts_dev, c->host_stride, c->d_slots, c->blob);
        if ((rc = cuda_status())) return rc;
        DecodePlan plan;
        if ((rc = decode_plan(l, x, T, flags, y, idx_out, gate_out, ws, &plan))) return rc;
        plan.a.experts = c->d_slots;
        plan.a.stride = c->blob;
        plan.a.use_map = 1;
        plan.a.slot_dev = c->d_lfu->where;
        plan.a.idx_pre = ws.idx;
        plan.a.gate_pre = ws.gate;
        return decode_launch(plan, kModeShared | kModeRouted | kModePre, stream);
    }
    const unsigned seq = ++c->seq == 0 ? ++c->seq : c->seq;  // never 0 (the flag's initial value)
    if ((rc = launch_route(l, ly, x, T, ws, ws.idx, ws.gate, nullptr, st, c->d_idx, c->d_flag, seq,
                           flags & MOE_PRENORM)))
        return rc;
    const int P2 = T * l->topk;
    {
        // the router's flag (bounded: 5 s; a failed stream ends the wait at once)
        volatile unsigned *flag = c->h_flag;
        const auto t0 = std::chrono::steady_clock::now();
        for (unsigned spin = 0; *flag != seq; spin++) {
            if ((spin & 1023u) == 1023u) {
                const cudaError_t q = cudaStreamQuery(st);
                if (q != cudaSuccess && q != cudaErrorNotReady) return cuda_status();
                if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(5)) return MOE_ETIMEOUT;
            }
        }
        std::atomic_thread_fence(std::memory_order_acquire);
    }
    int32_t req[kMaxPairs], slot[kMaxPairs];
    uint8_t hit[kMaxPairs];
    int n = 0;
    for (int p = 0; p < P2; p++) {
        bool seen = false;
        for (int i = 0; i < n && !seen; i++) seen = req[i] == c->h_idx[p];
        if (!seen) req[n++] = c->h_idx[p];
    }
    const moe::LfuPolicy before = c->policy;  // restored if the step cannot be carried out
    rc = c->policy.step(req, n, slot, hit);
    if (rc == 3) return MOE_ECAPACITY;
    if (rc) return MOE_EINVAL;
    // A failure from here on leaves the policy as it was before the step, except
    // that the slots whose copies were already issued are marked empty (their
    // contents are no longer the experts the policy had there).
    int issued[kMaxPairs], n_issued = 0;
    auto fail = [&](int status) {
        c->policy = before;
        for (int i = 0; i < n_issued; i++) c->policy.invalidate(issued[i]);
        return status;
    };
    DecodePlan plan;
    if ((rc = decode_plan(l, x, T, flags, y, idx_out, gate_out, ws, &plan))) return fail(rc);
    plan.a.experts = c->d_slots;
    plan.a.stride = c->blob;
    plan.a.use_map = 1;
    plan.a.idx_pre = ws.idx;
    plan.a.gate_pre = ws.gate;
    for (int e = 0; e < l->E; e++) plan.a.slot_map[e] = (short)c->policy.slot_of(e);
    int misses = 0;
    for (int i = 0; i < n; i++) {
        if (hit[i]) continue;
        if (take_inject(MOE_INJECT_COPY)) return fail(MOE_ECUDA);  // as if the copy had failed
        // The slot's previous expert was last read by work that precedes the
        // router launch on `stream`, which the host has just waited for.
        if (cudaMemcpyAsync(c->d_slots + (size_t)slot[i] * c->blob, c->h_experts + (size_t)req[i] * c->host_stride,
                            c->blob, cudaMemcpyHostToDevice, c->side) != cudaSuccess)
            return fail(cuda_status());
        issued[n_issued++] = slot[i];
        c->h2d_bytes += c->blob;
        misses++;
    }
    if (misses == 0) {
        rc = decode_launch(plan, kModeShared | kModeRouted | kModePre, stream);
        return rc ? fail(rc) : MOE_OK;
    }
    if (cudaEventRecord(c->ev_copies, c->side) != cudaSuccess) return fail(cuda_status());
    if ((rc = decode_launch(plan, kModeShared | kModePre, stream))) return fail(rc);
    if (cudaStreamWaitEvent(st, c->ev_copies, 0) != cudaSuccess) return fail(cuda_status());
    rc = decode_launch(plan, kModeRouted | kModePre, stream);
    return rc ? fail(rc) : MOE_OK;
}

// ------------------------------------------------------------------ allocation-free decode
// Scratch of moe_layer_decode_noalloc.  In host code this name is only a stand-in
// for the device array, so the host looks up its device address once per device
// and hands that address to the kernel like any workspace.
__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the current device's scratch array; the first call on a device
// looks it up and zeroes the array (then waits for the device).
int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status();
    if (dev < 0 || dev >= kMaxDevices) return MOE_EINVAL;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return cuda_status();
        if (cudaMemset(p, 0, MOE_NOALLOC_SCRATCH_BYTES) != cudaSuccess) return cuda_status();
        if (cudaDeviceSynchronize() != cudaSuccess) return cuda_status();
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

// Reads the error word at the start of a scratch area after `stream` is idle and,
// if a device-side wait gave up, zeroes the whole area (then waits for the
// device): MOE_ETIMEOUT; MOE_OK otherwise.
int scratch_status(void *d_ws, size_t ws_bytes, cudaStream_t st) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_status();
    unsigned err = 0;
    if (cudaMemcpy(&err, d_ws, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_status();
    if (err) {
        if (cudaMemset(d_ws, 0, ws_bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return cuda_status();
        return MOE_ETIMEOUT;
    }
    return MOE_OK;
}

}  // namespace


// ------------------------------------------------------------------ prepared host call
struct moe_host_call {
    moe_layer_t layer;
    int T = 0, flags = 0;
    void *ws = nullptr;
    size_t ws_bytes = 0, xb = 0;
    cudaStream_t st = nullptr, cap = nullptr;
    float *x_h = nullptr, *y_h = nullptr;           // page-locked, mapped staging rows
    unsigned *flag_h = nullptr;                      // completion word (page-locked, mapped)
    unsigned *count_d = nullptr;                     // steps completed (device memory)
    unsigned seq = 0;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

namespace {

// After the step: counts it and publishes the count to the host's completion word.
__global__ void k_host_signal(unsigned *count, volatile unsigned *flag) {
    const unsigned v = *count + 1u;
    *count = v;
    __threadfence_system();
    *flag = v;
}

void host_call_free(moe_host_call *c) {
    if (c->exec) cudaGraphExecDestroy(c->exec);
    if (c->graph) cudaGraphDestroy(c->graph);
    if (c->cap) cudaStreamDestroy(c->cap);
    if (c->x_h) cudaFreeHost(c->x_h);
    if (c->y_h) cudaFreeHost(c->y_h);
    if (c->flag_h) cudaFreeHost(c->flag_h);
    if (c->count_d) cudaFree(c->count_d);
    delete c;
}

}  // namespace

extern "C" {

const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_EINVAL: return "invalid argument (shape, size, flag or pointer)";
        case MOE_ECUDA: return "CUDA runtime error";
        case MOE_ECAPACITY: return "more distinct experts requested than cache slots";
        case MOE_ETIMEOUT: return "a bounded device-side wait gave up";
        case MOE_EWORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ENOTREADY: return "handle not ready";
        default: return "unknown status";
    }
}

size_t moe_expert_blob_bytes(int H, int I) {
    if (H <= 0 || I <= 0 || H % kGroup || I % kGroup) return 0;
    return blob_layout(H, I).total;
}

int moe_expert_blob_offsets(int H, int I, size_t offsets_out[6]) {
    if (!offsets_out || H <= 0 || I <= 0 || H % kGroup || I % kGroup) return MOE_EINVAL;
    BlobLayout L = blob_layout(H, I);
    offsets_out[0] = L.gu_q;
    offsets_out[1] = L.gu_s;
    offsets_out[2] = L.gu_b;
    offsets_out[3] = L.d_q;
    offsets_out[4] = L.d_s;
    offsets_out[5] = L.d_b;
    return MOE_OK;
}

size_t moe_tile_blob_bytes(int H, int I) {
    if (H <= 0 || I <= 0 || H % 128 || I % kGroup) return 0;
    return tile_layout(H, I).total;
}

int moe_expert_tile(const void *mlx_blob, int H, int I, void *tile_blob, void *stream) {
    if (!mlx_blob || !tile_blob || !moe_tile_blob_bytes(H, I) || mlx_blob == tile_blob) return MOE_EINVAL;
    if (!aligned(mlx_blob, 16) || !aligned(tile_blob, 16)) return MOE_EINVAL;
    const TileLayout T = tile_layout(H, I);
    const long long threads = 32ll * ((long long)T.Ti * T.G + (long long)T.R * T.Gi);
    const int block = 256;
    k_tile_expert<<<(unsigned)((threads + block - 1) / block), block, 0, as_stream(stream)>>>(
        (const uint8_t *)mlx_blob, (uint8_t *)tile_blob, H, I);
    return cuda_status();
}

size_t moe_workspace_bytes(const moe_layer_t *layer, int T_max) {
    if (!layer_ok(layer) || T_max < 1 || T_max > MOE_MAX_PREFILL_TOKENS) return 0;
    return ws_layout(*layer, T_max).total;
}

int moe_workspace_init(void *d_ws, size_t ws_bytes, void *stream) {
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes == 0) return MOE_EINVAL;
    cudaMemsetAsync(d_ws, 0, ws_bytes, as_stream(stream));
    return cuda_status();
}

int moe_workspace_status(void *d_ws, size_t ws_bytes, void *stream) {
    if (!d_ws || ws_bytes < 16) return MOE_EINVAL;
    return scratch_status(d_ws, ws_bytes, as_stream(stream));
}

size_t moe_decode_workspace_bytes(const moe_layer_t *layer, int T_max) {
    if (!layer_ok(layer) || T_max < 1 || T_max > MOE_MAX_DECODE_TOKENS) return 0;
    return ws_layout(*layer, T_max).decode_total;
}

int moe_debug_inject(int what) {
    if (what != MOE_INJECT_NONE && what != MOE_INJECT_WAIT && what != MOE_INJECT_COPY && what != MOE_INJECT_ATTN_WAIT)
        return MOE_EINVAL;
    g_inject.store(what);
    return MOE_OK;
}

int affine_quantise(const float *w, int N, int K, int bits, uint32_t *q, uint16_t *s, uint16_t *b,
                    void *stream) {
    if (!w || !q || !s || !b || N < 1 || K < kGroup || K % kGroup || (bits != 4 && bits != 8))
        return MOE_EINVAL;
    long long groups = (long long)N * (K / kGroup);
    int threads = 256;
    long long blocks = (groups + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return MOE_EINVAL;
    k_quantise<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(w, N, K, bits, q, (__half *)s,
                                                                    (__half *)b);
    return cuda_status();
}

int moe_sample(const float *logits, int T, int V, float temperature, int top_k, float top_p, const float *u,
               int32_t *tokens, void *stream) {
    if (!logits || !u || !tokens || T < 1 || V < 1 || !(top_p > 0.f && top_p <= 1.f) || temperature != temperature)
        return MOE_EINVAL;
    if (!aligned(logits, 4) || !aligned(u, 4) || !aligned(tokens, 4)) return MOE_EINVAL;
    const int K = (top_k <= 0 || top_k >= V) ? V : top_k;
    if (temperature > 0.f && K > kSampleMaxK) return MOE_EINVAL;
    // one cluster of kSampleCluster CTAs per row (the kernel's static cluster shape)
    k_sample<<<T * kSampleCluster, kSampleThreads, 0, as_stream(stream)>>>(logits, V, temperature, K, top_p, u,
                                                                        tokens);
    return cuda_status();
}

int moe_rmsnorm(const float *x, const float *w, float eps, int T, int H, float *y, void *stream) {
    if (!x || !w || !y || T < 1 || H < 4 || H % 4 || !(eps >= 0.f)) return MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16)) return MOE_EINVAL;
    k_rmsnorm<<<T, 256, 0, as_stream(stream)>>>(x, w, eps, H, y);
    return cuda_status();
}

int qgemv_affine4(const uint32_t *q, const uint16_t *s, const uint16_t *b, int N, int K,
                  const float *x, float *y, void *stream) {
    if (!q || !s || !b || !x || !y || N < 1 || K < kGroup || K % kGroup) return MOE_EINVAL;
    if (!aligned(q, 16) || !aligned(x, 16)) return MOE_EINVAL;
    if (N % 16 == 0 && K <= 8192 && aligned(s, 16) && aligned(b, 16) && aligned(y, 16))
        return qgemv_rows16(q, (const __half *)s, (const __half *)b, N, K, x, y, as_stream(stream));
    QMat m{q, (const __half *)s, (const __half *)b, N, K};
    k_qgemv4_mma<<<(N + 15) / 16, kGemvWarps * 32, 0, as_stream(stream)>>>(m, x, y);
    return cuda_status();
}

int moe_route(const moe_layer_t *layer, const float *x, int T, int32_t *idx, float *gate,
              float *logits, void *d_ws, size_t ws_bytes, void *stream) {
    if (!layer_ok(layer) || !x || !idx || !gate || T < 1 || T > MOE_MAX_PREFILL_TOKENS)
        return MOE_EINVAL;
    if (!aligned(x, 16)) return MOE_EINVAL;
    Ws ws;
    int rc = bind_ws(layer, T, d_ws, ws_bytes, &ws);
    if (rc) return rc;
    LayerDev ly = layer_dev(layer);
    return launch_route(layer, ly, x, T, ws, idx, gate, logits, as_stream(stream));
}

int moe_layer_decode(const moe_layer_t *layer, const float *x, int T, int flags, float *y,
                     int32_t *idx_out, float *gate_out, moe_cache_t *cache, void *d_ws,
                     size_t ws_bytes, void *stream) {
    if (cache) {
        if (!layer_ok(layer) || !x || !y || T < 1 || T > MOE_MAX_DECODE_TOKENS || !flags_ok(layer, flags) ||
            !aligned(x, 16) || !aligned(y, 16) || x == y)
            return MOE_EINVAL;
        return run_decode_cached(layer, x, T, flags, y, idx_out, gate_out, cache, d_ws, ws_bytes, stream);
    }
    int rc = check_layer_call(layer, x, T, MOE_MAX_DECODE_TOKENS, flags, y);
    if (rc) return rc;
    return run_decode(layer, x, T, flags, y, idx_out, gate_out, d_ws, ws_bytes, stream);
}

// Host buffers: x is staged in the workspace, the decode step runs on the stream,
// y (and the routing) come back; the call returns once the stream is idle.  Where a
// host buffer is page-locked and mapped into the device's address space, the copies
// are kernels' plain accesses instead of DMA transfers (whose set-up dominates at
// these sizes): a small kernel reads x into the workspace, and the decode kernel
// writes y, idx and gate straight into host memory.
int moe_layer_decode_host(const moe_layer_t *layer, const float *x_host, int T, int flags, float *y_host,
                          int32_t *idx_host, float *gate_host, moe_cache_t *cache, void *d_ws, size_t ws_bytes,
                          void *stream) {
    if (!layer_ok(layer) || !x_host || !y_host || T < 1 || T > MOE_MAX_DECODE_TOKENS || !flags_ok(layer, flags))
        return MOE_EINVAL;
    Ws ws;
    int rc = bind_ws(layer, T, d_ws, ws_bytes, &ws);
    if (rc) return rc;
    cudaStream_t st = as_stream(stream);
    const size_t xb = sizeof(float) * (size_t)T * layer->H, rb = (size_t)T * layer->topk;
    const float *xd = mapped_alias(x_host);
    float *yd = mapped_alias(y_host), *gd = mapped_alias(gate_host);
    int32_t *id = mapped_alias(idx_host);
    if (xd && aligned(xd, 16)) {
        k_copy16<<<(unsigned)((xb / 16 + 255) / 256), 256, 0, st>>>(reinterpret_cast<const uint4 *>(xd),
                                                                  reinterpret_cast<uint4 *>(ws.xh), xb / 16);
        if ((rc = cuda_status())) return rc;
    } else if (cudaMemcpyAsync(ws.xh, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        return cuda_status();
    }
    const bool y_direct = yd && aligned(yd, 16) && !cache;
    const bool i_direct = id && !cache, g_direct = gd && !cache;
    rc = moe_layer_decode(layer, ws.xh, T, flags, y_direct ? yd : ws.yh,
                          idx_host ? (i_direct ? id : ws.ih) : nullptr, gate_host ? (g_direct ? gd : ws.gh) : nullptr,
                          cache, d_ws, ws_bytes, stream);
    if (rc) return rc;
    if (!y_direct && cudaMemcpyAsync(y_host, ws.yh, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return cuda_status();
    if (idx_host && !i_direct &&
        cudaMemcpyAsync(idx_host, ws.ih, sizeof(int32_t) * rb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return cuda_status();
    if (gate_host && !g_direct &&
        cudaMemcpyAsync(gate_host, ws.gh, sizeof(float) * rb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return cuda_status();
    // wait for the stream by polling it: a decode step is a few tens of
    // microseconds, shorter than the wake-up of a blocking wait
    cudaError_t q;
    while ((q = cudaStreamQuery(st)) == cudaErrorNotReady) {
    }
    if (q != cudaSuccess) return cuda_status();
    return MOE_OK;
}

int moe_layer_prefill_chunk(const moe_layer_t *layer, const float *x, int T, int flags, float *y,
                            int32_t *idx_out, float *gate_out, void *d_ws, size_t ws_bytes,
                            void *stream) {
    int rc = check_layer_call(layer, x, T, MOE_MAX_PREFILL_TOKENS, flags, y);
    if (rc) return rc;
    return run_layer_chunk(layer, x, T, flags, y, idx_out, gate_out, d_ws, ws_bytes, stream);
}

int moe_lfu_create(moe_lfu_t **out, int slots, int E) {
    if (!out) return MOE_EINVAL;
    *out = nullptr;
    if (slots < 1 || slots > MOE_MAX_CACHE_SLOTS || E < 1 || E > MOE_MAX_EXPERTS) return MOE_EINVAL;
    *out = new (std::nothrow) moe_lfu(slots, E);
    return *out ? MOE_OK : MOE_EINVAL;
}

int moe_lfu_destroy(moe_lfu_t *lfu) {
    delete lfu;
    return MOE_OK;
}

int moe_lfu_step(moe_lfu_t *lfu, const int32_t *req, int n, int32_t *slot_out, uint8_t *hit_out) {
    if (!lfu) return MOE_EINVAL;
    const int rc = lfu->policy.step(req, n, slot_out, hit_out);
    return rc == 3 ? MOE_ECAPACITY : rc ? MOE_EINVAL : MOE_OK;
}

static void policy_state(const moe::LfuPolicy &p, int32_t *expert_of_slot, uint32_t *counts, int64_t *last) {
    for (int s = 0; s < p.slots(); s++) {
        if (expert_of_slot) expert_of_slot[s] = p.expert_in(s);
        if (counts) counts[s] = p.count_of(s);
        if (last) last[s] = p.last_of(s);
    }
}

int moe_lfu_state(const moe_lfu_t *lfu, int32_t *expert_of_slot, uint32_t *counts, int64_t *last,
                  uint64_t *hits, uint64_t *misses) {
    if (!lfu) return MOE_EINVAL;
    policy_state(lfu->policy, expert_of_slot, counts, last);
    if (hits) *hits = lfu->policy.hits();
    if (misses) *misses = lfu->policy.misses();
    return MOE_OK;
}

int moe_cache_create(moe_cache_t **out, int H, int E, int I, const void *h_experts,
                     size_t host_stride, int slots) {
    if (!out) return MOE_EINVAL;
    *out = nullptr;
    const size_t blob = moe_tile_blob_bytes(H, I);
    if (!blob || !h_experts || E < 1 || E > MOE_MAX_EXPERTS || slots < 1 || slots > MOE_MAX_CACHE_SLOTS ||
        host_stride < blob)
        return MOE_EINVAL;
    moe_cache *c = new (std::nothrow) moe_cache(slots, E);
    if (!c) return MOE_EINVAL;
    c->H = H; c->E = E; c->I = I; c->slots = slots;
    c->blob = blob;
    c->host_stride = host_stride;
    c->h_experts = (const uint8_t *)h_experts;
    // the routing buffer and, after it, the router's flag: page-locked, mapped
    const size_t idx_bytes = sizeof(int32_t) * kMaxPairs + 64;
    bool ok = cudaGetDevice(&c->device) == cudaSuccess &&
              cudaMalloc((void **)&c->d_slots, blob * (size_t)slots) == cudaSuccess &&
              cudaHostAlloc((void **)&c->h_idx, idx_bytes, cudaHostAllocMapped) == cudaSuccess &&
              cudaHostGetDevicePointer((void **)&c->d_idx, c->h_idx, 0) == cudaSuccess &&
              cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&c->ev_copies, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cache_free(c);
        (void)cudaGetLastError();
        return MOE_ECUDA;
    }
    c->h_flag = reinterpret_cast<unsigned *>(c->h_idx + kMaxPairs);
    c->d_flag = reinterpret_cast<unsigned *>(c->d_idx + kMaxPairs);
    *c->h_flag = 0u;
    *out = c;
    return MOE_OK;
}

int moe_cache_destroy(moe_cache_t *cache) {
    if (!cache) return MOE_OK;
    cudaStreamSynchronize(cache->side);
    if (cache->dev_policy) cudaDeviceSynchronize();
    cache_free(cache);
    return cuda_status();
}

int moe_cache_slots(const moe_cache_t *cache, int32_t *expert_of_slot, uint32_t *counts) {
    if (!cache) return MOE_EINVAL;
    const int rc = cache_pull(const_cast<moe_cache *>(cache));
    if (rc) return rc;
    policy_state(cache->policy, expert_of_slot, counts, nullptr);
    return MOE_OK;
}

int moe_cache_stats(const moe_cache_t *cache, uint64_t *hits, uint64_t *misses, uint64_t *h2d_bytes) {
    if (!cache) return MOE_EINVAL;
    const int rc = cache_pull(const_cast<moe_cache *>(cache));
    if (rc) return rc;
    if (hits) *hits = cache->policy.hits();
    if (misses) *misses = cache->policy.misses();
    if (h2d_bytes) *h2d_bytes = cache->h2d_bytes;
    return MOE_OK;
}

int moe_cache_set_device_policy(moe_cache_t *cache, int enable) {
    if (!cache) return MOE_EINVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status();
    if (dev != cache->device) return MOE_EINVAL;
    if (!enable) {
        const int rc = cache_pull(cache);
        if (rc) return rc;
        cache->dev_policy = 0;
        return MOE_OK;
    }
    if (cache->dev_policy) return MOE_OK;
    // the host blobs must be readable by the device (page-locked and mapped)
    void *hd = nullptr;
    if (cudaHostGetDevicePointer(&hd, const_cast<uint8_t *>(cache->h_experts), 0) != cudaSuccess || !hd) {
        (void)cudaGetLastError();
        return MOE_EINVAL;
    }
    if (!aligned(hd, 16) || cache->host_stride % 16) return MOE_EINVAL;
    if (!cache->d_lfu && cudaMalloc((void **)&cache->d_lfu, sizeof(moe::DevLfu)) != cudaSuccess) return cuda_status();
    const moe::DevLfu d = dev_state_of(cache->policy, cache->h2d_bytes);
    if (cudaStreamSynchronize(cache->side) != cudaSuccess ||
        cudaMemcpy(cache->d_lfu, &d, sizeof(d), cudaMemcpyHostToDevice) != cudaSuccess)
        return cuda_status();
    cache->h_experts_dev = (const uint8_t *)hd;
    cache->dev_policy = 1;
    return MOE_OK;
}

int moe_layer_decode_noalloc(const moe_layer_t *layer, const float *x, int T, int flags, float *y,
                             int32_t *idx_out, float *gate_out, void *stream) {
    int rc = check_layer_call(layer, x, T, MOE_MAX_DECODE_TOKENS, flags, y);
    if (rc) return rc;
    if (ws_layout(*layer, T).decode_total > MOE_NOALLOC_SCRATCH_BYTES) {
        if (getenv("MOE_DEBUG"))
            fprintf(stderr, "libmoe: layer needs %zu bytes of scratch at T=%d, more than %u\n",
                    ws_layout(*layer, T).decode_total, T, MOE_NOALLOC_SCRATCH_BYTES);
        return MOE_EWORKSPACE;
    }
    void *ws = nullptr;
    if ((rc = noalloc_scratch(&ws))) return rc;
    return run_decode(layer, x, T, flags, y, idx_out, gate_out, ws, MOE_NOALLOC_SCRATCH_BYTES, stream);
}

int moe_noalloc_status(void *stream) {
    void *ws = nullptr;
    const int rc = noalloc_scratch(&ws);
    if (rc) return rc;
    return scratch_status(ws, MOE_NOALLOC_SCRATCH_BYTES, as_stream(stream));
}


int moe_host_call_create(moe_host_call_t **out, const moe_layer_t *layer, int T, int flags, void *d_ws,
                         size_t ws_bytes, void *stream) {
    if (!out) return MOE_EINVAL;
    *out = nullptr;
    if (!layer_ok(layer) || T < 1 || T > MOE_MAX_DECODE_TOKENS || !flags_ok(layer, flags)) return MOE_EINVAL;
    Ws w;
    int rc = bind_ws(layer, T, d_ws, ws_bytes, &w);
    if (rc) return rc;
    moe_host_call *c = new (std::nothrow) moe_host_call();
    if (!c) return MOE_EINVAL;
    c->layer = *layer;
    c->T = T;
    c->flags = flags;
    c->ws = d_ws;
    c->ws_bytes = ws_bytes;
    c->xb = sizeof(float) * (size_t)T * layer->H;
    c->st = as_stream(stream);
    void *xd = nullptr, *yd = nullptr, *fd = nullptr;
    if (cudaHostAlloc(&c->x_h, c->xb, cudaHostAllocMapped) != cudaSuccess ||
        cudaHostAlloc(&c->y_h, c->xb, cudaHostAllocMapped) != cudaSuccess ||
        cudaHostAlloc(&c->flag_h, 256, cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer(&xd, c->x_h, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&yd, c->y_h, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&fd, c->flag_h, 0) != cudaSuccess || cudaMalloc(&c->count_d, 256) != cudaSuccess ||
        cudaMemset(c->count_d, 0, 256) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking) != cudaSuccess) {
        rc = cuda_status();
        host_call_free(c);
        return rc ? rc : MOE_ECUDA;
    }
    memset(c->x_h, 0, c->xb);
    *(volatile unsigned *)c->flag_h = 0u;
    // the step, recorded once: x from its staging row into the workspace, the decode
    // kernel writing y into its staging row, the completion word
    if (cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        rc = cuda_status();
        host_call_free(c);
        return rc ? rc : MOE_ECUDA;
    }
    k_copy16<<<(unsigned)((c->xb / 16 + 255) / 256), 256, 0, c->cap>>>(reinterpret_cast<const uint4 *>(xd),
                                                                      reinterpret_cast<uint4 *>(w.xh), c->xb / 16);
    rc = cuda_status();
    if (!rc)
        rc = moe_layer_decode(layer, w.xh, T, flags, static_cast<float *>(yd), nullptr, nullptr, nullptr, d_ws,
                              ws_bytes, c->cap);
    if (!rc) {
        k_host_signal<<<1, 1, 0, c->cap>>>(c->count_d, static_cast<volatile unsigned *>(fd));
        rc = cuda_status();
    }
    const cudaError_t ec = cudaStreamEndCapture(c->cap, &c->graph);
    if (!rc && (ec != cudaSuccess || cudaGraphInstantiate(&c->exec, c->graph, 0) != cudaSuccess)) rc = MOE_ECUDA;
    if (rc) {
        (void)cudaGetLastError();
        host_call_free(c);
        return rc;
    }
    *out = c;
    return MOE_OK;
}

int moe_host_call_run(moe_host_call_t *c, const float *x_host, float *y_host) {
    if (!c || !x_host || !y_host) return MOE_EINVAL;
    if (x_host != c->x_h) memcpy(c->x_h, x_host, c->xb);
    if (cudaGraphLaunch(c->exec, c->st) != cudaSuccess) return cuda_status();
    const unsigned want = ++c->seq;
    volatile unsigned *flag = c->flag_h;
    // wait for the completion word: host memory, no driver call per test; the stream
    // is asked now and then so that a failed step ends the wait
    const auto t0 = std::chrono::steady_clock::now();
    for (unsigned spins = 1;; spins++) {
        if (*flag == want) break;
        if ((spins & 1023u) == 0) {
            const cudaError_t q = cudaStreamQuery(c->st);
            if (q != cudaSuccess && q != cudaErrorNotReady) return cuda_status();
            if (q == cudaSuccess && *flag != want) return MOE_ECUDA;  // the step ended without its signal
            if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(5)) return MOE_ETIMEOUT;
        }
    }
    std::atomic_thread_fence(std::memory_order_acquire);
    if (y_host != c->y_h) memcpy(y_host, c->y_h, c->xb);
    return MOE_OK;
}

int moe_host_call_rows(moe_host_call_t *c, float **x_row, float **y_row) {
    if (!c) return MOE_EINVAL;
    if (x_row) *x_row = c->x_h;
    if (y_row) *y_row = c->y_h;
    return MOE_OK;
}

int moe_host_call_destroy(moe_host_call_t *c) {
    if (!c) return MOE_OK;
    if (cudaStreamSynchronize(c->st) != cudaSuccess) (void)cudaGetLastError();
    host_call_free(c);
    return MOE_OK;
}

}  // extern "C"

bool moe::take_injection(int what) { return take_inject(what); }
