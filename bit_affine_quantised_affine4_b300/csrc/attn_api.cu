// attn_api.cu -- C ABI of the attention block (include/moe.h, moe_attn_*):
// argument checks, workspace layout and the three launches of attn.cuh.
#include <cuda_runtime.h>

#include <atomic>
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "attn.cuh"

using namespace moe;

namespace {


int attn_cuda_status() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (getenv("MOE_DEBUG")) fprintf(stderr, "libmoe: CUDA error %s\n", cudaGetErrorString(e));
        return MOE_ECUDA;
    }
    return MOE_OK;
}

bool al(const void *p, size_t n) { return ((uintptr_t)p % n) == 0; }

bool shape_ok(const moe_attn_t *a) {
    if (!a) return false;
    if (a->H < 64 || a->H % 64 || a->H > MOE_ATTN_MAX_HIDDEN) return false;
    if (a->nq < 1 || a->nkv < 1 || a->nq % a->nkv) return false;
    if (a->d != 64 && a->d != 128 && a->d != 256 && a->d != 512) return false;
    if ((long long)a->nq * a->d > MOE_ATTN_MAX_HIDDEN) return false;
    if (a->window < 0 || a->kv_len < 1 || a->kv_len > MOE_ATTN_MAX_KV) return false;
    if (!(a->theta > 0.f) || !std::isfinite(a->theta) || !std::isfinite(a->scale)) return false;
    if (!a->wqkv_q || !a->wqkv_s || !a->wqkv_b || !a->wo_q || !a->wo_s || !a->wo_b) return false;
    if (!al(a->wqkv_q, 16) || !al(a->wo_q, 16) || !al(a->wqkv_s, 16) || !al(a->wqkv_b, 16) || !al(a->wo_s, 16) ||
        !al(a->wo_b, 16))
        return false;
    if (!a->k_cache || !a->v_cache || !al(a->k_cache, 16) || !al(a->v_cache, 16)) return false;
    return true;
}

int group_of(const moe_attn_t *a) { return a->nq / a->nkv; }
// Rows of an attention tile: the smallest power of two that holds the call's
// T x G (token, query head) rows of one key/value head, at most kAttnRows.
int rows_of(const moe_attn_t *a, int T) {
    const int n = T * group_of(a);
    int rt = 1;
    while (rt < n && rt < kAttnRows) rt *= 2;
    return rt;
}
int tiles_of(const moe_attn_t *a, int T) { return (T * group_of(a) + rows_of(a, T) - 1) / rows_of(a, T); }

// The widest position range one tile can attend to in a call of T tokens.
long long range_max(const moe_attn_t *a, int T) {
    const int tpt = std::min(T, (rows_of(a, T) - 1) / group_of(a) + 2);  // tokens a tile can touch
    return a->window > 0 ? (long long)a->window + tpt - 1 : (long long)a->kv_len;
}

// Slices of a tile's positions: one shared-memory block of kAttnSlice positions
// each, at most kAttnMaxSlices (longer ranges give a slice several blocks).
int slices_for(long long range) {
    return (int)std::max(1LL, std::min((range + kAttnSlice - 1) / kAttnSlice, (long long)kAttnMaxSlices));
}
int slices_max(const moe_attn_t *a, int T) { return slices_for(range_max(a, T)); }

struct AttnWs {
    unsigned *err, *ticket;
    float *qr, *ao, *part_o;
    float2 *part_ml;
};

struct AttnLayout {
    size_t err, ticket, qr, ao, part_o, part_ml, total;
};

AttnLayout attn_layout(const moe_attn_t *a, int T) {
    AttnLayout L;
    const size_t nt = (size_t)a->nkv * tiles_of(a, T), S = slices_max(a, T), rt = rows_of(a, T);
    const size_t od = (size_t)T * a->nq * a->d;
    size_t max_tickets = 0;  // the ticket words sit at the front whatever the call's T
    for (int t = 1; t <= MOE_MAX_PREFILL_TOKENS; t++) max_tickets = std::max(max_tickets, (size_t)tiles_of(a, t));
    size_t off = 0;
    L.err = off;    off = up256(off + sizeof(unsigned));
    L.ticket = off; off = up256(off + sizeof(unsigned) * a->nkv * max_tickets);
    L.qr = off;     off = up256(off + sizeof(float) * od);
    L.ao = off;     off = up256(off + sizeof(float) * od);
    L.part_o = off; off = up256(off + sizeof(float) * nt * S * rt * a->d);
    L.part_ml = off; off = up256(off + sizeof(float2) * nt * S * rt);
    L.total = off;
    return L;
}

size_t ws_bytes_for(const moe_attn_t *a, int T) {
    size_t m = 0;
    for (int t = 1; t <= T; t++) m = std::max(m, attn_layout(a, t).total);
    return m;
}

// Dynamic shared memory above the default 48 KB is opted into once per kernel.
template <int MODE>
int proj_smem_optin() {
    static std::atomic<int> done{0};
    if (done.load()) return MOE_OK;
    const size_t most = proj_smem_bytes<MODE>(MOE_ATTN_MAX_HIDDEN, kProjTokens);
    if (cudaFuncSetAttribute(k_attn_proj<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most) !=
            cudaSuccess ||
        (MODE == kProjPlain &&
         cudaFuncSetAttribute(k_attn_proj<kProjPlain, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most) !=
             cudaSuccess))
        return attn_cuda_status();
    done.store(1);
    return MOE_OK;
}

// Every launch asks for programmatic dependent launch, so that a kernel can load
// what does not depend on its predecessor (weights, key/value rows into L2) while
// that one finishes; each kernel waits (griddepcontrol.wait) before it reads the
// predecessor's output.  If the runtime refuses the attribute, plain launches are
// used from then on.
// `cluster` > 1 launches thread block clusters of that many CTAs along x.
template <typename Args>
int launch_pdl(void (*fn)(Args), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Args &args,
               int cluster = 1) {
    static std::atomic<int> pdl_ok{1};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        n++;
    }
    if (pdl_ok.load()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = n + 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, args);
        if (e == cudaSuccess) return attn_cuda_status();
        if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return attn_cuda_status();
        (void)cudaGetLastError();
        pdl_ok.store(0);
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (cudaLaunchKernelEx(&cfg, fn, args) != cudaSuccess) return attn_cuda_status();
    return attn_cuda_status();
}

// RoPE frequencies theta^(-2i/d) for i < d/2, in fp64, kept for the last few
// (theta, d) pairs seen (a decoder has one or two).
void rope_freqs(float theta, int d, double *out) {
    struct Entry {
        float theta;
        int d;
        double f[256];
    };
    static Entry cache[4];
    static int used = 0, next = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int e = 0; e < used; e++)
        if (cache[e].theta == theta && cache[e].d == d) {
            memcpy(out, cache[e].f, sizeof(double) * (d / 2));
            return;
        }
    Entry &n = cache[next];
    next = (next + 1) % 4;
    used = std::min(used + 1, 4);
    n.theta = theta;
    n.d = d;
    for (int i = 0; i < d / 2; i++) n.f[i] = std::pow((double)theta, -(double)(2 * i) / (double)d);
    memcpy(out, n.f, sizeof(double) * (d / 2));
}

// The largest cluster of k_attn<D, RT> CTAs the device co-schedules: 16 (a
// non-portable size) when it can, else 8; found once per kernel.
template <int D, int RT>
int attn_max_cluster() {
    static std::atomic<int> cmax{0};
    int c = cmax.load();
    if (c) return c;
    if (cudaFuncSetAttribute(k_attn<D, RT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_smem_bytes(D, RT)) != cudaSuccess)
        return -attn_cuda_status();
    c = 8;
    if (cudaFuncSetAttribute(k_attn<D, RT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kAttnMaxCluster, 1, 1);
        cfg.blockDim = dim3(kAttnThreads);
        cfg.dynamicSmemBytes = attn_smem_bytes(D, RT);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = kAttnMaxCluster;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_attn<D, RT>, &cfg) == cudaSuccess && n > 0) c = kAttnMaxCluster;
    }
    (void)cudaGetLastError();
    cmax.store(c);
    return c;
}

// Slices of a call whose tiles attend to at most `range` positions.  When two
// shared-memory blocks per slice let one cluster (of up to cmax CTAs) cover a
// tile, that is the launch (*nst = 2, *cluster = the slices rounded up to a power
// of two): no partial leaves the cluster.  Otherwise one block per slice, at most
// kAttnMaxSlices, each CTA its own cluster (*nst = 1, *cluster = 1) and the
// partials merged through the workspace: larger clusters measured slower there
// (co-scheduling 16 CTAs per GPC left SMs idle).
int attn_slices(long long range, int cmax, int *cluster, int *nst) {
    const long long two = (range + 2 * kAttnSlice - 1) / (2 * kAttnSlice);
    if (two <= cmax) {
        int cs = 1;
        while (cs < two) cs *= 2;
        *cluster = cs;
        *nst = kAttnStages;
        return cs;
    }
    *cluster = 1;
    *nst = 1;
    return (int)std::min((range + kAttnSlice - 1) / kAttnSlice, (long long)kAttnMaxSlices);
}

template <int D, int RT>
int launch_attn_rt(AttnArgs args, long long range, int tiles, int nkv, int max_partials, cudaStream_t st) {
    const int cmax = attn_max_cluster<D, RT>();
    if (cmax < 0) return -cmax;
    int cs, nst;
    args.S = attn_slices(range, cmax, &cs, &nst);
    args.nst = nst;
    // a chunk's call range can exceed one tile's: fewer, longer slices then
    if (cs == 1) args.S = std::min(args.S, max_partials);
    if (args.S / cs > max_partials) return MOE_EWORKSPACE;  // cannot happen with moe_attn_workspace_bytes
    return launch_pdl(k_attn<D, RT>, dim3(args.S, tiles, nkv), dim3(kAttnThreads), attn_smem_bytes(D, RT, nst), st,
                      args, cs);
}

template <int D>
int launch_attn(const AttnArgs &args, long long range, int rt, int tiles, int nkv, int max_partials,
                cudaStream_t st) {
    switch (rt) {
        case 1: return launch_attn_rt<D, 1>(args, range, tiles, nkv, max_partials, st);
        case 2: return launch_attn_rt<D, 2>(args, range, tiles, nkv, max_partials, st);
        case 4: return launch_attn_rt<D, 4>(args, range, tiles, nkv, max_partials, st);
        default: return launch_attn_rt<D, 8>(args, range, tiles, nkv, max_partials, st);
    }
}

__device__ unsigned g_qgemv_err;  // bounded-wait report word of the standalone GEMV

}  // namespace

int moe::qgemv_rows16(const uint32_t *q, const __half *s, const __half *b, int N, int K, const float *x, float *y,
                      cudaStream_t st) {
    static unsigned *err = nullptr;
    int rc;
    if (!err && cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_qgemv_err) != cudaSuccess)
        return attn_cuda_status();
    if ((rc = proj_smem_optin<kProjPlain>())) return rc;
    ProjArgs o{};
    o.q = q;
    o.s = s;
    o.b = b;
    o.N = N;
    o.K = K;
    o.x = x;
    o.T = 1;
    o.y = y;
    o.err = err;
    // more tiles than two waves of 2 CTAs per SM: the build that fits 4 per SM
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return attn_cuda_status();
    }
    if (N / 16 > 2 * sms)
        return launch_pdl(k_attn_proj<kProjPlain, 4>, dim3(N / 16, 1), dim3(proj_threads<kProjPlain>()),
                          proj_smem_bytes<kProjPlain>(K, 1), st, o);
    return launch_pdl(k_attn_proj<kProjPlain>, dim3(N / 16, 1), dim3(proj_threads<kProjPlain>()),
                      proj_smem_bytes<kProjPlain>(K, 1), st, o);
}

extern "C" {

size_t moe_attn_workspace_bytes(const moe_attn_t *attn, int T) {
    if (!shape_ok(attn) || T < 1 || T > MOE_MAX_PREFILL_TOKENS) return 0;
    return ws_bytes_for(attn, T);
}

int moe_attn_step(const moe_attn_t *attn, const float *x, int T, int pos, int flags, float *y, float *attn_out,
                  void *d_ws, size_t ws_bytes, void *stream) {
    const moe_attn_t *a = attn;
    if (!shape_ok(a) || !x || !y || !al(x, 16) || !al(y, 16) || (attn_out && !al(attn_out, 16))) return MOE_EINVAL;
    if (T < 1 || T > MOE_MAX_PREFILL_TOKENS || pos < 0 || pos > INT_MAX - 2 * MOE_MAX_PREFILL_TOKENS)
        return MOE_EINVAL;
    if (flags & ~(MOE_RESIDUAL | MOE_PRENORM)) return MOE_EINVAL;
    const bool prenorm = flags & MOE_PRENORM;
    if (prenorm && (!a->norm_w || !al(a->norm_w, 16) || !(a->norm_eps >= 0.f))) return MOE_EINVAL;
    if (a->window > 0 ? (long long)a->kv_len < (long long)a->window + T - 1 : (long long)pos + T > a->kv_len)
        return MOE_ECAPACITY;
    if (!d_ws || !al(d_ws, 256) || ws_bytes < ws_bytes_for(a, T)) return MOE_EWORKSPACE;

    const AttnLayout L = attn_layout(a, T);
    uint8_t *base = static_cast<uint8_t *>(d_ws);
    AttnWs w;
    w.err = reinterpret_cast<unsigned *>(base + L.err);
    w.ticket = reinterpret_cast<unsigned *>(base + L.ticket);
    w.qr = reinterpret_cast<float *>(base + L.qr);
    w.ao = reinterpret_cast<float *>(base + L.ao);
    w.part_o = reinterpret_cast<float *>(base + L.part_o);
    w.part_ml = reinterpret_cast<float2 *>(base + L.part_ml);
    cudaStream_t st = (cudaStream_t)stream;
    int rc;
    if ((rc = proj_smem_optin<kProjQKV>()) || (rc = proj_smem_optin<kProjPlain>())) return rc;
    const int tok_groups = (T + kProjTokens - 1) / kProjTokens;

    // 1. [q; k; v] = Wqkv xn, RoPE, the cache store
    ProjArgs p{};
    p.q = a->wqkv_q;
    p.s = reinterpret_cast<const __half *>(a->wqkv_s);
    p.b = reinterpret_cast<const __half *>(a->wqkv_b);
    p.N = (a->nq + 2 * a->nkv) * a->d;
    p.K = a->H;
    p.x = x;
    p.T = T;
    p.norm_w = prenorm ? a->norm_w : nullptr;
    p.norm_eps = a->norm_eps;
    p.nq = a->nq; p.nkv = a->nkv; p.d = a->d; p.window = a->window; p.kv_len = a->kv_len; p.p0 = pos;
    rope_freqs(a->theta, a->d, p.freq);
    p.scale = a->scale;
    p.qr = w.qr;
    p.err = w.err;
    p.kc = reinterpret_cast<__half *>(a->k_cache);
    p.vc = reinterpret_cast<__half *>(a->v_cache);
    if ((rc = launch_pdl(k_attn_proj<kProjQKV>, dim3(p.N / 16, tok_groups), dim3(proj_threads<kProjQKV>()),
                         proj_smem_bytes<kProjQKV>(a->H, T), st, p)))
        return rc;

    // 2. attention over the slices of each tile's positions, merged in-kernel
    const int G = group_of(a), tiles = tiles_of(a, T);
    const long long lo = a->window > 0 ? std::max(0, pos - a->window + 1) : 0;
    const long long range = (long long)pos + T - lo;
    AttnArgs g{};
    g.qr = w.qr;
    g.kc = reinterpret_cast<const __half *>(a->k_cache);
    g.vc = reinterpret_cast<const __half *>(a->v_cache);
    g.nq = a->nq; g.nkv = a->nkv; g.G = G; g.kv_len = a->kv_len; g.window = a->window; g.p0 = pos; g.T = T;
    g.S = 0;  // set with the cluster size at the launch
    g.part_o = w.part_o;
    g.part_ml = w.part_ml;
    g.ticket = w.ticket;
    g.err = w.err;
    g.wait_ns = kWaitNs;
    if (take_injection(MOE_INJECT_ATTN_WAIT)) {  // the blocks' barriers wait for 16 bytes that never come
        g.extra_tx = 16;
        g.wait_ns = 2ull * 1000 * 1000;
    }
    g.ao = w.ao;
    g.ao_user = attn_out;
    const int rt = rows_of(a, T);
    const int mp = slices_max(a, T);
    switch (a->d) {
        case 64: rc = launch_attn<64>(g, range, rt, tiles, a->nkv, mp, st); break;
        case 128: rc = launch_attn<128>(g, range, rt, tiles, a->nkv, mp, st); break;
        case 256: rc = launch_attn<256>(g, range, rt, tiles, a->nkv, mp, st); break;
        default: rc = launch_attn<512>(g, range, rt, tiles, a->nkv, mp, st); break;
    }
    if (rc) return rc;

    // 3. y = Wo o (+ x)
    ProjArgs o{};
    o.q = a->wo_q;
    o.s = reinterpret_cast<const __half *>(a->wo_s);
    o.b = reinterpret_cast<const __half *>(a->wo_b);
    o.N = a->H;
    o.K = a->nq * a->d;
    o.x = w.ao;
    o.T = T;
    o.y = y;
    o.resid = (flags & MOE_RESIDUAL) ? x : nullptr;
    o.err = w.err;
    return launch_pdl(k_attn_proj<kProjPlain>, dim3(a->H / 16, tok_groups), dim3(proj_threads<kProjPlain>()),
                      proj_smem_bytes<kProjPlain>(o.K, T), st, o);
}

int moe_attn_workspace_status(void *d_ws, size_t ws_bytes, void *stream) {
    if (!d_ws || !al(d_ws, 256) || ws_bytes < 256) return MOE_EWORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    unsigned err = 0;
    if (cudaMemcpyAsync(&err, d_ws, sizeof(err), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return attn_cuda_status();
    if (err && (cudaMemsetAsync(d_ws, 0, sizeof(err), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess))
        return attn_cuda_status();
    return err ? MOE_ETIMEOUT : MOE_OK;
}

}  // extern "C"
