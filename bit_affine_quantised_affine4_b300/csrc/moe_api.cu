// moe_api.cu -- the C ABI of libmoe (include/moe.h): argument checks, workspace
// layout and kernel launches.  All arithmetic runs in the kernels included below.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "route.cuh"
#include "simple_kernels.cuh"
#include "decode.cuh"
#include "gemv.cuh"

using namespace moe;

namespace {

cudaStream_t as_stream(void *s) { return (cudaStream_t)s; }

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
           l->expert_stride >= blob_layout(l->H, l->I).total;
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
// fits in ws_bytes (it is what the caller sized it for, or larger).
WsLayout ws_fit(const moe_layer_t *l, size_t ws_bytes) {
    WsLayout best = ws_layout(*l, 1);
    for (int t = 2; t <= MOE_MAX_PREFILL_TOKENS; t++) {
        WsLayout w = ws_layout(*l, t);
        if (w.total > ws_bytes) break;
        best = w;
    }
    return best;
}

// Binds the caller's workspace: the layout is the one for the largest T_max whose
// size fits ws_bytes (what moe_workspace_bytes was asked for, or more).
int bind_ws(const moe_layer_t *l, int T, void *d_ws, size_t ws_bytes, Ws *out) {
    if (!d_ws || !aligned(d_ws, 256)) return MOE_EWORKSPACE;
    WsLayout W = ws_fit(l, ws_bytes);
    if (W.total > ws_bytes || W.Tmax < T) return MOE_EWORKSPACE;
    *out = ws_bind(d_ws, W, *l);
    return MOE_OK;
}

int launch_route(const moe_layer_t *l, const LayerDev &ly, const float *x, int T, Ws ws,
                 int32_t *idx, float *gate, float *logits, cudaStream_t st) {
    const int grid = (l->E + kRouteWarps - 1) / kRouteWarps;
    if (T == 1)
        k_route<1><<<grid, kRouteWarps * 32, 0, st>>>(ly, x, T, ws, idx, gate, logits);
    else
        k_route<4><<<grid, kRouteWarps * 32, 0, st>>>(ly, x, T, ws, idx, gate, logits);
    return cuda_status();
}

int check_layer_call(const moe_layer_t *l, const float *x, int T, int Tlimit, int flags,
                     const float *y) {
    if (!layer_ok(l) || !experts_ok(l) || !x || !y || T < 1 || T > Tlimit) return MOE_EINVAL;
    if (flags & ~MOE_RESIDUAL) return MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(y, 16) || x == y) return MOE_EINVAL;
    return MOE_OK;
}

// Prefill chunk (and any T beyond the decode kernel): router + gather + expert
// kernels launched in sequence.
int run_layer_chunk(const moe_layer_t *l, const float *x, int T, int flags, float *y,
                    int32_t *idx_out, float *gate_out, void *d_ws, size_t ws_bytes, void *stream) {
    Ws ws;
    int rc = bind_ws(l, T, d_ws, ws_bytes, &ws);
    if (rc) return rc;
    LayerDev ly = layer_dev(l);
    cudaStream_t st = as_stream(stream);
    rc = launch_route(l, ly, x, T, ws, idx_out, gate_out, nullptr, st);
    if (rc) return rc;
    const int up_items = ws.Umax * (l->I / 16) + l->Is / 16;
    k_expert_up_simple<<<up_items, 128, 0, st>>>(ly, x, T, ws);
    if ((rc = cuda_status())) return rc;
    const int down_items = (ws.Umax + 1) * (l->H / 16);
    k_expert_down_simple<<<down_items, 128, 0, st>>>(ly, x, T, flags, y, ws);
    return cuda_status();
}

struct DecodeLaunch {
    int device = -1;
    int sms = 0;
    int occ[2] = {0, 0};
    size_t smem[2] = {0, 0};
};

// Grid of the persistent decode kernel: every SM times the CTAs that fit.
int decode_grid(const moe_layer_t *l, int nch, size_t smem, int *grid) {
    static thread_local DecodeLaunch cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status();
    if (cache.device != dev) {
        cache = DecodeLaunch();
        cache.device = dev;
        if (cudaDeviceGetAttribute(&cache.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cuda_status();
    }
    int k = nch - 1;
    if (cache.smem[k] != smem || cache.occ[k] == 0) {
        int occ = 0;
        auto fn = nch == 1 ? k_decode<1> : k_decode<2>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return cuda_status();
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kDecThreads, smem) != cudaSuccess)
            return cuda_status();
        if (occ < 1) return MOE_EINVAL;
        cache.occ[k] = occ;
        cache.smem[k] = smem;
    }
    (void)l;
    *grid = cache.sms * cache.occ[k];
    return MOE_OK;
}

int run_decode(const moe_layer_t *l, const float *x, int T, int flags, float *y, int32_t *idx_out,
               float *gate_out, void *d_ws, size_t ws_bytes, void *stream) {
    Ws ws;
    int rc = bind_ws(l, T, d_ws, ws_bytes, &ws);
    if (rc) return rc;
    DecodeArgs a;
    a.ly = layer_dev(l);
    a.x = x;
    a.T = T;
    a.flags = flags;
    a.y = y;
    a.idx_out = idx_out;
    a.gate_out = gate_out;
    a.ws = ws;
    a.R = (l->E + kRouterRows - 1) / kRouterRows;
    const int nch = T > 8 ? 2 : 1;
    const size_t smem = decode_smem_bytes(*l, nch);
    int grid = 0;
    if ((rc = decode_grid(l, nch, smem, &grid))) return rc;
    cudaStream_t st = as_stream(stream);
    if (nch == 1)
        k_decode<1><<<grid, kDecThreads, smem, st>>>(a);
    else
        k_decode<2><<<grid, kDecThreads, smem, st>>>(a);
    return cuda_status();
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
    cudaStream_t st = as_stream(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_status();
    unsigned err = 0;
    if (cudaMemcpy(&err, d_ws, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_status();
    if (err) {
        cudaMemset(d_ws, 0, ws_bytes);
        cudaDeviceSynchronize();
        return MOE_ETIMEOUT;
    }
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

int qgemv_affine4(const uint32_t *q, const uint16_t *s, const uint16_t *b, int N, int K,
                  const float *x, float *y, void *stream) {
    if (!q || !s || !b || !x || !y || N < 1 || K < kGroup || K % kGroup) return MOE_EINVAL;
    if (!aligned(q, 16) || !aligned(x, 16)) return MOE_EINVAL;
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
    if (cache) return MOE_ENOTREADY;
    int rc = check_layer_call(layer, x, T, MOE_MAX_DECODE_TOKENS, flags, y);
    if (rc) return rc;
    return run_decode(layer, x, T, flags, y, idx_out, gate_out, d_ws, ws_bytes, stream);
}

int moe_layer_prefill_chunk(const moe_layer_t *layer, const float *x, int T, int flags, float *y,
                            int32_t *idx_out, float *gate_out, void *d_ws, size_t ws_bytes,
                            void *stream) {
    int rc = check_layer_call(layer, x, T, MOE_MAX_PREFILL_TOKENS, flags, y);
    if (rc) return rc;
    return run_layer_chunk(layer, x, T, flags, y, idx_out, gate_out, d_ws, ws_bytes, stream);
}

int moe_cache_create(moe_cache_t **out, int H, int E, int I, const void *h_experts,
                     size_t host_stride, int slots) {
    (void)H; (void)E; (void)I; (void)h_experts; (void)host_stride; (void)slots;
    if (out) *out = nullptr;
    return MOE_ENOTREADY;
}
int moe_cache_destroy(moe_cache_t *cache) { return cache ? MOE_ENOTREADY : MOE_OK; }
int moe_cache_slots(const moe_cache_t *, int32_t *, uint32_t *) { return MOE_ENOTREADY; }
int moe_cache_stats(const moe_cache_t *, uint64_t *, uint64_t *, uint64_t *) { return MOE_ENOTREADY; }

int moe_layer_decode_noalloc(const moe_layer_t *layer, const float *x, int T, int flags, float *y,
                             int32_t *idx_out, float *gate_out, void *stream) {
    int rc = check_layer_call(layer, x, T, MOE_MAX_DECODE_TOKENS, flags, y);
    if (rc) return rc;
    if (ws_layout(*layer, T).total > MOE_NOALLOC_SCRATCH_BYTES) {
        if (getenv("MOE_DEBUG"))
            fprintf(stderr, "libmoe: layer needs %zu bytes of scratch at T=%d, more than %u\n",
                    ws_layout(*layer, T).total, T, MOE_NOALLOC_SCRATCH_BYTES);
        return MOE_EWORKSPACE;
    }
    void *ws = nullptr;
    if ((rc = noalloc_scratch(&ws))) return rc;
    return run_decode(layer, x, T, flags, y, idx_out, gate_out, ws, MOE_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
