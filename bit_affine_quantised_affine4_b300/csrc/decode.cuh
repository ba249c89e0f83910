// decode.cuh -- the whole MoE layer for 1..16 decode tokens in one persistent,
// cooperative kernel (one CTA per SM).
//
// The layer (devtrends page, section "Qual e il trucco principale dell'architettura";
// remio.ai page, sections "Mac Gemma 4 26B entra nello spazio disponibile..." and
// "L'affermazione dei 2 GB..."): an 8-bit router picks the top-8 experts per
// token, the routed experts and an always-on shared expert run GeGLU FFNs on
// 4-bit affine weights, and the outputs are combined with the softmax gates.
//
// Each CTA has 15 compute warps and one producer warp.  Weights arrive through a
// ring of shared-memory stages filled by bulk copies (TMA) and guarded by
// mbarriers.
//
//   phase A  producer: copies this CTA's first shared-expert gate/up tiles,
//            prefetches a slice of the shared down matrix into L2, then (after the
//            previous kernel: programmatic dependent launch) publishes the CTA's
//            router logits and waits until all E rows are published.  compute
//            warps: this CTA's router rows (CUDA cores, 8-bit; each row split over
//            the warps), then the token vectors' MMA fragments.
//   routing  every CTA ranks the logits itself, one warp per token (identical
//            results everywhere), and builds the schedule: distinct experts U in
//            ascending id, the tokens using each, and a compact slot per (token,
//            choice).  Nothing else competes for the SM meanwhile.
//   phase B  gate/up: the CTA's tiles j = b, b+nC, ... of [shared | routed u=0..U-1]
//            (one tile = 8 gate rows + the 8 matching up rows, full K); the shared
//            ones are already in the ring while the routed ones are copied.  The
//            warps split K and leave their partial sums in shared memory; a tile
//            is reduced (GeGLU, h written in fp16, compact slots for routed
//            experts) by the first warp that finds it complete after its next
//            tile, the CTA's last tile by its last arriver.
//            down: units (matrix, 16 output rows) in matrix-major order, a
//            contiguous range per CTA, one unit per warp with full K; h of the
//            CTA's matrices is copied to shared memory once every CTA's gate/up
//            tiles are done.  Each unit writes fp32 partial rows and counts itself
//            into its 16-row tile's ticket.
//   combine  CTA b owns the 16-row tiles b, b + nC, ...; once a tile's ticket
//            shows every contribution, the owner sums the partials in a fixed
//            order: y = sum_k gate_k * routed_k + sum_parts shared (+ x).
// All cross-CTA waits are bounded (sync.cuh); results do not depend on timing.
#pragma once

#include "common.cuh"
#include "mma_core.cuh"
#include "route.cuh"
#include "sync.cuh"
#include "tile.cuh"

namespace moe {

// 15 compute warps + the producer warp: 16 warps, 4 per SM sub-partition, so a
// thread may hold up to 128 registers
constexpr int kCW = 15;                       // compute warps
constexpr int kCThreads = kCW * 32;           // compute threads
constexpr int kDecThreads = kCThreads + 32;   // + producer warp
constexpr int kMaxStages = 4;
constexpr int kMaxUnitsPerCta = 512;
constexpr int kMaxPairs = MOE_MAX_DECODE_TOKENS * MOE_MAX_TOPK;
constexpr int kMaxRouterRows = 4;  // router rows per CTA (E <= 4 x grid size)

// What one launch does: the shared expert, the routed experts, or both; and
// whether the routing comes from an earlier router launch (idx_pre/gate_pre)
// instead of the kernel's own router.  A launch with the routed experts also
// combines the output tiles (reading the shared partials an earlier launch may
// have written).
constexpr int kModeShared = 1, kModeRouted = 2, kModePre = 4;

struct DecodeArgs {
    // layer
    int H, E, topk, I, Is;
    const uint32_t *rq;
    const __half *rs, *rb;
    const float *bias;
    const uint8_t *experts;
    size_t stride;
    const uint8_t *shared;
    TileLayout Lr, Ls;  // routed and shared expert tile layouts
    int P;              // shared down matrix split in P parts of <= Lr.Gi groups
    // call
    const float *x;
    int T, flags;
    float *y;
    int32_t *idx_out;
    float *gate_out;
    // workspace
    unsigned *ctrl, *ticket;
    float *logits;
    __half *h16;   // routed h: per distinct expert u a block [Gi][n_u][64] at slot base * I
    __half *hs16;  // shared h: [Gs][T][64]
    float *pr;     // routed partials [T*topk][H]
    float *ps;     // shared partials [P][T][H]
    // launch
    int stages, SB, UPS, red_off, hsm_off, hsm_mat_bytes, hsum_off;
    int mode;
    const int *idx_pre;      // [T][topk] routing of an earlier router launch (kModePre)
    const float *gate_pre;   // [T][topk]
    int use_map;             // expert e's blob is experts + slot_map[e] * stride (cache slots)
    short slot_map[MOE_MAX_EXPERTS];
    const short *slot_dev;   // or, when non-null, the slot of expert e in device memory
    // fault injection (tests of the error path): extra router rows the routing
    // wait expects (0 normally; > 0 makes it unreachable) and that wait's limit
    unsigned route_extra;
    unsigned long long route_wait_ns;
    // RMSNorm in front of the layer (flags & MOE_PRENORM): the router and the
    // experts read x * norm_w / rms(x); 1 / rms is applied to their sums
    const float *norm_w;
    float norm_eps;
};

// x / d for x < 2^24 and 1 <= d <= 256: magic = 0xFFFFFFFF / d + 1 (d > 1), exact
// in that range; d == 1 is passed through.
__device__ __forceinline__ int udiv_small(int x, int d, unsigned magic) {
    return d == 1 ? x : (int)__umulhi((unsigned)x, magic);
}
__device__ __forceinline__ unsigned udiv_magic(int d) { return d > 1 ? 0xFFFFFFFFu / (unsigned)d + 1u : 0u; }

// fp16 pair (lo, hi) of a 32-bit word -> floats
__device__ __forceinline__ float lo_half(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float hi_half(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// acc += s*2^24*D + b*S with S given per token column (2c, 2c+1).
__device__ __forceinline__ void affine_acc(float (&acc)[4], const float (&d)[4], float S0, float S1,
                                           float sa, float ba, float sb, float bb) {
    acc[0] = fmaf(sa, d[0], fmaf(ba, S0, acc[0]));
    acc[1] = fmaf(sa, d[1], fmaf(ba, S1, acc[1]));
    acc[2] = fmaf(sb, d[2], fmaf(bb, S0, acc[2]));
    acc[3] = fmaf(sb, d[3], fmaf(bb, S1, acc[3]));
}

// Position of column k of a group (fragment order) in a 128-byte h row of slot j:
// the row's 16-byte chunks are swapped pairwise for odd slots, which makes the
// B-fragment loads of 8 consecutive lanes hit 8 distinct bank groups.
__host__ __device__ __forceinline__ int h_pos(int k, int j) { return frag_pos(k) ^ ((j & 1) << 3); }

struct DecodeSmem {
    uint64_t full[kMaxStages], empty[kMaxStages], hbar;
    int idx[kMaxPairs];
    float gate[kMaxPairs];
    int pidx[kMaxPairs];
    unsigned mask[MOE_MAX_EXPERTS];
    short uid[MOE_MAX_EXPERTS];
    int uexp[kMaxPairs], ubase[kMaxPairs], ucnt[kMaxPairs], uslot[kMaxPairs];
    float rpart[kMaxRouterRows][kCW > MOE_MAX_DECODE_TOKENS ? kCW : MOE_MAX_DECODE_TOKENS];
    unsigned wsum[MOE_MAX_EXPERTS / 32];  // schedule: experts << 16 | slots of 32 experts
    unsigned tcnt[kMaxStages + 2];         // gate/up partial-sum slots: warps arrived (+1: claimed)
    float xss[kCW][MOE_MAX_DECODE_TOKENS];  // RMSNorm: partial sums of squares of x per warp
    float inv_r[MOE_MAX_DECODE_TOKENS];     // RMSNorm: 1 / rms(x_t)
    int U;
    int err;
};

template <int NCH, int GPW>
__global__ void __launch_bounds__(kDecThreads, 1) k_decode(const DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ DecodeSmem S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gl = lane >> 2, c = lane & 3;
    const int b = blockIdx.x, nC = gridDim.x;
    const bool producer = warp == kCW;
    const int T = a.T, H = a.H;
    const int Ti = a.Lr.Ti, G = a.Lr.G, Gi = a.Lr.Gi, Gs = a.Ls.Gi, R = a.Lr.R;
    const bool do_shared = a.mode & kModeShared, do_routed = a.mode & kModeRouted, pre = a.mode & kModePre;
    const int Ts = do_shared ? a.Ls.Ti : 0;  // shared gate/up tiles of this launch
    const int Pe = do_shared ? a.P : 0;      // shared down parts of this launch
    uint8_t *ring = dsm;
    float *red = reinterpret_cast<float *>(dsm + a.red_off);
    uint8_t *hsm = dsm + a.hsm_off;
    volatile int *err = &S.err;

    // the next decode kernel on the stream may start on SMs this one leaves; it
    // waits for this one (pdl_wait) before it touches the workspace or x
    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < a.stages; s++) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], kCW);
        }
        mbar_init(&S.hbar, 1);
        for (int i = 0; i < kMaxStages + 2; i++) S.tcnt[i] = 0u;
        S.err = 0;
        mbar_fence_init();
    }
    __syncthreads();

    // ---- ring bookkeeping (the producer and the consumers count fills alike)
    int fill = 0;
    int last_fill[kMaxStages] = {-1, -1, -1, -1};
    auto producer_slot = [&](int k) -> int {  // lane 0 of the producer
        const int s = k % a.stages;
        if (k >= a.stages && !*err) {
            if (!mbar_wait(&S.empty[s], ((k / a.stages) - 1) & 1, err)) {
                *err = 1;
                atomicExch(&a.ctrl[kErr], 1u);
            }
        }
        return s;
    };
    auto consumer_wait = [&](int k) -> int {
        const int s = k % a.stages;
        // a non-blocking test first: the stage has usually landed already
        unsigned done;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(smem_addr(&S.full[s])), "r"((unsigned)((k / a.stages) & 1))
                     : "memory");
        if (!done && !*err && !mbar_wait(&S.full[s], (k / a.stages) & 1, err)) {
            *err = 1;
            atomicExch(&a.ctrl[kErr], 1u);
        }
        return s;
    };
    auto consumer_release = [&](int s) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[s]);
    };

    // gate/up tile t of the global list: shared tiles first, then routed (u, it).
    auto gu_src = [&](int j) -> const uint8_t * {
        if (j < Ts) return a.shared + (size_t)kTileBytes * G * j;
        const int u = (j - Ts) / Ti, it = (j - Ts) % Ti;
        return a.experts + (size_t)S.uslot[u] * a.stride + (size_t)kTileBytes * G * it;
    };
    const unsigned gu_bytes = (unsigned)(kTileBytes * G);
    const int n_shared_mine = b < Ts ? (Ts - 1 - b) / nC + 1 : 0;

    // ---- compute warps: x fragments for this warp's K slice, and their group sums
    // (of x * norm_w with MOE_PRENORM)
    const bool prenorm = a.flags & MOE_PRENORM;
    const int g0w = warp * G / kCW, g1w = (warp + 1) * G / kCW;
    uint32_t xb[GPW][NCH][8];
    float xs[GPW][NCH][2];
    auto load_x = [&]() {
#pragma unroll
        for (int gi = 0; gi < GPW; gi++)
#pragma unroll
            for (int ch = 0; ch < NCH; ch++) {
                const int g = g0w + gi, t = 8 * ch + gl;
                if (g < g1w && t < T)
                    load_b_f32(xb[gi][ch], a.x + (size_t)t * H + g * kGroup + 16 * c,
                               prenorm ? a.norm_w + g * kGroup + 16 * c : nullptr);
                else
                    zero_b(xb[gi][ch]);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_group_sums(d, xb[gi][ch]);
                xs[gi][ch][0] = d[0];
                xs[gi][ch][1] = d[1];
            }
    };

    // One gate/up tile by the compute warps: each warp takes its K slice and puts
    // its partial sums in one of stages + 2 slots of shared memory and counts
    // itself in (a counter per slot).  A tile is reduced (the 15 partials added up
    // in warp order, GeGLU, h stored in fp16) by the first warp that, having
    // written its partial of the next tile, finds all 15 partials of this one in
    // and claims it -- usually a fast warp, so no warp is both the slowest and the
    // one that reduces.  The CTA's last tile is reduced by its last arriver.  A slot
    // is reused only after the warp that reduced its previous tile has released a
    // later ring stage.  u < 0 marks the shared expert, it is the tile's row block.
    int slot = 0;
    const int nslot = a.stages + 2;
    auto reduce_tile = [&](int sl, int u, int it) {
        const float *rw = red + (size_t)sl * kCW * NCH * 128;
        __threadfence_block();
        // lane L holds rows (L / 4, L / 4 + 8) = (gate, up) of row block it, token
        // columns 2(L % 4), 2(L % 4) + 1 of each chunk
        const int row = 8 * it + gl, g = row / kGroup, k = row % kGroup;
#pragma unroll
        for (int ch = 0; ch < NCH; ch++) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 5
            for (int w = 0; w < kCW; w++) {
                const float4 p = reinterpret_cast<const float4 *>(rw + (size_t)(w * NCH + ch) * 128)[lane];
                v.x += p.x;
                v.y += p.y;
                v.z += p.z;
                v.w += p.w;
            }
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const int t = 8 * ch + 2 * c + i;
                if (t >= T || *err) continue;
                const float f = prenorm ? S.inv_r[t] : 1.f;
                const __half hv = __float2half_rn(gelu_tanh(f * (i ? v.y : v.x)) * (f * (i ? v.w : v.z)));
                if (u < 0) {
                    a.hs16[((size_t)g * T + t) * kGroup + h_pos(k, t)] = hv;
                } else {
                    const unsigned m = S.mask[S.uexp[u]];
                    if ((m >> t) & 1u) {
                        const int sl2 = __popc(m & ((1u << t) - 1u)), nu = S.ucnt[u];
                        a.h16[(size_t)S.ubase[u] * a.I + ((size_t)g * nu + sl2) * kGroup + h_pos(k, sl2)] = hv;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) S.tcnt[sl] = 0u;
    };
    int p_slot = -1, p_u = 0, p_it = 0;  // the previous tile (a reduction candidate)
    auto gateup_tile = [&](int s, int u, int it, bool final_tile) {
        float acc[NCH][4];
#pragma unroll
        for (int ch = 0; ch < NCH; ch++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[ch][i] = 0.f;
        if (!*err) {
            const uint8_t *st = ring + (size_t)s * a.SB;
#pragma unroll
            for (int gi = 0; gi < GPW; gi++) {
                const int g = g0w + gi;
                if (g < g1w) {
                    const uint4 q = *reinterpret_cast<const uint4 *>(st + g * kTileBytes + 16 * lane);
                    const uint2 e = *reinterpret_cast<const uint2 *>(st + g * kTileBytes + 512 + 8 * gl);
                    const float sa = lo_half(e.x) * kTwo24, ba = hi_half(e.x);
                    const float sb = lo_half(e.y) * kTwo24, bb = hi_half(e.y);
#pragma unroll
                    for (int ch = 0; ch < NCH; ch++) {
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_group_codes(d, make_uint2(q.x, q.y), make_uint2(q.z, q.w), xb[gi][ch]);
                        affine_acc(acc[ch], d, xs[gi][ch][0], xs[gi][ch][1], sa, ba, sb, bb);
                    }
                }
            }
        }
        consumer_release(s);
        float *rw = red + (size_t)slot * kCW * NCH * 128;
#pragma unroll
        for (int ch = 0; ch < NCH; ch++)
            reinterpret_cast<float4 *>(rw + (size_t)(warp * NCH + ch) * 128)[lane] =
                make_float4(acc[ch][0], acc[ch][1], acc[ch][2], acc[ch][3]);
        __syncwarp();
        unsigned claim = 0;  // bit 0: reduce the previous tile; bit 1: reduce this one
        if (lane == 0) {
            __threadfence_block();
            // both atomics issued before either result is used
            const unsigned n = atomicAdd(&S.tcnt[slot], 1u) + 1u;
            const unsigned pc = p_slot >= 0 ? atomicCAS(&S.tcnt[p_slot], (unsigned)kCW, (unsigned)kCW + 1u) : 0u;
            if (final_tile && n == (unsigned)kCW) claim |= 2u;
            if (p_slot >= 0 && pc == (unsigned)kCW) claim |= 1u;
        }
        claim = __shfl_sync(0xffffffffu, claim, 0);
        if (claim & 1u) reduce_tile(p_slot, p_u, p_it);
        if (claim & 2u) reduce_tile(slot, u, it);
        p_slot = slot;
        p_u = u;
        p_it = it;
        if (++slot == nslot) slot = 0;
    };
    // ---- routing helpers (one warp): rank token t from the logits staged in
    // shared memory; build the schedule from S.idx
    auto rank_token = [&](int t) {
        const float *lg = reinterpret_cast<const float *>(hsm);
        warp_topk_softmax<true>(lg + (size_t)t * a.E, a.E, a.topk, S.idx + t * a.topk, S.gate + t * a.topk,
                                b == 0 ? a.idx_out + (a.idx_out ? t * a.topk : 0) : nullptr,
                                b == 0 ? a.gate_out + (a.gate_out ? t * a.topk : 0) : nullptr);
    };
    // The schedule, by every thread of the CTA (called between barriers): the
    // distinct experts U in ascending id, the tokens using each (mask), a compact
    // slot per (token, choice).
    const unsigned topk_magic = udiv_magic(a.topk);
    auto build_schedule = [&]() {
        const int P2 = T * a.topk;
        for (int e = tid; e < a.E; e += kDecThreads) S.mask[e] = 0u;
        __syncthreads();
        if (!*err)
            for (int p = tid; p < P2; p += kDecThreads)
                atomicOr(&S.mask[S.idx[p]], 1u << udiv_small(p, a.topk, topk_magic));
        __syncthreads();
        // warp w < nw scans experts 32w..32w+31
        const int nw = (a.E + 31) >> 5;
        unsigned m = 0u, bal = 0u;
        int cnt = 0, incl = 0;
        if (warp < nw) {
            const int e = warp * 32 + lane;
            m = e < a.E ? S.mask[e] : 0u;
            bal = __ballot_sync(0xffffffffu, m != 0u);
            cnt = __popc(m);
            incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (lane == 31) S.wsum[warp] = ((unsigned)__popc(bal) << 16) | (unsigned)incl;
        }
        __syncthreads();
        if (warp < nw) {
            int ub = 0, sb = 0;
            for (int w = 0; w < warp; w++) {
                const unsigned v = S.wsum[w];
                ub += (int)(v >> 16);
                sb += (int)(v & 0xFFFFu);
            }
            const int e = warp * 32 + lane;
            if (m) {
                const int u = ub + __popc(bal & ((1u << lane) - 1u));
                S.uid[e] = (short)u;
                S.uexp[u] = e;
                S.ucnt[u] = cnt;
                S.ubase[u] = sb + incl - cnt;
                S.uslot[u] = a.use_map ? (a.slot_dev ? a.slot_dev[e] : a.slot_map[e]) : e;
            }
            if (warp == nw - 1 && lane == 31) S.U = *err ? 0 : ub + __popc(bal);
        }
        __syncthreads();
        for (int p = tid; p < P2 && !*err; p += kDecThreads) {
            const int t = udiv_small(p, a.topk, topk_magic), e = S.idx[p];
            S.pidx[p] = S.ubase[S.uid[e]] + __popc(S.mask[e] & ((1u << t) - 1u));
        }
    };

    // the counters' values at the start of this call (cumulative counters: no
    // reset between calls)
    uint2 base = make_uint2(0u, 0u);
    // =========================== phase A ===========================
    if (producer) {
        if (lane == 0) {
            // this CTA's shared gate/up tiles, and a slice of the shared down matrix into
            // L2 (weights only: this may run before the previous kernel has finished)
            for (int k = 0; k < n_shared_mine && k < a.stages; k++) {
                const int s = producer_slot(fill);
                mbar_arrive_expect_tx(&S.full[s], gu_bytes);
                bulk_g2s(ring + (size_t)s * a.SB, gu_src(b + k * nC), gu_bytes, &S.full[s]);
                last_fill[s] = fill++;
            }
            for (int r = b; r < R && do_shared; r += nC)
                prefetch_l2(a.shared + a.Ls.gu_bytes + (size_t)kTileBytes * Gs * r, kTileBytes * Gs);
        }
        __syncwarp();
        pdl_wait();
        if (lane == 0) {
            base = __ldcg(reinterpret_cast<const uint2 *>(a.ctrl + kRouteBase));
            if (base.x == 0xFFFFFFFFu && base.y == 0xFFFFFFFFu) __nanosleep(0);  // the load has landed
        }
        if (!pre) {
            // this CTA's router logits from the compute warps' partial sums
            named_sync(2, kDecThreads);
            const int nchk = T >= kCW ? 1 : kCW / T;
            int j = 0;
            for (int e = b; e < a.E; e += nC, j++) {
                if (lane < T) {
                    float acc = 0.f;
                    for (int k = 0; k < nchk; k++) acc += S.rpart[j][lane * nchk + k];
                    // with MOE_PRENORM the sum is of x * norm_w: every CTA applies
                    // 1 / rms and the bias when it ranks
                    a.logits[(size_t)lane * a.E + e] = prenorm ? acc : acc + (a.bias ? a.bias[e] : 0.f);
                }
            }
            if (j > 0) {
                fence_acq_rel_gpu();
                __syncwarp();
                if (lane == 0) atomicAdd(&a.ctrl[kRouteCnt], (unsigned)j);
            }
        }
        if (lane == 0 && !pre &&
            !spin_reach(&a.ctrl[kRouteCnt], base.x, (unsigned)a.E + a.route_extra, &a.ctrl[kErr], a.route_wait_ns))
            *err = 1;
        __syncwarp();
        // the routing (an earlier launch's choices, or every token's logits) into
        // shared memory
        if (pre) {
            for (int p = lane; p < T * a.topk; p += 32) {
                S.idx[p] = a.idx_pre[p];
                S.gate[p] = a.gate_pre[p];
                if (b == 0 && a.idx_out) a.idx_out[p] = S.idx[p];
                if (b == 0 && a.gate_out) a.gate_out[p] = S.gate[p];
            }
        } else if (!*err) {
            float *lg = reinterpret_cast<float *>(hsm);
            const int n = T * a.E;
            for (int i = lane; i < n / 4; i += 32)
                reinterpret_cast<float4 *>(lg)[i] = __ldcg(reinterpret_cast<const float4 *>(a.logits) + i);
            for (int i = (n & ~3) + lane; i < n; i += 32) lg[i] = __ldcg(a.logits + i);
        }
    } else {
        if (!pre) {
            // router rows e = b, b + nC, ...: warp w takes chunk w % nchk of the row
            // for tokens w / nchk, w / nchk + kCW / nchk, ..., so every lane issues
            // its few loads at once; the producer warp adds the partial sums up and
            // publishes the logits.  The chunk's weight lines are prefetched into L2
            // before the wait for the previous kernel.
            const int nchk = T >= kCW ? 1 : kCW / T;
            const int np = H / 8;  // 8-code word pairs per row
            const int t0 = warp / nchk, ck = warp % nchk, tstep = kCW / nchk;
            const int p0 = ck * np / nchk, p1 = (ck + 1) * np / nchk;
            if (t0 < T)
                for (int e = b; e < a.E; e += nC) {
                    const uint8_t *row = reinterpret_cast<const uint8_t *>(a.rq) + (size_t)e * H;
                    const int l0 = (8 * p0) >> 7, l1 = (8 * p1 + 127) >> 7;
                    if (l0 + lane < l1) prefetch_line_l2(row + (size_t)(l0 + lane) * 128);
                    if (lane == 31 && ck == 0) {
                        prefetch_line_l2(a.rs + (size_t)e * (H / kGroup));
                        prefetch_line_l2(a.rb + (size_t)e * (H / kGroup));
                    }
                }
            pdl_wait();
            int j = 0;
            for (int e = b; e < a.E; e += nC, j++)
                for (int t = t0; t < T; t += tstep) {
                    const float v = router_dot(a.rq, a.rs, a.rb, H, a.x, e, t, p0, p1, prenorm ? a.norm_w : nullptr);
                    if (lane == 0) S.rpart[j][t * nchk + ck] = v;
                }
            named_arrive(2, kDecThreads);
        } else {
            pdl_wait();
        }
        if (prenorm) {
            // this warp's share of every token's sum of squares
            for (int t = 0; t < T; t++) {
                const float4 *xt = reinterpret_cast<const float4 *>(a.x + (size_t)t * H);
                float sq = 0.f;
                for (int i = warp * 32 + lane; i < H / 4; i += kCThreads) {
                    const float4 v = __ldg(xt + i);
                    sq += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                }
                sq = warp_sum(sq);
                if (lane == 0) S.xss[warp][t] = sq;
            }
        }
        load_x();
    }
    __syncthreads();
    if (prenorm) {
        // 1 / rms(x_t) from the warps' partial sums (in warp order), then the staged
        // logits become (1 / rms) sum + bias
        if (tid < T) {
            float sq = 0.f;
            for (int w = 0; w < kCW; w++) sq += S.xss[w][tid];
            S.inv_r[tid] = rms_inv(sq, H, a.norm_eps);
        }
        __syncthreads();
        if (!pre && !*err) {
            float *lg = reinterpret_cast<float *>(hsm);
            for (int i = tid; i < T * a.E; i += kDecThreads) {
                const int t = i / a.E, e = i - t * a.E;
                lg[i] = lg[i] * S.inv_r[t] + (a.bias ? a.bias[e] : 0.f);
            }
        }
        __syncthreads();
    }
    // routing with the whole CTA (nothing else runs meanwhile): one warp per token
    // ranks the staged logits, then every thread helps to build the schedule
    if (!pre && !*err)
        for (int t = warp; t < T; t += kCW + 1) rank_token(t);
    __syncthreads();
    build_schedule();
    __syncthreads();

    const int U = do_routed ? S.U : 0;  // routed experts of this launch
    const int NGU = Ts + U * Ti;
    const int NDN = (Pe + U) * R;
    const int ulo = (int)((long long)NDN * b / nC), uhi = (int)((long long)NDN * (b + 1) / nC);
    const int nunits = uhi - ulo;
    const int nstg = (nunits + a.UPS - 1) / a.UPS;
    const int m_first = ulo / R;
    auto unit_src = [&](int m, int r, int *ng) -> const uint8_t * {
        if (m < Pe) {
            const int g0 = m * Gi;
            *ng = min(Gi, Gs - g0);
            return a.shared + a.Ls.gu_bytes + (size_t)kTileBytes * ((size_t)r * Gs + g0);
        }
        *ng = Gi;
        return a.experts + (size_t)S.uslot[m - Pe] * a.stride + a.Lr.gu_bytes + (size_t)kTileBytes * Gi * r;
    };
    // first gate/up tile index of this CTA among the routed ones
    const int j_first = b + n_shared_mine * nC;
    const int n_routed_mine = j_first < NGU ? (NGU - 1 - j_first) / nC + 1 : 0;

    // =========================== phase B ===========================
    if (producer) {
        if (lane == 0) {
            // the shared gate/up tiles that did not fit the ring at the start, then the
            // routed ones (bulk copies stream better on their own than behind L2
            // prefetches of the same data)
            for (int k = a.stages; k < n_shared_mine; k++) {
                const int s = producer_slot(fill);
                if (!*err) {
                    mbar_arrive_expect_tx(&S.full[s], gu_bytes);
                    bulk_g2s(ring + (size_t)s * a.SB, gu_src(b + k * nC), gu_bytes, &S.full[s]);
                    last_fill[s] = fill;
                }
                fill++;
            }
            for (int k = 0; k < n_routed_mine; k++) {
                const int s = producer_slot(fill);
                if (!*err) {
                    mbar_arrive_expect_tx(&S.full[s], gu_bytes);
                    bulk_g2s(ring + (size_t)s * a.SB, gu_src(j_first + k * nC), gu_bytes, &S.full[s]);
                    last_fill[s] = fill;
                }
                fill++;
            }
            // down units: the first `stages` stages now; h of this CTA's matrices once
            // every gate/up tile of the layer is done; then the remaining stages
            const int early = min(nstg, a.stages);
            bool h_armed = false;                      // the h copies were issued
            int um = m_first, ur = ulo - m_first * R;  // (matrix, row tile) of the next unit
#pragma unroll 1
            for (int k = 0; k <= nstg; k++) {
                if (k == early) {
                    if (!*err && !spin_reach(&a.ctrl[kGuDone], base.y, (unsigned)NGU, &a.ctrl[kErr])) *err = 1;
                    if (!*err && nunits > 0) {
                        unsigned bytes = 0;
#pragma unroll 1
                        for (int m = m_first; m <= (uhi - 1) / R; m++) {
                            const bool sh = m < Pe;
                            const unsigned nb = sh ? (unsigned)(min(Gi, Gs - m * Gi) * T * 128)
                                                   : (unsigned)(Gi * S.ucnt[m - Pe] * 128);
                            const __half *src = sh ? a.hs16 + (size_t)m * Gi * T * kGroup
                                                   : a.h16 + (size_t)S.ubase[m - Pe] * a.I;
                            bulk_g2s(hsm + (size_t)(m - m_first) * a.hsm_mat_bytes, src, nb, &S.hbar);
                            bytes += nb;
                        }
                        // the arrival (with the byte count) comes after the copies: the
                        // phase cannot complete before it
                        mbar_arrive_expect_tx(&S.hbar, bytes);
                        h_armed = true;
                    }
                }
                if (k == nstg) break;
                const int s = producer_slot(fill);
                if (!*err) {
                    const int u0 = k * a.UPS, u1 = min(nunits, u0 + a.UPS);
                    unsigned bytes = 0;
#pragma unroll 1
                    for (int i = u0; i < u1; i++) {
                        int ng;
                        const uint8_t *src = unit_src(um, ur, &ng);
                        if (++ur == R) {
                            ur = 0;
                            um++;
                        }
                        bulk_g2s(ring + (size_t)s * a.SB + (size_t)(i - u0) * Gi * kTileBytes, src,
                                 kTileBytes * ng, &S.full[s]);
                        bytes += kTileBytes * ng;
                    }
                    mbar_arrive_expect_tx(&S.full[s], bytes);
                    last_fill[s] = fill;
                }
                fill++;
            }
            // drain: every copy this CTA issued has landed before the CTA exits
            volatile int never = 0;
            for (int s = 0; s < a.stages; s++)
                if (last_fill[s] >= 0) mbar_wait(&S.full[s], (last_fill[s] / a.stages) & 1, &never);
            if (h_armed) mbar_wait(&S.hbar, 0, &never);
            // every CTA has read the bases (all gate/up tiles are counted): the next
            // call's bases
            if (b == 0) {
                a.ctrl[kRouteBase] = base.x + (pre ? 0u : (unsigned)a.E);
                a.ctrl[kGuBase] = base.y + (unsigned)NGU;
            }
        }
        __syncwarp();
    } else {
        // ---- the shared gate/up tiles (in the ring since the start) while the routed
        // ones are on their way
        for (int k = 0; k < n_shared_mine; k++) {
            const int s = consumer_wait(fill++);
            gateup_tile(s, -1, b + k * nC, n_routed_mine == 0 && k == n_shared_mine - 1);
        }
        // ---- routed gate/up tiles: (expert u, row block it) of tile j_first + k nC
        int gu_u = (j_first - Ts) / Ti, gu_it = j_first - Ts - gu_u * Ti;
        for (int k = 0; k < n_routed_mine; k++) {
            const int s = consumer_wait(fill++);
            gateup_tile(s, gu_u, gu_it, k == n_routed_mine - 1);
            gu_it += nC;
            while (gu_it >= Ti) {
                gu_it -= Ti;
                gu_u++;
            }
        }
        fence_acq_rel_gpu();
        named_sync(1, kCThreads);
        if (tid == 0) atomicAdd(&a.ctrl[kGuDone], (unsigned)(n_shared_mine + n_routed_mine));
        // ---- down units
        if (nunits > 0 && !*err && !mbar_wait(&S.hbar, 0, err)) {
            *err = 1;
            atomicExch(&a.ctrl[kErr], 1u);
        }
        // T > 8: the group sums of h (the bias term b * sum h) once per (matrix,
        // group, 8-token chunk) of this CTA's matrices, by an MMA with a ones matrix;
        // at T <= 8 each unit computes its own (one chunk: cheaper than a barrier)
        float *hsum = reinterpret_cast<float *>(dsm + a.hsum_off);  // [matrix][Gi][16]
        if constexpr (NCH > 1) {
            const int nm = nunits > 0 ? (uhi - 1) / R - m_first + 1 : 0;
            for (int task = warp; task < nm * Gi * NCH && !*err; task += kCW) {
                const int ch = task % NCH, mg = task / NCH, mi = mg / Gi, g = mg - mi * Gi, m = m_first + mi;
                const int ng = m < Pe ? min(Gi, Gs - m * Gi) : Gi;
                const int nsl = m < Pe ? T : S.ucnt[m - Pe];
                if (g >= ng || 8 * ch >= nsl) continue;
                uint32_t hb[8];
                const int j = 8 * ch + gl;
                if (j < nsl) {
                    const uint8_t *hr = hsm + (size_t)mi * a.hsm_mat_bytes + ((size_t)g * nsl + j) * 128;
                    const int sw = (j & 1);
                    const uint4 v0 = *reinterpret_cast<const uint4 *>(hr + 16 * ((2 * c) ^ sw));
                    const uint4 v1 = *reinterpret_cast<const uint4 *>(hr + 16 * ((2 * c + 1) ^ sw));
                    hb[0] = v0.x; hb[1] = v0.y; hb[2] = v0.z; hb[3] = v0.w;
                    hb[4] = v1.x; hb[5] = v1.y; hb[6] = v1.z; hb[7] = v1.w;
                } else {
                    zero_b(hb);
                }
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_group_sums(d, hb);
                if (gl == 0) {
                    hsum[(size_t)mg * 16 + 8 * ch + 2 * c] = d[0];
                    hsum[(size_t)mg * 16 + 8 * ch + 2 * c + 1] = d[1];
                }
            }
            named_sync(1, kCThreads);
        }
        int wm = (ulo + warp) / R, wr = ulo + warp - wm * R;  // this warp's next unit
        for (int k = 0; k < nstg; k++) {
            const int s = consumer_wait(fill++);
            for (int i = 0; i < a.UPS; i++) {
                const int lu = k * a.UPS + i;
                if (lu >= nunits || (lu % kCW) != warp || *err) continue;
                const int m = wm, r = wr;
                wr += kCW;
                while (wr >= R) {
                    wr -= R;
                    wm++;
                }
                int ng, nsl;
                float *dst;
                size_t dstride;
                if (m < Pe) {
                    ng = min(Gi, Gs - m * Gi);
                    nsl = T;
                    dst = a.ps + (size_t)m * T * H;
                } else {
                    ng = Gi;
                    nsl = S.ucnt[m - Pe];
                    dst = a.pr + (size_t)S.ubase[m - Pe] * H;
                }
                dstride = H;
                const uint8_t *wst = ring + (size_t)s * a.SB + (size_t)i * Gi * kTileBytes;
                const uint8_t *hm = hsm + (size_t)(m - m_first) * a.hsm_mat_bytes;
                float acc[NCH][4];
#pragma unroll
                for (int ch = 0; ch < NCH; ch++)
#pragma unroll
                    for (int v = 0; v < 4; v++) acc[ch][v] = 0.f;
#pragma unroll 2
                for (int g = 0; g < ng; g++) {
                    const uint4 q = *reinterpret_cast<const uint4 *>(wst + g * kTileBytes + 16 * lane);
                    const uint2 e = *reinterpret_cast<const uint2 *>(wst + g * kTileBytes + 512 + 8 * gl);
                    const float sa = lo_half(e.x) * kTwo24, ba = hi_half(e.x);
                    const float sb = lo_half(e.y) * kTwo24, bb = hi_half(e.y);
#pragma unroll
                    for (int ch = 0; ch < NCH; ch++) {
                        if (8 * ch < nsl) {
                            uint32_t hb[8];
                            const int j = 8 * ch + gl;
                            if (j < nsl) {
                                const uint8_t *hr = hm + ((size_t)g * nsl + j) * 128;
                                const int sw = (j & 1);
                                const uint4 v0 = *reinterpret_cast<const uint4 *>(hr + 16 * ((2 * c) ^ sw));
                                const uint4 v1 = *reinterpret_cast<const uint4 *>(hr + 16 * ((2 * c + 1) ^ sw));
                                hb[0] = v0.x; hb[1] = v0.y; hb[2] = v0.z; hb[3] = v0.w;
                                hb[4] = v1.x; hb[5] = v1.y; hb[6] = v1.z; hb[7] = v1.w;
                            } else {
                                zero_b(hb);
                            }
                            // the group sums of h for token columns 2c, 2c+1 (the bias term
                            // b * sum h), on the tensor cores like those of x
                            float s0, s1;
                            if constexpr (NCH > 1) {
                                const float *hg = hsum + ((size_t)(m - m_first) * Gi + g) * 16 + 8 * ch + 2 * c;
                                s0 = hg[0];
                                s1 = hg[1];
                            } else {
                                float hq[4] = {0.f, 0.f, 0.f, 0.f};
                                mma_group_sums(hq, hb);
                                s0 = hq[0];
                                s1 = hq[1];
                            }
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_group_codes(d, make_uint2(q.x, q.y), make_uint2(q.z, q.w), hb);
                            affine_acc(acc[ch], d, s0, s1, sa, ba, sb, bb);
                        }
                    }
                }
#pragma unroll
                for (int ch = 0; ch < NCH; ch++) {
                    const int j0 = 8 * ch + 2 * c, na = 16 * r + gl;
                    if (j0 < nsl) {
                        dst[(size_t)j0 * dstride + na] = acc[ch][0];
                        dst[(size_t)j0 * dstride + na + 8] = acc[ch][2];
                    }
                    if (j0 + 1 < nsl) {
                        dst[(size_t)(j0 + 1) * dstride + na] = acc[ch][1];
                        dst[(size_t)(j0 + 1) * dstride + na + 8] = acc[ch][3];
                    }
                }
            }
            consumer_release(s);
        }
        // ---- tickets: this CTA's down units are counted into their 16-row tiles
        fence_acq_rel_gpu();
        named_sync(1, kCThreads);
        if (do_routed && !*err)
            for (int lu = tid; lu < nunits; lu += kCThreads) atomicAdd(&a.ticket[(ulo + lu) % R], 1u);
        // ---- combine the tiles this CTA owns (r = b, b + nC, ...) once every
        // contribution to them is in: y = sum_k gate_k * routed_k + sum_parts shared (+ x)
        if (do_routed) {
            const unsigned target = (unsigned)(Pe + U);
            const int nown = b < R ? (R - 1 - b) / nC + 1 : 0;
            for (int c = tid; c < nown && !*err; c += kCThreads) {
                const int r = b + c * nC;
                if (!spin_geq(&a.ticket[r], target, &a.ctrl[kErr])) *err = 1;
                a.ticket[r] = 0u;  // every contribution is in: ready for the next call
            }
            named_sync(1, kCThreads);
            const unsigned T_magic = udiv_magic(T);
            // element v = (owned tile c, token t, row n % 16), v >> 4 = c * T + t
            for (int v = tid; v < nown * 16 * T && !*err; v += kCThreads) {
                const int ct = v >> 4, c = udiv_small(ct, T, T_magic), t = ct - c * T;
                const int n = 16 * (b + c * nC) + (v & 15);
                float pv[MOE_MAX_TOPK];
#pragma unroll
                for (int k = 0; k < MOE_MAX_TOPK; k++)
                    pv[k] = k < a.topk ? __ldcg(a.pr + (size_t)S.pidx[t * a.topk + k] * H + n) : 0.f;
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < MOE_MAX_TOPK; k++)
                    if (k < a.topk) acc = fmaf(S.gate[t * a.topk + k], pv[k], acc);
                for (int p0 = 0; p0 < a.P; p0 += 4) {
                    float sv[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) sv[q] = p0 + q < a.P ? __ldcg(a.ps + ((size_t)(p0 + q) * T + t) * H + n) : 0.f;
#pragma unroll
                    for (int q = 0; q < 4; q++) acc += sv[q];
                }
                if (a.flags & MOE_RESIDUAL) acc += __ldg(a.x + (size_t)t * H + n);
                a.y[(size_t)t * H + n] = acc;
            }
        }
    }

}

}  // namespace moe
