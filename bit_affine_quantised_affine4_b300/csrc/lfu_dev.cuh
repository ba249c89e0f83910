// lfu_dev.cuh -- the per-layer expert cache policy run on the device, and the
// kernel that fetches missing experts from page-locked host memory.
//
// The policy is lfu.h's (16 slots, least frequently used, per layer: devtrends page
// "Come eseguire un modello da 26 miliardi...", section "Qual e il trucco
// principale dell'architettura"; remio.ai page, section "Mac Gemma 4 26B entra
// nello spazio disponibile..."; the tie rules are this library's reading), step for
// step: a request list R of the step's distinct experts in first-appearance order;
// every resident member of R is a hit (count + 1, last use = step); then each
// missing member, in order, takes the lowest empty slot or else evicts the slot,
// among those not holding a member of R, with the smallest (count, last use, slot),
// and starts at count 1.  The pages have the CPU decide the reads while the GPU
// computes; here the decision stays on the GPU, so a layer call needs no host round
// trip: the router's ranking CTA runs the step, a fetch kernel copies the misses
// from host memory (read by the SMs through its device mapping) into their slots,
// and the decode kernel reads the slot of each expert from device memory.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kDevLfuMaxSlots = MOE_MAX_CACHE_SLOTS;

// Policy state and the last step's outcome, in device memory.
struct DevLfu {
    int slots, E;
    long long step;
    unsigned long long hits, misses, h2d_bytes;
    int nmiss;                         // the last step's misses, in request order
    int miss_e[kDevLfuMaxSlots], miss_s[kDevLfuMaxSlots];
    int expert_of[kDevLfuMaxSlots];    // -1 = empty
    unsigned count[kDevLfuMaxSlots];
    long long last[kDevLfuMaxSlots];
    short where[MOE_MAX_EXPERTS];      // slot of each expert, -1 = not resident
};

// One step by one thread, on the routing idx[T][topk].  The caller guarantees that
// T * topk <= slots, so the request list always fits.
__device__ void dev_lfu_step(DevLfu *p, const int *idx, int P2) {
    int req[kDevLfuMaxSlots];
    unsigned wanted[MOE_MAX_EXPERTS / 32] = {};
    int n = 0;
    for (int q = 0; q < P2; q++) {
        const int e = idx[q];
        if ((wanted[e >> 5] >> (e & 31)) & 1u) continue;
        wanted[e >> 5] |= 1u << (e & 31);
        req[n++] = e;
    }
    const long long step = p->step;
    for (int i = 0; i < n; i++) {
        const int s = p->where[req[i]];
        if (s >= 0) {
            p->count[s]++;
            p->last[s] = step;
            p->hits++;
        }
    }
    int nm = 0;
    for (int i = 0; i < n; i++) {
        const int e = req[i];
        if (p->where[e] >= 0) continue;
        int v = -1;
        for (int s = 0; s < p->slots && v < 0; s++)
            if (p->expert_of[s] < 0) v = s;
        if (v < 0)
            for (int s = 0; s < p->slots; s++) {
                const int o = p->expert_of[s];  // every slot is occupied here
                if (o >= 0 && ((wanted[o >> 5] >> (o & 31)) & 1u)) continue;
                if (v < 0 || p->count[s] < p->count[v] || (p->count[s] == p->count[v] && p->last[s] < p->last[v]))
                    v = s;
            }
        if (p->expert_of[v] >= 0) p->where[p->expert_of[v]] = -1;
        p->expert_of[v] = e;
        p->where[e] = (short)v;
        p->count[v] = 1u;
        p->last[v] = step;
        p->misses++;
        p->miss_e[nm] = e;
        p->miss_s[nm] = v;
        nm++;
    }
    p->nmiss = nm;
    p->step = step + 1;
}

// Copies the last step's missing experts (blob bytes each, a multiple of 64) from
// host memory (h_experts: the device's address of the page-locked blobs, blob e at
// e * host_stride) into their slots.  Grid-stride over 16-byte chunks, four loads
// in flight per thread; loads go around L1 (the source is read once).
__global__ void __launch_bounds__(256) k_cache_fetch(DevLfu *p, const uint8_t *h_experts, size_t host_stride,
                                                    uint8_t *slots, size_t blob) {
    const int nm = p->nmiss;
    const unsigned per = (unsigned)(blob / 16), step = gridDim.x * blockDim.x;
    const unsigned first = blockIdx.x * blockDim.x + threadIdx.x;
    for (int m = 0; m < nm; m++) {
        const uint4 *src = reinterpret_cast<const uint4 *>(h_experts + (size_t)p->miss_e[m] * host_stride);
        uint4 *dst = reinterpret_cast<uint4 *>(slots + (size_t)p->miss_s[m] * blob);
        unsigned k = first;
        for (; k + 3 * step < per; k += 4 * step) {
            const uint4 a = __ldcg(src + k), b = __ldcg(src + k + step), c = __ldcg(src + k + 2 * step),
                        d = __ldcg(src + k + 3 * step);
            dst[k] = a;
            dst[k + step] = b;
            dst[k + 2 * step] = c;
            dst[k + 3 * step] = d;
        }
        for (; k < per; k += step) dst[k] = __ldcg(src + k);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) p->h2d_bytes += (unsigned long long)nm * blob;
}

}  // namespace moe
