// sample.cuh -- one token per row of logits: temperature, top-K, top-P, and a draw
// with a caller-supplied uniform number.
//
// The engine samples with temperature, top-K and top-P (defaults 0.2, 64, 0.95:
// "Correr un modelo de 26.000 millones...", section "Como empezar"); the order of
// the steps is the plain one: the K largest logits (ties to the lower index), the
// softmax of those at the temperature, the shortest prefix (in that order) whose
// probability reaches top-P, and the first token of the prefix whose cumulative
// weight exceeds u times the prefix's total.  Temperature <= 0 is greedy.
//
// One cluster of 8 CTAs (1024 threads each) per row, CTA r taking the r-th eighth
// of the row, so that 8 SMs stream it; the CTAs meet through distributed shared
// memory and cluster barriers (hardware barriers: every CTA of a cluster runs at
// the same time).  The candidates are the K largest (key, index) packs, key =
// route.cuh's order-preserving topk_key, larger key first, then lower index:
//   count    each CTA: a 4096-bin histogram of its keys' top 12 bits (sign,
//            exponent, 3 mantissa bits: 1/8 of a binade per bin), warp-aggregated
//            shared atomics (lanes with the same bin add once);
//   choose   the leader CTA (rank 0) adds the 8 histograms and finds the bin
//            holding the K-th largest key by a block scan from the top;
//   compact  each CTA appends every pack of its eighth in that bin or above (at
//            most 4096 in all) to the leader's shared memory (remote atomics on
//            the leader's counter); the leader sorts them, bitonic;
//   fallback when more than 4096 keys reach the chosen bin: a four-pass radix
//            select on 8-bit digits finds the K-th key, the keys above it plus the
//            lowest-index ties at it are collected (threads own contiguous chunks
//            of the row and a scan of their tie counts orders the ties) and sorted;
//   draw     softmax weights at the temperature, an inclusive scan, the top-P cut
//            and the draw, each a block-wide minimum.
// The leader alone runs the fallback and the draw.  Everything is fp32 and
// deterministic (atomics only count, pick slots or minima; the sorted order does
// not depend on which slot a pack took).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "route.cuh"

namespace moe {

constexpr int kSampleThreads = 1024;
constexpr int kSampleMaxK = 1024;
constexpr int kSamplePool = 4096;  // packs the compacting path keeps in shared memory
constexpr int kSampleBatch = 32;   // logits a thread loads before it uses any of them
constexpr int kSampleCluster = 8;  // CTAs (SMs) per row

// (key, index) packed so that a larger value means a larger key, then a lower index.
__device__ __forceinline__ unsigned long long sample_pack(unsigned key, int i) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)i);
}
__device__ __forceinline__ int sample_index(unsigned long long p) { return (int)(0xFFFFFFFFu - (unsigned)p); }

// Inclusive scan of v over the CTA's threads (in thread order); wsum: 32 floats.
__device__ __forceinline__ float block_scan_incl(float v, float *wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    return warp > 0 ? v + wsum[warp - 1] : v;
}

__device__ __forceinline__ unsigned block_scan_excl_u(unsigned v, unsigned *wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        unsigned w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    return (warp > 0 ? wsum[warp - 1] : 0u) + x - v;
}

// Bitonic sort of pool[0, n) into descending order (n a power of two <= 4096).
__device__ __forceinline__ void sample_sort_desc(unsigned long long *pool, int n) {
    for (int k2 = 2; k2 <= n; k2 <<= 1) {
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += kSampleThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long a = pool[i], b = pool[l];
                    const bool desc = (i & k2) == 0;
                    if (desc ? a < b : a > b) {
                        pool[i] = b;
                        pool[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kSampleThreads)
    k_sample(const float *__restrict__ logits, int V, float temp, int K, float top_p, const float *__restrict__ u,
             int32_t *__restrict__ tok) {
    namespace cg = cooperative_groups;
    // the candidates (sorted, largest first) end in the leader's pool[0, K); the
    // count pass uses the same memory as its histogram, the fallback keeps its 256
    // bins at the end
    __shared__ __align__(16) unsigned long long pool[kSamplePool];
    __shared__ float cum[kSampleMaxK];
    __shared__ float fsum[32];
    __shared__ unsigned usum[32];
    __shared__ unsigned long long wbest[32], cbest[kSampleCluster];
    __shared__ unsigned prefix, need, nabove, sel_bin, sel_total, nbuf;
    __shared__ int ncut, pick;
    cg::cluster_group cl = cg::this_cluster();
    const unsigned rank = cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rowi = blockIdx.x / kSampleCluster;
    const float *row = logits + (size_t)rowi * V;
    const int c0 = (int)((long long)V * rank / kSampleCluster), c1 = (int)((long long)V * (rank + 1) / kSampleCluster);

    if (temp <= 0.f || K == 1) {
        // greedy: the largest key, then the lowest index
        unsigned long long best = 0ull;
        for (int base = c0; base < c1; base += kSampleThreads * kSampleBatch) {
            float v[kSampleBatch];
#pragma unroll
            for (int k = 0; k < kSampleBatch; k++) {
                const int i = base + k * kSampleThreads + tid;
                v[k] = i < c1 ? row[i] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kSampleBatch; k++) {
                const int i = base + k * kSampleThreads + tid;
                const unsigned long long p = i < c1 ? sample_pack(topk_key(v[k]), i) : 0ull;
                best = p > best ? p : best;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
            best = y > best ? y : best;
        }
        if (lane == 0) wbest[warp] = best;
        __syncthreads();
        if (warp == 0) {
            best = wbest[lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
                best = y > best ? y : best;
            }
            if (lane == 0) cl.map_shared_rank(cbest, 0)[rank] = best;
        }
        cl.sync();
        if (rank == 0 && tid == 0) {
            best = 0ull;
            for (int r = 0; r < kSampleCluster; r++) best = cbest[r] > best ? cbest[r] : best;
            tok[rowi] = sample_index(best);
        }
        return;
    }

    // ---- count: histogram of the top 12 key bits of this CTA's eighth
    unsigned *hist = reinterpret_cast<unsigned *>(pool);  // [4096]
    for (int i = tid; i < 4096; i += kSampleThreads) hist[i] = 0u;
    __syncthreads();
    for (int base = c0; base < c1; base += kSampleThreads * kSampleBatch) {
        float v[kSampleBatch];
#pragma unroll
        for (int k = 0; k < kSampleBatch; k++) {
            const int i = base + k * kSampleThreads + tid;
            v[k] = i < c1 ? row[i] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kSampleBatch; k++) {
            const bool ok = base + k * kSampleThreads + tid < c1;
            const unsigned d = ok ? topk_key(v[k]) >> 20 : 0xFFFFFFFFu;
            const unsigned peers = __match_any_sync(0xffffffffu, d);
            if (ok && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (unsigned)__popc(peers));
        }
    }
    cl.sync();  // every eighth counted
    // ---- choose (leader): thread t holds bins 4095 - 4t .. 4092 - 4t (largest first)
    if (rank == 0) {
        unsigned c4[4], tot = 0u;
#pragma unroll
        for (int j = 0; j < 4; j++) c4[j] = 0u;
        for (int r = 0; r < kSampleCluster; r++) {
            const unsigned *h = cl.map_shared_rank(hist, r);
#pragma unroll
            for (int j = 0; j < 4; j++) c4[j] += h[4095 - 4 * tid - j];
        }
#pragma unroll
        for (int j = 0; j < 4; j++) tot += c4[j];
        const unsigned before = block_scan_excl_u(tot, usum);  // keys in larger bins
        if (before < (unsigned)K && before + tot >= (unsigned)K) {
            unsigned acc = before;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                if (acc + c4[j] >= (unsigned)K) {
                    sel_bin = 4095u - 4u * tid - j;
                    sel_total = acc + c4[j];
                    break;
                }
                acc += c4[j];
            }
        }
        if (tid == 0) nbuf = 0u;
    }
    cl.sync();  // the choice is made; no histogram is read any more
    const unsigned bsel = *cl.map_shared_rank(&sel_bin, 0), total = *cl.map_shared_rank(&sel_total, 0);

    if (total <= (unsigned)kSamplePool) {
        // ---- compact this eighth's packs of bin bsel and above into the leader's pool
        unsigned long long *lpool = cl.map_shared_rank(pool, 0);
        unsigned *lnbuf = cl.map_shared_rank(&nbuf, 0);
        for (int base = c0; base < c1; base += kSampleThreads * kSampleBatch) {
            float v[kSampleBatch];
#pragma unroll
            for (int k = 0; k < kSampleBatch; k++) {
                const int i = base + k * kSampleThreads + tid;
                v[k] = i < c1 ? row[i] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kSampleBatch; k++) {
                const int i = base + k * kSampleThreads + tid;
                const unsigned key = i < c1 ? topk_key(v[k]) : 0u;
                const bool take = i < c1 && (key >> 20) >= bsel;
                const unsigned m = __ballot_sync(0xffffffffu, take);
                if (m) {  // warp-uniform
                    unsigned slot0 = 0u;
                    if (lane == 0) slot0 = atomicAdd(lnbuf, (unsigned)__popc(m));
                    slot0 = __shfl_sync(0xffffffffu, slot0, 0);
                    if (take) lpool[slot0 + __popc(m & ((1u << lane) - 1u))] = sample_pack(key, i);
                }
            }
        }
    }
    cl.sync();  // the leader's pool is complete; from here the leader works alone, in its own memory
    if (rank != 0) return;
    if (total <= (unsigned)kSamplePool) {
        int n2 = 2;
        while (n2 < (int)total) n2 <<= 1;
        for (int i = (int)total + tid; i < n2; i += kSampleThreads) pool[i] = 0ull;  // padding sorts last
        __syncthreads();
        sample_sort_desc(pool, n2);
    } else {
        // ---- fallback: radix select of the K-th largest key, most significant digit first
        unsigned *hist8 = reinterpret_cast<unsigned *>(pool + kSamplePool - 128);  // 256 bins past the candidates
        if (tid == 0) {
            prefix = 0u;
            need = (unsigned)K;
        }
        unsigned mask = 0u;
        for (int d = 3; d >= 0; d--) {
            if (tid < 256) hist8[tid] = 0u;
            __syncthreads();
            const unsigned pf = prefix;
            for (int i = tid; i < V; i += kSampleThreads) {
                const unsigned key = topk_key(row[i]);
                if ((key & mask) == pf) atomicAdd(&hist8[(key >> (8 * d)) & 255u], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                const unsigned nd = need;  // read by every lane before any lane writes it
                __syncwarp();
                // lane l holds bins 255 - 8l .. 248 - 8l (largest first)
                unsigned cnt[8], tot = 0u;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    cnt[j] = hist8[255 - 8 * lane - j];
                    tot += cnt[j];
                }
                unsigned above = tot;  // exclusive prefix over the lanes of larger bins
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(0xffffffffu, above, o);
                    if (lane >= o) above += y;
                }
                above -= tot;
                if (above < nd && above + tot >= nd) {
                    unsigned acc = above;
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        if (acc + cnt[j] >= nd) {
                            prefix = pf | ((unsigned)(255 - 8 * lane - j) << (8 * d));
                            need = nd - acc;
                            break;
                        }
                        acc += cnt[j];
                    }
                }
            }
            mask |= 255u << (8 * d);
            __syncthreads();
        }
        const unsigned kth = prefix, ties = need;  // take the `ties` lowest-index keys equal to kth
        // collect: contiguous chunks per thread so that ties are ordered by index
        const int chunk = (V + kSampleThreads - 1) / kSampleThreads;
        const int i0 = min(V, tid * chunk), i1 = min(V, i0 + chunk);
        unsigned my_ties = 0u;
        for (int i = i0; i < i1; i++) my_ties += topk_key(row[i]) == kth;
        if (tid == 0) nabove = 0u;
        const unsigned tie_base = block_scan_excl_u(my_ties, usum);
        const unsigned n_above = (unsigned)K - ties;
        for (int i = tid; i < kSampleMaxK; i += kSampleThreads) pool[i] = 0ull;
        __syncthreads();
        unsigned r = tie_base;
        for (int i = i0; i < i1; i++) {
            const unsigned key = topk_key(row[i]);
            if (key > kth) {
                const unsigned sl = atomicAdd(&nabove, 1u);  // < n_above by the selection
                if (sl < n_above) pool[sl] = sample_pack(key, i);
            } else if (key == kth) {
                if (r < ties && n_above + r < (unsigned)kSampleMaxK) pool[n_above + r] = sample_pack(key, i);
                r++;
            }
        }
        __syncthreads();
        sample_sort_desc(pool, kSampleMaxK);
    }

    // ---- softmax weights at the temperature, their inclusive scan, top-P, draw
    const float m = row[sample_index(pool[0])];
    const float w = tid < K ? expf((row[sample_index(pool[tid])] - m) / temp) : 0.f;
    const float c = block_scan_incl(w, fsum);
    if (tid < K) cum[tid] = c;
    if (tid == 0) ncut = K;
    __syncthreads();
    const float total_w = cum[K - 1];
    if (top_p < 1.f && tid < K && cum[tid] >= top_p * total_w) atomicMin(&ncut, tid + 1);
    __syncthreads();
    const int n = ncut;
    if (tid == 0) pick = n - 1;
    __syncthreads();
    const float thr = u[rowi] * cum[n - 1];
    if (tid < n && cum[tid] > thr) atomicMin(&pick, tid);
    __syncthreads();
    if (tid == 0) tok[rowi] = sample_index(pool[pick]);
}

}  // namespace moe
