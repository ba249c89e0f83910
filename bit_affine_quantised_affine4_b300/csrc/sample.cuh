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
// One CTA of 1024 threads per row:
//   select   the K-th largest order-preserving key (route.cuh's topk_key) by a
//            four-pass radix select on 8-bit digits (a shared 256-bin histogram per
//            pass over the row);
//   collect  the keys above it, plus the lowest-index ties at it (threads own
//            contiguous chunks of the row, and a scan of their tie counts orders
//            the ties by index);
//   sort     the K candidates by (key desc, index asc), bitonic in shared memory;
//   draw     softmax weights at the temperature, an inclusive scan, the top-P cut
//            and the draw, each a block-wide minimum.
// Everything is fp32 and deterministic (atomics only pick slots or minima).
#pragma once

#include "common.cuh"
#include "route.cuh"

namespace moe {

constexpr int kSampleThreads = 1024;
constexpr int kSampleMaxK = 1024;

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

__global__ void __launch_bounds__(kSampleThreads) k_sample(const float *__restrict__ logits, int V, float temp,
                                                         int K, float top_p, const float *__restrict__ u,
                                                         int32_t *__restrict__ tok) {
    __shared__ unsigned hist[256];
    __shared__ unsigned long long cand[kSampleMaxK];
    __shared__ float cum[kSampleMaxK];
    __shared__ float fsum[32];
    __shared__ unsigned usum[32];
    __shared__ unsigned long long wbest[32];
    __shared__ unsigned prefix, need, nabove;
    __shared__ int ncut, pick;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *row = logits + (size_t)blockIdx.x * V;

    if (temp <= 0.f || K == 1) {
        // greedy: the largest key, then the lowest index
        unsigned long long best = 0ull;
        for (int i = tid; i < V; i += kSampleThreads) {
            const unsigned long long p = sample_pack(topk_key(row[i]), i);
            best = p > best ? p : best;
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
            if (lane == 0) tok[blockIdx.x] = sample_index(best);
        }
        return;
    }

    // ---- radix select: the K-th largest key, most significant digit first
    if (tid == 0) {
        prefix = 0u;
        need = (unsigned)K;
    }
    unsigned mask = 0u;
    for (int d = 3; d >= 0; d--) {
        if (tid < 256) hist[tid] = 0u;
        __syncthreads();
        const unsigned pf = prefix;
        for (int i = tid; i < V; i += kSampleThreads) {
            const unsigned key = topk_key(row[i]);
            if ((key & mask) == pf) atomicAdd(&hist[(key >> (8 * d)) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            const unsigned nd = need;  // read by every lane before any lane writes it
            __syncwarp();
            // lane l holds bins 255 - 8l .. 248 - 8l (largest first)
            unsigned cnt[8], tot = 0u;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                cnt[j] = hist[255 - 8 * lane - j];
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
    // ---- collect: contiguous chunks per thread so that ties are ordered by index
    const int chunk = (V + kSampleThreads - 1) / kSampleThreads;
    const int i0 = min(V, tid * chunk), i1 = min(V, i0 + chunk);
    unsigned my_ties = 0u;
    for (int i = i0; i < i1; i++) my_ties += topk_key(row[i]) == kth;
    if (tid == 0) nabove = 0u;
    const unsigned tie_base = block_scan_excl_u(my_ties, usum);
    const unsigned n_above = (unsigned)K - ties;
    for (int i = tid; i < kSampleMaxK; i += kSampleThreads) cand[i] = 0ull;
    __syncthreads();
    unsigned r = tie_base;
    for (int i = i0; i < i1; i++) {
        const unsigned key = topk_key(row[i]);
        if (key > kth) {
            const unsigned sl = atomicAdd(&nabove, 1u);  // < n_above by the selection
            if (sl < n_above) cand[sl] = sample_pack(key, i);
        } else if (key == kth) {
            if (r < ties && n_above + r < (unsigned)kSampleMaxK) cand[n_above + r] = sample_pack(key, i);
            r++;
        }
    }
    __syncthreads();
    // ---- bitonic sort, descending (padding entries are 0: last)
    for (int k2 = 2; k2 <= kSampleMaxK; k2 <<= 1) {
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const int i = tid, l = i ^ j;
            if (l > i) {
                const unsigned long long a = cand[i], b = cand[l];
                const bool desc = (i & k2) == 0;
                if (desc ? a < b : a > b) {
                    cand[i] = b;
                    cand[l] = a;
                }
            }
            __syncthreads();
        }
    }
    // ---- softmax weights at the temperature, their inclusive scan, top-P, draw
    const float m = row[sample_index(cand[0])];
    const float w = tid < K ? expf((row[sample_index(cand[tid])] - m) / temp) : 0.f;
    const float c = block_scan_incl(w, fsum);
    if (tid < K) cum[tid] = c;
    if (tid == 0) ncut = K;
    __syncthreads();
    const float total = cum[K - 1];
    if (top_p < 1.f && tid < K && cum[tid] >= top_p * total) atomicMin(&ncut, tid + 1);
    __syncthreads();
    const int n = ncut;
    if (tid == 0) pick = n - 1;
    __syncthreads();
    const float thr = u[blockIdx.x] * cum[n - 1];
    if (tid < n && cum[tid] > thr) atomicMin(&pick, tid);
    __syncthreads();
    if (tid == 0) tok[blockIdx.x] = sample_index(cand[pick]);
}

}  // namespace moe
