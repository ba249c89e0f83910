// quantise.cuh -- the affine group quantiser (builds packed weights; not on the
// layer's hot path).
#pragma once

#include "common.cuh"

namespace moe {

// ------------------------------------------------------------------ quantiser
// One thread per (row, group of 64).  Same fp32 operations, in the same order,
// as the definition in moe.h, with explicitly rounded intrinsics so that the
// compiler cannot contract them.
__global__ void k_quantise(const float *__restrict__ w, int N, int K, int bits, uint32_t *q,
                           __half *s, __half *b) {
    const int G = K / kGroup;
    long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)N * G) return;
    const int n = (int)(gid / G), g = (int)(gid % G);
    const float *v = w + (size_t)n * K + (size_t)g * kGroup;
    float mn = v[0], mx = v[0];
    for (int j = 1; j < kGroup; j++) {
        float a = v[j];
        if (a < mn) mn = a;
        if (a > mx) mx = a;
    }
    const unsigned qmax = (1u << bits) - 1u;
    float step = __fdiv_rn(__fsub_rn(mx, mn), (float)qmax);
    __half sh = __float2half_rn(step);
    __half bh = __float2half_rn(mn);
    s[(size_t)n * G + g] = sh;
    b[(size_t)n * G + g] = bh;
    const float sf = __half2float(sh), bf = __half2float(bh);
    const int per_word = 32 / bits;
    uint32_t *out = q + (size_t)n * (K * bits / 32) + (size_t)g * (kGroup / per_word);
    for (int wi = 0; wi < kGroup / per_word; wi++) {
        uint32_t word = 0;
        for (int i = 0; i < per_word; i++) {
            unsigned code = 0;
            if (sf != 0.0f) {
                float t = rintf(__fdiv_rn(__fsub_rn(v[wi * per_word + i], bf), sf));
                t = fminf(fmaxf(t, 0.0f), (float)qmax);
                code = (unsigned)t;
            }
            word |= code << (bits * i);
        }
        out[wi] = word;
    }
}

}  // namespace moe
