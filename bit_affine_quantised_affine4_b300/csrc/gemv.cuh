// gemv.cuh -- the standalone 4-bit affine GEMV, y = deq(W) x, on the tensor cores.
#pragma once

#include "common.cuh"
#include "mma_core.cuh"

namespace moe {

constexpr int kGemvWarps = 4;

// One CTA per 16-row tile; its 4 warps split the K groups.  Rows past N read the
// last row (in bounds) and are not written.
__global__ void __launch_bounds__(kGemvWarps * 32) k_qgemv4_mma(QMat m, const float *__restrict__ x,
                                                                float *__restrict__ y) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
    const int r0 = blockIdx.x * 16;
    const int ra = min(r0 + gl, m.rows - 1), rb = min(r0 + gl + 8, m.rows - 1);
    const int G = m.K / kGroup, wpr = m.K / 8;
    const int g0 = warp * G / kGemvWarps, g1 = (warp + 1) * G / kGemvWarps;
    const uint32_t *qa = m.q + (size_t)ra * wpr + 2 * c, *qb = m.q + (size_t)rb * wpr + 2 * c;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = g0; g < g1; g++) {
        const uint2 wa = ldg_u2(qa + g * 8), wb = ldg_u2(qb + g * 8);
        uint32_t xb[8];
        if (gl == 0)
            load_b_f32(xb, x + g * kGroup + 16 * c);
        else
            zero_b(xb);
        float d[4] = {0.f, 0.f, 0.f, 0.f}, sm[4] = {0.f, 0.f, 0.f, 0.f};
        mma_group_sums(sm, xb);
        mma_group_codes(d, wa, wb, xb);
        apply_affine(acc, d, sm, __half2float(m.s[(size_t)ra * G + g]) * kTwo24,
                     __half2float(m.b[(size_t)ra * G + g]), __half2float(m.s[(size_t)rb * G + g]) * kTwo24,
                     __half2float(m.b[(size_t)rb * G + g]));
    }
    __shared__ float red[kGemvWarps][16];
    if (c == 0) {  // token column 0 lives in accumulator slots 0 (row g) and 2 (row g+8)
        red[warp][gl] = acc[0];
        red[warp][gl + 8] = acc[2];
    }
    __syncthreads();
    if (threadIdx.x < 16 && r0 + (int)threadIdx.x < m.rows) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kGemvWarps; w++) v += red[w][threadIdx.x];
        y[r0 + threadIdx.x] = v;
    }
}

}  // namespace moe
