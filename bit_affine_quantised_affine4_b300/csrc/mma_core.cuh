// mma_core.cuh -- tensor-core dot products on packed 4-bit affine weights.
//
// A 16-row x 64-column tile (one quantisation group) is multiplied by up to 8
// token columns with four m16n8k16 MMAs (fp16 operands, fp32 accumulation):
//   * A (weights): each lane holds, for rows g and g+8 (g = lane/4), the two
//     32-bit words 2c, 2c+1 (c = lane%4) of the group -- 16 consecutive columns
//     16c..16c+15.  A nibble pair (n_s, n_{s+4}) of a word is turned into an
//     fp16x2 register with one AND: (w >> 4s) & 0x000F000F puts each code in the
//     low mantissa bits of a zero-exponent half, i.e. the value q * 2^-24 exactly.
//   * B (tokens): the same columns of the token vectors in fp16, stored in
//     "fragment order": within each aligned run of 8 columns the halves are kept as
//     (0,4, 1,5, 2,6, 3,7), so one 16-byte load gives the four B registers that
//     pair with the four nibble pairs of one word.
// The k order inside an MMA is a permutation of the group's 64 columns, applied
// identically to A and B, so the dot product is unchanged.
// Per group:  D = sum_j q_j x_j * 2^-24  and  S = sum_j x_j (an MMA with A = 1),
// and the affine weight w = s q + b gives  s * 2^24 * D + b * S.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Position of column k in fragment order (a permutation within each aligned run of 8).
__host__ __device__ __forceinline__ int frag_pos(int k) {
    return (k & ~7) | (2 * (k & 3) + ((k >> 2) & 1));
}

// D += (q * 2^-24) x over one group for rows (g, g+8): qa/qb = the lane's two words
// of rows g and g+8; xb = the lane's 8 B registers (two 16-byte loads).
__device__ __forceinline__ void mma_group_codes(float (&d)[4], uint2 qa, uint2 qb,
                                                const uint32_t (&xb)[8]) {
    // two independent accumulator chains (words 2c and 2c+1), added at the end
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const uint32_t wa = j ? qa.y : qa.x, wb = j ? qb.y : qb.x;
#pragma unroll
        for (int h = 0; h < 2; h++) {
            uint32_t a[4];
            a[0] = (wa >> (8 * h)) & 0x000F000Fu;
            a[1] = (wb >> (8 * h)) & 0x000F000Fu;
            a[2] = (wa >> (8 * h + 4)) & 0x000F000Fu;
            a[3] = (wb >> (8 * h + 4)) & 0x000F000Fu;
            if (j == 0)
                mma16816(d, a, xb[4 * j + 2 * h], xb[4 * j + 2 * h + 1]);
            else
                mma16816(e, a, xb[4 * j + 2 * h], xb[4 * j + 2 * h + 1]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) d[i] += e[i];
}

// S += sum of the group's 64 token values, for token columns (2c, 2c+1) in d[0], d[1]
// (d[2], d[3] repeat them for rows g+8).
__device__ __forceinline__ void mma_group_sums(float (&d)[4], const uint32_t (&xb)[8]) {
    const uint32_t one2 = 0x3C003C00u;  // fp16x2 (1, 1)
    const uint32_t a[4] = {one2, one2, one2, one2};
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; h++) {
        mma16816(d, a, xb[2 * h], xb[2 * h + 1]);
        mma16816(e, a, xb[4 + 2 * h], xb[4 + 2 * h + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; i++) d[i] += e[i];
}

// acc += s * 2^24 * D + b * S for the lane's four accumulator slots.
__device__ __forceinline__ void apply_affine(float (&acc)[4], const float (&d)[4],
                                             const float (&sum)[4], float sa, float ba, float sb,
                                             float bb) {
    acc[0] = fmaf(sa, d[0], fmaf(ba, sum[0], acc[0]));
    acc[1] = fmaf(sa, d[1], fmaf(ba, sum[1], acc[1]));
    acc[2] = fmaf(sb, d[2], fmaf(bb, sum[0], acc[2]));
    acc[3] = fmaf(sb, d[3], fmaf(bb, sum[1], acc[3]));
}

constexpr float kTwo24 = 16777216.0f;

__device__ __forceinline__ uint2 ldg_u2(const uint32_t *p) {
    return __ldg(reinterpret_cast<const uint2 *>(p));
}

// Two 16-byte loads of a fragment-ordered fp16 token row (plain cached loads: the
// rows may have been written earlier in the same kernel, before a flag was read).
__device__ __forceinline__ void load_b(uint32_t (&xb)[8], const __half *row16) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row16);
    uint4 v0 = p[0], v1 = p[1];
    xb[0] = v0.x; xb[1] = v0.y; xb[2] = v0.z; xb[3] = v0.w;
    xb[4] = v1.x; xb[5] = v1.y; xb[6] = v1.z; xb[7] = v1.w;
}

__device__ __forceinline__ void zero_b(uint32_t (&xb)[8]) {
#pragma unroll
    for (int i = 0; i < 8; i++) xb[i] = 0u;
}

// Sixteen fp32 columns 16c..16c+15 of one group -> the lane's 8 B registers;
// scaled elementwise by the matching columns of w when w is non-null.
__device__ __forceinline__ void load_b_f32(uint32_t (&xb)[8], const float *cols16, const float *w = nullptr) {
    const float4 *p = reinterpret_cast<const float4 *>(cols16);
    const float4 *q = reinterpret_cast<const float4 *>(w);
#pragma unroll
    for (int j = 0; j < 2; j++) {
        float4 lo = __ldg(p + 2 * j), hi = __ldg(p + 2 * j + 1);  // columns 8j..8j+3, 8j+4..8j+7
        if (q) {
            const float4 wl = __ldg(q + 2 * j), wh = __ldg(q + 2 * j + 1);
            lo = make_float4(lo.x * wl.x, lo.y * wl.y, lo.z * wl.z, lo.w * wl.w);
            hi = make_float4(hi.x * wh.x, hi.y * wh.y, hi.z * wh.z, hi.w * wh.w);
        }
        __half2 r0 = __floats2half2_rn(lo.x, hi.x);
        __half2 r1 = __floats2half2_rn(lo.y, hi.y);
        __half2 r2 = __floats2half2_rn(lo.z, hi.z);
        __half2 r3 = __floats2half2_rn(lo.w, hi.w);
        xb[4 * j + 0] = *reinterpret_cast<uint32_t *>(&r0);
        xb[4 * j + 1] = *reinterpret_cast<uint32_t *>(&r1);
        xb[4 * j + 2] = *reinterpret_cast<uint32_t *>(&r2);
        xb[4 * j + 3] = *reinterpret_cast<uint32_t *>(&r3);
    }
}

}  // namespace moe
