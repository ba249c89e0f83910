// tile.cuh -- the tile layout of an expert blob, and the kernel that builds it
// from the MLX row-major layout.
//
// A tile is 16 matrix rows by one quantisation group (64 columns): 512 bytes of
// 4-bit codes in the register order of an m16n8k16 A fragment, then 64 bytes of
// fp16 scale/bias.  For row pair r = 0..7 and column lane c = 0..3, lane
// L = 4r + c holds at bytes 16L..16L+15 the words 2c, 2c+1 of the group in row
// a(r), then the same two words of row b(r); bytes 512+8r..512+8r+7 hold
// (scale a, bias a, scale b, bias b).  One warp therefore reads a tile as one
// 128-bit load per lane (512 contiguous bytes) plus one 64-bit load of its pair's
// scales, and the tile sizes are exactly 4.5 bits per weight.
//
//   gate/up part (byte 0):  tile (it, g) at 576 (it G + g), a(r) = gate row 8it + r,
//                           b(r) = up row 8it + r            (it < I/8, g < G = H/64)
//   down part:              tile (rt, g) at gu_bytes + 576 (rt Gi + g),
//                           a(r) = row 16rt + r, b(r) = row 16rt + 8 + r
//                                                            (rt < H/16, g < Gi = I/64)
// Pairing each gate row with its up row in one tile lets one MMA produce both
// halves of a GeGLU unit in the same lane.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kTileBytes = 576;

struct TileLayout {
    int G, Gi;         // groups per gate/up row (H/64) and per down row (I/64)
    int Ti, R;         // gate/up tiles per row block (I/8), down row tiles (H/16)
    size_t gu_bytes;   // size of the gate/up part = offset of the down part
    size_t total;
};

__host__ __device__ inline TileLayout tile_layout(int H, int I) {
    TileLayout t;
    t.G = H / kGroup;
    t.Gi = I / kGroup;
    t.Ti = I / 8;
    t.R = H / 16;
    t.gu_bytes = (size_t)kTileBytes * t.Ti * t.G;
    t.total = t.gu_bytes + (size_t)kTileBytes * t.R * t.Gi;
    return t;
}

// One thread per (tile, lane): copies 4 code words and, for lanes with c == 0,
// the 8-byte scale/bias entry.  src is an MLX-layout blob (BlobLayout), dst a
// tile-layout blob of the same expert.
__global__ void k_tile_expert(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int H, int I) {
    const BlobLayout L = blob_layout(H, I);
    const TileLayout T = tile_layout(H, I);
    const long long ntiles = (long long)T.Ti * T.G + (long long)T.R * T.Gi;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= ntiles * 32) return;
    const long long tile = gid >> 5;
    const int lane = (int)(gid & 31), r = lane >> 2, c = lane & 3;
    int ra, rb, g, wpr, groups;
    const uint32_t *q;
    const uint16_t *s, *b;
    uint8_t *out;
    if (tile < (long long)T.Ti * T.G) {
        const int it = (int)(tile / T.G);
        g = (int)(tile % T.G);
        ra = 8 * it + r;
        rb = I + 8 * it + r;
        wpr = H / 8;
        groups = T.G;
        q = (const uint32_t *)(src + L.gu_q);
        s = (const uint16_t *)(src + L.gu_s);
        b = (const uint16_t *)(src + L.gu_b);
        out = dst + (size_t)kTileBytes * tile;
    } else {
        const long long dt = tile - (long long)T.Ti * T.G;
        const int rt = (int)(dt / T.Gi);
        g = (int)(dt % T.Gi);
        ra = 16 * rt + r;
        rb = 16 * rt + 8 + r;
        wpr = I / 8;
        groups = T.Gi;
        q = (const uint32_t *)(src + L.d_q);
        s = (const uint16_t *)(src + L.d_s);
        b = (const uint16_t *)(src + L.d_b);
        out = dst + T.gu_bytes + (size_t)kTileBytes * dt;
    }
    uint4 w;
    w.x = q[(size_t)ra * wpr + 8 * g + 2 * c];
    w.y = q[(size_t)ra * wpr + 8 * g + 2 * c + 1];
    w.z = q[(size_t)rb * wpr + 8 * g + 2 * c];
    w.w = q[(size_t)rb * wpr + 8 * g + 2 * c + 1];
    reinterpret_cast<uint4 *>(out)[lane] = w;
    if (c == 0) {
        uint2 e;
        e.x = (uint32_t)s[(size_t)ra * groups + g] | ((uint32_t)b[(size_t)ra * groups + g] << 16);
        e.y = (uint32_t)s[(size_t)rb * groups + g] | ((uint32_t)b[(size_t)rb * groups + g] << 16);
        reinterpret_cast<uint2 *>(out + 512)[r] = e;
    }
}

}  // namespace moe
