/*
 * moe_oracle.c -- plain, slow CPU oracle for one routed Mixture-of-Experts layer
 * over MLX-style affine group-quantised weights.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA path is checked
 * against; it is never linked into, called by, or shipped as part of the product
 * library.  Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no code, header, table or constant generator with
 * the CUDA path.
 *
 * What it computes, and where the pages fix it (pages are cited by title and
 * section):
 *   - Affine 4-bit weights, group 64, w = scale*q + bias; the router at 8 bits
 *     ("TurboFieldfare esegue Mac Gemma 4 26B in 2 GB...", section "L'affermazione
 *     dei 2 GB trasforma la larghezza di banda dell'SSD nel nuovo vincolo";
 *     "Correr un modelo de 26.000 millones...", section "Detalles tecnicos y
 *     rendimiento").
 *   - The router picks 8 experts per token per layer, a shared expert is always
 *     used, and the outputs of both branches are combined ("Come eseguire un
 *     modello da 26 miliardi...", section "Qual e il trucco principale
 *     dell'architettura"; the remio.ai page, sections "Mac Gemma 4 26B entra nello
 *     spazio disponibile..." and "L'affermazione dei 2 GB...").
 *   - Chunked prefill of up to 128 tokens is only an efficiency device, so a chunk
 *     is defined as that many independent decodes (devtrends page, section
 *     "Prestazioni nel mondo reale"; remio.ai page, same section as above).
 *   - A 16-slot least-frequently-used expert cache per layer (devtrends page,
 *     "Qual e il trucco principale..."; remio.ai page, "Mac Gemma 4 26B entra...").
 *
 * Readings taken where the pages are silent (each one is listed in the design
 * notes of the repository):
 *   - GeGLU with the tanh form of GELU, h = gelu(gate) * up.
 *   - Gates are the softmax over the selected logits; shared expert weight 1.
 *   - Top-k order: larger logit first, equal logits -> lower expert index; the
 *     selection is made on the logits rounded to fp32 (the precision the kernels
 *     decide in); sums are fp64.
 *   - MLX nibble order: element j of a row lives in bits 4*(j%8) of 32-bit word
 *     j/8 (8-bit: bits 8*(j%4) of word j/4); scale and bias are fp16, one pair per
 *     group of 64 consecutive elements of a row.
 *   - The quantiser (encoding, used only to build test data): per group
 *     s = fp16((max-min)/(2^bits-1)), b = fp16(min), q = clamp(rint((w-b)/s)),
 *     all in fp32; s == 0 -> q = 0.
 *   - In-cache LFU, ties broken by (count, last use, slot); see orc_lfu_step.
 *
 * Arithmetic: every dot product is summed in fp64 in ascending index order.  The
 * only library primitives are tanh and exp from libm and the compiler's
 * IEEE binary16 conversions.  OpenMP splits independent output rows across
 * threads; no sum is reordered.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ECAPACITY 3

#define GROUP 64

/* ---- IEEE binary16 <-> host floats (compiler-provided _Float16, RNE) ---- */

double orc_half_to_double(uint16_t h) {
    _Float16 v;
    memcpy(&v, &h, 2);
    return (double)v;
}

static float half_to_float(uint16_t h) {
    _Float16 v;
    memcpy(&v, &h, 2);
    return (float)v;
}

uint16_t orc_float_to_half(float f) {
    _Float16 v = (_Float16)f;
    uint16_t h;
    memcpy(&h, &v, 2);
    return h;
}

/* ---- affine code extraction (MLX layout) ---- */

/* Code q of element j of one row whose packed words start at `row`. */
static unsigned code_at(const uint32_t *row, int j, int bits) {
    if (bits == 4) return (row[j / 8] >> (4 * (j % 8))) & 0xFu;
    return (row[j / 4] >> (8 * (j % 4))) & 0xFFu;
}

static int words_per_row(int K, int bits) { return K * bits / 32; }

/* w[n][j] = scale[n][j/64] * q[n][j] + bias[n][j/64], in fp64. */
static double deq_at(const uint32_t *q, const uint16_t *s, const uint16_t *b, int K, int bits,
                     int n, int j) {
    const uint32_t *row = q + (size_t)n * words_per_row(K, bits);
    size_t gi = (size_t)n * (K / GROUP) + j / GROUP;
    return orc_half_to_double(s[gi]) * (double)code_at(row, j, bits) + orc_half_to_double(b[gi]);
}

static int shape_ok(int N, int K, int bits) {
    return N >= 0 && K > 0 && K % GROUP == 0 && (bits == 4 || bits == 8);
}

/* Dense dequantisation of an N x K matrix into out[n*K + j]. */
int orc_dequant(const uint32_t *q, const uint16_t *s, const uint16_t *b, int N, int K, int bits,
                double *out) {
    if (!shape_ok(N, K, bits)) return ORC_EINVAL;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++)
        for (int j = 0; j < K; j++) out[(size_t)n * K + j] = deq_at(q, s, b, K, bits, n, j);
    return ORC_OK;
}

/* Encoding used to build test data: min/max affine quantiser, fp32 arithmetic. */
int orc_quantise(const float *w, int N, int K, int bits, uint32_t *q, uint16_t *s, uint16_t *b) {
    if (!shape_ok(N, K, bits)) return ORC_EINVAL;
    const unsigned qmax = (1u << bits) - 1u;
    const int wpr = words_per_row(K, bits);
    const int G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        uint32_t *row = q + (size_t)n * wpr;
        memset(row, 0, sizeof(uint32_t) * (size_t)wpr);
        for (int g = 0; g < G; g++) {
            const float *v = w + (size_t)n * K + (size_t)g * GROUP;
            float mn = v[0], mx = v[0];
            for (int j = 1; j < GROUP; j++) {
                if (v[j] < mn) mn = v[j];
                if (v[j] > mx) mx = v[j];
            }
            float range = mx - mn;
            float step = range / (float)qmax;
            uint16_t sh = orc_float_to_half(step);
            uint16_t bh = orc_float_to_half(mn);
            s[(size_t)n * G + g] = sh;
            b[(size_t)n * G + g] = bh;
            float sf = half_to_float(sh);
            float bf = half_to_float(bh);
            for (int j = 0; j < GROUP; j++) {
                unsigned code = 0;
                if (sf != 0.0f) {
                    float t = rintf((v[j] - bf) / sf);
                    if (t < 0.0f) t = 0.0f;
                    if (t > (float)qmax) t = (float)qmax;
                    code = (unsigned)t;
                }
                int col = g * GROUP + j;
                if (bits == 4)
                    row[col / 8] |= (uint32_t)code << (4 * (col % 8));
                else
                    row[col / 4] |= (uint32_t)code << (8 * (col % 4));
            }
        }
    }
    return ORC_OK;
}

/* y[t][n] = sum_j w[n][j] * x[t][j], fp64, j ascending. */
int orc_qgemv(const uint32_t *q, const uint16_t *s, const uint16_t *b, int N, int K, int bits,
              const float *x, int T, double *y) {
    if (!shape_ok(N, K, bits) || T < 0) return ORC_EINVAL;
    for (int t = 0; t < T; t++) {
#pragma omp parallel for schedule(static)
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (int j = 0; j < K; j++) acc += deq_at(q, s, b, K, bits, n, j) * (double)x[(size_t)t * K + j];
            y[(size_t)t * N + n] = acc;
        }
    }
    return ORC_OK;
}

/* ---- router: logits, top-k, softmax gates ---- */

/*
 * For each token t: logit[e] = sum_j Wr[e][j] x[t][j] (+ bias[e] if given), fp64.
 * The k experts chosen are the k largest logits rounded to fp32, larger first,
 * equal values -> lower index first.  Gate g_k = exp(l_k - l_max) / sum exp(...)
 * over the chosen k, using the fp64 logits.
 */
int orc_route(const uint32_t *rq, const uint16_t *rs, const uint16_t *rb, int E, int H,
              const float *x, int T, const float *logit_bias, int topk, double *logits_out,
              int32_t *idx, double *gate) {
    if (!shape_ok(E, H, 8) || E <= 0 || topk <= 0 || topk > E || T < 0) return ORC_EINVAL;
    double *l = (double *)malloc(sizeof(double) * (size_t)E);
    float *lf = (float *)malloc(sizeof(float) * (size_t)E);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!l || !lf || !taken) {
        free(l); free(lf); free(taken);
        return ORC_EINVAL;
    }
    for (int t = 0; t < T; t++) {
#pragma omp parallel for schedule(static)
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int j = 0; j < H; j++) acc += deq_at(rq, rs, rb, H, 8, e, j) * (double)x[(size_t)t * H + j];
            if (logit_bias) acc += (double)logit_bias[e];
            l[e] = acc;
        }
        for (int e = 0; e < E; e++) {
            lf[e] = (float)l[e];
            taken[e] = 0;
            if (logits_out) logits_out[(size_t)t * E + e] = l[e];
        }
        /* selection: repeatedly take the best remaining (value desc, index asc) */
        for (int k = 0; k < topk; k++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e]) continue;
                if (best < 0 || lf[e] > lf[best]) best = e;
            }
            taken[best] = 1;
            idx[(size_t)t * topk + k] = best;
        }
        double m = l[idx[(size_t)t * topk]];
        for (int k = 1; k < topk; k++) {
            double v = l[idx[(size_t)t * topk + k]];
            if (v > m) m = v;
        }
        double z = 0.0;
        for (int k = 0; k < topk; k++) z += exp(l[idx[(size_t)t * topk + k]] - m);
        for (int k = 0; k < topk; k++) gate[(size_t)t * topk + k] = exp(l[idx[(size_t)t * topk + k]] - m) / z;
    }
    free(l);
    free(lf);
    free(taken);
    return ORC_OK;
}

/* ---- expert blob layout ----
 * One expert (gate/up rows [gate; up] = 2I x H, then down H x I) is one contiguous
 * blob; each sub-array starts on a 256-byte boundary:
 *   gu_q [2I][H/8] u32 | gu_s [2I][H/64] f16 | gu_b [2I][H/64] f16 |
 *   d_q  [H][I/8]  u32 | d_s  [H][I/64]  f16 | d_b  [H][I/64]  f16
 */
static size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

typedef struct {
    size_t gu_q, gu_s, gu_b, d_q, d_s, d_b, total;
} blob_layout;

static blob_layout layout_of(int H, int I) {
    blob_layout L;
    size_t off = 0;
    L.gu_q = off; off = up256(off + (size_t)2 * I * H / 2);
    L.gu_s = off; off = up256(off + (size_t)2 * I * (H / GROUP) * 2);
    L.gu_b = off; off = up256(off + (size_t)2 * I * (H / GROUP) * 2);
    L.d_q = off;  off = up256(off + (size_t)H * I / 2);
    L.d_s = off;  off = up256(off + (size_t)H * (I / GROUP) * 2);
    L.d_b = off;  off = up256(off + (size_t)H * (I / GROUP) * 2);
    L.total = off;
    return L;
}

size_t orc_expert_blob_bytes(int H, int I) { return layout_of(H, I).total; }

void orc_expert_blob_offsets(int H, int I, size_t *off6) {
    blob_layout L = layout_of(H, I);
    off6[0] = L.gu_q; off6[1] = L.gu_s; off6[2] = L.gu_b;
    off6[3] = L.d_q;  off6[4] = L.d_s;  off6[5] = L.d_b;
}

/*
 * The library's tile layout of an expert (a storage order of the same codes,
 * scales and biases; the pages give no layout, this one is the library's own).
 * A tile is 16 matrix rows (an "a" row and a "b" row for each r = 0..7) by one
 * group of 64 columns, 576 bytes:
 *   bytes 16L..16L+15 (lane L = 4r + c, r = 0..7, c = 0..3): four 32-bit words,
 *     words 2c and 2c+1 of the group in row a(r), then the same two words of
 *     row b(r)  (word w of a group holds columns 8w..8w+7, MLX nibble order);
 *   bytes 512 + 8r .. 512 + 8r + 7: four fp16 values, scale and bias of row a(r)
 *     for this group, then scale and bias of row b(r).
 * Gate/up part, at byte 0: tile (it, g), it = 0..I/8-1, g = 0..H/64-1, at
 *   576 (it (H/64) + g), with a(r) = gate row 8 it + r and b(r) = up row 8 it + r
 *   (row I + 8 it + r of the [2I][H] gate/up matrix).
 * Down part, at byte 576 (I/8)(H/64): tile (rt, g), rt = 0..H/16-1,
 *   g = 0..I/64-1, at 576 (rt (I/64) + g) from the part's start, with
 *   a(r) = row 16 rt + r and b(r) = row 16 rt + 8 + r of the [H][I] down matrix.
 */
#define TILE_BYTES 576

size_t orc_tile_blob_bytes(int H, int I) {
    if (H <= 0 || I <= 0 || H % 128 || I % GROUP) return 0;
    return (size_t)TILE_BYTES * ((size_t)(I / 8) * (H / GROUP) + (size_t)(H / 16) * (I / GROUP));
}

/* Copies one tile's words and scale/bias pairs back to MLX row-major arrays. */
static void untile_one(const uint8_t *tile, int g, const int rows_a[8], const int rows_b[8],
                       uint32_t *q, uint16_t *s, uint16_t *b, int words_per_row, int groups) {
    for (int L = 0; L < 32; L++) {
        const int r = L / 4, c = L % 4;
        const uint32_t *w = (const uint32_t *)(tile + 16 * L);
        q[(size_t)rows_a[r] * words_per_row + 8 * g + 2 * c] = w[0];
        q[(size_t)rows_a[r] * words_per_row + 8 * g + 2 * c + 1] = w[1];
        q[(size_t)rows_b[r] * words_per_row + 8 * g + 2 * c] = w[2];
        q[(size_t)rows_b[r] * words_per_row + 8 * g + 2 * c + 1] = w[3];
    }
    for (int r = 0; r < 8; r++) {
        const uint16_t *h = (const uint16_t *)(tile + 512 + 8 * r);
        s[(size_t)rows_a[r] * groups + g] = h[0];
        b[(size_t)rows_a[r] * groups + g] = h[1];
        s[(size_t)rows_b[r] * groups + g] = h[2];
        b[(size_t)rows_b[r] * groups + g] = h[3];
    }
}

/* Tile-layout blob -> MLX-layout blob (orc_expert_blob_bytes(H, I) bytes). */
int orc_untile_expert(const uint8_t *tiled, int H, int I, uint8_t *blob) {
    if (!orc_tile_blob_bytes(H, I)) return ORC_EINVAL;
    blob_layout L = layout_of(H, I);
    memset(blob, 0, L.total);
    const int G = H / GROUP, Gi = I / GROUP;
    uint32_t *guq = (uint32_t *)(blob + L.gu_q);
    uint16_t *gus = (uint16_t *)(blob + L.gu_s), *gub = (uint16_t *)(blob + L.gu_b);
    uint32_t *dq = (uint32_t *)(blob + L.d_q);
    uint16_t *ds = (uint16_t *)(blob + L.d_s), *db = (uint16_t *)(blob + L.d_b);
    int ra[8], rb[8];
    for (int it = 0; it < I / 8; it++)
        for (int g = 0; g < G; g++) {
            for (int r = 0; r < 8; r++) {
                ra[r] = 8 * it + r;
                rb[r] = I + 8 * it + r;
            }
            untile_one(tiled + (size_t)TILE_BYTES * ((size_t)it * G + g), g, ra, rb, guq, gus, gub,
                       H / 8, G);
        }
    const uint8_t *down = tiled + (size_t)TILE_BYTES * (I / 8) * G;
    for (int rt = 0; rt < H / 16; rt++)
        for (int g = 0; g < Gi; g++) {
            for (int r = 0; r < 8; r++) {
                ra[r] = 16 * rt + r;
                rb[r] = 16 * rt + 8 + r;
            }
            untile_one(down + (size_t)TILE_BYTES * ((size_t)rt * Gi + g), g, ra, rb, dq, ds, db,
                       I / 8, Gi);
        }
    return ORC_OK;
}

/* GELU, tanh form: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))). */
double orc_gelu_tanh(double z) {
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)));
}

/*
 * One expert applied to one token:  a = Wg x, u = Wu x, h = gelu(a) * u,
 * out = Wd h.  Optionally returns h.
 */
int orc_expert(const uint8_t *blob, int H, int I, const float *x, double *out, double *h_out) {
    if (!shape_ok(2 * I, H, 4) || !shape_ok(H, I, 4)) return ORC_EINVAL;
    blob_layout L = layout_of(H, I);
    const uint32_t *guq = (const uint32_t *)(blob + L.gu_q);
    const uint16_t *gus = (const uint16_t *)(blob + L.gu_s);
    const uint16_t *gub = (const uint16_t *)(blob + L.gu_b);
    const uint32_t *dq = (const uint32_t *)(blob + L.d_q);
    const uint16_t *ds = (const uint16_t *)(blob + L.d_s);
    const uint16_t *db = (const uint16_t *)(blob + L.d_b);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    if (!h) return ORC_EINVAL;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < I; i++) {
        double a = 0.0, u = 0.0;
        for (int j = 0; j < H; j++) a += deq_at(guq, gus, gub, H, 4, i, j) * (double)x[j];
        for (int j = 0; j < H; j++) u += deq_at(guq, gus, gub, H, 4, I + i, j) * (double)x[j];
        h[i] = orc_gelu_tanh(a) * u;
    }
#pragma omp parallel for schedule(static)
    for (int n = 0; n < H; n++) {
        double acc = 0.0;
        for (int i = 0; i < I; i++) acc += deq_at(dq, ds, db, I, 4, n, i) * h[i];
        out[n] = acc;
    }
    if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)I);
    free(h);
    return ORC_OK;
}

/*
 * The layer.  For each token t:
 *   (idx, g) = route(x_t);  y_t = sum_k g_k * expert_{idx_k}(x_t) + shared(x_t)
 * and, if `residual` is set, y_t += x_t.  `experts[e]` is expert e's blob (only
 * the routed ones are read; a routed NULL is an error).  idx/gate outputs are
 * optional.
 */
int orc_moe_layer(int H, int E, int topk, int I, int Is, const uint32_t *rq, const uint16_t *rs,
                  const uint16_t *rb, const uint8_t *const *experts, const uint8_t *shared,
                  const float *x, int T, const float *logit_bias, int residual, double *y,
                  int32_t *idx_out, double *gate_out) {
    if (T < 0 || topk <= 0 || topk > E || !shape_ok(2 * I, H, 4) || !shape_ok(2 * Is, H, 4) ||
        !shape_ok(H, I, 4) || !shape_ok(H, Is, 4) || !shared)
        return ORC_EINVAL;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)topk);
    double *g = (double *)malloc(sizeof(double) * (size_t)topk);
    double *o = (double *)malloc(sizeof(double) * (size_t)H);
    int rc = ORC_OK;
    if (!idx || !g || !o) { rc = ORC_EINVAL; goto done; }
    for (int t = 0; t < T; t++) {
        const float *xt = x + (size_t)t * H;
        double *yt = y + (size_t)t * H;
        rc = orc_route(rq, rs, rb, E, H, xt, 1, logit_bias, topk, NULL, idx, g);
        if (rc) goto done;
        for (int n = 0; n < H; n++) yt[n] = 0.0;
        for (int k = 0; k < topk; k++) {
            const uint8_t *blob = experts[idx[k]];
            if (!blob) { rc = ORC_EINVAL; goto done; }
            rc = orc_expert(blob, H, I, xt, o, NULL);
            if (rc) goto done;
            for (int n = 0; n < H; n++) yt[n] += g[k] * o[n];
        }
        rc = orc_expert(shared, H, Is, xt, o, NULL);
        if (rc) goto done;
        for (int n = 0; n < H; n++) yt[n] += o[n];
        if (residual)
            for (int n = 0; n < H; n++) yt[n] += (double)xt[n];
        if (idx_out) memcpy(idx_out + (size_t)t * topk, idx, sizeof(int32_t) * (size_t)topk);
        if (gate_out) memcpy(gate_out + (size_t)t * topk, g, sizeof(double) * (size_t)topk);
    }
done:
    free(idx);
    free(g);
    free(o);
    return rc;
}

/*
 * RMSNorm of T rows of H values:
 *   out[t][j] = x[t][j] * g[j] / sqrt(mean over j of x[t][j]^2 + eps).
 * The pages list an RMSNorm kernel among the engine's own kernels ("Come eseguire
 * un modello da 26 miliardi...", section "Senza dipendenze da llama.cpp e MLX";
 * "TurboFieldfare: движок с открытым кодом...", main technical paragraph) without
 * its formula; this is the plain root-mean-square normalisation (Zhang and
 * Sennrich, 2019): no mean subtraction, g applied as is.  The MoE block around it
 * is y = x + MoE(RMSNorm(x)) (pre-norm with the residual).  fp64, the sum of
 * squares in index order.
 */
int orc_rmsnorm(const float *x, const float *g, double eps, int T, int H, double *out) {
    if (T < 0 || H <= 0 || eps < 0.0 || !x || !g || !out) return ORC_EINVAL;
    for (int t = 0; t < T; t++) {
        const float *xt = x + (size_t)t * H;
        double ss = 0.0;
        for (int j = 0; j < H; j++) ss += (double)xt[j] * (double)xt[j];
        const double rms = sqrt(ss / (double)H + eps);
        for (int j = 0; j < H; j++) out[(size_t)t * H + j] = rms > 0.0 ? (double)xt[j] * (double)g[j] / rms : 0.0;
    }
    return ORC_OK;
}

/*
 * Token sampling from one row of V logits (the engine's defaults are temperature
 * 0.2, top-K 64, top-P 0.95: "Correr un modelo de 26.000 millones...", section
 * "Como empezar"; the pages give the parameters, not the procedure).  The plain
 * reading, in this order:
 *   1. top-K: the K largest logits, larger first, equal -> lower index (K <= 0 or
 *      K >= V keeps all V);
 *   2. softmax of the kept logits at the temperature: p_i = exp((l_i - l_max) / temp)
 *      / sum, in fp64;
 *   3. top-P: the kept tokens in that order; keep the shortest prefix whose
 *      cumulative probability reaches top_p (at least one token; top_p >= 1 keeps
 *      all);
 *   4. draw: with the caller's uniform u in [0, 1), the first kept token j whose
 *      cumulative probability exceeds u times the prefix's total.
 * temperature <= 0 is greedy: the largest logit, equal -> lower index.
 * Writes the token; *margin (if non-null) receives the smallest distance, in
 * units of the prefix total, between u * total and a cumulative sum, or between
 * top_p and a cumulative probability -- the decisions a rounding could flip.
 */
typedef struct {
    float v;
    int i;
} orc_vi;

static int vi_desc(const void *a, const void *b) {
    const orc_vi *x = (const orc_vi *)a, *y = (const orc_vi *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return x->i < y->i ? -1 : (x->i > y->i);
}

int orc_sample(const float *logits, int V, double temperature, int top_k, double top_p, double u,
               int32_t *token, double *margin) {
    if (V <= 0 || !logits || !token || !(u >= 0.0 && u < 1.0)) return ORC_EINVAL;
    orc_vi *s = (orc_vi *)malloc(sizeof(orc_vi) * (size_t)V);
    double *c = (double *)malloc(sizeof(double) * (size_t)V);
    if (!s || !c) {
        free(s);
        free(c);
        return ORC_EINVAL;
    }
    for (int i = 0; i < V; i++) {
        s[i].v = logits[i];
        s[i].i = i;
    }
    qsort(s, (size_t)V, sizeof(orc_vi), vi_desc);
    if (temperature <= 0.0) {
        *token = s[0].i;
        if (margin) *margin = 1.0;
        free(s);
        free(c);
        return ORC_OK;
    }
    const int K = (top_k <= 0 || top_k >= V) ? V : top_k;
    double total = 0.0;
    for (int j = 0; j < K; j++) {
        total += exp(((double)s[j].v - (double)s[0].v) / temperature);
        c[j] = total;
    }
    int n = K;
    double m = 1.0;
    if (top_p < 1.0) {
        for (int j = 0; j < K; j++) {
            const double d = c[j] / total - top_p;
            if (fabs(d) < m) m = fabs(d);
            if (d >= 0.0) {
                n = j + 1;
                break;
            }
        }
    }
    const double thr = u * c[n - 1];
    int pick = n - 1;
    for (int j = 0; j < n; j++) {
        const double d = (c[j] - thr) / c[n - 1];
        if (fabs(d) < m) m = fabs(d);
        if (c[j] > thr) {
            pick = j;
            break;
        }
    }
    *token = s[pick].i;
    if (margin) *margin = m;
    free(s);
    free(c);
    return ORC_OK;
}

/* ---- per-layer LFU expert cache ----
 *
 * One call = one step with the request list R (router order; for a batch, the
 * union of the tokens' choices in first-appearance order).
 *   1. every requested expert already resident is a hit: count += 1, last = step;
 *   2. every requested expert not resident, in request order, is a miss: it goes
 *      into the lowest-numbered empty slot, else it evicts, among the slots whose
 *      expert is not in R, the one with the smallest (count, last, slot); it is
 *      installed with count = 1, last = step.  The evicted expert's count is
 *      forgotten.
 * |R| > slots is ORC_ECAPACITY; an index outside [0, E) or a repeated index is
 * ORC_EINVAL.  On an error nothing changes.
 */
typedef struct {
    int slots, E;
    int64_t step;
    uint64_t hits, misses;
    int32_t *expert_of_slot; /* -1 = empty */
    uint32_t *count;
    int64_t *last;
} orc_lfu;

orc_lfu *orc_lfu_create(int slots, int E) {
    if (slots <= 0 || E <= 0) return NULL;
    orc_lfu *c = (orc_lfu *)calloc(1, sizeof(orc_lfu));
    if (!c) return NULL;
    c->slots = slots;
    c->E = E;
    c->expert_of_slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)slots);
    c->count = (uint32_t *)calloc((size_t)slots, sizeof(uint32_t));
    c->last = (int64_t *)calloc((size_t)slots, sizeof(int64_t));
    if (!c->expert_of_slot || !c->count || !c->last) {
        free(c->expert_of_slot); free(c->count); free(c->last); free(c);
        return NULL;
    }
    for (int i = 0; i < slots; i++) c->expert_of_slot[i] = -1;
    return c;
}

void orc_lfu_destroy(orc_lfu *c) {
    if (!c) return;
    free(c->expert_of_slot);
    free(c->count);
    free(c->last);
    free(c);
}

static int slot_of(const orc_lfu *c, int e) {
    for (int i = 0; i < c->slots; i++)
        if (c->expert_of_slot[i] == e) return i;
    return -1;
}

/* slot_out[r] = slot now holding request r; hit_out[r] = 1 on a hit. */
int orc_lfu_step(orc_lfu *c, const int32_t *req, int n, int32_t *slot_out, uint8_t *hit_out) {
    if (!c || n < 0) return ORC_EINVAL;
    for (int r = 0; r < n; r++) {
        if (req[r] < 0 || req[r] >= c->E) return ORC_EINVAL;
        for (int p = 0; p < r; p++)
            if (req[p] == req[r]) return ORC_EINVAL;
    }
    if (n > c->slots) return ORC_ECAPACITY;
    int64_t step = c->step;
    /* 1. hits */
    for (int r = 0; r < n; r++) {
        int s = slot_of(c, req[r]);
        hit_out[r] = (uint8_t)(s >= 0);
        if (s >= 0) {
            c->count[s] += 1;
            c->last[s] = step;
            slot_out[r] = s;
            c->hits++;
        }
    }
    /* 2. misses in request order */
    for (int r = 0; r < n; r++) {
        if (hit_out[r]) continue;
        int victim = -1;
        for (int i = 0; i < c->slots; i++)
            if (c->expert_of_slot[i] < 0) { victim = i; break; }
        if (victim < 0) {
            for (int i = 0; i < c->slots; i++) {
                int e = c->expert_of_slot[i];
                int requested = 0;
                for (int p = 0; p < n; p++)
                    if (req[p] == e) requested = 1;
                if (requested) continue;
                if (victim < 0 || c->count[i] < c->count[victim] ||
                    (c->count[i] == c->count[victim] && c->last[i] < c->last[victim]))
                    victim = i;
            }
        }
        /* victim >= 0 always: n <= slots and requested experts occupy < slots. */
        c->expert_of_slot[victim] = req[r];
        c->count[victim] = 1;
        c->last[victim] = step;
        slot_out[r] = victim;
        c->misses++;
    }
    c->step++;
    return ORC_OK;
}

void orc_lfu_state(const orc_lfu *c, int32_t *expert_of_slot, uint32_t *count, int64_t *last,
                   uint64_t *hits, uint64_t *misses) {
    for (int i = 0; i < c->slots; i++) {
        if (expert_of_slot) expert_of_slot[i] = c->expert_of_slot[i];
        if (count) count[i] = c->count[i];
        if (last) last[i] = c->last[i];
    }
    if (hits) *hits = c->hits;
    if (misses) *misses = c->misses;
}

/* ---- attention block with an FP16 key/value cache ---- */

/*
 * One attention block over T consecutive tokens of one sequence, at positions
 * pos .. pos+T-1.  The pages name the pieces: the engine's own kernels compute a
 * quantised GEMV, attention, RMSNorm and RoPE; the projections are 4-bit MLX affine
 * weights; the key/value cache is FP16, a bounded ring for the 25 sliding-window
 * layers and a linear store for the 5 full-attention layers, 4096 tokens in the
 * measured setup ("TurboFieldfare: движок с открытым кодом...", main technical
 * paragraph; "TurboFieldfare esegue Mac Gemma 4 26B in 2 GB...", section "Mac Gemma 4
 * 26B entra nello spazio disponibile...").  They give no shapes or formulas, so the
 * plain readings (each listed in the design notes) are:
 *   - tokens are taken one after another; each is written into the cache before
 *     it attends, so it sees itself;
 *   - xn = RMSNorm(x) when norm_w is given (pre-norm), else x;
 *   - [q; k; v] = Wqkv xn, Wqkv [(nq + 2 nkv) d][H] with the nq query heads, then
 *     the nkv key heads, then the nkv value heads, d rows each;
 *   - RoPE, rotate-half pairing: for i < d/2 and angle a = p * theta^(-2i/d),
 *     (u_i, u_{i+d/2}) -> (u_i cos a - u_{i+d/2} sin a, u_{i+d/2} cos a + u_i sin a),
 *     applied to every query and key head at the token's own position p;
 *   - the cache holds the rotated keys and the values rounded to binary16, laid
 *     out [nkv][kv_len][d]; a sliding layer (window > 0) keeps position j in slot
 *     j mod kv_len and attends to positions max(0, p - window + 1) .. p; a full
 *     layer (window == 0) keeps j in slot j and attends to 0 .. p;
 *   - query head h reads key/value head h / (nq / nkv) (grouped queries);
 *     scores s_j = scale * q_h . k_j, weights softmax(s) over the attended
 *     positions, o_h = sum_j w_j v_j;
 *   - y = Wo o (+ x when residual), Wo [H][nq d].
 * Everything in fp64 except the cache, which is binary16 as the pages state.
 * The cache arrays are read and updated in place; attn_out (optional) receives
 * o [T][nq d].
 */
static double pow_neg(double theta, int i2, int d) { return pow(theta, -(double)i2 / (double)d); }

static void rope_fp64(double *u, int d, int p, double theta) {
    for (int i = 0; i < d / 2; i++) {
        const double a = (double)p * pow_neg(theta, 2 * i, d);
        const double c = cos(a), s = sin(a);
        const double lo = u[i], hi = u[i + d / 2];
        u[i] = lo * c - hi * s;
        u[i + d / 2] = hi * c + lo * s;
    }
}

static uint16_t double_to_half(double v) {
    _Float16 h = (_Float16)v;
    uint16_t r;
    memcpy(&r, &h, 2);
    return r;
}

int orc_attn_step(int H, int nq, int nkv, int d, int window, int kv_len, double theta, double scale,
                  const uint32_t *wqkv_q, const uint16_t *wqkv_s, const uint16_t *wqkv_b,
                  const uint32_t *wo_q, const uint16_t *wo_s, const uint16_t *wo_b,
                  const float *norm_w, double eps, int residual, uint16_t *k_cache, uint16_t *v_cache,
                  const float *x, int T, int pos, double *y, double *attn_out) {
    if (H <= 0 || H % GROUP || nq <= 0 || nkv <= 0 || nq % nkv || d <= 0 || d % 2 || (nq * d) % GROUP ||
        window < 0 || kv_len <= 0 || T < 0 || pos < 0 || !k_cache || !v_cache || !x || !y || theta <= 0.0)
        return ORC_EINVAL;
    if (window > 0 ? kv_len < window : pos + T > kv_len) return ORC_ECAPACITY;
    const int G = nq / nkv, nqkv = (nq + 2 * nkv) * d, no = nq * d;
    double *xn = malloc(sizeof(double) * H), *qkv = malloc(sizeof(double) * nqkv);
    double *o = malloc(sizeof(double) * no), *sc = malloc(sizeof(double) * (size_t)(pos + T));
    if (!xn || !qkv || !o || !sc) {
        free(xn); free(qkv); free(o); free(sc);
        return ORC_EINVAL;
    }
    for (int t = 0; t < T; t++) {
        const int p = pos + t;
        const float *xt = x + (size_t)t * H;
        if (norm_w) {
            double ss = 0.0;
            for (int j = 0; j < H; j++) ss += (double)xt[j] * (double)xt[j];
            const double rms = sqrt(ss / (double)H + eps);
            for (int j = 0; j < H; j++) xn[j] = rms > 0.0 ? (double)xt[j] * (double)norm_w[j] / rms : 0.0;
        } else {
            for (int j = 0; j < H; j++) xn[j] = (double)xt[j];
        }
#pragma omp parallel for schedule(static)
        for (int n = 0; n < nqkv; n++) {
            double acc = 0.0;
            for (int j = 0; j < H; j++) acc += deq_at(wqkv_q, wqkv_s, wqkv_b, H, 4, n, j) * xn[j];
            qkv[n] = acc;
        }
        for (int h = 0; h < nq + nkv; h++) rope_fp64(qkv + (size_t)h * d, d, p, theta);
        const int slot = window > 0 ? p % kv_len : p;
        for (int g = 0; g < nkv; g++)
            for (int i = 0; i < d; i++) {
                const size_t at = ((size_t)g * kv_len + slot) * d + i;
                k_cache[at] = double_to_half(qkv[(size_t)(nq + g) * d + i]);
                v_cache[at] = double_to_half(qkv[(size_t)(nq + nkv + g) * d + i]);
            }
        const int lo = window > 0 ? (p - window + 1 > 0 ? p - window + 1 : 0) : 0;
        for (int h = 0; h < nq; h++) {
            const int g = h / G;
            const double *qh = qkv + (size_t)h * d;
            double m = -INFINITY;
            for (int j = lo; j <= p; j++) {
                const int sl = window > 0 ? j % kv_len : j;
                const uint16_t *kj = k_cache + ((size_t)g * kv_len + sl) * d;
                double s = 0.0;
                for (int i = 0; i < d; i++) s += qh[i] * orc_half_to_double(kj[i]);
                sc[j] = scale * s;
                if (sc[j] > m) m = sc[j];
            }
            double den = 0.0;
            for (int j = lo; j <= p; j++) den += exp(sc[j] - m);
            double *oh = o + (size_t)h * d;
            for (int i = 0; i < d; i++) oh[i] = 0.0;
            for (int j = lo; j <= p; j++) {
                const int sl = window > 0 ? j % kv_len : j;
                const uint16_t *vj = v_cache + ((size_t)g * kv_len + sl) * d;
                const double w = exp(sc[j] - m) / den;
                for (int i = 0; i < d; i++) oh[i] += w * orc_half_to_double(vj[i]);
            }
        }
        if (attn_out)
            for (int i = 0; i < no; i++) attn_out[(size_t)t * no + i] = o[i];
#pragma omp parallel for schedule(static)
        for (int n = 0; n < H; n++) {
            double acc = residual ? (double)xt[n] : 0.0;
            for (int i = 0; i < no; i++) acc += deq_at(wo_q, wo_s, wo_b, no, 4, n, i) * o[i];
            y[(size_t)t * H + n] = acc;
        }
    }
    free(xn); free(qkv); free(o); free(sc);
    return ORC_OK;
}
