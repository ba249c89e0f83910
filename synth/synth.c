/*
 * synth.c -- seeded synthetic inputs for the MoE layer workloads.
 *
 * Holds none of the layer's arithmetic: only random numbers.  Both the CPU oracle
 * and the CUDA path receive the arrays made here, so they see identical inputs.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; the constants are the published
 * ones).  Output c of the stream keyed by k is mix(k + (c+1) * 0x9E3779B97F4A7C15).
 *
 * Normal draws: the Irwin-Hall sum of twelve uniforms minus six (mean 0, variance
 * 1), the uniforms being the twelve 16-bit pieces of three consecutive SplitMix64
 * outputs, u = (a + 1/2) / 65536.  The value z = (S + 6)/65536 - 6, S the integer
 * sum, is exact in binary64, and sigma * z is one correctly rounded product, so the
 * same bits come out on any IEEE machine and in any thread split.  The tails stop
 * at six sigma, which these workloads do not need.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output number c (from 0) of the SplitMix64 stream seeded with key. */
uint64_t synth_splitmix64_at(uint64_t key, uint64_t c) { return mix64(key + (c + 1) * GOLDEN); }

/* Key of a sub-stream: folds the ids in one at a time. */
uint64_t synth_key(uint64_t seed, int64_t a, int64_t b, int64_t c, int64_t d) {
    uint64_t k = synth_splitmix64_at(seed, 0);
    k = synth_splitmix64_at(k ^ (uint64_t)a, 1);
    k = synth_splitmix64_at(k ^ (uint64_t)b, 2);
    k = synth_splitmix64_at(k ^ (uint64_t)c, 3);
    k = synth_splitmix64_at(k ^ (uint64_t)d, 4);
    return k;
}

static inline double irwin_hall12(uint64_t key, uint64_t i) {
    uint64_t s = 0;
    for (int m = 0; m < 3; m++) {
        uint64_t r = synth_splitmix64_at(key, 3 * i + (uint64_t)m);
        s += (r & 0xFFFF) + ((r >> 16) & 0xFFFF) + ((r >> 32) & 0xFFFF) + (r >> 48);
    }
    return ((double)(s + 6)) / 65536.0 - 6.0;
}

/* out[i] = (float)(sigma * z_{first + i}) */
void synth_normal_f32(uint64_t key, uint64_t first, int64_t n, double sigma, float *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = (float)(sigma * irwin_hall12(key, first + (uint64_t)i));
}

void synth_normal_f64(uint64_t key, uint64_t first, int64_t n, double *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = irwin_hall12(key, first + (uint64_t)i);
}

/* Seeded Fisher-Yates permutation of 0..n-1. */
void synth_permutation(uint64_t key, int n, int32_t *perm) {
    for (int i = 0; i < n; i++) perm[i] = i;
    for (int i = n - 1; i > 0; i--) {
        uint64_t r = synth_splitmix64_at(key, (uint64_t)i);
        int j = (int)(r % (uint64_t)(i + 1));
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
}

/*
 * Router logit bias that makes expert popularity Zipf(s): expert e gets rank
 * perm[e] + 1 and bias ln p_rank with p_r = r^-s / sum_r r^-s.  Adding ln p to
 * logits with Gumbel-like noise approximates drawing experts with probabilities p
 * (the Gumbel-top-k construction).
 */
void synth_zipf_bias(uint64_t key, int E, double s, float *bias) {
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!perm) return;
    synth_permutation(key, E, perm);
    double z = 0.0;
    for (int r = 1; r <= E; r++) z += pow((double)r, -s);
    for (int e = 0; e < E; e++) bias[e] = (float)(log(pow((double)(perm[e] + 1), -s) / z));
    free(perm);
}

/*
 * AR(1) token sequence: x_0 = eps_0, x_{t+1} = rho x_t + sqrt(1 - rho^2) eps_{t+1},
 * eps ~ N(0, 1) per coordinate; out is [steps][dim] fp32 (the recursion runs in fp64).
 */
void synth_ar1(uint64_t key, int steps, int dim, double rho, float *out) {
    double *cur = (double *)malloc(sizeof(double) * (size_t)dim);
    double *eps = (double *)malloc(sizeof(double) * (size_t)dim);
    if (!cur || !eps) { free(cur); free(eps); return; }
    double c = sqrt(1.0 - rho * rho);
    for (int t = 0; t < steps; t++) {
        synth_normal_f64(key, (uint64_t)t * (uint64_t)dim, dim, eps);
        for (int i = 0; i < dim; i++) {
            cur[i] = (t == 0) ? eps[i] : rho * cur[i] + c * eps[i];
            out[(size_t)t * dim + i] = (float)cur[i];
        }
    }
    free(cur);
    free(eps);
}
