/*
 * Seeded synthetic inputs for the speculative-decoding verification sampler.
 *
 * This module is shared by the tests, the benchmark and the smoke check. It produces
 * target logits, draft distributions and draft token ids with the shapes and value
 * distributions of the verification workloads; it contains none of the verifier's own
 * arithmetic (no temperature softmax of the target, no acceptance test, no race).
 *
 * Every value is a pure function of (seed, stream, row, column) through a counter-based
 * hash (the SplitMix64 output function of Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), so results do not depend on the number
 * of OpenMP threads or on the machine. Normals use the Box-Muller transform in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z)
{
    z += 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t hash4(uint64_t seed, uint64_t stream, uint64_t a, uint64_t b)
{
    return mix64(mix64(mix64(mix64(seed) + stream) + a) + b);
}

/* Uniform in the open interval (0, 1) with 53 random bits. */
static inline double u01(uint64_t h) { return ((double)(h >> 11) + 0.5) * 0x1p-53; }

static inline double normal(uint64_t seed, uint64_t stream, uint64_t row, uint64_t col)
{
    double u1 = u01(hash4(seed, stream, row, 2 * col));
    double u2 = u01(hash4(seed, stream, row, 2 * col + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

/* binary32 -> bfloat16 bits, round to nearest even (finite inputs). */
static inline uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static inline float load_logit(const void *p, int bf16, size_t idx)
{
    return bf16 ? bf16_to_f32(((const uint16_t *)p)[idx]) : ((const float *)p)[idx];
}

/* Open-interval uniforms, n of them, for small host-side draws (temperatures, draft
 * lengths, group shuffles). */
void gen_uniform(uint64_t seed, uint64_t stream, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = u01(hash4(seed, stream, 0, (uint64_t)i));
}

/*
 * Target logits [rows, V]:  sigma * N(0,1)  -  zipf_coef * ln(rank)  +  boost on n_boost tokens.
 * rank is 1 + the position of the token under a random permutation of the row (drawn by a
 * Fisher-Yates shuffle); zipf_coef = 0 disables it. The n_boost boosted tokens are distinct
 * and drawn uniformly per row. Output is bf16 bits (out_bf16 != 0) or binary32.
 */
void gen_target_logits(uint64_t seed, uint64_t stream, int64_t rows, int64_t V, double sigma,
                       double zipf_coef, int n_boost, double boost, int out_bf16, void *out)
{
#pragma omp parallel
    {
        int32_t *perm = zipf_coef != 0.0 ? (int32_t *)malloc(sizeof(int32_t) * (size_t)V) : NULL;
        int32_t *rankpos = zipf_coef != 0.0 ? (int32_t *)malloc(sizeof(int32_t) * (size_t)V) : NULL;
        int64_t boosted[64];
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < rows; ++r) {
            if (perm) {
                for (int64_t v = 0; v < V; ++v) perm[v] = (int32_t)v;
                for (int64_t k = V - 1; k > 0; --k) {
                    uint64_t h = hash4(seed, stream + 1, (uint64_t)r, (uint64_t)k);
                    int64_t j = (int64_t)(((unsigned __int128)h * (uint64_t)(k + 1)) >> 64);
                    int32_t t = perm[k];
                    perm[k] = perm[j];
                    perm[j] = t;
                }
                for (int64_t k = 0; k < V; ++k) rankpos[perm[k]] = (int32_t)k;
            }
            int nb = n_boost < 64 ? n_boost : 64;
            if (nb > V) nb = (int)V;
            for (int b = 0, attempt = 0; b < nb; ++attempt) {
                uint64_t h = hash4(seed, stream + 2, (uint64_t)r, (uint64_t)attempt);
                int64_t cand = (int64_t)(((unsigned __int128)h * (uint64_t)V) >> 64);
                int dup = 0;
                for (int c = 0; c < b; ++c) dup |= boosted[c] == cand;
                if (!dup) boosted[b++] = cand;
            }
            for (int64_t v = 0; v < V; ++v) {
                double x = sigma * normal(seed, stream, (uint64_t)r, (uint64_t)v);
                if (perm) x -= zipf_coef * log((double)rankpos[v] + 1.0);
                for (int c = 0; c < nb; ++c)
                    if (boosted[c] == v) x += boost;
                float f = (float)x;
                size_t idx = (size_t)r * (size_t)V + (size_t)v;
                if (out_bf16) ((uint16_t *)out)[idx] = f32_to_bf16(f);
                else ((float *)out)[idx] = f;
            }
        }
        free(perm);
        free(rankpos);
    }
}

/*
 * Draft distributions q [n_qrows, V] (binary32), each a softmax computed in double of the
 * draft model's logits. With independent == 0 the draft logits are the target row
 * src_row[k] plus noise_sigma * N(0,1); otherwise they are an independent
 * indep_sigma * N(0,1) draw. This is the draft model's side of the problem: the verifier
 * receives q as an input.
 */
void gen_draft_probs(uint64_t seed, uint64_t stream, int64_t n_qrows, int64_t V,
                     const int32_t *src_row, const void *target, int target_bf16,
                     double noise_sigma, int independent, double indep_sigma, float *q)
{
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 4)
        for (int64_t k = 0; k < n_qrows; ++k) {
            double zmax = -INFINITY;
            for (int64_t v = 0; v < V; ++v) {
                double n = normal(seed, stream, (uint64_t)k, (uint64_t)v);
                double x = independent
                               ? indep_sigma * n
                               : (double)load_logit(target, target_bf16,
                                                    (size_t)src_row[k] * (size_t)V + (size_t)v) +
                                     noise_sigma * n;
                z[v] = x;
                if (x > zmax) zmax = x;
            }
            double sum = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                z[v] = exp(z[v] - zmax);
                sum += z[v];
            }
            for (int64_t v = 0; v < V; ++v) q[(size_t)k * (size_t)V + (size_t)v] = (float)(z[v] / sum);
        }
        free(z);
    }
}

/* Draft token ids drawn from q by inverse CDF in double (one uniform per row). */
/* Draft logits: the target row plus N(0, noise^2) per entry, rounded to the logits' type. */
void gen_draft_logits(uint64_t seed, uint64_t stream, int64_t n_qrows, int64_t V,
                      const int32_t *src_row, const void *target, int bf16, double noise_sigma,
                      void *out)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t k = 0; k < n_qrows; ++k) {
        for (int64_t v = 0; v < V; ++v) {
            const size_t idx = (size_t)k * (size_t)V + (size_t)v;
            const double x = (double)load_logit(target, bf16, (size_t)src_row[k] * (size_t)V + (size_t)v) +
                             noise_sigma * normal(seed, stream, (uint64_t)k, (uint64_t)v);
            if (bf16)
                ((uint16_t *)out)[idx] = f32_to_bf16((float)x);
            else
                ((float *)out)[idx] = (float)x;
        }
    }
}

/* Draft ids drawn by the draft model: from softmax(dl / T) of each draft row (inverse CDF in
 * double with a uniform of (seed, stream, row)); inv_temp[k] = 1 / T of row k's request. */
void gen_sample_from_logits(uint64_t seed, uint64_t stream, int64_t n_qrows, int64_t V,
                            const void *dl, int bf16, const double *inv_temp, int32_t *ids)
{
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 8)
        for (int64_t k = 0; k < n_qrows; ++k) {
            double zmax = -INFINITY;
            for (int64_t v = 0; v < V; ++v) {
                z[v] = (double)load_logit(dl, bf16, (size_t)k * (size_t)V + (size_t)v) * inv_temp[k];
                if (z[v] > zmax) zmax = z[v];
            }
            double total = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                z[v] = exp(z[v] - zmax);
                total += z[v];
            }
            const double target = u01(hash4(seed, stream, (uint64_t)k, 0)) * total;
            double cum = 0.0;
            int64_t pick = V - 1;
            for (int64_t v = 0; v < V; ++v) {
                cum += z[v];
                if (cum > target) {
                    pick = v;
                    break;
                }
            }
            ids[k] = (int32_t)pick;
        }
        free(z);
    }
}

void gen_sample_from_q(uint64_t seed, uint64_t stream, int64_t n_qrows, int64_t V, const float *q,
                       int32_t *ids)
{
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t k = 0; k < n_qrows; ++k) {
        const float *row = q + (size_t)k * (size_t)V;
        double total = 0.0;
        int64_t last_pos = 0;
        for (int64_t v = 0; v < V; ++v) {
            total += (double)row[v];
            if (row[v] > 0.0f) last_pos = v;
        }
        double target = u01(hash4(seed, stream, (uint64_t)k, 0)) * total;
        double cum = 0.0;
        int64_t pick = last_pos;
        for (int64_t v = 0; v < V; ++v) {
            cum += (double)row[v];
            if (cum > target && row[v] > 0.0f) {
                pick = v;
                break;
            }
        }
        ids[k] = (int32_t)pick;
    }
}

/* Draft token ids without a draft distribution: with probability p_argmax the argmax of the
 * target row src_row[k] (lowest index on ties), otherwise uniform over [0, V). */
void gen_argmax_or_uniform(uint64_t seed, uint64_t stream, int64_t n_qrows, int64_t V,
                           const int32_t *src_row, const void *target, int target_bf16,
                           double p_argmax, int32_t *ids)
{
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t k = 0; k < n_qrows; ++k) {
        double coin = u01(hash4(seed, stream, (uint64_t)k, 0));
        if (coin < p_argmax) {
            size_t base = (size_t)src_row[k] * (size_t)V;
            float best = load_logit(target, target_bf16, base);
            int64_t bi = 0;
            for (int64_t v = 1; v < V; ++v) {
                float x = load_logit(target, target_bf16, base + (size_t)v);
                if (x > best) {
                    best = x;
                    bi = v;
                }
            }
            ids[k] = (int32_t)bi;
        } else {
            uint64_t h = hash4(seed, stream, (uint64_t)k, 1);
            ids[k] = (int32_t)(((unsigned __int128)h * (uint64_t)V) >> 64);
        }
    }
}
