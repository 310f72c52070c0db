/*
 * datagen.c — seeded synthetic inputs for the MoE layer (weights, tokens,
 * router bias ranks).
 *
 * This module holds no step of the MoE method: it only draws numbers. Both
 * the CPU oracle (tests) and the CUDA path (tests, bench) consume the bytes
 * it writes, so the two sides always see identical inputs.
 *
 * Generator (the pages name none, so this is a stated choice):
 *   h(seed, tag, i) = splitmix64(key(seed, tag) + i * GOLDEN)
 *   key(seed, tag)  = splitmix64(seed ^ splitmix64(tag + 1))
 * splitmix64 is Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators" (OOPSLA 2014), finaliser constants as published there.
 * Uniforms take the top 53 bits. Normals come in pairs from Box-Muller
 * (element 2p and 2p+1 from counters 2p and 2p+1), evaluated in double with
 * the host libm, scaled by sigma, rounded to fp32 and then to bf16 with
 * round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define DG_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t splitmix64(uint64_t z)
{
    z += DG_GOLDEN;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t dg_key(uint64_t seed, uint64_t tag)
{
    return splitmix64(seed ^ splitmix64(tag + 1));
}

static inline uint64_t dg_hash(uint64_t key, uint64_t i)
{
    return splitmix64(key + i * DG_GOLDEN);
}

/* uniform in (0, 1]: never 0, so log() below is finite */
static inline double dg_u01_open0(uint64_t r)
{
    return (double)((r >> 11) + 1) * (1.0 / 9007199254740992.0);
}

/* uniform in [0, 1) */
static inline double dg_u01(uint64_t r)
{
    return (double)(r >> 11) * (1.0 / 9007199254740992.0);
}

static inline uint16_t dg_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static inline double dg_normal_at(uint64_t key, uint64_t i)
{
    uint64_t p = i >> 1;
    double u1 = dg_u01_open0(dg_hash(key, 2 * p));
    double u2 = dg_u01(dg_hash(key, 2 * p + 1));
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? rad * sin(ang) : rad * cos(ang);
}

/* out[i] = bf16(fp32(sigma * N_i)) for i in [start, start + n) of stream (seed, tag) */
void dg_normal_bf16(uint64_t seed, uint64_t tag, uint64_t start, uint64_t n,
                    double sigma, uint16_t *out)
{
    uint64_t key = dg_key(seed, tag);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < nn; ++j) {
        double z = dg_normal_at(key, start + (uint64_t)j);
        out[j] = dg_f32_to_bf16_rne((float)(sigma * z));
    }
}

/* out[i] = fp32(sigma * N_i) */
void dg_normal_f32(uint64_t seed, uint64_t tag, uint64_t start, uint64_t n,
                   double sigma, float *out)
{
    uint64_t key = dg_key(seed, tag);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < nn; ++j)
        out[j] = (float)(sigma * dg_normal_at(key, start + (uint64_t)j));
}

/* out[i] = uniform [0,1) as double */
void dg_uniform_f64(uint64_t seed, uint64_t tag, uint64_t start, uint64_t n, double *out)
{
    uint64_t key = dg_key(seed, tag);
    for (uint64_t j = 0; j < n; ++j)
        out[j] = dg_u01(dg_hash(key, start + j));
}

/* Fisher-Yates shuffle of 0..n-1 driven by stream (seed, tag). */
void dg_permutation(uint64_t seed, uint64_t tag, int n, int32_t *out)
{
    uint64_t key = dg_key(seed, tag);
    for (int i = 0; i < n; ++i)
        out[i] = i;
    for (int i = n - 1; i > 0; --i) {
        uint64_t r = dg_hash(key, (uint64_t)i);
        int j = (int)(dg_u01(r) * (double)(i + 1));
        if (j > i)
            j = i;
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}

/* raw 64-bit counter hash, exposed for the generator's own tests */
uint64_t dg_raw(uint64_t seed, uint64_t tag, uint64_t i)
{
    return dg_hash(dg_key(seed, tag), i);
}
