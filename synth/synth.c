/*
 * Seeded synthetic inputs for the routed-expert MoE FFN workloads.
 *
 * This module only produces input data: pseudo-random streams, normal
 * deviates, canonical Q4 weight blocks, permutations and Gumbel-perturbed
 * router logits.  It holds none of the method's arithmetic (no routing,
 * quantization, dot product or cache policy) and is shared, as data, by the
 * CPU oracle and by the CUDA path.
 *
 * Generators (published definitions, restated here):
 *   - splitmix64 (Steele, Lea, Flood 2014) to derive stream keys and seeds;
 *   - xoshiro256** (Blackman, Vigna 2018) as the stream generator;
 *   - Box-Muller (1958) for N(0,1), in double precision, rounded to float;
 *   - Gumbel(0,1) as -ln(-ln U).
 *
 * Every stream is keyed by a tuple (seed, stream id, a, b, c), so any part
 * of a workload can be generated on its own, in parallel, in any order.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

static uint64_t sm64_next(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Mix a tuple into one 64-bit stream key. */
uint64_t synth_key(uint64_t seed, uint64_t stream, uint64_t a, uint64_t b, uint64_t c) {
    uint64_t s = seed;
    uint64_t k = sm64_next(&s);
    uint64_t parts[4] = {stream, a, b, c};
    for (int i = 0; i < 4; ++i) {
        s = k ^ (parts[i] + 0x632BE59BD9B4E019ull * (uint64_t)(i + 1));
        k = sm64_next(&s);
    }
    return k;
}

typedef struct {
    uint64_t s[4];
} xo_t;

static inline uint64_t rotl64(uint64_t x, int k) { return (x << k) | (x >> (64 - k)); }

static void xo_init(xo_t *g, uint64_t key) {
    uint64_t s = key;
    for (int i = 0; i < 4; ++i) g->s[i] = sm64_next(&s);
}

static inline uint64_t xo_next(xo_t *g) {
    uint64_t *s = g->s;
    const uint64_t result = rotl64(s[1] * 5, 7) * 9;
    const uint64_t t = s[1] << 17;
    s[2] ^= s[0];
    s[3] ^= s[1];
    s[1] ^= s[2];
    s[0] ^= s[3];
    s[2] ^= t;
    s[3] = rotl64(s[3], 45);
    return result;
}

/* Uniform in [0,1) with 53 random bits. */
static inline double xo_unit(xo_t *g) { return (double)(xo_next(g) >> 11) * 0x1.0p-53; }
/* Uniform in (0,1]. */
static inline double xo_unit_open(xo_t *g) { return (double)((xo_next(g) >> 11) + 1) * 0x1.0p-53; }

/* float -> IEEE binary16 bits, round to nearest even.  Used only to store the
 * generated Q4 block scales in their on-disk format. */
static uint16_t gen_f16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x200u : 0u));
    if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* >= 65520 rounds to inf */
    if (ax < 0x38800000u) {                                  /* below 2^-14: subnormal */
        float v;
        memcpy(&v, &ax, 4);
        double r = nearbyint((double)v * 16777216.0);
        return (uint16_t)(sign | (uint32_t)r);
    }
    uint32_t e = (ax >> 23) - 127u + 15u;
    uint32_t m = ax & 0x7fffffu;
    uint32_t h = (e << 10) | (m >> 13);
    uint32_t rem = m & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++;
    return (uint16_t)(sign | h);
}

void synth_uniform_f64(uint64_t key, double *out, size_t n) {
    xo_t g;
    xo_init(&g, key);
    for (size_t i = 0; i < n; ++i) out[i] = xo_unit(&g);
}

/* N(0,1) deviates (Box-Muller, both outputs of each pair used). */
void synth_normal_f32(uint64_t key, float *out, size_t n) {
    xo_t g;
    xo_init(&g, key);
    const double two_pi = 6.283185307179586476925286766559;
    size_t i = 0;
    while (i < n) {
        double u1 = xo_unit_open(&g);
        double u2 = xo_unit(&g);
        double r = sqrt(-2.0 * log(u1));
        out[i++] = (float)(r * cos(two_pi * u2));
        if (i < n) out[i++] = (float)(r * sin(two_pi * u2));
    }
}

/*
 * Canonical Q4 blocks of 32 weights, 18 bytes each: a little-endian binary16
 * scale d ~ U(dlo, dhi) (rounded to binary16), then 16 bytes of 4-bit codes
 * q ~ U{0..15}.  Byte j holds element j in its low nibble and element j+16 in
 * its high nibble.  The generator draws the 16 code bytes as two 64-bit words.
 */
void synth_q4_blocks(uint64_t key, uint8_t *out, size_t n_blocks, double dlo, double dhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_blocks; ++b) {
        uint8_t *blk = out + b * 18;
        double d = dlo + (dhi - dlo) * xo_unit(&g);
        uint16_t h = gen_f16_bits((float)d);
        blk[0] = (uint8_t)(h & 0xff);
        blk[1] = (uint8_t)(h >> 8);
        uint64_t w0 = xo_next(&g), w1 = xo_next(&g);
        for (int j = 0; j < 8; ++j) {
            blk[2 + j] = (uint8_t)(w0 >> (8 * j));
            blk[10 + j] = (uint8_t)(w1 >> (8 * j));
        }
    }
}

/*
 * Canonical Q8_0 blocks of 32 weights, 34 bytes each: a little-endian
 * binary16 scale d ~ U(dlo, dhi) (rounded to binary16), then 32 signed code
 * bytes q ~ U{-127..127} in element order.  Each 64-bit draw gives four codes
 * from its 16-bit quarters c as (c * 255) >> 16, minus 127.
 */
void synth_q8_blocks(uint64_t key, uint8_t *out, size_t n_blocks, double dlo, double dhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_blocks; ++b) {
        uint8_t *blk = out + b * 34;
        double d = dlo + (dhi - dlo) * xo_unit(&g);
        uint16_t h = gen_f16_bits((float)d);
        blk[0] = (uint8_t)(h & 0xff);
        blk[1] = (uint8_t)(h >> 8);
        for (int w = 0; w < 8; ++w) {
            uint64_t v = xo_next(&g);
            for (int j = 0; j < 4; ++j) {
                uint32_t c = (uint32_t)((v >> (16 * j)) & 0xffffu);
                int q = (int)((c * 255u) >> 16) - 127;
                blk[2 + 4 * w + j] = (uint8_t)(int8_t)q;
            }
        }
    }
}

/*
 * Canonical Q5_0 blocks of 32 weights, 22 bytes each: a little-endian
 * binary16 scale d ~ U(dlo, dhi) (rounded to binary16), then 4 bytes of high
 * bits and 16 bytes of low nibbles (codes q ~ U{0..31}: every bit uniform).
 */
void synth_q5_blocks(uint64_t key, uint8_t *out, size_t n_blocks, double dlo, double dhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_blocks; ++b) {
        uint8_t *blk = out + b * 22;
        double d = dlo + (dhi - dlo) * xo_unit(&g);
        uint16_t h = gen_f16_bits((float)d);
        blk[0] = (uint8_t)(h & 0xff);
        blk[1] = (uint8_t)(h >> 8);
        uint64_t w0 = xo_next(&g), w1 = xo_next(&g), w2 = xo_next(&g);
        for (int j = 0; j < 4; ++j) blk[2 + j] = (uint8_t)(w2 >> (8 * j));
        for (int j = 0; j < 8; ++j) {
            blk[6 + j] = (uint8_t)(w0 >> (8 * j));
            blk[14 + j] = (uint8_t)(w1 >> (8 * j));
        }
    }
}

/*
 * Canonical Q4_K super-blocks of 256 weights, 144 bytes each: binary16
 * d ~ U(dlo, dhi) and dmin ~ U(mlo, mhi) (rounded to binary16), then 140
 * uniform bytes (12 bytes of packed 6-bit sub-block scales and mins, every
 * pattern valid and every 6-bit value equally likely, and 128 code bytes).
 */
/*
 * Q5_K super-blocks of 256 weights in the published layout, 176 bytes each:
 * d ~ U(dlo, dhi) and dmin ~ U(mlo, mhi) as binary16, then 172 uniform bytes
 * (packed 6-bit scales and mins, the fifth-bit bytes qh, the code bytes).
 */
void synth_q5k_blocks(uint64_t key, uint8_t *out, size_t n_super, double dlo, double dhi, double mlo, double mhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_super; ++b) {
        uint8_t *sb = out + b * 176;
        uint16_t h = gen_f16_bits((float)(dlo + (dhi - dlo) * xo_unit(&g)));
        uint16_t hm = gen_f16_bits((float)(mlo + (mhi - mlo) * xo_unit(&g)));
        sb[0] = (uint8_t)(h & 0xff);
        sb[1] = (uint8_t)(h >> 8);
        sb[2] = (uint8_t)(hm & 0xff);
        sb[3] = (uint8_t)(hm >> 8);
        for (int w = 0; w < 172; w += 4) {
            uint64_t v = xo_next(&g);
            for (int j = 0; j < 4; ++j) sb[4 + w + j] = (uint8_t)(v >> (8 * j));
        }
    }
}

/*
 * Q2_K super-blocks of 256 weights in the published layout, 84 bytes each:
 * 80 uniform bytes (16 bytes of 4-bit scales and mins, 64 code bytes), then
 * d ~ U(dlo, dhi) and dmin ~ U(mlo, mhi) as binary16.
 */
void synth_q2k_blocks(uint64_t key, uint8_t *out, size_t n_super, double dlo, double dhi, double mlo, double mhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_super; ++b) {
        uint8_t *sb = out + b * 84;
        for (int w = 0; w < 80; w += 4) {
            uint64_t v = xo_next(&g);
            for (int j = 0; j < 4; ++j) sb[w + j] = (uint8_t)(v >> (8 * j));
        }
        uint16_t h = gen_f16_bits((float)(dlo + (dhi - dlo) * xo_unit(&g)));
        uint16_t hm = gen_f16_bits((float)(mlo + (mhi - mlo) * xo_unit(&g)));
        sb[80] = (uint8_t)(h & 0xff);
        sb[81] = (uint8_t)(h >> 8);
        sb[82] = (uint8_t)(hm & 0xff);
        sb[83] = (uint8_t)(hm >> 8);
    }
}

/*
 * Q3_K super-blocks of 256 weights in the published layout, 110 bytes each:
 * 108 uniform bytes (hmask, code bytes, packed 6-bit scales), then a
 * binary16 d ~ U(dlo, dhi).
 */
void synth_q3k_blocks(uint64_t key, uint8_t *out, size_t n_super, double dlo, double dhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_super; ++b) {
        uint8_t *sb = out + b * 110;
        for (int w = 0; w < 108; w += 4) {
            uint64_t v = xo_next(&g);
            for (int j = 0; j < 4; ++j) sb[w + j] = (uint8_t)(v >> (8 * j));
        }
        uint16_t h = gen_f16_bits((float)(dlo + (dhi - dlo) * xo_unit(&g)));
        sb[108] = (uint8_t)(h & 0xff);
        sb[109] = (uint8_t)(h >> 8);
    }
}

void synth_q4k_blocks(uint64_t key, uint8_t *out, size_t n_super, double dlo, double dhi, double mlo, double mhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_super; ++b) {
        uint8_t *sb = out + b * 144;
        uint16_t h = gen_f16_bits((float)(dlo + (dhi - dlo) * xo_unit(&g)));
        uint16_t hm = gen_f16_bits((float)(mlo + (mhi - mlo) * xo_unit(&g)));
        sb[0] = (uint8_t)(h & 0xff);
        sb[1] = (uint8_t)(h >> 8);
        sb[2] = (uint8_t)(hm & 0xff);
        sb[3] = (uint8_t)(hm >> 8);
        for (int w = 0; w < 140; w += 4) {
            uint64_t v = xo_next(&g);
            for (int j = 0; j < 4; ++j) sb[4 + w + j] = (uint8_t)(v >> (8 * j));
        }
    }
}

/*
 * Q6_K super-blocks of 256 weights in the published block layout, 210 bytes
 * each: 192 uniform bytes of 6-bit codes (ql, qh: every code equally likely
 * whatever the element order), 16 signed scales ~ U{-64..63}, then a
 * binary16 d ~ U(dlo, dhi).
 */
void synth_q6k_blocks(uint64_t key, uint8_t *out, size_t n_super, double dlo, double dhi) {
    xo_t g;
    xo_init(&g, key);
    for (size_t b = 0; b < n_super; ++b) {
        uint8_t *sb = out + b * 210;
        for (int w = 0; w < 192; w += 8) {
            uint64_t v = xo_next(&g);
            for (int j = 0; j < 8; ++j) sb[w + j] = (uint8_t)(v >> (8 * j));
        }
        uint64_t v0 = xo_next(&g), v1 = xo_next(&g);
        for (int j = 0; j < 16; ++j) {
            const unsigned byte = (unsigned)(((j < 8 ? v0 : v1) >> (8 * (j & 7))) & 0xff);
            sb[192 + j] = (uint8_t)(int8_t)((int)(byte % 128) - 64);
        }
        uint16_t h = gen_f16_bits((float)(dlo + (dhi - dlo) * xo_unit(&g)));
        sb[208] = (uint8_t)(h & 0xff);
        sb[209] = (uint8_t)(h >> 8);
    }
}

typedef struct {
    uint64_t seed, tag;
    int e0, e1, fmt;
    size_t blocks_per_expert;
    uint8_t *out;
    double dlo, dhi;
} q4_job_t;

static void *q4_worker(void *arg) {
    q4_job_t *j = (q4_job_t *)arg;
    const size_t bb = j->fmt == 1   ? 34
                      : j->fmt == 2 ? 22
                      : j->fmt == 3 ? 144
                      : j->fmt == 4 ? 210
                      : j->fmt == 5 ? 176
                      : j->fmt == 6 ? 84
                      : j->fmt == 7 ? 110
                                    : 18;
    for (int e = j->e0; e < j->e1; ++e) {
        uint64_t key = synth_key(j->seed, 1, j->tag, (uint64_t)e, 0);
        uint8_t *dst = j->out + (size_t)e * j->blocks_per_expert * bb;
        if (j->fmt == 7)
            synth_q3k_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi);
        else if (j->fmt == 6)
            synth_q2k_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi, 0.002, 0.0106);
        else if (j->fmt == 5)
            synth_q5k_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi, 0.0006, 0.0025);
        else if (j->fmt == 4)
            synth_q6k_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi);
        else if (j->fmt == 3)
            synth_q4k_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi, 0.0006, 0.0025);
        else if (j->fmt == 1)
            synth_q8_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi);
        else if (j->fmt == 2)
            synth_q5_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi);
        else
            synth_q4_blocks(key, dst, j->blocks_per_expert, j->dlo, j->dhi);
    }
    return NULL;
}

/*
 * All experts of one expert tensor, expert-major: out[e][block] (18 B each
 * for Q4, fmt 0; 34 B for Q8_0, fmt 1; 22 B for Q5_0, fmt 2; 144-byte
 * super-blocks of 256 weights for Q4_K, fmt 3, with dmin ~ U(0.0006, 0.0025);
 * 210-byte super-blocks for Q6_K, fmt 4; 176-byte super-blocks for Q5_K,
 * fmt 5, dmin as for Q4_K; 84-byte super-blocks for Q2_K, fmt 6, with
 * dmin ~ U(0.002, 0.0106); 110-byte super-blocks for Q3_K, fmt 7).
 * Expert e is drawn from its own stream keyed by (seed, 1, tensor_tag, e), so
 * the result does not depend on n_threads and any expert can be regenerated
 * alone with synth_experts(seed, tag, e, e+1, ...).
 */
void synth_experts(uint64_t seed, uint64_t tensor_tag, int e_begin, int e_end, size_t blocks_per_expert,
                   uint8_t *out, double dlo, double dhi, int n_threads, int fmt) {
    const size_t bb = fmt == 1   ? 34
                      : fmt == 2 ? 22
                      : fmt == 3 ? 144
                      : fmt == 4 ? 210
                      : fmt == 5 ? 176
                      : fmt == 6 ? 84
                      : fmt == 7 ? 110
                                 : 18;
    int n = e_end - e_begin;
    if (n <= 0) return;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 64) n_threads = 64;
    if (n_threads > n) n_threads = n;
    q4_job_t jobs[64];
    pthread_t th[64];
    for (int t = 0; t < n_threads; ++t) {
        jobs[t].seed = seed;
        jobs[t].tag = tensor_tag;
        jobs[t].e0 = e_begin + (int)((long)n * t / n_threads);
        jobs[t].e1 = e_begin + (int)((long)n * (t + 1) / n_threads);
        jobs[t].fmt = fmt;
        jobs[t].blocks_per_expert = blocks_per_expert;
        jobs[t].out = out - (size_t)e_begin * blocks_per_expert * bb;
        jobs[t].dlo = dlo;
        jobs[t].dhi = dhi;
    }
    for (int t = 1; t < n_threads; ++t) pthread_create(&th[t], NULL, q4_worker, &jobs[t]);
    q4_worker(&jobs[0]);
    for (int t = 1; t < n_threads; ++t) pthread_join(th[t], NULL);
}

void synth_q4_experts(uint64_t seed, uint64_t tensor_tag, int e_begin, int e_end, size_t blocks_per_expert,
                      uint8_t *out, double dlo, double dhi, int n_threads) {
    synth_experts(seed, tensor_tag, e_begin, e_end, blocks_per_expert, out, dlo, dhi, n_threads, 0);
}

/* Uniform random permutation of 0..n-1 (Fisher-Yates, Lemire-free modulo with
 * rejection so every permutation is equally likely). */
void synth_permutation(uint64_t key, int32_t *perm, int n) {
    xo_t g;
    xo_init(&g, key);
    for (int i = 0; i < n; ++i) perm[i] = i;
    for (int i = n - 1; i > 0; --i) {
        uint64_t bound = (uint64_t)(i + 1);
        uint64_t lim = UINT64_MAX - UINT64_MAX % bound;
        uint64_t r;
        do r = xo_next(&g);
        while (r >= lim);
        int j = (int)(r % bound);
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
}

/*
 * Router logits with a given popularity: out[t][e] = base[e] + G[t][e], with
 * G ~ Gumbel(0,1) i.i.d.  When base[e] = ln p(e), the top-k of a row is a
 * sample of k experts without replacement from p (the Gumbel-top-k trick,
 * Kool, van Hoof, Welling 2019), so each token's first pick follows p exactly.
 */
void synth_gumbel_logits(uint64_t key, const double *base, int T, int E, float *out) {
    xo_t g;
    xo_init(&g, key);
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double u = xo_unit_open(&g);
            if (u >= 1.0) u = 0x1.fffffffffffffp-1;
            out[(size_t)t * E + e] = (float)(base[e] - log(-log(u)));
        }
}
