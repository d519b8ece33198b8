/*
 * ORACLE for the routed-expert MoE feed-forward with a quantized expert cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded CPU
 * restatement of what the hot path computes, used to check the CUDA path.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or constant with the CUDA
 * library, and the CUDA library never calls it.
 *
 * Sources (page titles and sections):
 *  [A2] Zapdev-labs/a6000-custom-kernels -- the pointer-table GEMV diagram
 *       ("router (top-8 of 512 experts, per layer)", moe_cache_gemv) and the
 *       paragraph on the MMVQ dot kernels, which keep every fusion argument
 *       of the stock path, the GLU among them.
 *  [M4] mx-llama.cpp FEATURES.md -- activation quantization to q8_1 reused
 *       by the matmuls that share one input (router and gate/up).
 *  [S5] mihailescu2m/llama.cpp -- "the graph-shape problem" (top-k of 512
 *       expert scores).
 *  Format of the weights (fmt): 0 = Q4 blocks of 32 weights with one
 *  binary16 scale d and 4-bit codes q, w = d * (q - 8) (the block-quantized
 *  weight format of the workloads); byte j of the 16 code bytes holds element
 *  j in its low nibble and element j+16 in its high nibble (the canonical Q4
 *  block order).  1 = Q8_0, one of the other block formats the
 *  Zapdev-labs/a6000-custom-kernels dot kernels accept: blocks of 32 with one
 *  binary16 scale d and 32 signed 8-bit codes q, w = d * q; the pages give no
 *  byte layout, the reading is d (little endian) followed by code bytes 0..31
 *  in element order (34 bytes).  2 = Q5_0, another of those formats: blocks
 *  of 32 with one binary16 scale d and 5-bit codes q, w = d * (q - 16); the
 *  reading of the layout is d, then 4 bytes of high bits (bit j of the
 *  little-endian word = bit 4 of element j), then 16 bytes of low nibbles in
 *  the Q4 order (22 bytes).  3 = Q4_K, one of the K-quant formats those
 *  kernels accept: super-blocks of 256 weights = 8 sub-blocks of 32 with a
 *  binary16 scale d and min scale dmin per super-block, a 6-bit scale sc_j
 *  and 6-bit min m_j per sub-block and 4-bit codes q, w = d*sc_j*q - dmin*m_j.
 *  Reading of the 144-byte layout: d, dmin, 12 bytes of packed (sc, m) (for
 *  j < 4: sc = b[j] & 63, m = b[j+4] & 63; for j >= 4: sc = (b[j+4] & 15) |
 *  (b[j-4] >> 6) << 4, m = (b[j+4] >> 4) | (b[j] >> 6) << 4), then 128 code
 *  bytes in 4 chunks of 32: chunk c holds sub-block 2c in its low nibbles and
 *  sub-block 2c+1 in its high nibbles (byte i of a chunk = element i of each).
 *  Per 32 weights that is 18 bytes, as for Q4.  4 = Q6_K, another K-quant:
 *  super-blocks of 256 weights = 16 sub-blocks of 16 with a signed 8-bit
 *  scale sc_j each, one binary16 scale d and 6-bit codes q,
 *  w = d * sc_j * (q - 32).  The 210-byte layout is the one the format is
 *  published with (the pages name Q6_K but print no layout): 128 bytes of
 *  low nibbles ql, 64 bytes of high bit pairs qh, the 16 scales, then d;
 *  each 128-weight half n owns ql[64n .. 64n + 63] and qh[32n .. 32n + 31],
 *  and its element 32m + l (m = 0..3, l < 32) keeps its low four bits in
 *  ql[64n + l + 32 (m & 1)] (the low nibble for m < 2, the high one for
 *  m >= 2) and its high two bits in bits 2m..2m+1 of qh[32n + l].
 *  5 = Q5_K, another K-quant: the Q4_K super-block with a fifth code bit,
 *  w = d*sc_j*q - dmin*m_j, q in 0..31.  The 176-byte layout is the one the
 *  format is published with: d, dmin, the 12 scale/min bytes packed as for
 *  Q4_K, 32 bytes qh, then 128 code bytes qs in the Q4_K chunk order; bit j
 *  of qh[l] is the fifth bit of element l of sub-block j.
 *  6 = Q2_K, the K-quant of the pages' headline model (Q2_K_S): super-blocks
 *  of 256 weights = 16 sub-blocks of 16, each with a 4-bit scale sc_j and a
 *  4-bit min m_j, 2-bit codes, binary16 d and dmin, w = d*sc_j*q - dmin*m_j.
 *  The 84-byte layout is the published one: 16 bytes scales (byte j: sc_j in
 *  the low nibble, m_j in the high one), 64 code bytes qs, then d and dmin;
 *  element i = 128n + 32m + t (half n, quarter m, t < 32) is bits 2m..2m+1
 *  of qs[32n + t].
 *  7 = Q3_K: super-blocks of 256 weights = 16 sub-blocks of 16 with signed
 *  6-bit scales sc_j, binary16 d, 3-bit codes q in -4..3, w = d*sc_j*q.  The
 *  110-byte layout is the published one: 32 bytes hmask, 64 code bytes qs,
 *  12 scale bytes, d.  Element 128n + 32m + t has the low two bits
 *  (qs[32n + t] >> 2m) & 3 and q = low - 4 unless bit 4n + m of hmask[t] is
 *  set (then q = low).  Scale j: low four bits = byte j & 15 (j < 8) or byte
 *  j - 8 >> 4 (j >= 8), high two = bits 2(j/4)..2(j/4)+1 of byte 8 + j mod 4,
 *  sc_j = that 6-bit value - 32.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - top-k order is (logit descending, expert index ascending): ties go to
 *    the lower index; -0.0 and +0.0 tie;
 *  - routing weights are the softmax over the k selected logits
 *    (renormalized top-k); renorm=0 gives the softmax over all E logits;
 *  - activation blocks of 32: d = binary16(amax / 127) computed in binary32,
 *    q_i = clamp(rint(x_i / d), -127, 127) in binary32 with round-half-even,
 *    using the stored binary16 scale; an all-zero block (d == 0) gives q = 0;
 *  - SwiGLU: h = silu(gate) * up = g * u / (1 + exp(-g));
 *  - the expert FFN output is combined as y[t] = sum_j w[t,j] * o[t,j].
 *
 * Precision: the exact values of the method are computed in binary64.  The
 * two places where floating point decides an integer (the code of an
 * activation element and the binary16 scale of a block) take that decision
 * in binary32, the precision the CUDA path uses, after rounding the binary64
 * value of h to binary32.  Compile with -ffp-contract=off.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_BLOCK 32
#define ORC_BLOCK_BYTES 18
#define ORC_Q8_BLOCK_BYTES 34
#define ORC_Q5_BLOCK_BYTES 22

#define ORC_K4_SUPER_BYTES 144
#define ORC_K6_SUPER_BYTES 210
#define ORC_K5_SUPER_BYTES 176
#define ORC_K2_SUPER_BYTES 84
#define ORC_K3_SUPER_BYTES 110

double orc_h2d(uint16_t h);

/* Bytes per 32 weights (Q4_K: a 144-byte super-block holds 256). */
static size_t orc_bbytes(int fmt) {
    return fmt == 1 ? ORC_Q8_BLOCK_BYTES : fmt == 2 ? ORC_Q5_BLOCK_BYTES : ORC_BLOCK_BYTES;
}

/* Bytes of a row of nb 32-weight blocks (super-block formats: nb / 8 of them). */
static size_t orc_row_bytes(int fmt, int nb) {
    if (fmt == 3) return (size_t)(nb / 8) * ORC_K4_SUPER_BYTES;
    if (fmt == 4) return (size_t)(nb / 8) * ORC_K6_SUPER_BYTES;
    if (fmt == 5) return (size_t)(nb / 8) * ORC_K5_SUPER_BYTES;
    if (fmt == 6) return (size_t)(nb / 8) * ORC_K2_SUPER_BYTES;
    if (fmt == 7) return (size_t)(nb / 8) * ORC_K3_SUPER_BYTES;
    return (size_t)nb * orc_bbytes(fmt);
}

/* Q6_K: 6-bit code of element i (0..255) of a super-block: half n = i / 128,
 * quarter m of that half, position l in the quarter. */
static int orc_k6_code(const uint8_t *sb, int i) {
    const uint8_t *ql = sb, *qh = sb + 128;
    const int n = i / 128, m = (i % 128) / 32, l = i % 32;
    const uint8_t lb = ql[64 * n + 32 * (m & 1) + l];
    const int lo = m < 2 ? (lb & 15) : (lb >> 4);
    const int hi = (qh[32 * n + l] >> (2 * m)) & 3;
    return lo | (hi << 4);
}

/* Q6_K: signed scale of 16-weight sub-block j (0..15) and the super-block's d. */
static int orc_k6_scale(const uint8_t *sb, int j) { return (int)(int8_t)sb[192 + j]; }
static double orc_k6_d(const uint8_t *sb) { return orc_h2d((uint16_t)(sb[208] | (sb[209] << 8))); }

/* Q6_K: the integer dot of each 32-weight block against 32 int8
 * activations: sc_2b * sum_{i<16} (q-32) a + sc_2b+1 * sum_{16<=i<32} (q-32) a
 * (exact in int32: |.| <= 2 * 128 * 16 * 32 * 127). */
void orc_k6_blockdots(const uint8_t *sb, const int8_t *qa, int32_t *out) {
    for (int b = 0; b < 8; ++b) {
        int32_t s = 0;
        for (int h = 0; h < 2; ++h) {
            int32_t t = 0;
            for (int i = 0; i < 16; ++i) {
                const int e = 32 * b + 16 * h + i;
                t += (int32_t)(orc_k6_code(sb, e) - 32) * (int32_t)qa[e];
            }
            s += orc_k6_scale(sb, 2 * b + h) * t;
        }
        out[b] = s;
    }
}

/* Q4_K: scale and min of sub-block j (0..7) of a super-block. */
static void orc_k4_scale_min(const uint8_t *sb, int j, int *sc, int *m) {
    const uint8_t *b = sb + 4;
    if (j < 4) {
        *sc = b[j] & 63;
        *m = b[j + 4] & 63;
    } else {
        *sc = (b[j + 4] & 15) | ((b[j - 4] >> 6) << 4);
        *m = (b[j + 4] >> 4) | ((b[j] >> 6) << 4);
    }
}

/* Q4_K: 4-bit code of element i (0..255) of a super-block. */
static int orc_k4_code(const uint8_t *sb, int i) {
    const uint8_t *qs = sb + 16;
    const int c = i / 64, r = i % 64;
    return r < 32 ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);
}

/* Q5_K: 5-bit code of element i (0..255) of a super-block: the low four bits
 * as in Q4_K (from the code bytes after qh), the fifth from qh. */
static int orc_k5_code(const uint8_t *sb, int i) {
    const uint8_t *qh = sb + 16, *qs = sb + 48;
    const int c = i / 64, r = i % 64, j = i / 32, l = i % 32;
    const int lo = r < 32 ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);
    return lo | (((qh[l] >> j) & 1) << 4);
}

/* Q5_K: raw integer dots sum_i q_i * a_i of the 8 sub-blocks against 256
 * int8 activations (exact in int32: |sum| <= 32 * 31 * 127). */
void orc_k5_subdots(const uint8_t *sb, const int8_t *qa, int32_t *out) {
    for (int j = 0; j < 8; ++j) {
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)orc_k5_code(sb, 32 * j + i) * (int32_t)qa[32 * j + i];
        out[j] = s;
    }
}

/* Q3_K: signed 3-bit code of element i (0..255), signed scale of its
 * 16-weight sub-block j = i / 16, and d. */
static int orc_k3_code(const uint8_t *sb, int i) {
    const uint8_t *hm = sb, *qs = sb + 32;
    const int n = i / 128, m = (i % 128) / 32, t = i % 32;
    const int low = (qs[32 * n + t] >> (2 * m)) & 3;
    return ((hm[t] >> (4 * n + m)) & 1) ? low : low - 4;
}
static int orc_k3_scale(const uint8_t *sb, int j) {
    const uint8_t *b = sb + 96;
    const int low4 = j < 8 ? (b[j] & 15) : (b[j - 8] >> 4);
    const int high2 = (b[8 + j % 4] >> (2 * (j / 4))) & 3;
    return (low4 | (high2 << 4)) - 32;
}
static double orc_k3_d(const uint8_t *sb) { return orc_h2d((uint16_t)(sb[108] | (sb[109] << 8))); }

/* Q3_K: the integer dot of each 32-weight block against 32 int8
 * activations: sc_2b * sum_{i<16} q a + sc_2b+1 * sum_{16<=i<32} q a
 * (exact in int32: |.| <= 2 * 32 * 16 * 4 * 127). */
void orc_k3_blockdots(const uint8_t *sb, const int8_t *qa, int32_t *out) {
    for (int b = 0; b < 8; ++b) {
        int32_t s = 0;
        for (int h = 0; h < 2; ++h) {
            int32_t part = 0;
            for (int i = 0; i < 16; ++i) {
                const int e = 32 * b + 16 * h + i;
                part += (int32_t)orc_k3_code(sb, e) * (int32_t)qa[e];
            }
            s += orc_k3_scale(sb, 2 * b + h) * part;
        }
        out[b] = s;
    }
}

/* Q2_K: 2-bit code of element i (0..255), and scale / min of its 16-weight
 * sub-block j = i / 16. */
static int orc_k2_code(const uint8_t *sb, int i) {
    const uint8_t *qs = sb + 16;
    const int n = i / 128, m = (i % 128) / 32, t = i % 32;
    return (qs[32 * n + t] >> (2 * m)) & 3;
}
static void orc_k2_scale_min(const uint8_t *sb, int j, int *sc, int *m) {
    *sc = sb[j] & 15;
    *m = sb[j] >> 4;
}

/* Q2_K: raw integer dots sum_i q_i * a_i of the 16 sub-blocks against 256
 * int8 activations (exact in int32: |sum| <= 16 * 3 * 127). */
void orc_k2_subdots(const uint8_t *sb, const int8_t *qa, int32_t *out) {
    for (int j = 0; j < 16; ++j) {
        int32_t s = 0;
        for (int i = 0; i < 16; ++i) s += (int32_t)orc_k2_code(sb, 16 * j + i) * (int32_t)qa[16 * j + i];
        out[j] = s;
    }
}

/* Q4_K: raw integer dots sum_i q_i * a_i of the 8 sub-blocks against 256
 * int8 activations (exact in int32: |sum| <= 32 * 15 * 127). */
void orc_k4_subdots(const uint8_t *sb, const int8_t *qa, int32_t *out) {
    for (int j = 0; j < 8; ++j) {
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)orc_k4_code(sb, 32 * j + i) * (int32_t)qa[32 * j + i];
        out[j] = s;
    }
}

/* ---- binary16 <-> binary64/32 from the IEEE 754 definition ------------- */

/* Value of binary16 bits h: (-1)^s * 2^(e-15) * 1.m for 1 <= e <= 30,
 * (-1)^s * 2^-14 * 0.m for e = 0, inf/NaN for e = 31. */
double orc_h2d(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return s ? -v : v;
}

/* binary32 -> binary16, round to nearest, ties to even.  The quantum of the
 * binade holding |f| is 2^(max(e,-14)-10); |f| divided by it is exact in
 * binary64, and rounding that quotient to an integer (ties to even) picks the
 * nearest binary16 value.  A carry to 2048 moves into the next binade, which
 * the encoding handles by itself. */
uint16_t orc_f2h(float f) {
    double v = (double)f;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7e00);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) -> binade exponent ex-1 */
    int e = ex - 1;
    if (e < -14) e = -14;
    double quantum = ldexp(1.0, e - 10);
    double r = nearbyint(a / quantum); /* default rounding: ties to even */
    uint32_t bits;
    if (r < 1024.0) /* subnormal: value r * 2^-24, encoding is r */
        bits = (uint32_t)r;
    else
        bits = ((uint32_t)(e + 15) << 10) + ((uint32_t)r - 1024u);
    return (uint16_t)(sign | bits);
}

/* ---- [S5]/[A2] router top-k ---------------------------------------------- */

/* For each token t: idx[t][0..k) = the k experts with the largest logits,
 * in order (logit desc, index asc); w[t][j] = routing weight.  O(k*E). */
void orc_topk(const float *logits, int T, int E, int k, int renorm, int32_t *idx, double *w) {
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        int32_t *id = idx + (size_t)t * k;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int i = 0; i < j; ++i)
                    if (id[i] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: ties keep the lower index */
            }
            id[j] = best;
        }
        double m = (double)l[id[0]];
        double den = 0.0;
        if (renorm) {
            for (int j = 0; j < k; ++j) den += exp((double)l[id[j]] - m);
        } else {
            for (int e = 0; e < E; ++e) den += exp((double)l[e] - m);
        }
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = exp((double)l[id[j]] - m) / den;
    }
}

/* ---- [M4] activation quantization, int8 blocks of 32 + binary16 scale ---- */

void orc_quantize_blocks(const float *x, int n, int8_t *q, uint16_t *d) {
    for (int b = 0; b < n / ORC_BLOCK; ++b) {
        const float *xb = x + (size_t)b * ORC_BLOCK;
        float amax = 0.0f;
        for (int i = 0; i < ORC_BLOCK; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        float d32 = amax / 127.0f;
        uint16_t dh = orc_f2h(d32);
        float dd = (float)orc_h2d(dh);
        d[b] = dh;
        for (int i = 0; i < ORC_BLOCK; ++i) {
            int v = 0;
            if (dd != 0.0f) {
                float r = rintf(xb[i] / dd);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                v = (int)r;
            }
            q[(size_t)b * ORC_BLOCK + i] = (int8_t)v;
        }
    }
}

/* ---- quantized weights ------------------------------------------------------ */

/* 4-bit code of element i (0..31) of a canonical 18-byte block. */
static int orc_code(const uint8_t *blk, int i) {
    const uint8_t *qs = blk + 2;
    return i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4);
}

/* 5-bit code of element i of a canonical 22-byte Q5_0 block: low nibble
 * from the 16 code bytes (Q4 order, after the 4 high-bit bytes), bit 4 from
 * bit i of the high-bit word. */
static int orc_code5(const uint8_t *blk, int i) {
    const uint8_t *qh = blk + 2, *qs = blk + 6;
    const int lo = i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4);
    const int hi = (qh[i / 8] >> (i % 8)) & 1;
    return lo | (hi << 4);
}

/* Signed weight code of element i: q - 8 (Q4), q (Q8_0) or q - 16 (Q5_0),
 * so w = d * code. */
static int orc_wcode(const uint8_t *blk, int i, int fmt) {
    if (fmt == 1) return (int)(int8_t)blk[2 + i];
    if (fmt == 2) return orc_code5(blk, i) - 16;
    return orc_code(blk, i) - 8;
}

static uint16_t orc_block_scale(const uint8_t *blk) { return (uint16_t)(blk[0] | (blk[1] << 8)); }

/* Dequantized weights of nb blocks: w = d * (q - 8) (Q4), d * q (Q8_0) or
 * d * (q - 16) (Q5_0). */
void orc_dequant_fmt(const uint8_t *blocks, int nb, int fmt, double *out) {
    if (fmt == 4) { /* Q6_K: w = d * sc_j * (q - 32), sub-blocks of 16 */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = blocks + (size_t)s * ORC_K6_SUPER_BYTES;
            const double d = orc_k6_d(sb);
            for (int i = 0; i < 256; ++i)
                out[(size_t)s * 256 + i] = d * orc_k6_scale(sb, i / 16) * (double)(orc_k6_code(sb, i) - 32);
        }
        return;
    }
    if (fmt == 7) { /* Q3_K: w = d * sc_j * q, sub-blocks of 16 */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = blocks + (size_t)s * ORC_K3_SUPER_BYTES;
            const double d = orc_k3_d(sb);
            for (int i = 0; i < 256; ++i)
                out[(size_t)s * 256 + i] = d * orc_k3_scale(sb, i / 16) * (double)orc_k3_code(sb, i);
        }
        return;
    }
    if (fmt == 6) { /* Q2_K: w = d * sc_j * q - dmin * m_j, sub-blocks of 16 */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = blocks + (size_t)s * ORC_K2_SUPER_BYTES;
            const double d = orc_h2d(orc_block_scale(sb + 80)), dmin = orc_h2d(orc_block_scale(sb + 82));
            for (int i = 0; i < 256; ++i) {
                int sc, m;
                orc_k2_scale_min(sb, i / 16, &sc, &m);
                out[(size_t)s * 256 + i] = d * sc * (double)orc_k2_code(sb, i) - dmin * m;
            }
        }
        return;
    }
    if (fmt == 5) { /* Q5_K: w = d * sc_j * q - dmin * m_j, q in 0..31 */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = blocks + (size_t)s * ORC_K5_SUPER_BYTES;
            const double d = orc_h2d(orc_block_scale(sb)), dmin = orc_h2d(orc_block_scale(sb + 2));
            for (int i = 0; i < 256; ++i) {
                int sc, m;
                orc_k4_scale_min(sb, i / 32, &sc, &m);
                out[(size_t)s * 256 + i] = d * sc * (double)orc_k5_code(sb, i) - dmin * m;
            }
        }
        return;
    }
    if (fmt == 3) { /* nb counts 32-weight blocks; super-blocks of 8 */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = blocks + (size_t)s * ORC_K4_SUPER_BYTES;
            const double d = orc_h2d(orc_block_scale(sb)), dmin = orc_h2d(orc_block_scale(sb + 2));
            for (int i = 0; i < 256; ++i) {
                int sc, m;
                orc_k4_scale_min(sb, i / 32, &sc, &m);
                out[(size_t)s * 256 + i] = d * sc * (double)orc_k4_code(sb, i) - dmin * m;
            }
        }
        return;
    }
    for (int b = 0; b < nb; ++b) {
        const uint8_t *blk = blocks + (size_t)b * orc_bbytes(fmt);
        double d = orc_h2d(orc_block_scale(blk));
        for (int i = 0; i < ORC_BLOCK; ++i) out[(size_t)b * ORC_BLOCK + i] = d * (double)orc_wcode(blk, i, fmt);
    }
}

void orc_dequant(const uint8_t *blocks, int nb, double *out) { orc_dequant_fmt(blocks, nb, 0, out); }

/* [A2] integer block dot: sum_i code_w,i * q_a,i, exact in int32
 * (|sum| <= 32 * 8 * 127 for Q4, 32 * 16 * 127 for Q5_0, 32 * 128 * 127 for
 * Q8_0). */
int32_t orc_block_dot_fmt(const uint8_t *blk, const int8_t *qa, int fmt) {
    int32_t s = 0;
    for (int i = 0; i < ORC_BLOCK; ++i) s += (int32_t)orc_wcode(blk, i, fmt) * (int32_t)qa[i];
    return s;
}

int32_t orc_block_dot(const uint8_t *blk, const int8_t *qa) { return orc_block_dot_fmt(blk, qa, 0); }

/* One weight row (nb blocks) against one quantized activation vector:
 * r = sum_b d_w,b * d_a,b * sumi_b, in binary64, block order.  abs_sum gets
 * sum_b |d_w,b * d_a,b * sumi_b| (for error bounds), if not NULL. */
double orc_row_dot_fmt(const uint8_t *row, const int8_t *qa, const uint16_t *da, int nb, int fmt, double *abs_sum) {
    double acc = 0.0, aacc = 0.0;
    if (fmt == 4) {
        /* per 32-weight block b: d_a,b * d * (its integer dot) */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = row + (size_t)s * ORC_K6_SUPER_BYTES;
            const double d = orc_k6_d(sb);
            int32_t dots[8];
            orc_k6_blockdots(sb, qa + (size_t)s * 256, dots);
            for (int j = 0; j < 8; ++j) {
                const double term = orc_h2d(da[8 * s + j]) * d * (double)dots[j];
                acc += term;
                aacc += fabs(term);
            }
        }
        if (abs_sum) *abs_sum = aacc;
        return acc;
    }
    if (fmt == 7) {
        /* per 32-weight block b: d_a,b * d * (its two-scale integer dot) */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = row + (size_t)s * ORC_K3_SUPER_BYTES;
            const double d3 = orc_k3_d(sb);
            int32_t dots3[8];
            orc_k3_blockdots(sb, qa + (size_t)s * 256, dots3);
            for (int j = 0; j < 8; ++j) {
                const double t3 = orc_h2d(da[8 * s + j]) * d3 * (double)dots3[j];
                acc += t3;
                aacc += fabs(t3);
            }
        }
        if (abs_sum) *abs_sum = aacc;
        return acc;
    }
    if (fmt == 6) {
        /* per 16-weight sub-block j (half of 32-block b = j / 2):
         * d_a,b * (d * sc_j * sum q*a - dmin * m_j * sum a) */
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = row + (size_t)s * ORC_K2_SUPER_BYTES;
            const double d = orc_h2d(orc_block_scale(sb + 80)), dmin = orc_h2d(orc_block_scale(sb + 82));
            int32_t raw[16];
            orc_k2_subdots(sb, qa + (size_t)s * 256, raw);
            for (int j = 0; j < 16; ++j) {
                const int b = 8 * s + j / 2;
                int sc, m;
                orc_k2_scale_min(sb, j, &sc, &m);
                int32_t asum16 = 0;
                for (int i = 0; i < 16; ++i) asum16 += qa[(size_t)s * 256 + 16 * j + i];
                const double da_s = orc_h2d(da[b]);
                const double sq = d * sc * (double)raw[j], mq = dmin * m * (double)asum16;
                acc += da_s * (sq - mq);
                aacc += fabs(da_s) * (fabs(sq) + fabs(mq));
            }
        }
        if (abs_sum) *abs_sum = aacc;
        return acc;
    }
    if (fmt == 3 || fmt == 5) {
        /* per sub-block b: d_a,b * (d * sc * sum q*a - dmin * m * sum a) */
        const size_t sbytes = fmt == 3 ? ORC_K4_SUPER_BYTES : ORC_K5_SUPER_BYTES;
        for (int s = 0; s < nb / 8; ++s) {
            const uint8_t *sb = row + (size_t)s * sbytes;
            const double d = orc_h2d(orc_block_scale(sb)), dmin = orc_h2d(orc_block_scale(sb + 2));
            int32_t raw[8];
            if (fmt == 3)
                orc_k4_subdots(sb, qa + (size_t)s * 256, raw);
            else
                orc_k5_subdots(sb, qa + (size_t)s * 256, raw);
            for (int j = 0; j < 8; ++j) {
                const int b = 8 * s + j;
                int sc, m;
                orc_k4_scale_min(sb, j, &sc, &m);
                int32_t asum = 0;
                for (int i = 0; i < 32; ++i) asum += qa[(size_t)b * 32 + i];
                const double da_b = orc_h2d(da[b]);
                const double p1 = d * sc * (double)raw[j], p2 = dmin * m * (double)asum;
                acc += da_b * (p1 - p2);
                aacc += fabs(da_b) * (fabs(p1) + fabs(p2));
            }
        }
        if (abs_sum) *abs_sum = aacc;
        return acc;
    }
    for (int b = 0; b < nb; ++b) {
        const uint8_t *blk = row + (size_t)b * orc_bbytes(fmt);
        int32_t s = orc_block_dot_fmt(blk, qa + (size_t)b * ORC_BLOCK, fmt);
        double term = orc_h2d(orc_block_scale(blk)) * orc_h2d(da[b]) * (double)s;
        acc += term;
        aacc += fabs(term);
    }
    if (abs_sum) *abs_sum = aacc;
    return acc;
}

double orc_row_dot(const uint8_t *row, const int8_t *qa, const uint16_t *da, int nb, double *abs_sum) {
    return orc_row_dot_fmt(row, qa, da, nb, 0, abs_sum);
}

/* ---- [A2] one routed expert on one token: gate/up, SwiGLU, quantize, down --- */

/* gate, up: F rows x (H/32) blocks; down: H rows x (F/32) blocks (canonical,
 * format fmt).
 * Outputs (any may be NULL except o): g, u, |terms| sums of g and u, h (binary64),
 * hq/hd (the quantized h), o (binary64, H values). */
void orc_expert(const uint8_t *gate, const uint8_t *up, const uint8_t *down, int H, int F, const int8_t *xq,
                const uint16_t *xd, double *g_out, double *u_out, double *gabs, double *uabs, double *h_out,
                int8_t *hq_out, uint16_t *hd_out, double *o, int fmt) {
    int nbh = H / ORC_BLOCK, nbf = F / ORC_BLOCK;
    size_t rowh = orc_row_bytes(fmt, nbh), rowf = orc_row_bytes(fmt, nbf);
    float h32[F > 0 ? F : 1];
    int8_t hq[F > 0 ? F : 1];
    uint16_t hd[F / ORC_BLOCK > 0 ? F / ORC_BLOCK : 1];
    for (int r = 0; r < F; ++r) {
        double ga, ua;
        double g = orc_row_dot_fmt(gate + r * rowh, xq, xd, nbh, fmt, &ga);
        double u = orc_row_dot_fmt(up + r * rowh, xq, xd, nbh, fmt, &ua);
        double h = g * u / (1.0 + exp(-g));
        if (g_out) g_out[r] = g;
        if (u_out) u_out[r] = u;
        if (gabs) gabs[r] = ga;
        if (uabs) uabs[r] = ua;
        if (h_out) h_out[r] = h;
        h32[r] = (float)h;
    }
    orc_quantize_blocks(h32, F, hq, hd);
    if (hq_out) memcpy(hq_out, hq, (size_t)F);
    if (hd_out) memcpy(hd_out, hd, sizeof(uint16_t) * (size_t)nbf);
    for (int i = 0; i < H; ++i) o[i] = orc_row_dot_fmt(down + i * rowf, hq, hd, nbf, fmt, NULL);
}

/* Down projection + combine from given quantized h (one entry per
 * assignment a = t*k + j): y[t] = sum_j w[t,j] * (W_down[idx[t,j]] . h_a). */
void orc_down_combine(int T, int H, int F, int k, const int32_t *idx, const double *w,
                      const uint8_t *const *down, const int8_t *hq, const uint16_t *hd, double *y, int fmt) {
    int nbf = F / ORC_BLOCK;
    size_t rowf = orc_row_bytes(fmt, nbf);
    for (int t = 0; t < T; ++t) {
        double *yt = y + (size_t)t * H;
        for (int i = 0; i < H; ++i) yt[i] = 0.0;
        for (int j = 0; j < k; ++j) {
            size_t a = (size_t)t * k + j;
            const uint8_t *dn = down[idx[a]];
            for (int i = 0; i < H; ++i)
                yt[i] += w[a] * orc_row_dot_fmt(dn + i * rowf, hq + a * F, hd + a * nbf, nbf, fmt, NULL);
        }
    }
}

/*
 * A whole MoE FFN layer on T tokens with given routing (idx, w):
 *   quantize x_t; for each j: expert idx[t,j] -> o; y[t] = sum_j w[t,j] o_j.
 * Expert tensors are passed as arrays of E pointers (entries not referenced
 * by idx may be NULL).  Per-assignment outputs (a = t*k + j) are optional.
 */
void orc_layer(int T, int H, int F, int k, const float *x, const int32_t *idx, const double *w,
               const uint8_t *const *gate, const uint8_t *const *up, const uint8_t *const *down, double *y,
               int8_t *xq_out, uint16_t *xd_out, double *g_out, double *u_out, double *gabs, double *uabs,
               double *h_out, int8_t *hq_out, uint16_t *hd_out, int fmt) {
    int nbh = H / ORC_BLOCK, nbf = F / ORC_BLOCK;
    int8_t xq[H];
    uint16_t xd[H / ORC_BLOCK];
    double o[H];
    for (int t = 0; t < T; ++t) {
        orc_quantize_blocks(x + (size_t)t * H, H, xq, xd);
        if (xq_out) memcpy(xq_out + (size_t)t * H, xq, (size_t)H);
        if (xd_out) memcpy(xd_out + (size_t)t * nbh, xd, sizeof(uint16_t) * (size_t)nbh);
        double *yt = y + (size_t)t * H;
        for (int i = 0; i < H; ++i) yt[i] = 0.0;
        for (int j = 0; j < k; ++j) {
            size_t a = (size_t)t * k + j;
            int e = idx[a];
            orc_expert(gate[e], up[e], down[e], H, F, xq, xd, g_out ? g_out + a * F : NULL,
                       u_out ? u_out + a * F : NULL, gabs ? gabs + a * F : NULL, uabs ? uabs + a * F : NULL,
                       h_out ? h_out + a * F : NULL, hq_out ? hq_out + a * F : NULL,
                       hd_out ? hd_out + a * nbf : NULL, o, fmt);
            for (int i = 0; i < H; ++i) yt[i] += w[a] * o[i];
        }
    }
}
