// Registration-time repack of canonical expert blocks into the plane blobs
// the kernels read (host code; the plane layouts are defined next to
// code_bytes / scale_plane_bytes in common.cuh).  Its own header so that it
// can be compiled for the host alone.
#pragma once
#include <algorithm>
#include <cstring>
#include <thread>
#include <vector>

#include "common.cuh"

namespace moe {

// Q4_K super-block (144 bytes, 256 weights) -> 8 sub-blocks: Q4-order
// nibbles (byte t = element t | element t + 16 << 4) and the exact fp32
// pairs (d * sc_j, dmin * m_j) (binary16 times a 6-bit integer fits fp32).
inline void repack_q4k_super(const uint8_t *sb, uint8_t *codes, float *sm) {
    auto h2f = [](const uint8_t *p) {
        __half h;
        uint16_t b = (uint16_t)(p[0] | (p[1] << 8));
        memcpy(&h, &b, 2);
        return __half2float(h);
    };
    const float d = h2f(sb), dmin = h2f(sb + 2);
    const uint8_t *sc = sb + 4, *qs = sb + 16;
    for (int j = 0; j < 8; ++j) {
        int s6, m6;
        if (j < 4) {
            s6 = sc[j] & 63;
            m6 = sc[j + 4] & 63;
        } else {
            s6 = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
            m6 = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
        }
        sm[2 * j] = d * (float)s6;
        sm[2 * j + 1] = dmin * (float)m6;
        const uint8_t *chunk = qs + 32 * (j / 2);
        const int shift = (j & 1) ? 4 : 0;
        for (int t = 0; t < 16; ++t) {
            const int lo = (chunk[t] >> shift) & 15, hi = (chunk[t + 16] >> shift) & 15;
            codes[16 * j + t] = (uint8_t)(lo | (hi << 4));
        }
    }
}

// Q5_K super-block (176 bytes, 256 weights, the published layout: d, dmin,
// the 12 packed scale/min bytes of Q4_K, 32 bytes qh whose byte l bit j is
// the fifth bit of element l of sub-block j, then the Q4_K code bytes) -> 8
// sub-blocks: Q4-order low nibbles, a fifth-bit word (bit t = element t),
// and the exact fp32 pair (d * sc_j, dmin * m_j).
inline void repack_q5k_super(const uint8_t *sb, uint8_t *codes, uint32_t *fifth, float *sm) {
    uint8_t q4[144];
    memcpy(q4, sb, 16);
    memcpy(q4 + 16, sb + 48, 128);
    repack_q4k_super(q4, codes, sm);
    const uint8_t *qh = sb + 16;
    for (int j = 0; j < 8; ++j) {
        uint32_t w = 0;
        for (int t = 0; t < 32; ++t) w |= (uint32_t)((qh[t] >> j) & 1u) << t;
        fifth[j] = w;
    }
}

// Q6_K super-block (210 bytes, 256 weights, the published layout: per
// 128-weight half n, element 32m + l has its low nibble in
// ql[64n + 32 (m & 1) + l] (low half of the byte for m < 2) and its high pair
// in bits 2m..2m+1 of qh[32n + l]; then 16 signed scales and d) -> 8 blocks
// of 32: Q4-order low nibbles, packed high pairs, the two scales; and d.
inline void repack_q6k_super(const uint8_t *sb, uint8_t *lo, uint32_t *hi, uint8_t *sc, uint8_t *d) {
    memset(lo, 0, 128);
    memset(hi, 0, 16 * sizeof(uint32_t));
    for (int n = 0; n < 2; ++n)
        for (int m = 0; m < 4; ++m)
            for (int l = 0; l < 32; ++l) {
                const uint8_t lb = sb[64 * n + 32 * (m & 1) + l];
                const uint32_t q_lo = m < 2 ? (lb & 15u) : (uint32_t)(lb >> 4);
                const uint32_t q_hi = (sb[128 + 32 * n + l] >> (2 * m)) & 3u;
                const int b = 4 * n + m, j = l & 15;  // block b, element l of it
                lo[16 * b + j] |= (uint8_t)(q_lo << (l < 16 ? 0 : 4));
                hi[2 * b + (l >> 4)] |= q_hi << (8 * (j & 3) + 2 * (j >> 2));
            }
    memcpy(sc, sb + 192, 16);
    memcpy(d, sb + 208, 2);
}

// Repack canonical blocks (binary16 d, then the code bytes: 18 bytes for
// Q4, 34 for Q8_0; d, 4 fifth-bit bytes, 16 nibble bytes = 22 for Q5_0;
// 144-byte super-blocks of 8 blocks for Q4_K, 210-byte ones for Q6_K) of
// n_experts experts into plane blobs.
inline void repack(const uint8_t *src, uint8_t *dst, int fmt, int n_experts, int rows, int nb, size_t stride) {
    const size_t nblk = (size_t)rows * nb, cb = (size_t)code_bytes(fmt), bb = cb + 2;
    auto work = [&](int e0, int e1) {
        for (int e = e0; e < e1; ++e) {
            if (fmt == kFmtQ4K) {
                const uint8_t *s = src + (size_t)e * (nblk / 8) * 144;
                uint8_t *q = dst + (size_t)e * stride;
                float *sm = (float *)(q + nblk * 16);
                for (size_t u = 0; u < nblk / 8; ++u) repack_q4k_super(s + 144 * u, q + 128 * u, sm + 16 * u);
                continue;
            }
            if (fmt == kFmtQ5K) {
                const uint8_t *s = src + (size_t)e * (nblk / 8) * 176;
                uint8_t *q = dst + (size_t)e * stride;
                uint32_t *fifth = (uint32_t *)(q + nblk * 16);
                float *sm = (float *)(q + nblk * 20);
                for (size_t u = 0; u < nblk / 8; ++u)
                    repack_q5k_super(s + 176 * u, q + 128 * u, fifth + 8 * u, sm + 16 * u);
                continue;
            }
            if (fmt == kFmtQ6K) {
                const uint8_t *s = src + (size_t)e * (nblk / 8) * 210;
                uint8_t *q = dst + (size_t)e * stride;
                for (size_t u = 0; u < nblk / 8; ++u)
                    repack_q6k_super(s + 210 * u, q + 128 * u, (uint32_t *)(q + 16 * nblk + 64 * u),
                                     q + 24 * nblk + 16 * u, q + 26 * nblk + 2 * u);
                continue;
            }
            const uint8_t *s = src + (size_t)e * nblk * bb;
            uint8_t *q = dst + (size_t)e * stride;
            uint8_t *d = q + nblk * cb;
            for (size_t b = 0; b < nblk; ++b) {
                d[2 * b] = s[bb * b];
                d[2 * b + 1] = s[bb * b + 1];
                if (fmt == kFmtQ5) {
                    memcpy(q + 16 * b, s + bb * b + 6, 16);              // nibbles
                    memcpy(q + 16 * nblk + 4 * b, s + bb * b + 2, 4);  // fifth bits
                } else {
                    memcpy(q + cb * b, s + bb * b + 2, cb);
                }
            }
        }
    };
    int nth = (int)std::min<unsigned>(16, std::max(1u, std::thread::hardware_concurrency()));
    if ((size_t)n_experts * nblk < (1u << 16) || nth == 1) {
        work(0, n_experts);
        return;
    }
    nth = std::min(nth, n_experts);
    std::vector<std::thread> th;
    for (int i = 0; i < nth; ++i) th.emplace_back(work, n_experts * i / nth, n_experts * (i + 1) / nth);
    for (auto &x : th) x.join();
}

}  // namespace moe
