// Device-side building blocks shared by the kernels of the expert-cache
// library: the Q4 x int8 block dot, the int8 block quantizer, warp
// reductions, the expert-blob plane layout and the miss / stamp recorder.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kBlock = 32;         // weights / activations per quantization block
constexpr int kBlockBytes = 18;    // canonical Q4 block: binary16 d + 16 code bytes
constexpr int kWarps = 8;          // warps per CTA of the mat-vec kernels
constexpr int kMaxChunk = 8;       // tokens per expert handled per weight pass

// Expert blob in the pool and in pinned host memory ("plane" layout, after
// the repacked quant/scale planes of mx-llama.cpp FEATURES.md):
//   [codes: rows x nb x 16 B][scales: rows x nb x binary16]
// Row r's codes are 16*nb contiguous bytes, so 8 lanes reading 16 B each
// cover 128 contiguous bytes: coalesced 128-bit loads, which the canonical
// 18-byte blocks (not 16-B aligned) do not allow.
__host__ __device__ inline size_t blob_scales_offset(int rows, int nb) { return (size_t)rows * nb * 16; }
__host__ __device__ inline size_t blob_bytes(int rows, int nb) { return (size_t)rows * nb * kBlockBytes; }

// Weight formats: Q4 (16 code bytes per block, w = d (q - 8)), Q8_0 (32
// signed code bytes per block in element order, w = d q) and Q5_0 (16 nibble
// bytes as Q4 plus a 32-bit word of fifth bits, w = d (q - 16)).  Blob
// layout, N = rows x nb blocks: [codes: N x 16 or 32 B][Q5_0 only: fifth
// bits, N x 4 B][scales: N x binary16]; code_bytes counts both code planes.
// Q4_K (256-weight super-blocks with 6-bit sub-block scales and mins) is
// repacked per 32-weight sub-block: Q4-order nibbles, and the exact fp32 pair
// (d * sc, dmin * m) in the scale plane (8 bytes per block instead of the
// canonical 2.25: decoding the packed 6-bit pairs in the kernel measured
// slower than reading the pairs).  Q6_K (16-weight sub-blocks with signed
// 8-bit scales, 6-bit codes) keeps per block the low nibbles in Q4 order
// (16 B), the high bit pairs (8 B: word h, byte b, bits 2i..2i+1 = element
// 16h + 4i + b) and the two sub-block scales (2 B) in its code planes, and
// the super-block's binary16 d in its scale plane: the canonical 26.25 bytes
// per 32 weights.  Q5_K (Q4_K with a fifth code bit) is repacked like Q4_K
// plus a plane of 32-bit fifth-bit words as for Q5_0 (28 bytes per 32).
constexpr int kFmtQ4 = 0, kFmtQ8 = 1, kFmtQ5 = 2, kFmtQ4K = 3, kFmtQ6K = 4, kFmtQ5K = 5;
__host__ __device__ constexpr int code_bytes(int fmt) {
    return fmt == kFmtQ8 ? 32 : (fmt == kFmtQ5 || fmt == kFmtQ5K) ? 20 : fmt == kFmtQ6K ? 26 : 16;
}
__host__ __device__ inline size_t blob_scales_offset_fmt(int fmt, int rows, int nb) {
    return (size_t)rows * nb * code_bytes(fmt);
}
// bytes of the scale plane of n blocks (n a multiple of 8 for the K-quants)
__host__ __device__ inline size_t scale_plane_bytes(int fmt, size_t n) {
    return (fmt == kFmtQ4K || fmt == kFmtQ5K) ? n * 8 : fmt == kFmtQ6K ? n / 8 * 2 : n * 2;
}
__host__ __device__ inline size_t blob_bytes_fmt(int fmt, int rows, int nb) {
    const size_t n = (size_t)rows * nb;
    return n * code_bytes(fmt) + scale_plane_bytes(fmt, n);
}

// Per-activation-block data kept next to the int8 codes: the binary16 scale
// (held as the exactly equal fp32 value) and the sum of the 32 codes, so that
// sum_i (q_w,i - 8) q_a,i = sum_i q_w,i q_a,i - 8 * sum_i q_a,i.
struct BlockScale {
    float d;
    int s;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Quantize one block of 32 values held one per lane: d = binary16(amax/127)
// in fp32, q = clamp(rint(v / d), -127, 127) with the stored binary16 scale
// (round-half-even, IEEE division; this translation unit is compiled without
// fast-math).  An all-zero block (d == 0) gives q = 0.  Lane 0 writes the
// scale and the code sum.
__device__ __forceinline__ void quantize_block_warp(float v, int lane, int8_t *q_out, BlockScale *ds_out) {
    // max of |v| over the warp: non-negative floats order like their bits
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
    float d32 = amax / 127.0f;
    float dd = __half2float(__float2half_rn(d32));
    int q = 0;
    if (dd != 0.0f) {
        float r = rintf(v / dd);
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        q = (int)r;
    }
    const int s = __reduce_add_sync(0xffffffffu, q);
    q_out[lane] = (int8_t)q;
    if (lane == 0) {
        ds_out->d = dd;
        ds_out->s = s;
    }
}

// Raw integer dot of one Q4 block (16 code bytes as 4 words) with 32 int8
// activations (8 words): sum_i q_w,i * q_a,i with q_w in 0..15.  Word i of the
// codes holds elements 4i..4i+3 in its low nibbles and 4i+16..4i+19 in its
// high nibbles.  The caller subtracts 8 * sum(q_a).
__device__ __forceinline__ int q4_dot_raw(const uint4 &w, const int4 &a0, const int4 &a1) {
    const uint32_t m = 0x0F0F0F0Fu;
    int s = 0;
    s = __dp4a((int)(w.x & m), a0.x, s);
    s = __dp4a((int)(w.y & m), a0.y, s);
    s = __dp4a((int)(w.z & m), a0.z, s);
    s = __dp4a((int)(w.w & m), a0.w, s);
    s = __dp4a((int)((w.x >> 4) & m), a1.x, s);
    s = __dp4a((int)((w.y >> 4) & m), a1.y, s);
    s = __dp4a((int)((w.z >> 4) & m), a1.z, s);
    s = __dp4a((int)((w.w >> 4) & m), a1.w, s);
    return s;
}

// Exact int32 block dot sum_i (q_w,i - 8) * q_a,i.
__device__ __forceinline__ int q4_block_dot(const uint4 &w, const int4 &a0, const int4 &a1, int a_sum) {
    return q4_dot_raw(w, a0, a1) - 8 * a_sum;
}

// Streaming 128-bit load of expert weights (read once per pass; works for
// pool slots in HBM and for pinned host memory mapped into the device).
__device__ __forceinline__ uint4 ld_weights(const uint4 *p) { return __ldcs(p); }

__device__ __forceinline__ float ld_scale(const __half *p) { return __half2float(__ldcs(p)); }

// Codes of one weight block held in registers, per format: load block i of a
// blob of n blocks (i = row * nb + block), and its exact int32 dot with 32
// int8 activations (two 16-byte halves a0 = elements 0..15, a1 = 16..31;
// a_sum = their sum).
template <int FMT>
struct WCodes;
template <>
struct WCodes<kFmtQ4> {
    uint4 c;
    __device__ __forceinline__ void load(const uint8_t *blob, size_t, size_t i) {
        c = ld_weights((const uint4 *)blob + i);
    }
    __device__ __forceinline__ int dot(const int4 &a0, const int4 &a1, int a_sum) const {
        return q4_block_dot(c, a0, a1, a_sum);
    }
};
template <>
struct WCodes<kFmtQ8> {
    uint4 lo, hi;  // elements 0..15, 16..31
    __device__ __forceinline__ void load(const uint8_t *blob, size_t, size_t i) {
        const uint4 *p = (const uint4 *)blob + 2 * i;
        lo = ld_weights(p);
        hi = ld_weights(p + 1);
    }
    __device__ __forceinline__ int dot(const int4 &a0, const int4 &a1, int) const {
        int s = __dp4a((int)lo.x, a0.x, 0);
        s = __dp4a((int)lo.y, a0.y, s);
        s = __dp4a((int)lo.z, a0.z, s);
        s = __dp4a((int)lo.w, a0.w, s);
        s = __dp4a((int)hi.x, a1.x, s);
        s = __dp4a((int)hi.y, a1.y, s);
        s = __dp4a((int)hi.z, a1.z, s);
        return __dp4a((int)hi.w, a1.w, s);
    }
};
template <>
struct WCodes<kFmtQ4K> {
    uint4 c;  // Q4-order nibbles of one sub-block
    __device__ __forceinline__ void load(const uint8_t *blob, size_t, size_t i) {
        c = ld_weights((const uint4 *)blob + i);
    }
    // raw sum q_w * q_a (the sub-block's min enters through its scale term)
    __device__ __forceinline__ int dot(const int4 &a0, const int4 &a1, int) const { return q4_dot_raw(c, a0, a1); }
};

// Scale of one weight block and its contribution to a row sum given the
// block's integer dot and the activation block's scale and code sum:
// d_w * d_a * dot, or for Q4_K d_a * (d*sc * dot - dmin*m * sum q_a).
template <int FMT>
struct WScale {
    float s;
    __device__ __forceinline__ void load(const uint8_t *scales, size_t i) {
        s = ld_scale((const __half *)scales + i);
    }
    __device__ __forceinline__ float term(int dot, const BlockScale &a) const { return (float)dot * (s * a.d); }
};
template <>
struct WScale<kFmtQ4K> {
    float2 sm;  // (d * sc_j, dmin * m_j) of the block's sub-block
    __device__ __forceinline__ void load(const uint8_t *scales, size_t i) {
        sm = __ldcs((const float2 *)scales + i);
    }
    __device__ __forceinline__ float term(int dot, const BlockScale &a) const {
        return a.d * (sm.x * (float)dot - sm.y * (float)a.s);
    }
};
template <>
struct WScale<kFmtQ6K> {
    float s;  // the super-block's d
    __device__ __forceinline__ void load(const uint8_t *scales, size_t i) { s = __half2float(__ldg((const __half *)scales + i / 8)); }
    __device__ __forceinline__ float term(int dot, const BlockScale &a) const { return (float)dot * (s * a.d); }
};
template <>
struct WCodes<kFmtQ6K> {
    uint4 lo;      // low nibbles of the 32 codes, Q4 order
    uint2 hi;      // high bit pairs: word h, byte b, bits 2i..2i+1 = element 16h + 4i + b
    int sc0, sc1;  // signed scales of elements 0..15 and 16..31
    __device__ __forceinline__ void load(const uint8_t *blob, size_t n, size_t i) {
        lo = ld_weights((const uint4 *)blob + i);
        hi = __ldcs((const uint2 *)(blob + 16 * n) + i);
        const unsigned s = __ldcs((const unsigned short *)(blob + 24 * n) + i);
        sc0 = (int)(int8_t)(s & 255u);
        sc1 = (int)(int8_t)(s >> 8);
    }
    // sc0 * sum_{i<16} (q_i - 32) a_i + sc1 * sum_{i>=16} (q_i - 32) a_i, with
    // q = low nibble + 16 * high pair (|result| < 2^24: exact in fp32 too)
    __device__ __forceinline__ int dot(const int4 &a0, const int4 &a1, int a_sum) const {
        const uint32_t m4 = 0x0F0F0F0Fu, m2 = 0x03030303u;
        const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w};
        const int aw0[4] = {a0.x, a0.y, a0.z, a0.w}, aw1[4] = {a1.x, a1.y, a1.z, a1.w};
        int l0 = 0, l1 = 0, h0 = 0, h1 = 0, s0 = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            l0 = __dp4a((int)(lw[k] & m4), aw0[k], l0);
            l1 = __dp4a((int)((lw[k] >> 4) & m4), aw1[k], l1);
            h0 = __dp4a((int)((hi.x >> (2 * k)) & m2), aw0[k], h0);
            h1 = __dp4a((int)((hi.y >> (2 * k)) & m2), aw1[k], h1);
            s0 = __dp4a(0x01010101, aw0[k], s0);
        }
        const int s1 = a_sum - s0;
        return sc0 * (l0 + 16 * h0 - 32 * s0) + sc1 * (l1 + 16 * h1 - 32 * s1);
    }
};

// Bits 0..3 of x moved to bit 0 of bytes 0..3 (the four shifted copies do
// not overlap, so the product carries nothing).
__device__ __forceinline__ uint32_t spread4(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }
template <>
struct WCodes<kFmtQ5> {
    uint4 c;     // low nibbles, Q4 order
    uint32_t h;  // bit j = bit 4 of element j
    __device__ __forceinline__ void load(const uint8_t *blob, size_t n, size_t i) {
        c = ld_weights((const uint4 *)blob + i);
        h = __ldcs((const unsigned int *)(blob + 16 * n) + i);
    }
    __device__ __forceinline__ int dot(const int4 &a0, const int4 &a1, int a_sum) const {
        const uint32_t m = 0x0F0F0F0Fu;
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
        const int aw0[4] = {a0.x, a0.y, a0.z, a0.w}, aw1[4] = {a1.x, a1.y, a1.z, a1.w};
        int s = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = (cw[k] & m) | (spread4((h >> (4 * k)) & 15u) << 4);
            const uint32_t hi = ((cw[k] >> 4) & m) | (spread4((h >> (16 + 4 * k)) & 15u) << 4);
            s = __dp4a((int)lo, aw0[k], s);
            s = __dp4a((int)hi, aw1[k], s);
        }
        return s - 16 * a_sum;
    }
};
// Q5_K: the codes of Q5_0 without its offset (raw sum q * a, q in 0..31); the
// sub-block's scale and min enter through WScale<kFmtQ5K>
template <>
struct WCodes<kFmtQ5K> : WCodes<kFmtQ5> {
    __device__ __forceinline__ int dot(const int4 &a0, const int4 &a1, int a_sum) const {
        return WCodes<kFmtQ5>::dot(a0, a1, a_sum) + 16 * a_sum;
    }
};
template <>
struct WScale<kFmtQ5K> : WScale<kFmtQ4K> {};

// Cache-state arrays of one forward: pointer tables, local slots, stamps and
// the miss log (Zapdev-labs/a6000-custom-kernels, pointer-table GEMV).
struct CacheView {
    const uint64_t *tbl;       // [n_tensors][E]: pool address (bit0 = 0) or host address | 1
    const int32_t *slot;       // [n_tensors][E]: stamp index of the expert's pool slot, or -1
    uint32_t *stamps;          // [n_tensors * slots_per_tensor], indexed by stamp index
    uint32_t *miss_bitmap;     // [n_tensors][ceil(E/32)]
    uint32_t *miss_list;       // [miss_cap]
    uint32_t *miss_count;      // [1]
    const uint32_t *clock;     // [1]: token clock after the last promotion pass
    unsigned long long *cold_reads;  // [1]: (tensor, expert) zero-copy passes
    uint32_t *hit_bitmap;      // [hit_words]: stamp indices hit since the last promotion pass (or null)
    int E, slots_per_tensor, bitmap_words, miss_cap, hit_words;
    int clock_tokens;          // tokens of the step this launch belongs to: reads stamp *clock + clock_tokens
};

// Record one (tensor, expert) read: a cold read sets its bit in the miss
// bitmap and, when newly set, appends (tensor << 12 | expert) to the miss
// list; a pool hit writes the step's clock into the slot's stamp and sets
// the slot's bit in the hit bitmap (the hit count of the step, read by the
// promotion pass without reading every stamp).  The host chooses the stamp
// index of a slot: tensor * slots_per_tensor + local slot for per-tensor
// pools, the arena slot for one pool shared by all layers.
__device__ __forceinline__ void record_read(const CacheView &cv, int tid, int e, uint64_t entry, uint32_t step_clock) {
    if (entry & 1ull) {
        uint32_t bit = 1u << (e & 31);
        uint32_t old = atomicOr(&cv.miss_bitmap[(size_t)tid * cv.bitmap_words + (e >> 5)], bit);
        if (!(old & bit)) {
            uint32_t pos = atomicAdd(cv.miss_count, 1u);
            if (pos < (uint32_t)cv.miss_cap) cv.miss_list[pos] = ((uint32_t)tid << 12) | (uint32_t)e;
        }
    } else {
        int s = cv.slot[(size_t)tid * cv.E + e];
        if (s >= 0) {
            cv.stamps[s] = step_clock;
            if (cv.hit_bitmap) atomicOr(&cv.hit_bitmap[s >> 5], 1u << (s & 31));
        }
    }
}

}  // namespace moe
