// Host build of the library's weight-format path for the CPU test suite: the
// registration repack (csrc/repack.h) and the per-block code and scale traits
// the kernels use (WCodes<FMT>, WScale<FMT> in csrc/common.cuh), compiled by
// the host compiler from the library's own sources.  The device intrinsics
// those headers name get host stand-ins here: loads read memory (and count
// any load outside the blob under test or off its natural alignment, which
// on the GPU would be an out-of-bounds read or a misaligned-address fault),
// and __dp4a is the four-way signed byte dot it is defined as.  The warp and
// atomic primitives are never reached from this file's entry points.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

namespace {
const unsigned char *g_lo = nullptr, *g_hi = nullptr;
long g_bad = 0;

template <class T>
T checked_load(const T *p) {
    const unsigned char *b = (const unsigned char *)p;
    if (b < g_lo || b + sizeof(T) > g_hi || ((uintptr_t)b % sizeof(T)) != 0) {
        ++g_bad;
        return T{};
    }
    T v;
    memcpy(&v, p, sizeof(T));
    return v;
}
}  // namespace

template <class T>
static inline T __ldcs(const T *p) { return checked_load(p); }
template <class T>
static inline T __ldg(const T *p) { return checked_load(p); }

// sum over the four byte lanes of a * b (both signed), plus c
static inline int __dp4a(int a, int b, int c) {
    int s = c;
    for (int i = 0; i < 4; ++i) s += (int)(int8_t)(a >> (8 * i)) * (int)(int8_t)(b >> (8 * i));
    return s;
}
static inline unsigned __float_as_uint(float f) {
    unsigned u;
    memcpy(&u, &f, 4);
    return u;
}
static inline float __uint_as_float(unsigned u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}
template <class T>
static inline T __shfl_xor_sync(unsigned, T, int) { abort(); }
static inline unsigned __reduce_max_sync(unsigned, unsigned) { abort(); }
static inline int __reduce_add_sync(unsigned, int) { abort(); }
static inline unsigned atomicOr(unsigned *, unsigned) { abort(); }
static inline unsigned atomicAdd(unsigned *, unsigned) { abort(); }

#include "repack.h"

namespace {

template <int FMT>
void block_terms(const uint8_t *blob, int rows, int nb, const int8_t *qa, const float *da, int32_t *dots,
                 float *terms) {
    const size_t n = (size_t)rows * nb;
    const uint8_t *scales = blob + moe::blob_scales_offset_fmt(FMT, rows, nb);
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const size_t i = (size_t)r * nb + b;
            int4 a0, a1;
            memcpy(&a0, qa + 32 * b, 16);
            memcpy(&a1, qa + 32 * b + 16, 16);
            int a_sum = 0;
            for (int t = 0; t < 32; ++t) a_sum += qa[32 * b + t];
            moe::WCodes<FMT> w;
            w.load(blob, n, i);
            moe::WScale<FMT> s;
            s.load(scales, i);
            const int dot = w.dot(a0, a1, a_sum);
            dots[i] = dot;
            terms[i] = s.term(dot, moe::BlockScale{da[b], a_sum});
        }
}

}  // namespace

extern "C" {

size_t fp_blob_bytes(int fmt, int rows, int nb) { return moe::blob_bytes_fmt(fmt, rows, nb); }

void fp_repack(const uint8_t *src, uint8_t *dst, int fmt, int n_experts, int rows, int nb, size_t stride) {
    moe::repack(src, dst, fmt, n_experts, rows, nb, stride);
}

// dots[r][b] = the block's integer dot as the kernels form it, terms[r][b] =
// its contribution to the row sum (d_a = da[b]); returns the number of loads
// that fell outside [blob, blob + blob_bytes) or off their alignment.
long fp_block_terms(int fmt, const uint8_t *blob, size_t blob_bytes, int rows, int nb, const int8_t *qa,
                    const float *da, int32_t *dots, float *terms) {
    g_lo = blob;
    g_hi = blob + blob_bytes;
    g_bad = 0;
    switch (fmt) {
        case moe::kFmtQ4: block_terms<moe::kFmtQ4>(blob, rows, nb, qa, da, dots, terms); break;
        case moe::kFmtQ8: block_terms<moe::kFmtQ8>(blob, rows, nb, qa, da, dots, terms); break;
        case moe::kFmtQ5: block_terms<moe::kFmtQ5>(blob, rows, nb, qa, da, dots, terms); break;
        case moe::kFmtQ4K: block_terms<moe::kFmtQ4K>(blob, rows, nb, qa, da, dots, terms); break;
        case moe::kFmtQ6K: block_terms<moe::kFmtQ6K>(blob, rows, nb, qa, da, dots, terms); break;
        case moe::kFmtQ5K: block_terms<moe::kFmtQ5K>(blob, rows, nb, qa, da, dots, terms); break;
        default: return -1;
    }
    return g_bad;
}

}  // extern "C"
