// Prefill path of the routed-expert FFN: a grouped per-expert GEMM on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM), over tokens
// sorted by expert, only over (expert, tile) pairs that hold tokens.
//
// Sources: mihailescu2m/llama.cpp, Metal kernels (MUL_MAT_ID restricted to the
// used tiles: no work is launched for an (expert, tile) pair without
// tokens); neurall/llama.cpp, "How it works" (prompts in few big passes, each
// expert upload serving many prompt tokens); the Q4 / q8_1 block formats of
// the mat-vec kernels (Zapdev-labs/a6000-custom-kernels; mx-llama.cpp
// FEATURES.md).
//
// Arithmetic.  sm_103a has no integer tcgen05 MMA (ptxas rejects kind::i8), so
// the MMA is kind::f16 with integer-valued fp16 operands: weight codes q-8 in
// [-8, 7] and activation codes in [-127, 127] are exact in fp16, and the fp32
// sum of the 32 products of one quantization block (|sum| <= 32512) is exact.
// Each 32-wide K block is accumulated into its own TMEM buffer, so the MMA
// produces exactly the int32 block dots of the mat-vec path; epilogue warps
// then add d_w * d_a * sumi in fp32 (fma.rn.f32x2), as the mat-vec does.
//
// Tile: M = 128 weight rows (TMEM lanes) x N tokens (TMEM columns), K staged
// 64 at a time (two quantization blocks = one 128-B swizzle row of fp16).
// Warp roles (10 warps): 0 TMA producer of the token tile; 1 TMEM owner and
// MMA issuer; 2-5 weight converters (Q4 codes read through the expert table,
// from the HBM pool or zero-copy from pinned host memory, turned into fp16
// and stored in the 128-B swizzled K-major layout); 6-9 epilogue (TMEM lane
// quarter = warp % 4).  Gate/up tiles hold two A operands (gate rows and up
// rows) so SwiGLU and the quantization of h happen in the epilogue; the 32
// rows of one h block are the 32 lanes of one epilogue warp.
//
// Every mbarrier wait is bounded (about 2 s of SM clock): on expiry the CTA
// sets an error bit, all roles leave their loops, in-flight copies and MMAs
// are drained with bounded waits and TMEM is freed before the CTA exits.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace gemm {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int W_TMA = 0, W_MMA = 1, W_CONV = 2, W_EPI = 6;
constexpr long long kTimeoutCycles = 4000000000ll;

template <bool DUAL>
struct Cfg {
    static constexpr int BN = DUAL ? 64 : 128;
    static constexpr int NA = DUAL ? 2 : 1;
    static constexpr int STAGES = DUAL ? 3 : 4;   // A/B pipeline slots
    static constexpr int RR = 8;                  // raw prefetch ring (converter cp.async)
    static constexpr int PD = RR - 1;             // prefetch distance in stages
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    // per-slot scales for the epilogue: weight scales [NA][BM][2] fp16 and
    // activation scales [2][BN] fp32 of the slot's two K blocks
    static constexpr int WS_BYTES = NA * BM * 2 * 2;
    static constexpr int AS_BYTES = 2 * BN * 4;
    static constexpr int SLOT_BYTES = NA * A_BYTES + B_BYTES + WS_BYTES + AS_BYTES;
    static constexpr int SLOT_STRIDE = (SLOT_BYTES + 1023) / 1024 * 1024;
    // raw ring entry: codes [NA][BM][32 B], weight scales, activation scales
    static constexpr int RAW_CODES = NA * BM * 32;
    static constexpr int RAW_BYTES = RAW_CODES + WS_BYTES + AS_BYTES;
    static constexpr int RAW_OFF = STAGES * SLOT_STRIDE;
    static constexpr int TBUF = NA * BN;          // TMEM columns per K-block buffer
    static constexpr int NTBUF = 512 / TBUF;      // K-block buffers in TMEM
    static constexpr int BAR_OFF = RAW_OFF + RR * RAW_BYTES;
    static constexpr int NBARS = 2 * STAGES + 2 * NTBUF;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = MISC_OFF + 16 + 1024;  // + alignment slack
    // epilogue warps: EPI_SPLIT per TMEM lane quarter, each owning BN / EPI_SPLIT
    // token columns (32 for gate/up with its two tensors, 64 for down)
    static constexpr int N_EPI = 8;
    static constexpr int EPI_SPLIT = N_EPI / 4;
    static constexpr int NTHREADS = (W_EPI + N_EPI) * 32;
};

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
// One try: the thread is suspended (not spinning) until the phase completes
// or about kSuspendNs pass, so waiting warps leave their issue slots to the
// converter and epilogue warps.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred P;\nmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, %3;\nselp.u32 %0, 1, 0, P;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Bounded wait: false when the CTA is aborting or the wait expired (then the
// abort flag and an error bit are set).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *err,
                                          int code) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try(bar, parity)) return true;
        // the abort flag and the clock are checked every 64 tests
        if ((n & 63) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kTimeoutCycles) {
                *abort_flag = 1;
                atomicOr(err, code);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void cp_async(uint32_t dst, const void *src, int bytes, bool valid) {
    const int n = valid ? bytes : 0;  // 0: zero fill, nothing read
    if (bytes == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-B swizzle, 8-row groups 1024 B
// apart (SBO), Blackwell descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: D fp32, A/B fp16, both K-major, N, M.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive TMEM columns of this warp's 32 lanes (raw fp32 bits)
__device__ __forceinline__ void tmem_ld16u(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 32 consecutive TMEM columns of this warp's 32 lanes (one fp32 per column)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Packed fp32 pairs (two IEEE round-to-nearest operations per instruction).
__device__ __forceinline__ unsigned long long pk2(uint32_t lo, uint32_t hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
// acc{0,1} += sum{0,1} * (dw * da{0,1}): the scale products and the
// accumulation as packed fp32 pairs (mul.rn.f32x2, fma.rn.f32x2).
__device__ __forceinline__ void fma_scaled2(float &acc0, float &acc1, uint32_t sum0, uint32_t sum1, float da0, float da1,
                                            float dw) {
    asm("{\n.reg .b64 a, p, d, w, s;\n"
        "mov.b64 a, {%0, %1};\nmov.b64 p, {%2, %3};\nmov.b64 d, {%4, %5};\nmov.b64 w, {%6, %6};\n"
        "mul.rn.f32x2 s, w, d;\nfma.rn.f32x2 a, p, s, a;\nmov.b64 {%0, %1}, a;\n}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(sum0), "r"(sum1), "f"(da0), "f"(da1), "f"(dw));
}


// acc{0,1} += p{0,1} * s{0,1}, two IEEE fp32 fused multiply-adds.
__device__ __forceinline__ void fma2(float &a0, float &a1, float p0, float p1, float s0, float s1) {
    unsigned long long acc, pp, ss;
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(pp) : "f"(p0), "f"(p1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(ss) : "f"(s0), "f"(s1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(pp), "l"(ss));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

// Q4 codes of one row and two quantization blocks (32 B) -> 64 fp16 values
// (q - 8) in K order, stored as 8 16-byte chunks of the row in the 128-B
// swizzled layout (chunk c of row r of an 8-row group sits at chunk c ^ r).
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int sel, int hi) {
    // two bytes of w (selected) -> their low (hi=0) or high (hi=1) nibbles as
    // the fp16 pair (1024 + n0, 1024 + n1), then minus (1032, 1032)
    uint32_t t = __byte_perm(w, 0, sel);
    if (hi) t >>= 4;
    t = (t & 0x000F000Fu) | 0x64006400u;
    __half2 h = *reinterpret_cast<__half2 *>(&t);
    h = __hsub2(h, __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408)));
    return *reinterpret_cast<uint32_t *>(&h);
}

// Four codes (one nibble per byte of n, values 0..15) -> two fp16 pairs
// (q0 - 8, q1 - 8), (q2 - 8, q3 - 8): the bytes are placed under the fp16
// exponent byte 0x64 (1024 + q, exact) and 1032 is subtracted (exact).
__device__ __forceinline__ void nib4(uint32_t n, uint32_t &p01, uint32_t &p23) {
    const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    uint32_t a = __byte_perm(n, 0x64646464u, 0x5150);  // (1024 + q0, 1024 + q1)
    uint32_t b = __byte_perm(n, 0x64646464u, 0x5352);  // (1024 + q2, 1024 + q3)
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), off);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), off);
    p01 = *reinterpret_cast<uint32_t *>(&ha);
    p23 = *reinterpret_cast<uint32_t *>(&hb);
}

__device__ __forceinline__ void convert_store_row(uint8_t *tile, int r, uint4 c0, uint4 c1) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint8_t *rowbase = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const uint32_t *q = w + 4 * blk;  // 16 code bytes of this block
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            // part 0: elements 0..7 (low nibbles of bytes 0..7), 1: 8..15
            // (low, bytes 8..15), 2: 16..23 (high, bytes 0..7), 3: 24..31
            const uint32_t wa = q[(part & 1) * 2], wb = q[(part & 1) * 2 + 1];
            const uint32_t na = (part >> 1) ? (wa >> 4) & 0x0F0F0F0Fu : wa & 0x0F0F0F0Fu;
            const uint32_t nb = (part >> 1) ? (wb >> 4) & 0x0F0F0F0Fu : wb & 0x0F0F0F0Fu;
            uint4 out;
            nib4(na, out.x, out.y);
            nib4(nb, out.z, out.w);
            const int chunk = blk * 4 + part;
            *reinterpret_cast<uint4 *>(rowbase + ((chunk ^ (r & 7)) << 4)) = out;
        }
    }
}

// tile index -> (used expert u, row tile, token tile, valid token columns),
// from the per-tile records the tiling kernel writes (token tile innermost).
__device__ __forceinline__ void decode_tile(const uint2 *rec, int t, int &u, int &row_tile, int &tok_tile,
                                            int &ncols) {
    const uint2 r = __ldg(rec + t);
    u = (int)(r.x & 0xffffu);
    row_tile = (int)(r.x >> 16);
    tok_tile = (int)(r.y & 0xffffu);
    ncols = (int)(r.y >> 16);
}

// Stage cursor over the flattened (tile, K stage) sequence of one CTA.
// The tile's expert-table entries (weight blobs) and first token position
// are looked up once per tile, not per stage.
struct StageCur {
    int t, kt, u, rt, tt, nc, pos0;
    const uint8_t *blob[2];
    bool valid;
};

template <int BN>
__device__ __forceinline__ void cur_tile(StageCur &c, const GemmParams &p, int n_uniq) {
    decode_tile(p.tile_rec, c.t, c.u, c.rt, c.tt, c.nc);
    const int e = p.uniq_e[c.u];
    c.blob[0] = (const uint8_t *)(uintptr_t)(p.tbl[0][e] & ~1ull);
    c.blob[1] = p.tbl[1] ? (const uint8_t *)(uintptr_t)(p.tbl[1][e] & ~1ull) : c.blob[0];
    c.pos0 = p.uniq_off[c.u] + c.tt * BN;
}

template <int BN>
__device__ __forceinline__ void cur_init(StageCur &c, const GemmParams &p, int n_uniq, int total) {
    c.t = blockIdx.x;
    c.kt = 0;
    c.valid = c.t < total;
    if (c.valid) cur_tile<BN>(c, p, n_uniq);
}

template <int BN>
__device__ __forceinline__ void cur_next(StageCur &c, const GemmParams &p, int n_uniq, int total, int nkt) {
    if (!c.valid) return;
    if (++c.kt == nkt) {
        c.kt = 0;
        c.t += gridDim.x;
        c.valid = c.t < total;
        if (c.valid) cur_tile<BN>(c, p, n_uniq);
    }
}

template <bool DUAL>
__global__ void __launch_bounds__(Cfg<DUAL>::NTHREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmB, GemmParams p) {
    using C = Cfg<DUAL>;
    constexpr int BN = C::BN, NA = C::NA, NTBUF = C::NTBUF, STAGES = C::STAGES;
    constexpr int N_EPI = C::N_EPI, EPI_SPLIT = C::EPI_SPLIT;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + C::BAR_OFF);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * STAGES, tfull0 = empty0 + 8 * STAGES,
                   tempty0 = tfull0 + 8 * NTBUF;
    volatile uint32_t *tmem_slot = (volatile uint32_t *)(smem + C::MISC_OFF);
    volatile int *abort_flag = (volatile int *)(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1 + 4);       // TMA expect-tx arrive + 4 converter warps
            mbar_init(empty0 + 8 * s, 1 + N_EPI);  // MMA commit + the epilogue warps
        }
        for (int j = 0; j < NTBUF; ++j) {
            mbar_init(tfull0 + 8 * j, 1);
            mbar_init(tempty0 + 8 * j, N_EPI);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32((const void *)tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_uniq = *p.n_uniq;
    const int total = n_uniq > 0 ? p.tile_off[n_uniq] : 0;
    const int nkt = p.K / BK;
    const int nbk = p.K / kBlock;
    const size_t scale_off = blob_scales_offset(p.rows, nbk);
    auto slot_ptr = [&](int slot) { return smem + slot * C::SLOT_STRIDE; };

    if (warp == W_TMA) {
        if (lane == 0) {
            int it = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                int u, rt, tt, nc;
                decode_tile(p.tile_rec, t, u, rt, tt, nc);
                const int pos0 = p.uniq_off[u] + tt * BN;
                for (int kt = 0; kt < nkt; ++kt, ++it) {
                    const int slot = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!mbar_wait(empty0 + 8 * slot, ph ^ 1u, abort_flag, p.error, 2)) goto tma_done;
                    mbar_arrive_tx(full0 + 8 * slot, C::B_BYTES);
                    tma_load_2d(smem_u32(slot_ptr(slot) + NA * C::A_BYTES), &tmB, kt * BK, pos0, full0 + 8 * slot);
                }
            }
        tma_done:;
        }
    } else if (warp == W_MMA) {
        if (lane == 0) {
            int it = 0, qc = 0;
            // the tile's MMA width: its valid token columns rounded up to 16
            // (the record of the next tile is requested a tile ahead)
            uint2 rec_next = blockIdx.x < total ? __ldg(p.tile_rec + blockIdx.x) : make_uint2(0, 0);
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                const int ncols = (int)(rec_next.y >> 16);
                if (t + (int)gridDim.x < total) rec_next = __ldg(p.tile_rec + t + gridDim.x);
                const int nmma = min(BN, (ncols + 15) & ~15);
                const uint32_t idesc = idesc_f16(BM, nmma < 16 ? 16 : nmma);
                for (int kt = 0; kt < nkt; ++kt, ++it) {
                    const int slot = it % STAGES;
                    if (!mbar_wait(full0 + 8 * slot, (uint32_t)(it / STAGES) & 1u, abort_flag, p.error, 4))
                        goto mma_done;
                    tc_fence_after();
                    uint8_t *st = slot_ptr(slot);
                    const uint64_t db = sdesc(smem_u32(st + NA * C::A_BYTES));
                    for (int blk = 0; blk < 2; ++blk, ++qc) {
                        const int j = qc % NTBUF;
                        if (!mbar_wait(tempty0 + 8 * j, ((uint32_t)(qc / NTBUF) & 1u) ^ 1u, abort_flag, p.error, 8))
                            goto mma_done;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t koff = (uint64_t)((blk * 32 + kk * 16) * 2) >> 4;
#pragma unroll
                            for (int a = 0; a < NA; ++a) {
                                const uint64_t da = sdesc(smem_u32(st + a * C::A_BYTES));
                                mma_f16(tmem + (uint32_t)(j * C::TBUF + a * BN), da + koff, db + koff, idesc,
                                        kk > 0 ? 1u : 0u);
                            }
                        }
                        mma_commit(tfull0 + 8 * j);
                    }
                    mma_commit(empty0 + 8 * slot);
                }
            }
        mma_done:;
        }
    } else if (warp < W_EPI) {
        // Converters: thread r owns row r of the A tiles.  Raw Q4 codes and
        // both scale sets of stage s are fetched with cp.async PD stages ahead
        // into raw ring entry s % RR; stage s is then converted into its slot.
        const int r = threadIdx.x - W_CONV * 32;
        uint8_t *raw = smem + C::RAW_OFF;
        StageCur fc;  // fetch cursor; conversion only counts stages
        cur_init<BN>(fc, p, n_uniq, total);
        const int n_stages = blockIdx.x < total ? ((total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1) * nkt : 0;
        auto fetch = [&](const StageCur &c, int rs) {
            uint8_t *ent = raw + rs * C::RAW_BYTES;
            if (c.valid) {
                const int row = c.rt * BM + r;
                const bool vrow = row < p.rows;
                const int srow = vrow ? row : 0;
#pragma unroll
                for (int a = 0; a < NA; ++a) {
                    const uint8_t *blob = c.blob[a];
                    const uint8_t *src = blob + ((size_t)srow * nbk + 2 * c.kt) * 16;
                    const uint32_t dst = smem_u32(ent + (a * BM + r) * 32);
                    cp_async(dst, src, 16, vrow);
                    cp_async(dst + 16, src + 16, 16, vrow);
                    const uint8_t *ssrc = blob + scale_off + ((size_t)srow * nbk + 2 * c.kt) * 2;
                    cp_async(smem_u32(ent + C::RAW_CODES + (a * BM + r) * 4), ssrc, 4, vrow);
                }
                const int pos0 = c.pos0;
                for (int i = r; i < 2 * BN; i += 128) {
                    const int q = i / BN, col = i - q * BN;
                    const int pos = pos0 + col;
                    const bool v = pos < p.A_pad;
                    const float *src = p.a_scaleT + (size_t)(2 * c.kt + q) * p.A_pad + (v ? pos : 0);
                    cp_async(smem_u32(ent + C::RAW_CODES + C::WS_BYTES + i * 4), src, 4, v);
                }
            }
            cp_commit();
        };
        for (int i = 0; i < C::PD; ++i) {
            fetch(fc, i % C::RR);
            cur_next<BN>(fc, p, n_uniq, total, nkt);
        }
        int it = 0;
        while (it < n_stages) {
            fetch(fc, (it + C::PD) % C::RR);
            cur_next<BN>(fc, p, n_uniq, total, nkt);
            cp_wait<C::PD>();
            const uint8_t *ent = raw + (it % C::RR) * C::RAW_BYTES;
            const int slot = it % STAGES;
            const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(empty0 + 8 * slot, ph ^ 1u, abort_flag, p.error, 16);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            uint8_t *st = slot_ptr(slot);
#pragma unroll
            for (int a = 0; a < NA; ++a) {
                const uint4 *cs = (const uint4 *)(ent + (a * BM + r) * 32);
                convert_store_row(st + a * C::A_BYTES, r, cs[0], cs[1]);
                // this row's two weight scales of the stage
                *(uint32_t *)(st + NA * C::A_BYTES + C::B_BYTES + (a * BM + r) * 4) =
                    *(const uint32_t *)(ent + C::RAW_CODES + (a * BM + r) * 4);
            }
            for (int i = r; i < 2 * BN; i += 128)
                *(float *)(st + NA * C::A_BYTES + C::B_BYTES + C::WS_BYTES + i * 4) =
                    *(const float *)(ent + C::RAW_CODES + C::WS_BYTES + i * 4);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full0 + 8 * slot);
            ++it;
        }
        cp_wait<0>();
    } else {
        // epilogue: TMEM lane quarter = warp % 4 (thread = weight row), half =
        // which HC token columns this warp owns.  Per K stage: one wait (the
        // MMA's commit after the stage's second block covers the first), the
        // activation scales of the warp's columns read once per block, the
        // block sums read 32 columns per TMEM load, and the scaling as packed
        // fp32 pairs: s = d_w * d_a (mul.f32x2), acc += sum * s (fma.f32x2).
        const int quarter = warp & 3;
        const int half = (warp - W_EPI) >> 2;  // which column part this warp owns
        constexpr int HC = BN / EPI_SPLIT;      // token columns per epilogue warp
        static_assert(HC % 32 == 0, "32-column groups per epilogue warp");
        const int r = quarter * 32 + lane;
        int qc = 0, it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int u, rt, tt, ncols;
            decode_tile(p.tile_rec, t, u, rt, tt, ncols);
            const int ncw = ncols - half * HC;  // this warp's valid columns (may be <= 0)
            const int row = rt * BM + r;
            const bool vrow = row < p.rows;
            const int pos0 = p.uniq_off[u] + tt * BN + half * HC;
            const int pos_end = p.uniq_off[u + 1];
            float acc[NA][HC];
#pragma unroll
            for (int a = 0; a < NA; ++a)
#pragma unroll
                for (int c = 0; c < HC; ++c) acc[a][c] = 0.0f;
            for (int kt = 0; kt < nkt; ++kt, ++it, qc += 2) {
                const int slot = it % STAGES;
                const uint8_t *st = slot_ptr(slot);
                const int j0 = qc % NTBUF, j1 = (qc + 1) % NTBUF;
                bool ok = true;
                // the slot's scales were written before its full barrier
                // completed; the second block's commit covers both blocks
                if (lane == 0) {
                    ok = mbar_wait(full0 + 8 * slot, (uint32_t)(it / STAGES) & 1u, abort_flag, p.error, 64) &&
                         mbar_wait(tfull0 + 8 * j1, (uint32_t)((qc + 1) / NTBUF) & 1u, abort_flag, p.error, 32);
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) goto epi_done;
                tc_fence_after();
                uint32_t wsc[NA];
#pragma unroll
                for (int a = 0; a < NA; ++a)
                    wsc[a] = *(const uint32_t *)(st + NA * C::A_BYTES + C::B_BYTES + (a * BM + r) * 4);
                const float *asc = (const float *)(st + NA * C::A_BYTES + C::B_BYTES + C::WS_BYTES) + half * HC;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const int j = blk ? j1 : j0;
                    const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(j * C::TBUF + half * HC);
                    float dw[NA];
#pragma unroll
                    for (int a = 0; a < NA; ++a) {
                        const uint32_t dwb = blk ? (wsc[a] >> 16) : (wsc[a] & 0xffffu);
                        dw[a] = __half2float(__ushort_as_half((unsigned short)dwb));
                    }
                    const float2 *dq2 = reinterpret_cast<const float2 *>(asc + blk * BN);
#pragma unroll
                    for (int cb = 0; cb < HC; cb += 16) {
                        if (cb >= ncw) break;  // columns past the tile's tokens (warp-uniform)
#pragma unroll
                        for (int a = 0; a < NA; ++a) {
                            // block sums of 16 columns of tensor a
                            uint32_t pv[16];
                            tmem_ld16u(tb + (uint32_t)(a * BN + cb), pv);
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const float2 d2 = dq2[(cb >> 1) + c];  // activation scales: broadcast reads
                                fma_scaled2(acc[a][cb + 2 * c], acc[a][cb + 2 * c + 1], pv[2 * c], pv[2 * c + 1], d2.x,
                                            d2.y, dw[a]);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(tempty0 + 8 * j0);
                    mbar_arrive(tempty0 + 8 * j1);
                    mbar_arrive(empty0 + 8 * slot);
                }
            }
            // tile outputs (this warp's token columns); the assignment ids of
            // the columns are fetched once (lane i: columns i, i + 32, ...)
            int asg_l[HC / 32];
#pragma unroll
            for (int i = 0; i < HC / 32; ++i) {
                const int pos = pos0 + i * 32 + lane;
                asg_l[i] = pos < pos_end ? __ldg(p.assign + pos) : 0;
            }
            if (DUAL) {
                const int fb = (rt * BM + quarter * 32) / kBlock;  // h block index along F
                const bool vblk = rt * BM + quarter * 32 < p.rows;
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    if (c >= ncw) break;  // warp-uniform
                    const int pos = pos0 + c;
                    const float g = acc[0][c], uu = acc[NA - 1][c];
                    const float h = g * uu / (1.0f + expf(-g));
                    const float amax = warp_max(fabsf(h));
                    const float dd = __half2float(__float2half_rn(amax / 127.0f));
                    int qv = 0;
                    if (dd != 0.0f) qv = (int)fminf(fmaxf(rintf(h / dd), -127.0f), 127.0f);
                    const int s = warp_sum_i(qv);
                    const int a = __shfl_sync(0xffffffffu, asg_l[c / 32], c % 32);
                    if (vblk && pos < pos_end) {
                        p.hq16[(size_t)pos * p.F_out + row] = __int2half_rn(qv);
                        p.hq[(size_t)a * p.F_out + row] = (int8_t)qv;
                        if (lane == 0) {
                            p.hdT[(size_t)fb * p.A_pad + pos] = dd;
                            p.hds[(size_t)a * (p.F_out / kBlock) + fb] = BlockScale{dd, s};
                        }
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    if (c >= ncw) break;  // warp-uniform
                    const int pos = pos0 + c;
                    const int a = __shfl_sync(0xffffffffu, asg_l[c / 32], c % 32);
                    if (vrow && pos < pos_end) p.o[(size_t)a * p.rows + row] = acc[0][c];
                }
            }
        }
    epi_done:;
    }

    // drain: after an abort, give the copies and MMAs this CTA issued a
    // bounded time (about 10 ms) to land, then free TMEM
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < 20000000ll) {
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

}  // namespace gemm

// ---------------------------------------------------------------- prefill helpers
// Per used expert: cumulative tile counts of the gate/up and down GEMMs, and
// the miss / stamp record of the layer's three tensors.
__global__ void tiling_kernel(TilingParams p) {
    __shared__ int warp_tot[33];
    const int n_uniq = *p.n_uniq;
    const uint32_t step_clock = *p.cv.clock + (uint32_t)p.cv.clock_tokens;
    for (int u = threadIdx.x; u < n_uniq; u += blockDim.x) {
        const int e = p.uniq_e[u];
        for (int kd = 0; kd < 3; ++kd) {
            const int tid = p.tid0 + kd;
            record_read(p.cv, tid, e, p.cv.tbl[(size_t)tid * p.cv.E + e], step_clock);
        }
    }
    int run_gu = 0, run_dn = 0;
    for (int base = 0; base < n_uniq; base += blockDim.x) {
        const int u = base + threadIdx.x;
        int tg = 0, td = 0;
        if (u < n_uniq) {
            const int n = p.uniq_off[u + 1] - p.uniq_off[u];
            tg = p.rt_gu * ((n + p.bn_gu - 1) / p.bn_gu);
            td = p.rt_dn * ((n + p.bn_dn - 1) / p.bn_dn);
        }
        // inclusive warp scans then block offsets, for both counts
        int ig = tg, id = td;
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int a = __shfl_up_sync(0xffffffffu, ig, o), b = __shfl_up_sync(0xffffffffu, id, o);
            if (lane >= o) {
                ig += a;
                id += b;
            }
        }
        __shared__ int wg[32], wd[32];
        if (lane == 31) {
            wg[wid] = ig;
            wd[wid] = id;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int sg = 0, sd = 0;
            for (int w = 0; w < nw; ++w) {
                int a = wg[w], b = wd[w];
                wg[w] = sg;
                wd[w] = sd;
                sg += a;
                sd += b;
            }
            warp_tot[0] = sg;
            warp_tot[1] = sd;
        }
        __syncthreads();
        if (u < n_uniq) {
            p.tile_off_gu[u] = run_gu + wg[wid] + ig - tg;
            p.tile_off_dn[u] = run_dn + wd[wid] + id - td;
        }
        run_gu += warp_tot[0];
        run_dn += warp_tot[1];
        __syncthreads();
    }
    __syncthreads();
    // per-tile records: (u | row tile << 16, token tile | valid columns << 16)
    for (int u = threadIdx.x; u < n_uniq; u += blockDim.x) {
        const int n = p.uniq_off[u + 1] - p.uniq_off[u];
        const int ng = (n + p.bn_gu - 1) / p.bn_gu, nd = (n + p.bn_dn - 1) / p.bn_dn;
        const int bg = p.tile_off_gu[u], bd = p.tile_off_dn[u];
        for (int i = 0; i < p.rt_gu * ng; ++i) {
            const int rt = i / ng, tt = i - rt * ng;
            if (bg + i < p.cap_gu)
                p.rec_gu[bg + i] = make_uint2((unsigned)u | ((unsigned)rt << 16),
                                              (unsigned)tt | ((unsigned)min(p.bn_gu, n - tt * p.bn_gu) << 16));
        }
        for (int i = 0; i < p.rt_dn * nd; ++i) {
            const int rt = i / nd, tt = i - rt * nd;
            if (bd + i < p.cap_dn)
                p.rec_dn[bd + i] = make_uint2((unsigned)u | ((unsigned)rt << 16),
                                              (unsigned)tt | ((unsigned)min(p.bn_dn, n - tt * p.bn_dn) << 16));
        }
    }
    if (threadIdx.x == 0) {
        p.tile_off_gu[n_uniq] = run_gu;
        p.tile_off_dn[n_uniq] = run_dn;
    }
}

// Sorted fp16 activation rows and transposed block scales: row pos of expert
// order = token of assignment assign[pos].
__global__ void gather_kernel(const int32_t *__restrict__ assign, int A, int k, int H, const int8_t *__restrict__ xq,
                              const BlockScale *__restrict__ xds, __half *__restrict__ xs16, float *__restrict__ xdT,
                              int A_pad) {
    const int nbx = H / kBlock;
    const size_t n = (size_t)A * (H / 8);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int pos = (int)(i / (H / 8)), c8 = (int)(i % (H / 8));
        const int t = assign[pos] / k;
        const uint2 q = *reinterpret_cast<const uint2 *>(xq + (size_t)t * H + c8 * 8);
        const int8_t *b = reinterpret_cast<const int8_t *>(&q);
        __half h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = __int2half_rn(b[j]);
        *reinterpret_cast<uint4 *>(xs16 + (size_t)pos * H + c8 * 8) = *reinterpret_cast<uint4 *>(h);
        if ((c8 & 3) == 0) xdT[(size_t)(c8 / 4) * A_pad + pos] = xds[(size_t)t * nbx + c8 / 4].d;
    }
}

// y[t][i] = sum_j w[t][j] * o[t*k + j][i], j in order, over this shard's
// assignments (global id - e_base in [0, E)).
__global__ void combine_kernel(const float *__restrict__ o, const float *__restrict__ w,
                               const int32_t *__restrict__ idx, int e_base, int E, float *__restrict__ y, int T, int k,
                               int H) {
    const size_t n = (size_t)T * H;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / H), c = (int)(i % H);
        float acc = 0.0f;
        for (int j = 0; j < k; ++j) {
            const size_t a = (size_t)t * k + j;
            if ((unsigned)(idx[a] - e_base) < (unsigned)E) acc += w[a] * o[a * H + c];
        }
        y[i] = acc;
    }
}

// ---------------------------------------------------------------- staging
// Cold expert tensors of the layer's used experts are copied once over the
// host link into the pool slots lent to this prompt pass, and the GEMMs read
// them from HBM through an effective copy of the layer's three table rows.
// Assignment is deterministic: used experts ascending, tensors gate/up/down;
// cold tensors beyond the lent slots stay zero-copy.
__global__ void stage_plan_kernel(StageParams p) {
    const int n_uniq = *p.n_uniq;
    for (int i = threadIdx.x; i < 3 * p.E; i += blockDim.x) p.etbl[i] = p.tbl[(size_t)p.tid0 * p.E + i];
    __syncthreads();
    if (threadIdx.x == 0) {
        int n = 0;
        for (int u = 0; u < n_uniq; ++u) {
            const int e = p.uniq_e[u];
            for (int kd = 0; kd < 3; ++kd) {
                const uint64_t ent = p.tbl[(size_t)(p.tid0 + kd) * p.E + e];
                if (!(ent & 1ull) || n >= p.n_slots) continue;
                const uint64_t dst = p.slot_base + (uint64_t)n * p.slot_stride;
                p.jobs[2 * n] = ent & ~1ull;
                p.jobs[2 * n + 1] = dst;
                p.etbl[(size_t)kd * p.E + e] = dst;
                ++n;
            }
        }
        *p.n_jobs = n;
    }
}

// Grid-stride copy of the staging jobs, 128-bit loads from pinned host memory.
__global__ void __launch_bounds__(256) stage_copy_kernel(const uint64_t *__restrict__ jobs, const int *n_jobs,
                                                         size_t blob16) {
    const int nj = *n_jobs;
    const size_t total = (size_t)nj * blob16;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t j = i / blob16, w = i - j * blob16;
        const uint4 *src = (const uint4 *)(uintptr_t)jobs[2 * j];
        uint4 *dst = (uint4 *)(uintptr_t)jobs[2 * j + 1];
        dst[w] = ld_weights(src + w);
    }
}

// Effective table rows of a layer whose cold experts were prefetched: an
// entry that is cold now (host tag) and has a copy in the prefetch buffer
// points at that copy; every other entry is the live table entry.
__global__ void prefetch_table_kernel(const uint64_t *__restrict__ tbl, const int32_t *__restrict__ map,
                                      uint64_t buf, int cap, size_t stride, int E, uint64_t *etbl) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 3 * E; i += gridDim.x * blockDim.x) {
        const uint64_t entry = tbl[i];
        const int m = map[i];
        const int kd = i / E;
        etbl[i] = ((entry & 1ull) && m >= 0) ? buf + ((size_t)kd * cap + (size_t)m) * stride : entry;
    }
}

int launch_prefetch_table(const uint64_t *tbl_rows, const int32_t *map, const void *buf, int cap, size_t stride,
                          int E, uint64_t *etbl, cudaStream_t st) {
    const int grid = (3 * E + 255) / 256;
    prefetch_table_kernel<<<grid, 256, 0, st>>>(tbl_rows, map, (uint64_t)(uintptr_t)buf, cap, stride, E, etbl);
    return (int)cudaGetLastError();
}

int launch_stage(const StageParams &p, size_t blob_bytes, int n_sm, cudaStream_t st) {
    stage_plan_kernel<<<1, 256, 0, st>>>(p);
    stage_copy_kernel<<<n_sm * 8, 256, 0, st>>>(p.jobs, p.n_jobs, blob_bytes / 16);
    return (int)cudaGetLastError();
}

int gemm_smem_bytes(bool dual) { return dual ? gemm::Cfg<true>::SMEM : gemm::Cfg<false>::SMEM; }
int gemm_bn(bool dual) { return dual ? gemm::Cfg<true>::BN : gemm::Cfg<false>::BN; }
// Weight rows of the layer's tensors covered by one row tile (TMEM lanes).
int gemm_rows_per_tile(bool) { return gemm::BM; }

int gemm_configure() {
    cudaError_t e1 = cudaFuncSetAttribute(gemm::grouped_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          gemm::Cfg<true>::SMEM);
    cudaError_t e2 = cudaFuncSetAttribute(gemm::grouped_gemm_kernel<false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, gemm::Cfg<false>::SMEM);
    return (int)(e1 != cudaSuccess ? e1 : e2);
}

// An event record that also works inside a stream capture (an external
// event node there).
static void record_event(cudaEvent_t e, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(st, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
        cudaEventRecord(e, st);
}

int launch_prefill(const PrefillLaunch &L, cudaStream_t st, cudaEvent_t const *ev) {
    tiling_kernel<<<1, 1024, 0, st>>>(L.tiling);
    const int A = L.gu.A;
    int g = (int)std::min<size_t>(((size_t)A * (L.H / 8) + 255) / 256, (size_t)L.n_sm * 16);
    if (g > 0) gather_kernel<<<g, 256, 0, st>>>(L.gu.assign, A, L.k, L.H, L.xq, L.xds, L.xs16, L.xdT, L.gu.A_pad);
    // timing hook: events around each GEMM launch
    if (ev) record_event(ev[0], st);
    gemm::grouped_gemm_kernel<true><<<L.n_sm, gemm::Cfg<true>::NTHREADS, gemm::Cfg<true>::SMEM, st>>>(L.tm_x, L.gu);
    if (ev) record_event(ev[1], st);
    if (ev) record_event(ev[2], st);
    gemm::grouped_gemm_kernel<false><<<L.n_sm, gemm::Cfg<false>::NTHREADS, gemm::Cfg<false>::SMEM, st>>>(L.tm_h, L.dn);
    if (ev) record_event(ev[3], st);
    const size_t n = (size_t)L.T * L.H;
    int gc = (int)std::min<size_t>((n + 255) / 256, (size_t)L.n_sm * 16);
    combine_kernel<<<gc, 256, 0, st>>>(L.dn.o, L.w, L.idx, L.e_base, L.E, L.y, L.T, L.k, L.H);
    return (int)cudaGetLastError();
}

}  // namespace moe
