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
// then add sum * (d_w * d_a) in fp32 (packed fp32x2 multiplies and fused
// multiply-adds), as the mat-vec does.
//
// Tile: M = 128 weight rows (TMEM lanes) x N = 128 sorted tokens (TMEM
// columns), K staged 64 at a time (two quantization blocks = one 128-B
// swizzle row of fp16), four 128-column K-block buffers in TMEM (all 512
// columns).  Gate/up tiles stack 64 gate rows over the same 64 up rows, so
// one MMA per K step serves both tensors and the tile's SwiGLU pairs lane l of
// TMEM quarter q with lane l of quarter q + 2.  Warp roles (28 warps): 0-7
// weight converters (Q4 codes and scales fetched with cp.async through the
// expert table -- HBM pool, staged slot or zero-copy host memory -- several
// stages ahead, expanded to fp16 in the 128-B swizzled K-major layout); 8 TMA
// producer of the token tile; 9 TMEM owner and MMA issuer; 12-27 epilogue:
// TMEM lane quarter = warp % 4, 32 token columns per warp.  Per K
// block an epilogue thread reads its row's 32 block sums with one TMEM load;
// the columns' activation scales are broadcast shared-memory reads.
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

constexpr int BM = 128;   // weight rows per tile (TMEM lanes)
constexpr int BN = 128;   // token columns per tile
constexpr int BK = 64;    // K per pipeline stage (two quantization blocks)
// Warp roles by warpgroup (setmaxnreg moves registers between warpgroups):
// warpgroups 0-1 = the 8 converter warps, warpgroup 2 = TMA producer, MMA
// issuer and two warps that only join the final barrier, warpgroups 3-6 =
// the 16 epilogue warps (4 lane quarters x 4 column groups).
// Warp roles by warpgroup (setmaxnreg moves registers between warpgroups):
// warpgroup 0 = the 4 converter warps (warp k writes TMEM lane quarter k),
// warpgroup 1 = TMA producer, MMA issuer and two warps that only join the
// final barrier, warpgroups 2-5 = the 16 epilogue warps (4 lane quarters x 4
// column groups).
constexpr int N_CONV = 4, W_CONV = 0, W_TMA = 4, W_MMA = 5, W_EPI = 8;
constexpr int N_EPI = 16;
constexpr int NTHREADS = (W_EPI + N_EPI) * 32;  // 768
// Register split: launched with kLaunchRegs per thread (ptxas' allocation for
// 768 threads, checked on the host before the first launch), warpgroups 0-1
// drop to kProdRegs and warpgroups 2-5 rise to kEpiRegs.
constexpr int kLaunchRegs = 80, kProdRegs = 56, kEpiRegs = 88;
static_assert(2 * 128 * kProdRegs + 4 * 128 * kEpiRegs <= NTHREADS * kLaunchRegs, "register split");
constexpr long long kTimeoutCycles = 4000000000ll;

// Operand slots: the weight tile (A, fp16) in TMEM columns written by the
// converters with tcgen05.st, the token tile (B) in shared memory by TMA;
// a slot is freed by the MMA's commit alone.  Scale ring: the stage's weight
// and activation scales, fetched by cp.async straight into their slot and
// freed by the epilogue.
constexpr int STAGES = 4;                        // operand slots
constexpr int SR = 16;                           // scale slots
constexpr int RR = 6;                            // raw code ring of the converters (cp.async)
constexpr int PD = RR - 1;                       // prefetch distance in stages
constexpr int B_BYTES = BN * BK * 2;             // fp16 token tile (TMA), 128-B swizzle
constexpr int WS_BYTES = BM * 2 * 2;             // weight scales [row][2 blocks] binary16
constexpr int CS_BYTES = 2 * BN * 4;             // activation scales [2 blocks][column] fp32
constexpr int SC_BYTES = WS_BYTES + CS_BYTES;
constexpr int SC_OFF = STAGES * B_BYTES;
constexpr int RAW_BYTES = BM * 32;               // raw ring entry: Q4 codes [row][32 B]
constexpr int RAW_OFF = SC_OFF + SR * SC_BYTES;
constexpr int XCH_OFF = RAW_OFF + RR * RAW_BYTES;  // SwiGLU exchange: [8 pairs][2][16 cols][32 lanes] fp32
constexpr int XCH_BYTES = 8 * 2 * 16 * 32 * 4;
// TMEM: columns [0, 384) hold 12 units of 32 columns for the K-block
// accumulators.  One K block of a tile takes w = 1, 2 or 4 units (its valid
// token columns rounded up); tile j of a batch owns 3 block slots of w units
// starting at unit 3 w j, used in turn by its consecutive K blocks, so every
// tile keeps up to 3 K blocks in flight and an epilogue warp reads only its
// own tile's units.  Columns [384, 512) hold the A operand of the 4 operand
// slots (32 columns = 64 fp16 of K per lane each).
constexpr int NUNIT = 12;
constexpr uint32_t A_TMEM_COL = NUNIT * 32;
constexpr int BAR_OFF = XCH_OFF + XCH_BYTES;
constexpr int NBARS = 2 * STAGES + SR + 2 * NUNIT;
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
constexpr int SMEM = MISC_OFF + 16 + 1024;       // + alignment slack
static_assert(SMEM <= 227 * 1024, "shared memory of the GEMM CTA");

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void st_release_cta(uint32_t addr, uint32_t v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Bounded wait until the MMA issuer has issued at least n K blocks (an
// acquire of its release-stored count): false when the CTA is aborting or
// the wait expired.
__device__ __forceinline__ bool wait_issued(uint32_t issued, uint32_t n, volatile int *abort_flag, int *err) {
    if (ld_acquire_cta(issued) >= n) return true;
    const long long t0 = clock64();
    for (uint32_t k = 1;; ++k) {
        __nanosleep(32);
        if (ld_acquire_cta(issued) >= n) return true;
        if ((k & 63) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kTimeoutCycles) {
                *abort_flag = 1;
                atomicOr(err, 128);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
// One test of an mbarrier phase (mbarrier.try_wait: the hardware may hold the
// thread for a short, system-dependent time while the phase is incomplete).
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred P;\nmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\nselp.u32 %0, 1, 0, P;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: false when the CTA is aborting or the wait expired (then the
// abort flag and an error bit are set).  The abort flag and the clock are
// checked every 64 tests, so a waiting warp issues little besides the tests.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *err,
                                          int code) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try(bar, parity)) return true;
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

// D (TMEM) [+]= A (TMEM, 128 lanes x 16 fp16 of K) x B (shared memory descriptor)
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes <- 32 registers
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive TMEM columns of this warp's 32 lanes (raw fp32 bits)
__device__ __forceinline__ void tmem_ld16u(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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

// Q4 codes of one row and one quantization block (16 B) -> 32 fp16 values
// (q - 8) in K order as 16 words (word m = elements 2m, 2m + 1).
__device__ __forceinline__ void convert_block(uint4 c, uint32_t *o) {
    const uint32_t q[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int part = 0; part < 4; ++part) {
        // part 0: elements 0..7 (low nibbles of bytes 0..7), 1: 8..15
        // (low, bytes 8..15), 2: 16..23 (high, bytes 0..7), 3: 24..31
        const uint32_t wa = q[(part & 1) * 2], wb = q[(part & 1) * 2 + 1];
        const uint32_t na = (part >> 1) ? (wa >> 4) & 0x0F0F0F0Fu : wa & 0x0F0F0F0Fu;
        const uint32_t nb = (part >> 1) ? (wb >> 4) & 0x0F0F0F0Fu : wb & 0x0F0F0F0Fu;
        nib4(na, o[4 * part], o[4 * part + 1]);
        nib4(nb, o[4 * part + 2], o[4 * part + 3]);
    }
}

// TMEM units of one K block of a tile with ncols valid columns.
__host__ __device__ __forceinline__ int block_units(int ncols) { return ncols <= 32 ? 1 : ncols <= 64 ? 2 : 4; }

// Work item ("batch") index -> (used expert u, first row tile, token tile,
// valid token columns, row tiles in the batch), from the records the tiling
// kernel writes.  A batch holds 4 / block_units(ncols) consecutive row tiles
// of one expert's token tile (fewer at the end of the rows): narrow token
// tiles are processed several row tiles at a time, their K stages
// interleaved, so that every epilogue column group has a tile to finish.
__device__ __forceinline__ void decode_tile(const uint2 *rec, int t, int &u, int &row_tile, int &tok_tile,
                                            int &ncols, int &nrt) {
    const uint2 r = __ldg(rec + t);
    u = (int)(r.x & 0xffffu);
    row_tile = (int)(r.x >> 16);
    tok_tile = (int)(r.y & 0xffffu);
    ncols = (int)((r.y >> 16) & 0xffu);
    nrt = (int)(r.y >> 24);
}

// A-tile row r of row tile rt: gate/up tiles hold gate rows 64 rt .. 64 rt + 63
// in tile rows 0..63 and the same up rows in tile rows 64..127; down tiles
// hold rows 128 rt .. 128 rt + 127.
template <bool DUAL>
__device__ __forceinline__ int tile_row(int rt, int r) {
    return DUAL ? rt * 64 + (r & 63) : rt * BM + r;
}

// Stage cursor of one converter thread over the flattened (tile, K stage)
// sequence of its CTA.  The expert-table entry of the thread's tensor and the
// tile's first sorted position are looked up once per tile.
struct StageCur {
    int t, kt, j, rt0, nrt, pos0;
    const uint8_t *blob;
    bool valid;
};

template <bool DUAL>
__device__ __forceinline__ void cur_tile(StageCur &c, const GemmParams &p, int r) {
    int u, tt, nc;
    decode_tile(p.tile_rec, c.t, u, c.rt0, tt, nc, c.nrt);
    const int e = p.uniq_e[u];
    const uint64_t *tb = (DUAL && r >= 64) ? p.tbl[1] : p.tbl[0];
    c.blob = (const uint8_t *)(uintptr_t)(tb[e] & ~1ull);
    c.pos0 = p.uniq_off[u] + tt * BN;
}

template <bool DUAL>
__device__ __forceinline__ void cur_init(StageCur &c, const GemmParams &p, int total, int r) {
    c.t = blockIdx.x;
    c.kt = 0;
    c.j = 0;
    c.valid = c.t < total;
    if (c.valid) cur_tile<DUAL>(c, p, r);
}

// stage order within a batch: K stage outer, row tile of the batch inner
template <bool DUAL>
__device__ __forceinline__ void cur_next(StageCur &c, const GemmParams &p, int total, int nkt, int r) {
    if (!c.valid) return;
    if (++c.j < c.nrt) return;
    c.j = 0;
    if (++c.kt == nkt) {
        c.kt = 0;
        c.t += gridDim.x;
        c.valid = c.t < total;
        if (c.valid) cur_tile<DUAL>(c, p, r);
    }
}

// Parities of the TMEM units' barriers after a batch of nrt tiles, each of
// nblk K blocks of w units: block b of tile j uses block slot b % 3, i.e.
// units 3 w j + w (b % 3) .. + w - 1; every use flips a unit's parity.
__device__ __forceinline__ uint32_t batch_unit_flips(int nrt, int w, int nblk) {
    uint32_t m = 0;
    for (int sl = 0; sl < 3; ++sl)
        if (((nblk - sl + 2) / 3) & 1)
            for (int j = 0; j < nrt; ++j) m |= ((1u << w) - 1u) << (3 * w * j + w * sl);
    return m;
}

__device__ __forceinline__ void bar_sync_named(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <bool DUAL>
__global__ void __launch_bounds__(NTHREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmB, GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + BAR_OFF);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * STAGES, sempty0 = empty0 + 8 * STAGES,
                   tfull0 = sempty0 + 8 * SR, tempty0 = tfull0 + 8 * NUNIT;
    volatile uint32_t *tmem_slot = (volatile uint32_t *)(smem + MISC_OFF);
    volatile int *abort_flag = (volatile int *)(smem + MISC_OFF + 4);
    const uint32_t issued = smem_u32(smem + MISC_OFF + 8);  // K blocks the MMA issuer has issued

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1 + N_CONV);  // TMA expect-tx arrive + the converter warps
            mbar_init(empty0 + 8 * s, 1);          // the MMA's commit
        }
        for (int s = 0; s < SR; ++s) mbar_init(sempty0 + 8 * s, N_EPI);  // 16 weighted reader arrivals
        for (int j = 0; j < NUNIT; ++j) {
            mbar_init(tfull0 + 8 * j, 1);
            mbar_init(tempty0 + 8 * j, 4);  // the four lane-quarter warps of the column group reading it
        }
        *abort_flag = 0;
        *(volatile uint32_t *)(smem + MISC_OFF + 8) = 0u;
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
    auto slot_ptr = [&](int slot) { return smem + slot * B_BYTES; };  // the slot's B tile
    auto sc_ptr = [&](int s) { return smem + SC_OFF + s * SC_BYTES; };

    if (warp >= W_TMA && warp < W_EPI) {
        // the TMA/MMA warpgroup: one setmaxnreg for all four warps, then the
        // TMA and MMA roles (its last two warps only join the final barrier)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
        if (warp == W_TMA && lane == 0) {
            int it = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                int u, rt, tt, nc, nrt;
                decode_tile(p.tile_rec, t, u, rt, tt, nc, nrt);
                const int pos0 = p.uniq_off[u] + tt * BN;
                for (int kt = 0; kt < nkt; ++kt)
                    for (int j = 0; j < nrt; ++j, ++it) {
                        const int slot = it % STAGES;
                        const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                        if (!mbar_wait(empty0 + 8 * slot, ph ^ 1u, abort_flag, p.error, 2)) goto tma_done;
                        mbar_arrive_tx(full0 + 8 * slot, B_BYTES);
                        tma_load_2d(smem_u32(slot_ptr(slot)), &tmB, kt * BK, pos0, full0 + 8 * slot);
                    }
            }
        tma_done:;
        }
        if (warp == W_MMA && lane == 0) {
            int it = 0;
            uint32_t ph = 0;  // per TMEM unit: parity of its next use
            // the tile's MMA width: its valid token columns rounded up to 16
            // (the record of the next tile is requested a tile ahead)
            uint2 rec_next = blockIdx.x < total ? __ldg(p.tile_rec + blockIdx.x) : make_uint2(0, 0);
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                const int ncols = (int)((rec_next.y >> 16) & 0xffu), nrt = (int)(rec_next.y >> 24);
                if (t + (int)gridDim.x < total) rec_next = __ldg(p.tile_rec + t + gridDim.x);
                const int nmma = min(BN, (ncols + 15) & ~15);
                const int w = block_units(ncols);
                const uint32_t idesc = idesc_f16(BM, nmma < 16 ? 16 : nmma);
                uint32_t slots = 0;  // block slot (0..2) of each tile of the batch, 2 bits per tile
                for (int ks = 0, j = 0; ks < nkt * nrt; ++ks, ++it, j = (j + 1 == nrt) ? 0 : j + 1) {
                    const int slot = it % STAGES;
                    if (!mbar_wait(full0 + 8 * slot, (uint32_t)(it / STAGES) & 1u, abort_flag, p.error, 4))
                        goto mma_done;
                    tc_fence_after();
                    const uint32_t ta = tmem + A_TMEM_COL + 32u * (uint32_t)slot;
                    const uint64_t db = sdesc(smem_u32(slot_ptr(slot)));
                    for (int blk = 0; blk < 2; ++blk) {
                        const int sl = (int)((slots >> (2 * j)) & 3u);
                        slots = (slots & ~(3u << (2 * j))) | ((uint32_t)(sl == 2 ? 0 : sl + 1) << (2 * j));
                        const int u0 = 3 * w * j + w * sl;
                        // the units' previous readers are done with them
                        for (int g = 0; g < w; ++g)
                            if (!mbar_wait(tempty0 + 8 * (u0 + g), ((ph >> (u0 + g)) & 1u) ^ 1u, abort_flag, p.error, 8))
                                goto mma_done;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t koff = (uint64_t)((blk * 32 + kk * 16) * 2) >> 4;
                            mma_f16_ts(tmem + (uint32_t)(u0 * 32), ta + (uint32_t)(blk * 16 + kk * 8), db + koff, idesc,
                                       kk > 0 ? 1u : 0u);
                        }
                        for (int g = 0; g < w; ++g) mma_commit(tfull0 + 8 * (u0 + g));
                        ph ^= ((1u << w) - 1u) << u0;
                        // K block 2 it + blk is issued: its units' previous uses are complete
                        // (the waits above), and the stage's scales are in place (full)
                        st_release_cta(issued, (uint32_t)(2 * it + blk + 1));
                    }
                    mma_commit(empty0 + 8 * slot);
                }
            }
        mma_done:;
        }
    } else if (warp < W_TMA) {
        // Converters: thread r owns row r of the A tile (TMEM lane r).  The
        // raw Q4 codes of stage s are fetched with cp.async PD stages ahead
        // into raw ring entry s % RR, the stage's weight and activation scales
        // straight into scale slot s % SR (once the epilogue has freed it);
        // stage s is then expanded to fp16 and stored into the slot's TMEM
        // columns with one tcgen05.st per thread.
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
        const int r = threadIdx.x - W_CONV * 32;
        uint8_t *raw = smem + RAW_OFF;
        StageCur fc;  // fetch cursor; conversion only counts stages
        cur_init<DUAL>(fc, p, total, r);
        int n_stages = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int u, rt, tt, nc, nrt;
            decode_tile(p.tile_rec, t, u, rt, tt, nc, nrt);
            n_stages += nkt * nrt;
        }
        bool ok = true;
        auto fetch = [&](const StageCur &cu, int q) {  // stage q
            if (cu.valid) {
                uint8_t *ent = raw + (q % RR) * RAW_BYTES;
                uint8_t *sc = sc_ptr(q % SR);
                if (lane == 0)
                    ok = ok && mbar_wait(sempty0 + 8 * (q % SR), ((uint32_t)(q / SR) & 1u) ^ 1u, abort_flag, p.error, 16);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                const int row = tile_row<DUAL>(cu.rt0 + cu.j, r);
                const bool vrow = ok && row < p.rows;
                const int srow = row < p.rows ? row : 0;
                const uint8_t *src = cu.blob + ((size_t)srow * nbk + 2 * cu.kt) * 16;
                cp_async(smem_u32(ent + r * 32), src, 16, vrow);
                cp_async(smem_u32(ent + r * 32 + 16), src + 16, 16, vrow);
                const uint8_t *ssrc = cu.blob + scale_off + ((size_t)srow * nbk + 2 * cu.kt) * 2;
                cp_async(smem_u32(sc + r * 4), ssrc, 4, vrow);
                // activation scales i of the stage: block i / BN, column i % BN
#pragma unroll
                for (int i = r; i < 2 * BN; i += BM) {
                    const int qb = i / BN, col = i - qb * BN;
                    const int pos = cu.pos0 + col;
                    const bool v = ok && pos < p.A_pad;
                    const float *asrc = p.a_scaleT + (size_t)(2 * cu.kt + qb) * p.A_pad + (pos < p.A_pad ? pos : 0);
                    cp_async(smem_u32(sc + WS_BYTES + i * 4), asrc, 4, v);
                }
            }
            cp_commit();
        };
        for (int i = 0; i < PD; ++i) {
            fetch(fc, i);
            cur_next<DUAL>(fc, p, total, nkt, r);
        }
        const uint32_t ta_lane = tmem + ((uint32_t)(warp * 32) << 16) + A_TMEM_COL;  // this warp's lane quarter
        int it = 0;
        while (it < n_stages && ok) {
            fetch(fc, it + PD);
            cur_next<DUAL>(fc, p, total, nkt, r);
            cp_wait<PD>();
            const int slot = it % STAGES;
            if (lane == 0)
                ok = mbar_wait(empty0 + 8 * slot, ((uint32_t)(it / STAGES) & 1u) ^ 1u, abort_flag, p.error, 16);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            tc_fence_after();
            const uint8_t *ent = raw + (it % RR) * RAW_BYTES;
            uint32_t a[32];
            convert_block(*(const uint4 *)(ent + r * 32), a);
            convert_block(*(const uint4 *)(ent + r * 32 + 16), a + 16);
            tmem_st32(ta_lane + 32u * (uint32_t)slot, a);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(full0 + 8 * slot);
            ++it;
        }
        cp_wait<0>();
    } else {
        // Epilogue: TMEM lane quarter = warp % 4 (thread = tile row), column
        // group = 32 token columns.  Per K block: one 32-column TMEM load
        // (the buffer is handed back to the MMA as soon as the load is
        // complete), s = d_w * d_a (mul.f32x2) and acc += sum * s (fma.f32x2),
        // the activation scales of four columns per 128-bit broadcast load.
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
        const int e = warp - W_EPI;
        const int quarter = warp & 3;
        const int grp = e >> 2;  // column group: tile grp / w of the batch, its columns [32 cu, 32 cu + 32)
        const int r = quarter * 32 + lane;
        float *xch = (float *)(smem + XCH_OFF);
        int it0 = 0;      // stage index of the batch's first stage
        uint32_t ph = 0;  // per TMEM unit: parity of its next use, at the start of the batch
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int u, rt0, tt, ncols, nrt;
            decode_tile(p.tile_rec, t, u, rt0, tt, ncols, nrt);
            const int w = block_units(ncols);
            const int tj = grp / w, cu = grp - tj * w;  // this group's tile in the batch and column unit
            const uint32_t ph_next = ph ^ batch_unit_flips(nrt, w, 2 * nkt);
            const int it_first = it0;
            it0 += nkt * nrt;
            if (tj >= nrt) {  // no tile of this batch for this group
                ph = ph_next;
                continue;
            }
            const int rt = rt0 + tj;
            const bool active = cu * 32 < ncols;  // this warp has valid columns (warp-uniform)
            const int pos0 = p.uniq_off[u] + tt * BN + cu * 32;
            const int pos_end = p.uniq_off[u + 1];
            const uint32_t sc_weight = 4u / (uint32_t)w;  // 4 w warps read a stage's scales; 16 arrivals free it
            float2 acc[16];
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) acc[cc] = make_float2(0.0f, 0.0f);
            uint32_t q = ph;  // parities of this tile's units, updated as they are read
            int sl = 0;       // block slot of the next K block
            for (int kt = 0; kt < nkt; ++kt) {
                const int it = it_first + kt * nrt + tj;  // this tile's stage
                const int ss = it % SR;
                const uint8_t *sc = sc_ptr(ss);
                bool ok = true;
                // the stage's first K block is issued: its scales are in place
                // (and no TMEM unit of the stage is more than a phase ahead)
                if (lane == 0) ok = wait_issued(issued, (uint32_t)(2 * it + 1), abort_flag, p.error);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) goto epi_done;
                const uint32_t wsc = *(const uint32_t *)(sc + r * 4);
                const float4 *cs4 = (const float4 *)(sc + WS_BYTES) + cu * 8;
#pragma unroll 1
                for (int blk = 0; blk < 2; ++blk) {
                    const int un = 3 * w * tj + w * sl + cu;  // this warp's unit of the block
                    sl = sl == 2 ? 0 : sl + 1;
                    {
                        if (lane == 0)
                            ok = wait_issued(issued, (uint32_t)(2 * it + blk + 1), abort_flag, p.error) &&
                                 mbar_wait(tfull0 + 8 * un, (q >> un) & 1u, abort_flag, p.error, 32);
                        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                        if (!ok) goto epi_done;
                        tc_fence_after();
                        if (active) {
                            const float dw = __half2float(
                                __ushort_as_half((unsigned short)(blk ? (wsc >> 16) : (wsc & 0xffffu))));
                            const float2 dw2 = make_float2(dw, dw);
                            const float4 *c4p = cs4 + blk * (BN / 4);
                            // the unit's 32 columns in two 16-column loads
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                uint32_t sv[16];
                                tmem_ld16u(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(un * 32 + half * 16),
                                           sv);
                                tmem_ld_wait();
#pragma unroll
                                for (int c4 = 0; c4 < 4; ++c4) {
                                    const float4 d4 = c4p[half * 4 + c4];  // broadcast read
                                    const float2 s01 = __fmul2_rn(dw2, make_float2(d4.x, d4.y));
                                    const float2 s23 = __fmul2_rn(dw2, make_float2(d4.z, d4.w));
                                    float2 &a0 = acc[half * 8 + 2 * c4], &a1 = acc[half * 8 + 2 * c4 + 1];
                                    a0 = __ffma2_rn(make_float2(__uint_as_float(sv[4 * c4]),
                                                                __uint_as_float(sv[4 * c4 + 1])), s01, a0);
                                    a1 = __ffma2_rn(make_float2(__uint_as_float(sv[4 * c4 + 2]),
                                                                __uint_as_float(sv[4 * c4 + 3])), s23, a1);
                                }
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty0 + 8 * un);
                    }
                    q ^= 1u << un;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_n(sempty0 + 8 * ss, sc_weight);
            }
            ph = ph_next;
            // tile outputs; the assignment id of column i of this warp's group
            // is held by lane i
            const int my_pos = pos0 + lane;
            const int my_asg = my_pos < pos_end ? __ldg(p.assign + my_pos) : 0;
            if (DUAL) {
                // SwiGLU pairs gate row f (quarter q < 2) with up row f (quarter
                // q + 2), same lane, same column group; the gate warp finishes
                // columns 0..15 of the group, the up warp columns 16..31, each
                // receiving the other tensor's values through shared memory.
                const int pair = grp * 2 + (quarter & 1);
                const bool is_gate = quarter < 2;
                float *to_partner = xch + ((size_t)(pair * 2 + (is_gate ? 0 : 1)) * 16) * 32;
                const float *from_partner = xch + ((size_t)(pair * 2 + (is_gate ? 1 : 0)) * 16) * 32;
                if (active) {
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        // the gate warp sends columns 16..31, the up warp 0..15
                        const float2 v = is_gate ? acc[8 + cc] : acc[cc];
                        to_partner[(2 * cc) * 32 + lane] = v.x;
                        to_partner[(2 * cc + 1) * 32 + lane] = v.y;
                    }
                }
                bar_sync_named(1 + pair, 64);
                if (active) {
                    // this warp's 16 columns of the group (gate warp: 0..15, up warp: 16..31)
                    float mine[16];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const float2 v = is_gate ? acc[cc] : acc[8 + cc];
                        mine[2 * cc] = v.x;
                        mine[2 * cc + 1] = v.y;
                    }
                    const int c0 = is_gate ? 0 : 16;
                    const int fb = (rt * 64 + (quarter & 1) * 32) / kBlock;  // h block index along F
                    const int f = rt * 64 + (quarter & 1) * 32 + lane;       // F row of this lane
                    const int nc = min(16, ncols - cu * 32 - c0);            // valid columns (warp-uniform)
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        if (cc < nc) {
                            const float other = from_partner[cc * 32 + lane];
                            const float g = is_gate ? mine[cc] : other, uu = is_gate ? other : mine[cc];
                            const float h = g * uu / (1.0f + expf(-g));
                            const float amax =
                                __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
                            const float dd = __half2float(__float2half_rn(amax / 127.0f));
                            int qv = 0;
                            if (dd != 0.0f) qv = (int)fminf(fmaxf(rintf(h / dd), -127.0f), 127.0f);
                            const int sum = __reduce_add_sync(0xffffffffu, qv);
                            const int col = c0 + cc;
                            const int pos = pos0 + col;
                            const int a = __shfl_sync(0xffffffffu, my_asg, col);
                            if (pos < pos_end) {
                                p.hq16[(size_t)pos * p.F_out + f] = __int2half_rn(qv);
                                p.hq[(size_t)a * p.F_out + f] = (int8_t)qv;
                                if (lane == 0) {
                                    p.hdT[(size_t)fb * p.A_pad + pos] = dd;
                                    p.hds[(size_t)a * (p.F_out / kBlock) + fb] = BlockScale{dd, sum};
                                }
                            }
                        }
                    }
                }
                // the exchange area is rewritten at the end of the next tile
                bar_sync_named(1 + pair, 64);
            } else if (active) {
                const int row = rt * BM + r;
                const bool vrow = row < p.rows;
                const int nc = min(32, ncols - cu * 32);  // valid columns (warp-uniform)
#pragma unroll
                for (int cc = 0; cc < 32; ++cc) {
                    if (cc < nc) {
                        const int pos = pos0 + cc;
                        const int a = __shfl_sync(0xffffffffu, my_asg, cc);
                        const float v = (cc & 1) ? acc[cc >> 1].y : acc[cc >> 1].x;
                        if (vrow && pos < pos_end) p.o[(size_t)a * p.rows + row] = v;
                    }
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
// Work items of one expert with n tokens: per token tile of bn columns, its
// rt row tiles in batches of 4 / block_units(valid columns).
__device__ __forceinline__ int gemm_batches(int n, int rt, int bn) {
    int cnt = 0;
    for (int tt = 0; tt * bn < n; ++tt) {
        const int per = 4 / gemm::block_units(min(bn, n - tt * bn));
        cnt += (rt + per - 1) / per;
    }
    return cnt;
}

__device__ __forceinline__ void gemm_batch_records(int u, int n, int rt, int bn, uint2 *out, int cap) {
    int i = 0;
    for (int tt = 0; tt * bn < n; ++tt) {
        const int nc = min(bn, n - tt * bn);
        const int per = 4 / gemm::block_units(nc);
        for (int r0 = 0; r0 < rt; r0 += per, ++i) {
            if (i < cap)
                out[i] = make_uint2((unsigned)u | ((unsigned)r0 << 16),
                                    (unsigned)tt | ((unsigned)nc << 16) | ((unsigned)min(per, rt - r0) << 24));
        }
    }
}

// Per used expert: cumulative tile counts of the gate/up and down GEMMs, and
// the miss / stamp record of the layer's three tensors.
__global__ void tiling_kernel(TilingParams p) {
    __shared__ int warp_tot[33];
    const int n_uniq = *p.n_uniq;
    const uint32_t step_clock = *p.cv.clock + (uint32_t)p.n_tokens;
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
            tg = gemm_batches(n, p.rt_gu, p.bn_gu);
            td = gemm_batches(n, p.rt_dn, p.bn_dn);
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
    // batch records: (u | first row tile << 16, token tile | valid columns
    // << 16 | row tiles << 24), token tile outer, row tiles inner
    for (int u = threadIdx.x; u < n_uniq; u += blockDim.x) {
        const int n = p.uniq_off[u + 1] - p.uniq_off[u];
        gemm_batch_records(u, n, p.rt_gu, p.bn_gu, p.rec_gu + p.tile_off_gu[u], p.cap_gu - p.tile_off_gu[u]);
        gemm_batch_records(u, n, p.rt_dn, p.bn_dn, p.rec_dn + p.tile_off_dn[u], p.cap_dn - p.tile_off_dn[u]);
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

// y[t][i] = sum_j w[t][j] * o[t*k + j][i], j in order.
__global__ void combine_kernel(const float *__restrict__ o, const float *__restrict__ w, float *__restrict__ y, int T,
                               int k, int H) {
    const size_t n = (size_t)T * H;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / H), c = (int)(i % H);
        float acc = 0.0f;
        for (int j = 0; j < k; ++j) acc += w[(size_t)t * k + j] * o[((size_t)t * k + j) * H + c];
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

int gemm_bn(bool) { return gemm::BN; }
// Weight rows of the layer's tensors covered by one row tile: 64 F rows for
// gate/up (64 gate + the same 64 up rows), 128 H rows for down.
int gemm_rows_per_tile(bool dual) { return dual ? 64 : gemm::BM; }

int gemm_configure() {
    // the kernels' register split assumes ptxas gave them kLaunchRegs per thread
    for (const void *fn : {(const void *)gemm::grouped_gemm_kernel<true>, (const void *)gemm::grouped_gemm_kernel<false>}) {
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return (int)e;
        if (fa.numRegs != gemm::kLaunchRegs) return (int)cudaErrorInvalidConfiguration;
    }
    cudaError_t e1 = cudaFuncSetAttribute(gemm::grouped_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          gemm::SMEM);
    cudaError_t e2 = cudaFuncSetAttribute(gemm::grouped_gemm_kernel<false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, gemm::SMEM);
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
    gemm::grouped_gemm_kernel<true><<<L.n_sm, gemm::NTHREADS, gemm::SMEM, st>>>(L.tm_x, L.gu);
    if (ev) record_event(ev[1], st);
    if (ev) record_event(ev[2], st);
    gemm::grouped_gemm_kernel<false><<<L.n_sm, gemm::NTHREADS, gemm::SMEM, st>>>(L.tm_h, L.dn);
    if (ev) record_event(ev[3], st);
    const size_t n = (size_t)L.T * L.H;
    int gc = (int)std::min<size_t>((n + 255) / 256, (size_t)L.n_sm * 16);
    combine_kernel<<<gc, 256, 0, st>>>(L.dn.o, L.w, L.y, L.T, L.k, L.H);
    return (int)cudaGetLastError();
}

}  // namespace moe
