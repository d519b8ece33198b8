// Decode-side kernels of the routed-expert FFN: router top-k, the per-layer
// plan (activation quantization + grouping of assignments by expert), the
// pointer-table gate/up mat-vec with fused SwiGLU and h quantization, the
// down mat-vec with the fused weighted combine, and test/measurement hooks.
//
// Sources: Zapdev-labs/a6000-custom-kernels (moe_cache_gemv: one routed
// expert sourced through d_tbl; cold reads logged to a miss buffer; stamps);
// mx-llama.cpp FEATURES.md (q8_1 activations quantized once and reused by the
// matmuls of one input; fused up/gate lanes for narrow batches);
// mihailescu2m/llama.cpp (work only over (expert, tile) pairs that hold
// tokens; top-k instead of a full sort of the 512 scores).
#include "common.cuh"
#include "kernels.h"

#include <map>
#include <mutex>

#include <float.h>

namespace moe {

static void record(cudaEvent_t e, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(st, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
        cudaEventRecord(e, st);
}


// Programmatic dependent launch for the chained small kernels (top-k, plan,
// gate/up, down): wait for the previous kernel in the stream (a no-op when
// launched without the attribute), then let the next one be scheduled.  The
// wait comes first, so nothing of the previous kernel's output is read early;
// what overlaps is the next launch's latency.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// --------------------------------------------------------------- top-k// --------------------------------------------------------------- top-k
// One warp per token; lane l holds logits l, l+32, ... (V per lane).  k
// rounds of a warp arg-max over (value desc, index asc).
template <int V>
__global__ void __launch_bounds__(256) topk_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                   int renorm, int32_t *__restrict__ idx, float *__restrict__ w) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *l = logits + (size_t)t * E;
    float v[V];
    uint32_t taken[(V + 31) / 32];
#pragma unroll
    for (int i = 0; i < (V + 31) / 32; ++i) taken[i] = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        int e = lane + 32 * i;
        v[i] = e < E ? l[e] : -INFINITY;
        if (e >= E) taken[i >> 5] |= 1u << (i & 31);
    }
    float my_v = -INFINITY;
    int my_i = 0x7fffffff;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            bool free_ = !(taken[i >> 5] & (1u << (i & 31)));
            int e = lane + 32 * i;
            if (free_ && (bi == 0x7fffffff || v[i] > bv)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi != 0x7fffffff && (bi & 31) == lane) {
            int i = bi >> 5;
#pragma unroll
            for (int ii = 0; ii < V; ++ii)
                if (ii == i) taken[ii >> 5] |= 1u << (ii & 31);
        }
        if (lane == j) {
            my_v = bv;
            my_i = bi;
        }
    }
    float m = __shfl_sync(0xffffffffu, my_v, 0);
    float ej = lane < k ? expf(my_v - m) : 0.0f;
    float den;
    if (renorm) {
        den = warp_sum_f(ej);
    } else {
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i)
            if (lane + 32 * i < E) s += expf(v[i] - m);
        den = warp_sum_f(s);
    }
    if (lane < k) {
        idx[(size_t)t * k + lane] = my_i;
        w[(size_t)t * k + lane] = ej / den;
    }
}

int launch_topk(const float *logits, int T, int E, int k, int renorm, int32_t *idx, float *w, cudaStream_t st) {
    if (T <= 0) return 0;
    dim3 block(256), grid((T + 7) / 8);
    cudaError_t e;
    if (E <= 32)
        e = launch_pdl(topk_kernel<1>, grid, block, 0, st, logits, T, E, k, renorm, idx, w);
    else if (E <= 128)
        e = launch_pdl(topk_kernel<4>, grid, block, 0, st, logits, T, E, k, renorm, idx, w);
    else if (E <= 512)
        e = launch_pdl(topk_kernel<16>, grid, block, 0, st, logits, T, E, k, renorm, idx, w);
    else if (E <= 1024)
        e = launch_pdl(topk_kernel<32>, grid, block, 0, st, logits, T, E, k, renorm, idx, w);
    else
        e = launch_pdl(topk_kernel<128>, grid, block, 0, st, logits, T, E, k, renorm, idx, w);
    return (int)e;
}

// --------------------------------------------------------------- quantize
// Warp per block of 32 activations, grid-stride.
__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ x, int n_blocks,
                                                       int8_t *__restrict__ q, BlockScale *__restrict__ ds) {
    const int lane = threadIdx.x & 31;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    for (int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < n_blocks; b += nw)
        quantize_block_warp(x[(size_t)b * kBlock + lane], lane, q + (size_t)b * kBlock, ds + b);
}

int launch_quantize(const float *x, int n_blocks, int8_t *q, BlockScale *ds, int n_sm, cudaStream_t st) {
    if (n_blocks <= 0) return 0;
    int grid = (n_blocks + 7) / 8;
    if (grid > n_sm * 8) grid = n_sm * 8;
    quantize_kernel<<<grid, 256, 0, st>>>(x, n_blocks, q, ds);
    return (int)cudaGetLastError();
}

// --------------------------------------------------------------- plan
// One CTA of 1024 threads: optionally quantize x (small batches), then group
// the T*k assignments by expert: counts per expert, the ascending list of
// used experts with the offsets of their assignment lists, and the
// assignment ids grouped by expert (order within an expert is not fixed and
// does not change any result: each assignment is computed on its own).
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int s = lane < nw ? warp_tot[lane] : 0;
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += n;
        }
        if (lane < nw) warp_tot[lane] = si - s;  // exclusive warp offsets
        if (lane == nw - 1) warp_tot[32] = si;   // block total
    }
    __syncthreads();
    int r = warp_tot[wid] + incl - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanParams p) {
    pdl_enter();
    extern __shared__ int sm[];
    int *cnt = sm;            // [E]
    int *cur = sm + p.E;      // [E]
    __shared__ int warp_tot[33];
    __shared__ int s_other;   // assignments to experts of other shards
    const int A = p.T * p.k;
    const int lane = threadIdx.x & 31;
    if (p.quantize_x) {
        const int nbx = p.H / kBlock, nblk = p.T * nbx;
        for (int b = threadIdx.x >> 5; b < nblk; b += blockDim.x >> 5)
            quantize_block_warp(p.x[(size_t)b * kBlock + lane], lane, p.xq + (size_t)b * kBlock, p.xds + b);
    }
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) cnt[e] = 0;
    if (threadIdx.x == 0) s_other = 0;
    __syncthreads();
    // local expert of assignment a: -1 for another shard's expert; ids outside
    // the layer's range set error bit 0 and are read as local expert 0
    auto local_e = [&](int a) {
        const int g = p.idx[a];
        if (g < 0 || g >= p.E_route) return 0;
        const int e = g - p.e_base;
        return e >= 0 && e < p.E ? e : -1;
    };
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        const int g = p.idx[a];
        if (g < 0 || g >= p.E_route) atomicOr(p.error, 1);
        const int e = local_e(a);
        if (e >= 0) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive scans over experts of counts and of "used" flags, in
    // chunks of blockDim experts.
    int run_off = 0, run_u = 0;
    for (int base = 0; base < p.E; base += blockDim.x) {
        int e = base + threadIdx.x;
        int c = e < p.E ? cnt[e] : 0;
        int used = c > 0;
        int off = block_excl_scan(c, warp_tot);
        int tot_c = warp_tot[32];
        __syncthreads();
        int uix = block_excl_scan(used, warp_tot);
        int tot_u = warp_tot[32];
        __syncthreads();
        if (e < p.E) {
            cur[e] = run_off + off;
            if (used) {
                p.uniq_e[run_u + uix] = e;
                p.uniq_off[run_u + uix] = run_off + off;
            }
        }
        run_off += tot_c;
        run_u += tot_u;
    }
    if (threadIdx.x == 0) {
        p.uniq_off[run_u] = run_off;
        *p.n_uniq = run_u;
    }
    __syncthreads();
    // other shards' assignments follow the grouped ones (in no used list)
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        const int e = local_e(a);
        const int pos = e >= 0 ? atomicAdd(&cur[e], 1) : run_off + atomicAdd(&s_other, 1);
        p.assign[pos] = a;
    }
}

int launch_plan(const PlanParams &p, cudaStream_t st) {
    size_t smem = (size_t)2 * p.E * sizeof(int);
    return (int)launch_pdl(plan_kernel, dim3(1), dim3(1024), smem, st, p);
}

// --------------------------------------------------------------- gate/up
// Work item = (used expert u, block of 32 rows of F).  8 warps; each row is
// split over 8 lanes (lane l of a row reads blocks l, l+8, ...: 8 lanes x 16 B
// = 128 contiguous bytes per round), so one warp covers 4 rows and the CTA 32
// rows.  gate row r and up row r are read by the same lanes, which gives
// h_r = silu(g_r) * u_r in registers; the 32 values of h per token are then
// quantized by one warp per token.
constexpr int kGULanes = 8;

template <int FMT>
__global__ void __launch_bounds__(256) gate_up_kernel(GemvParams p) {
    pdl_enter();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % kGULanes, grp = lane / kGULanes;
    const int rloc = warp * (32 / kGULanes) + grp;  // 0..31
    const int nbx = p.H / kBlock;
    const int rgs = p.F / kBlock;
    const int n_uniq = *p.n_uniq;
    const int n_items = n_uniq * rgs;
    const uint32_t step_clock = *p.cv.clock + (uint32_t)p.cv.clock_tokens;
    const size_t scale_off = blob_scales_offset_fmt(FMT, p.F, nbx);
    __shared__ float sh_h[kMaxChunk][32];

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int u = item / rgs, rg = item - u * rgs;
        const int e = p.uniq_e[u];
        const int a0 = p.uniq_off[u], a1 = p.uniq_off[u + 1];
        const uint64_t eg = p.cv.tbl[(size_t)p.tid_gate * p.cv.E + e];
        const uint64_t eu = p.cv.tbl[(size_t)p.tid_up * p.cv.E + e];
        if (rg == 0 && threadIdx.x == 0) {
            record_read(p.cv, p.tid_gate, e, eg, step_clock);
            record_read(p.cv, p.tid_up, e, eu, step_clock);
        }
        const uint8_t *bg = (const uint8_t *)(uintptr_t)(eg & ~1ull);
        const uint8_t *bu = (const uint8_t *)(uintptr_t)(eu & ~1ull);
        const int r = rg * 32 + rloc;
        const size_t nblk = (size_t)p.F * nbx, rb0 = (size_t)r * nbx;

        for (int c0 = a0; c0 < a1; c0 += kMaxChunk) {
            const int nt = min(kMaxChunk, a1 - c0);
            int tok[kMaxChunk];
#pragma unroll
            for (int t = 0; t < kMaxChunk; ++t) tok[t] = t < nt ? p.assign[c0 + t] / p.k : 0;
            float ag[kMaxChunk], au[kMaxChunk];
#pragma unroll
            for (int t = 0; t < kMaxChunk; ++t) ag[t] = au[t] = 0.0f;
            for (int b0 = sub; b0 < nbx; b0 += 4 * kGULanes) {
                WCodes<FMT> wg4[4], wu4[4];
                WScale<FMT> sg[4], su[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    int b = b0 + i * kGULanes;
                    if (b < nbx) {
                        wg4[i].load(bg, nblk, rb0 + b);
                        wu4[i].load(bu, nblk, rb0 + b);
                        sg[i].load(bg + scale_off, rb0 + b);
                        su[i].load(bu + scale_off, rb0 + b);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    int b = b0 + i * kGULanes;
                    if (b < nbx) {
#pragma unroll
                        for (int t = 0; t < kMaxChunk; ++t) {
                            if (t < nt) {
                                const int4 *xa = (const int4 *)(p.xq + (size_t)tok[t] * p.H + (size_t)b * kBlock);
                                int4 x0 = __ldg(xa), x1 = __ldg(xa + 1);
                                BlockScale xs = p.xds[(size_t)tok[t] * nbx + b];
                                int ig = wg4[i].dot(x0, x1, xs.s);
                                int iu = wu4[i].dot(x0, x1, xs.s);
                                ag[t] += sg[i].term(ig, xs);
                                au[t] += su[i].term(iu, xs);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kMaxChunk; ++t) {
#pragma unroll
                for (int o = kGULanes / 2; o > 0; o >>= 1) {
                    ag[t] += __shfl_xor_sync(0xffffffffu, ag[t], o);
                    au[t] += __shfl_xor_sync(0xffffffffu, au[t], o);
                }
            }
            if (sub == 0) {
#pragma unroll
                for (int t = 0; t < kMaxChunk; ++t)
                    if (t < nt) {
                        float g = ag[t], uu = au[t];
                        sh_h[t][rloc] = g * uu / (1.0f + expf(-g));
                    }
            }
            __syncthreads();
            if (warp < nt) {
                const int a = p.assign[c0 + warp];
                quantize_block_warp(sh_h[warp][lane], lane, p.hq + (size_t)a * p.F + (size_t)rg * kBlock,
                                    p.hds + (size_t)a * rgs + rg);
            }
            __syncthreads();
        }
    }
}

// --------------------------------------------------------------- down
// Work item = (used expert u, block of ROWS rows of H); L lanes per row
// (blocks of a row: F/32).  Each item writes o[a][rows] for the assignments
// of u; the last item of a row block to finish (counted with an atomic per
// row block) sums y[t][rows] = sum_j w[t][j] * o[t*k+j][rows] in j order.
template <int L, int FMT>
__global__ void __launch_bounds__(256) down_kernel(GemvParams p) {
    pdl_enter();
    constexpr int G = 32 / L;          // rows per warp
    constexpr int ROWS = kWarps * G;   // rows per item
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % L, grp = lane / L;
    const int rloc = warp * G + grp;
    const int nbf = p.F / kBlock;
    const int n_rb = p.H / ROWS;
    const int n_uniq = *p.n_uniq;
    const int n_items = n_uniq * n_rb;
    const uint32_t step_clock = *p.cv.clock + (uint32_t)p.cv.clock_tokens;
    const size_t scale_off = blob_scales_offset_fmt(FMT, p.H, nbf);
    __shared__ int sh_last;
    if (n_uniq == 0) {
        // no assignment of this shard: y = 0
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)p.n_tokens * p.H;
             i += (size_t)gridDim.x * blockDim.x)
            p.y[i] = 0.0f;
        return;
    }

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int u = item / n_rb, rb = item - u * n_rb;
        const int e = p.uniq_e[u];
        const int a0 = p.uniq_off[u], a1 = p.uniq_off[u + 1];
        const uint64_t ed = p.cv.tbl[(size_t)p.tid_down * p.cv.E + e];
        if (rb == 0 && threadIdx.x == 0) record_read(p.cv, p.tid_down, e, ed, step_clock);
        const uint8_t *bd = (const uint8_t *)(uintptr_t)(ed & ~1ull);
        const int r = rb * ROWS + rloc;
        const size_t nblk = (size_t)p.H * nbf, rb0 = (size_t)r * nbf;

        for (int c0 = a0; c0 < a1; c0 += kMaxChunk) {
            const int nt = min(kMaxChunk, a1 - c0);
            int asg[kMaxChunk];
#pragma unroll
            for (int t = 0; t < kMaxChunk; ++t) asg[t] = t < nt ? p.assign[c0 + t] : 0;
            float acc[kMaxChunk];
#pragma unroll
            for (int t = 0; t < kMaxChunk; ++t) acc[t] = 0.0f;
            for (int b0 = sub; b0 < nbf; b0 += 4 * L) {
                WCodes<FMT> w4[4];
                WScale<FMT> sw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    int b = b0 + i * L;
                    if (b < nbf) {
                        w4[i].load(bd, nblk, rb0 + b);
                        sw[i].load(bd + scale_off, rb0 + b);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    int b = b0 + i * L;
                    if (b < nbf) {
#pragma unroll
                        for (int t = 0; t < kMaxChunk; ++t) {
                            if (t < nt) {
                                const int4 *ha = (const int4 *)(p.hq + (size_t)asg[t] * p.F + (size_t)b * kBlock);
                                int4 h0 = __ldcg(ha), h1 = __ldcg(ha + 1);
                                BlockScale hs = p.hds[(size_t)asg[t] * nbf + b];
                                int id = w4[i].dot(h0, h1, hs.s);
                                acc[t] += sw[i].term(id, hs);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kMaxChunk; ++t) {
#pragma unroll
                for (int o = L / 2; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
            }
            if (sub == 0) {
#pragma unroll
                for (int t = 0; t < kMaxChunk; ++t)
                    if (t < nt) p.o[(size_t)asg[t] * p.H + r] = acc[t];
            }
        }
        // arrival count of this row block; the last item combines
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned prev = atomicAdd(&p.counters[rb], 1u);
            sh_last = (prev == (unsigned)(n_uniq - 1));
        }
        __syncthreads();
        if (sh_last) {
            __threadfence();
            const int n_out = p.n_tokens * ROWS;
            for (int i = threadIdx.x; i < n_out; i += blockDim.x) {
                const int t = i / ROWS, rr = rb * ROWS + (i - t * ROWS);
                float y = 0.0f;
                for (int j = 0; j < p.k; ++j) {
                    const size_t a = (size_t)t * p.k + j;
                    if ((unsigned)(p.idx[a] - p.e_base) >= (unsigned)p.cv.E) continue;  // another shard's
                    y += p.w[a] * __ldcg(p.o + a * p.H + rr);
                }
                p.y[(size_t)t * p.H + rr] = y;
            }
            if (threadIdx.x == 0) p.counters[rb] = 0u;
        }
        __syncthreads();
    }
}

int down_rows_per_item(int F) {
    int nbf = F / kBlock;
    int L = nbf <= 40 ? 4 : 8;
    return kWarps * (32 / L);
}

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvParams &p, int grid_gu, int grid_dn, cudaStream_t st, cudaEvent_t const *ev) {
    cudaError_t e = launch_pdl(gate_up_kernel<FMT>, dim3(grid_gu), dim3(256), 0, st, p);
    if (e != cudaSuccess) return e;
    if (ev) record(ev[1], st);
    if (ev) record(ev[2], st);
    if (p.F / kBlock <= 40) return launch_pdl(down_kernel<4, FMT>, dim3(grid_dn), dim3(256), 0, st, p);
    return launch_pdl(down_kernel<8, FMT>, dim3(grid_dn), dim3(256), 0, st, p);
}

// ev (optional): 4 events recorded around the gate/up and the down launch.
int launch_gemv(const GemvParams &p, int grid_gu, int grid_dn, cudaStream_t st, cudaEvent_t const *ev) {
    if (ev) record(ev[0], st);
    cudaError_t e;
    if (p.fmt == kFmtQ8)
        e = launch_gemv_fmt<kFmtQ8>(p, grid_gu, grid_dn, st, ev);
    else if (p.fmt == kFmtQ4K)
        e = launch_gemv_fmt<kFmtQ4K>(p, grid_gu, grid_dn, st, ev);
    else if (p.fmt == kFmtQ6K)
        e = launch_gemv_fmt<kFmtQ6K>(p, grid_gu, grid_dn, st, ev);
    else if (p.fmt == kFmtQ5K)
        e = launch_gemv_fmt<kFmtQ5K>(p, grid_gu, grid_dn, st, ev);
    else if (p.fmt == kFmtQ5)
        e = launch_gemv_fmt<kFmtQ5>(p, grid_gu, grid_dn, st, ev);
    else
        e = launch_gemv_fmt<kFmtQ4>(p, grid_gu, grid_dn, st, ev);
    if (ev) record(ev[3], st);
    return (int)e;
}

// --------------------------------------------------------------- fused layer
// One cooperative launch per layer for small batches (T*k <= kMaxFusedA).
// Every CTA derives the same plan from idx in shared memory (used experts
// ascending, assignments grouped by expert).  Gate/up items (used expert,
// 32 rows of F) issue all their weight loads first, quantize the x of their
// tokens into shared memory while the loads are in flight, then compute
// SwiGLU and quantize h, and publish completion per expert.  Down items
// (used expert, ROWS rows of H) issue their weight loads, then wait (bounded)
// until every gate/up row block of their expert is published, read h and
// write o; the last item of a row block sums y in j order.  Gate/up items
// never wait, and a cooperative launch keeps every CTA resident, so each wait
// ends; an expired wait sets an error bit and the item is skipped.
constexpr int kMaxFusedA = 256;
constexpr int kMaxRbA = 32;     // row-block mode: assignments per launch
constexpr int kMaxRbRows = 8;   // row-block mode: rows of H per down item
constexpr int kMaxRbOut = kMaxRbA * kMaxRbRows;
constexpr int kGURounds = 8;  // 128-bit loads per lane and tensor issued together
constexpr int kXBatch = 8;    // x blocks per warp loaded before they are quantized

__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Publish: a release-ordered add (the warp's prior writes, ordered before
// lane 0 by __syncwarp, become visible before the count does).
__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Shared staging of x (gate/up) or h (down) codes for one chunk of tokens,
// rounded up to 16 B; the down prefetch area follows it.
__host__ __device__ inline size_t fused_stage_bytes(int H, int F) {
    const size_t gu = (size_t)kMaxChunk * H + (size_t)kMaxChunk * (H / kBlock) * sizeof(BlockScale);
    const size_t dn = (size_t)kMaxChunk * F + (size_t)kMaxChunk * (F / kBlock) * sizeof(BlockScale);
    return ((gu > dn ? gu : dn) + 15) / 16 * 16;
}

// Top-k of one logits row by one warp, without a taken mask: round j picks
// the largest (value, -index) below the previous pick in the order (value
// desc, index asc), so ties go to the lower index.  Lane j < k returns pick
// j and its routing weight (softmax over the k picks, or over all E).
// Order-preserving unsigned key of a float (-0.0 and +0.0 map to one key).
__device__ __forceinline__ unsigned fkey(float v) {
    unsigned u = __float_as_uint(v == 0.0f ? 0.0f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one logits row by one warp.  Each logit is packed with its
// index into a 64-bit rank r = key(v) << 32 | ~e, so that larger r means
// (value desc, index asc).  Round j picks the largest r below the previous
// pick: a local log-depth max over the lane's values, then the warp maximum
// of the high word and, among the lanes holding it, of the low word.  Lane
// j < k returns pick j and its routing weight (softmax over the k picks, or
// over all E logits).
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

// Inverse of fkey (-0.0 comes back as +0.0, which exp treats alike).
__device__ __forceinline__ float funkey(unsigned key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

__device__ __forceinline__ void warp_topk_row(const float *l, int E, int k, int renorm, int lane, int &my_e,
                                              float &my_w) {
    constexpr int C = 16;  // logits per lane held in registers (one 512-wide chunk per warp)
    unsigned long long last = ~0ull;  // rank of the previous pick (first round: no bound)
    my_e = 0;
    unsigned my_key = 0u;
    unsigned long long rk[C];
    const bool resident = E <= 32 * C;
    if (resident) {
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const int e = lane + 32 * i;
            rk[i] = e < E ? ((unsigned long long)fkey(__ldg(l + e)) << 32) | (unsigned)(~(unsigned)e) : 0ull;
        }
    }
    for (int j = 0; j < k; ++j) {
        unsigned long long best = 0ull;
        for (int e0 = 0; e0 < (resident ? 32 * C : E); e0 += 32 * C) {
            unsigned long long c[C];
#pragma unroll
            for (int i = 0; i < C; ++i) {
                unsigned long long r;
                if (resident) {
                    r = rk[i];
                } else {
                    const int e = e0 + lane + 32 * i;
                    r = e < E ? ((unsigned long long)fkey(__ldg(l + e)) << 32) | (unsigned)(~(unsigned)e) : 0ull;
                }
                c[i] = r < last ? r : 0ull;
            }
#pragma unroll
            for (int w = C / 2; w > 0; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) c[i] = umax64(c[i], c[i + w]);
            best = umax64(best, c[0]);
        }
        const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(best >> 32));
        const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(best >> 32) == hi ? (unsigned)best : 0u);
        last = ((unsigned long long)hi << 32) | lo;
        if (lane == j) {
            my_e = (int)(~lo);
            my_key = hi;
        }
    }
    const float my_v = lane < k ? funkey(my_key) : -INFINITY;
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    const float ej = lane < k ? expf(my_v - m) : 0.0f;
    float den;
    if (renorm) {
        den = warp_sum_f(ej);
    } else {
        float sacc = 0.0f;
        for (int e0 = 0; e0 < E; e0 += 32 * C) {
            float v[C];
#pragma unroll
            for (int i = 0; i < C; ++i) {
                const int e = e0 + lane + 32 * i;
                v[i] = e < E ? __ldg(l + e) : -INFINITY;
            }
#pragma unroll
            for (int i = 0; i < C; ++i) sacc += e0 + lane + 32 * i < E ? expf(v[i] - m) : 0.0f;
        }
        den = warp_sum_f(sacc);
    }
    my_w = ej / den;
}

// Global expert id of an assignment -> this shard's local expert, or -1 for
// another shard's expert (ids outside the layer's range set error bit 0 and
// are read as local expert 0).
__device__ __forceinline__ int fused_local_e(const FusedParams &p, int g) {
    if (g < 0 || g >= p.n_route) {
        atomicOr(p.error, 1);
        return 0;
    }
    const int e = g - p.g.e_base;
    return e >= 0 && e < p.g.cv.E ? e : -1;
}

// The launch's plan in shared memory: s_e[a] = local expert of assignment a
// (-1: another shard's, left out), s_uniq / s_off / s_asg = used experts
// ascending, their assignment ranges and the assignments grouped by expert.
__device__ void fused_plan(const FusedParams &p, int *s_e, int *s_uniq, int *s_off, int *s_asg, int *s_nu,
                           int *s_cnt, int *s_first, float *s_w) {
    const int A = p.g.n_tokens * p.g.k;
    if (A <= 32) {
        // one warp: bitonic sort of (expert, assignment) keys, then the
        // used experts are the positions where the expert changes
        __syncthreads();  // routing / x prologue writes
        if (p.logits && p.g.n_tokens == 1) {
            // one routed token: its k picks are distinct experts already;
            // this shard's picks in pick order
            if (threadIdx.x < 32) {
                const int lane = threadIdx.x;
                const int e = lane < p.g.k ? fused_local_e(p, s_e[lane]) : -1;
                const unsigned mine = __ballot_sync(0xffffffffu, e >= 0);
                const int u = __popc(mine & ((1u << lane) - 1u));
                if (lane < p.g.k) s_e[lane] = e;
                if (e >= 0) {
                    s_asg[u] = lane;
                    s_uniq[u] = e;
                    s_off[u] = u;
                }
                if (lane == 0) {
                    s_off[__popc(mine)] = __popc(mine);
                    *s_nu = __popc(mine);
                }
            }
        } else if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int e = -1;
            if (lane < A) {
                e = fused_local_e(p, p.logits ? s_e[lane] : p.idx[lane]);
                s_e[lane] = e;
                if (!p.logits) s_w[lane] = p.g.w[lane];
            }
            const unsigned mine = __ballot_sync(0xffffffffu, e >= 0);
            const int An = __popc(mine);  // this shard's assignments (sorted first)
            unsigned key = e >= 0 ? ((unsigned)e << 8) | (unsigned)lane : 0xffffffffu;
#pragma unroll
            for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    const unsigned other = __shfl_xor_sync(0xffffffffu, key, stride);
                    const bool up = (lane & size) == 0;
                    const bool lower = (lane & stride) == 0;
                    const unsigned lo = min(key, other), hi = max(key, other);
                    key = (lower == up) ? lo : hi;
                }
            }
            const int se = (int)(key >> 8), sa = (int)(key & 0xffu);
            const int prev = __shfl_up_sync(0xffffffffu, se, 1);
            const bool head = lane < An && (lane == 0 || prev != se);
            const unsigned heads = __ballot_sync(0xffffffffu, head);
            const int u = __popc(heads & ((1u << lane) - 1u)) + (head ? 0 : -1);
            if (lane < An) s_asg[lane] = sa;
            if (head) {
                s_uniq[u] = se;
                s_off[u] = lane;
            }
            if (lane == 0) {
                const int nu = __popc(heads);
                s_off[nu] = An;
                *s_nu = nu;
            }
        }
        __syncthreads();
        return;
    }
    __syncthreads();  // routing writes
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        s_e[a] = fused_local_e(p, p.logits ? s_e[a] : p.idx[a]);
        if (!p.logits) s_w[a] = p.g.w[a];
    }
    __syncthreads();
    int n_first = 0;
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        const int e = s_e[a];
        int first = e >= 0;
        for (int b = 0; first && b < a; ++b)
            if (s_e[b] == e) {
                first = 0;
                break;
            }
        s_first[a] = first;
        n_first += first;
    }
    (void)n_first;
    __syncthreads();
    // rank of each first occurrence among the distinct experts, and its count
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        if (!s_first[a]) continue;
        const int e = s_e[a];
        int smaller = 0, cnt = 0;
        for (int b = 0; b < A; ++b) {
            const int eb = s_e[b];
            cnt += eb == e;
            smaller += (eb < e) && s_first[b];
        }
        s_uniq[smaller] = e;
        s_cnt[smaller] = cnt;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int n = 0, off = 0;
        for (int a = 0; a < A; ++a) n += s_first[a];
        for (int u = 0; u < n; ++u) {
            s_off[u] = off;
            off += s_cnt[u];
        }
        s_off[n] = off;
        *s_nu = n;
    }
    __syncthreads();
    // assignments grouped by expert, ascending assignment id within an expert
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        const int e = s_e[a];
        if (e < 0) continue;  // another shard's
        int lo = 0, hi = *s_nu - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s_uniq[mid] < e)
                lo = mid + 1;
            else
                hi = mid;
        }
        int before = 0;
        for (int b = 0; b < a; ++b) before += s_e[b] == e;
        s_asg[s_off[lo] + before] = a;
    }
    __syncthreads();
}

// One chunk (nt <= NT tokens of one used expert) of a gate/up item: issue
// the item's weight loads, quantize the chunk's x rows into shared memory
// while they fly, block dots, SwiGLU, quantize h (one warp per token).
template <int NT, class Prefetch>
__device__ __forceinline__ void gu_chunk(const FusedParams &p, int c0, int nt, int rg, int rloc, int sub, int lane,
                                         int warp, const uint4 *qg, const uint4 *qu, const __half *dg,
                                         const __half *du, int8_t *xq_s, BlockScale *xds_s, float (*sh_h)[32],
                                         const int *s_asg, Prefetch &&prefetch, bool xpre, const int *s_e) {
    const GemvParams &g = p.g;
    const int H = g.H, F = g.F, k = g.k;
    const int nbx = H / kBlock, rgs = F / kBlock;
    constexpr int XB = NT == 1 ? 12 : kXBatch;  // x blocks per warp loaded ahead of the weights
    // xpre: every token's x is already quantized in xq_s (row = token id)
    int xrow[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) xrow[t] = xpre ? (t < nt ? s_asg[c0 + t] / k : 0) : t;
    float ag[NT], au[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) ag[t] = au[t] = 0.0f;
    const int nblk = nt * nbx;
    for (int bb = 0; bb * kGULanes * kGURounds < nbx; ++bb) {
        // x of the chunk is requested before the weights, so the tiny x loads
        // are not queued behind the item's weight stream
        float xv[XB];
        if (bb == 0 && !xpre) {
#pragma unroll
            for (int i = 0; i < XB; ++i) {
                const int q = warp + i * kWarps;
                if (q < nblk) {
                    const int t = q / nbx, b = q - t * nbx;
                    const int tok = s_asg[c0 + t] / k;
                    xv[i] = __ldg(p.x + (size_t)tok * H + (size_t)b * kBlock + lane);
                }
            }
        }
        uint4 wg4[kGURounds], wu4[kGURounds];
        float sg[kGURounds], su[kGURounds];
#pragma unroll
        for (int i = 0; i < kGURounds; ++i) {
            const int b = sub + kGULanes * (bb * kGURounds + i);
            if (b < nbx) {
                wg4[i] = ld_weights(qg + b);
                wu4[i] = ld_weights(qu + b);
                sg[i] = ld_scale(dg + b);
                su[i] = ld_scale(du + b);
            }
        }
        if (bb == 0) prefetch();  // the down item's weights, behind the gate/up weights
        if (bb == 0 && !xpre) {
            // quantize the x rows of this chunk while the weights fly
            for (int q0 = warp; q0 < nblk; q0 += kWarps * XB) {
                if (q0 != warp) {
#pragma unroll
                    for (int i = 0; i < XB; ++i) {
                        const int q = q0 + i * kWarps;
                        if (q < nblk) {
                            const int t = q / nbx, b = q - t * nbx;
                            const int tok = s_asg[c0 + t] / k;
                            xv[i] = __ldg(p.x + (size_t)tok * H + (size_t)b * kBlock + lane);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < XB; ++i) {
                    const int q = q0 + i * kWarps;
                    if (q < nblk) {
                        const int t = q / nbx, b = q - t * nbx;
                        const int a = s_asg[c0 + t];
                        const int tok = a / k;
                        quantize_block_warp(xv[i], lane, xq_s + (size_t)t * H + (size_t)b * kBlock,
                                            xds_s + (size_t)t * nbx + b);
                        // the context's copy of x: written by the token's
                        // first assignment of this shard (s_e < 0: another's)
                        bool first = rg == 0;
                        for (int j = 0; first && j < a % k; ++j) first = s_e[tok * k + j] < 0;
                        if (first) {
                            g.xq_out[(size_t)tok * H + (size_t)b * kBlock + lane] =
                                xq_s[(size_t)t * H + (size_t)b * kBlock + lane];
                            if (lane == 0) g.xds_out[(size_t)tok * nbx + b] = xds_s[(size_t)t * nbx + b];
                        }
                    }
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < kGURounds; ++i) {
            const int b = sub + kGULanes * (bb * kGURounds + i);
            if (b < nbx) {
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (NT == 1 || t < nt) {
                        const int4 *xa = (const int4 *)(xq_s + (size_t)xrow[t] * H + (size_t)b * kBlock);
                        const int4 x0 = xa[0], x1 = xa[1];
                        const BlockScale xs = xds_s[(size_t)xrow[t] * nbx + b];
                        ag[t] += (float)q4_block_dot(wg4[i], x0, x1, xs.s) * (sg[i] * xs.d);
                        au[t] += (float)q4_block_dot(wu4[i], x0, x1, xs.s) * (su[i] * xs.d);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int o = kGULanes / 2; o > 0; o >>= 1) {
            ag[t] += __shfl_xor_sync(0xffffffffu, ag[t], o);
            au[t] += __shfl_xor_sync(0xffffffffu, au[t], o);
        }
    }
    if (sub == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
            if (NT == 1 || t < nt) sh_h[t][rloc] = ag[t] * au[t] / (1.0f + expf(-ag[t]));
    }
    __syncthreads();
    if (warp < nt) {
        const int a = s_asg[c0 + warp];
        quantize_block_warp(sh_h[warp][lane], lane, g.hq + (size_t)a * F + (size_t)rg * kBlock,
                            g.hds + (size_t)a * rgs + rg);
        __threadfence();  // h is published by the item's counter after the barrier
    }
    __syncthreads();
}

// One chunk of a down item: weight loads (or the shared-memory prefetch),
// a bounded wait for the expert's h (first chunk only), h staged in shared
// memory, block dots, o written per assignment.
template <int NT, int LD>
__device__ __forceinline__ void dn_chunk(const FusedParams &p, int c0, int nt, int e, int r, int rloc, int sub,
                                         const uint4 *qd, const __half *dd, int8_t *hq_s, BlockScale *hds_s,
                                         const uint8_t *dpre, bool from_smem, bool waited, const int *s_asg) {
    constexpr int DG = 32 / LD, DROWS = kWarps * DG;
    constexpr int RD = 12;  // loads per lane issued together (<= 12 rounds)
    const GemvParams &g = p.g;
    const int H = g.H, F = g.F;
    const int nbf = F / kBlock, rgs = F / kBlock;
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    for (int bb = 0; bb * LD * RD < nbf; ++bb) {
        uint4 w4[RD];
        float sw[RD];
        if (!from_smem) {
#pragma unroll
            for (int i = 0; i < RD; ++i) {
                const int b = sub + LD * (bb * RD + i);
                if (b < nbf) {
                    w4[i] = ld_weights(qd + b);
                    sw[i] = ld_scale(dd + b);
                }
            }
        }
        if (bb == 0) {
            if (from_smem) cp_async_wait_all();
            if (!waited) {
                // wait (bounded) for all gate/up row blocks of expert e
                if (threadIdx.x == 0) {
                    const long long t0 = clock64();
                    while (ld_acquire(&p.done_gu[e]) < (unsigned)rgs) {
                        if (clock64() - t0 > 4000000000ll) {
                            atomicOr(p.error, 2);
                            break;
                        }
                        __nanosleep(64);
                    }
                }
                __syncthreads();
            }
            // stage the chunk's h codes and scales
            for (int i = threadIdx.x; i < nt * (F / 16); i += blockDim.x) {
                const int t = i / (F / 16), c = i - t * (F / 16);
                const int a = s_asg[c0 + t];
                reinterpret_cast<int4 *>(hq_s + (size_t)t * F)[c] =
                    __ldcg(reinterpret_cast<const int4 *>(g.hq + (size_t)a * F) + c);
            }
            for (int i = threadIdx.x; i < nt * nbf; i += blockDim.x) {
                const int t = i / nbf, c = i - t * nbf;
                const int a = s_asg[c0 + t];
                const int2 v = __ldcg(reinterpret_cast<const int2 *>(g.hds + (size_t)a * nbf + c));
                hds_s[(size_t)t * nbf + c] = BlockScale{__int_as_float(v.x), v.y};
            }
            __syncthreads();
        }
        if (from_smem) {
            const uint4 *pc = (const uint4 *)dpre + (size_t)rloc * nbf;
            const __half *ps = (const __half *)(dpre + (size_t)DROWS * nbf * 16) + (size_t)rloc * nbf;
#pragma unroll
            for (int i = 0; i < RD; ++i) {
                const int b = sub + LD * (bb * RD + i);
                if (b < nbf) {
                    w4[i] = pc[b];
                    sw[i] = __half2float(ps[b]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < RD; ++i) {
            const int b = sub + LD * (bb * RD + i);
            if (b < nbf) {
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (NT == 1 || t < nt) {
                        const int4 *ha = (const int4 *)(hq_s + (size_t)t * F + (size_t)b * kBlock);
                        const BlockScale hs = hds_s[(size_t)t * nbf + b];
                        acc[t] += (float)q4_block_dot(w4[i], ha[0], ha[1], hs.s) * (sw[i] * hs.d);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int o = LD / 2; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    }
    if (sub == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
            if (NT == 1 || t < nt) g.o[(size_t)s_asg[c0 + t] * H + r] = acc[t];
    }
    __syncthreads();
}


// ------------------------------------------------ one routed token, early start
// T = 1, routed, row-block mode, E <= kT1MaxE.  Warp 0 routes and publishes
// each pick the moment it is known; warps 1..7 meanwhile copy the layer's
// gate and up table rows into shared memory and quantize x.  Gate/up item i
// is (pick i mod k, row group i / k), so every CTA starts its weight loads as
// soon as its own pick is out, and the later picks overlap the weight
// stream.  Rows 0..27 of an item belong to warps 1..7, rows 28..31 to warp
// 0, which takes them (and issues the CTA's down staging) after routing.
__device__ __forceinline__ void bar_sync_n(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void bar_arrive_n(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Lookahead prediction (mihailescu2m/llama.cpp, MoE expert streaming,
// lookahead prefetch: layer L+1's router predicts its experts from layer L's
// input, so their reads start a layer early).  Warp-level dot of one router
// row (bf16) with the layer's input x (fp32); the warp that writes the last
// predicted logit of the launch takes their top-k and publishes it; every
// CTA then prefetches a share of the picked experts' pool-resident gate, up
// and down blobs into L2 (lookahead_prefetch).
__device__ __forceinline__ void l2_prefetch(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void lookahead_predict(const FusedParams &p, int e, int lane) {
    const int H = p.g.H, E = p.g.cv.E, k = p.g.k;
    const uint4 *w = reinterpret_cast<const uint4 *>(p.pr_w + (size_t)e * H);  // 8 bf16 per uint4
    const float4 *x = reinterpret_cast<const float4 *>(p.x);
    float acc = 0.0f;
    for (int i = lane; i < H / 8; i += 32) {
        const uint4 wv = __ldg(w + i);
        const float4 x0 = __ldg(x + 2 * i), x1 = __ldg(x + 2 * i + 1);
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&wv);
        const float2 w01 = __bfloat1622float2(b2[0]), w23 = __bfloat1622float2(b2[1]);
        const float2 w45 = __bfloat1622float2(b2[2]), w67 = __bfloat1622float2(b2[3]);
        acc += w01.x * x0.x + w01.y * x0.y + w23.x * x0.z + w23.y * x0.w;
        acc += w45.x * x1.x + w45.y * x1.y + w67.x * x1.z + w67.y * x1.w;
    }
    acc = warp_sum_f(acc);
    unsigned last = 0;
    if (lane == 0) {
        p.pr_z[e] = p.pr_b[e] + acc;
        __threadfence();
        last = atomicAdd(p.pr_count, 1u) == (unsigned)(E - 1);
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    // top-k of the predicted logits (value desc, index asc): the logits are
    // read once into registers (16 per lane; E <= 512 on this path)
    unsigned long long rk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e2 = lane + 32 * i;
        rk[i] = e2 < E ? ((unsigned long long)fkey(__ldcg(p.pr_z + e2)) << 32) | (unsigned)(~(unsigned)e2) : 0ull;
    }
    unsigned long long prev = ~0ull;
    int my_e = -1;
    for (int j = 0; j < k; ++j) {
        unsigned long long c[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) c[i] = rk[i] < prev ? rk[i] : 0ull;
#pragma unroll
        for (int w2 = 8; w2 > 0; w2 >>= 1)
#pragma unroll
            for (int i = 0; i < w2; ++i) c[i] = umax64(c[i], c[i + w2]);
        const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(c[0] >> 32));
        const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(c[0] >> 32) == hi ? (unsigned)c[0] : 0u);
        prev = ((unsigned long long)hi << 32) | lo;
        if (lane == j) my_e = (int)(~lo);
    }
    if (lane < k) p.pr_set[lane] = my_e;
    __syncwarp();
    if (lane == 0) {
        *p.pr_count = 0u;  // for the next launch
        __threadfence();
        atomicExch(p.pr_flag, 1u);  // the prediction is out
    }
}

// This CTA's share of the L2 prefetch of the predicted experts (64 KB
// chunks of the pool-resident gate, up and down blobs, spread over every
// thread of the grid); nothing when the prediction is not out yet.
__device__ void lookahead_prefetch(const FusedParams &p) {
    if (!ld_acquire(p.pr_flag)) return;
    const int E = p.g.cv.E, k = p.g.k;
    constexpr uint32_t CH = 64u << 10;
    const int nch = (int)((p.pr_blob + CH - 1) / CH);
    const int total = k * 3 * nch;
    for (int c = (int)blockIdx.x + (int)gridDim.x * (int)threadIdx.x; c < total; c += (int)(gridDim.x * blockDim.x)) {
        const int j = c / (3 * nch), rem = c - j * 3 * nch, kd = rem / nch, ci = rem - kd * nch;
        const int pe = __ldcg(p.pr_set + j);
        if (pe < 0 || pe >= E) continue;
        const uint64_t ent = p.pr_tbl[(size_t)kd * E + pe];
        if (ent & 1ull) continue;  // cold: read zero-copy by the next layer, not prefetched
        const size_t off = (size_t)ci * CH;
        const size_t n = p.pr_blob - off < CH ? p.pr_blob - off : CH;
        l2_prefetch((const uint8_t *)(uintptr_t)ent + off, (uint32_t)n);
    }
}

// 128-bit loads per lane and tensor that a single-token gate/up item issues
// together, per weight format (the wider formats hold more registers per
// block: Q8_0 two uint4, Q6_K a uint4, a uint2 and two scales)
template <int FMT>
__host__ __device__ constexpr int t1_gu_rounds() {
    return FMT == kFmtQ4 ? kGURounds : (FMT == kFmtQ5 || FMT == kFmtQ4K) ? 6 : 4;
}

template <int FMT>
__device__ __forceinline__ void t1_route_gate_up(const FusedParams &p, int *s_e, float *s_w, int *s_uniq, int *s_off,
                                                 int *s_asg, int *s_nu, int *s_npick, float (*sh_h)[32], uint8_t *dsm,
                                                 uint32_t step_clock) {
    const GemvParams &g = p.g;
    const int H = g.H, F = g.F, k = g.k, E = g.cv.E;
    // with a shared expert (n_shared = 1): kr routed picks of the Er routed
    // experts, then the shared expert as pick kr (table column Er, weight 1),
    // known at kernel entry
    const int kr = k - p.n_shared, Er = E - p.n_shared;
    const int nbx = H / kBlock, rgs = F / kBlock;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int8_t *xq_s = (int8_t *)dsm;
    BlockScale *xds_s = (BlockScale *)(dsm + kMaxChunk * H);
    const uint64_t *s_tg = (const uint64_t *)(dsm + p.tbl_off);  // [gate row E][up row E][down row E]
    const uint64_t *s_tu = s_tg + E;
    volatile int *v_npick = s_npick;
    volatile int *v_e = s_e;
    if (warp == 0) {
        // ---- routing: top-k over packed ranks, each pick published at once
        const float *l = p.logits;
        unsigned long long rk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = lane + 32 * i;
            rk[i] = e < Er ? ((unsigned long long)fkey(__ldg(l + e)) << 32) | (unsigned)(~(unsigned)e) : 0ull;
        }
        unsigned long long last = ~0ull;
        int my_e = 0;
        unsigned my_key = 0u;
        for (int j = 0; j < kr; ++j) {
            unsigned long long c[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) c[i] = rk[i] < last ? rk[i] : 0ull;
#pragma unroll
            for (int w = 8; w > 0; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) c[i] = umax64(c[i], c[i + w]);
            const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(c[0] >> 32));
            const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(c[0] >> 32) == hi ? (unsigned)c[0] : 0u);
            last = ((unsigned long long)hi << 32) | lo;
            if (lane == 0) {
                v_e[j] = (int)(~lo);
                __threadfence_block();
                *v_npick = j + 1;
            }
            if (lane == j) {
                my_e = (int)(~lo);
                my_key = hi;
            }
        }
        const float my_v = lane < kr ? funkey(my_key) : -INFINITY;
        const float m = __shfl_sync(0xffffffffu, my_v, 0);
        const float ej = lane < kr ? expf(my_v - m) : 0.0f;
        float den;
        if (p.renorm) {
            den = warp_sum_f(ej);
        } else {
            float sacc = 0.0f;
            for (int e = lane; e < Er; e += 32) sacc += expf(__ldg(l + e) - m);
            den = warp_sum_f(sacc);
        }
        const float my_w = ej / den;
        if (lane < kr) {
            s_w[lane] = my_w;
            s_uniq[lane] = my_e;
            s_off[lane] = lane;
            s_asg[lane] = lane;
            if (blockIdx.x == 0) {
                p.idx_out[lane] = my_e;
                p.w_out[lane] = my_w;
            }
        } else if (lane < k) {
            // the shared expert: assignment kr, weight 1
            v_e[lane] = Er;
            s_w[lane] = 1.0f;
            s_uniq[lane] = Er;
            s_off[lane] = lane;
            s_asg[lane] = lane;
        }
        if (p.pr_mine && blockIdx.x == 0) {
            // how many of this layer's picks the previous layer predicted
            bool hit = false;
            if (lane < kr)
                for (int j = 0; j < kr; ++j) hit |= __ldcg(p.pr_mine + j) == my_e;
            const int hits = __popc(__ballot_sync(0xffffffffu, hit));
            if (lane == 0) {
                atomicAdd(p.pr_stats, (unsigned long long)kr);
                atomicAdd(p.pr_stats + 1, (unsigned long long)hits);
            }
        }
        if (lane == 0) {
            s_off[k] = k;
            *s_nu = k;
        }
        bar_sync_n(2, 256);  // x and the table rows are in shared memory
    } else {
        // ---- gate, up and down table rows (contiguous: tensor ids 3l .. 3l + 2)
        {
            // 16-byte copies when the three rows are 16-byte aligned (E even),
            // else 8-byte ones (an odd row length: a shared expert's column)
            uint8_t *dst = dsm + p.tbl_off;
            if (E % 2 == 0) {
                const uint4 *src = reinterpret_cast<const uint4 *>(g.cv.tbl + (size_t)g.tid_gate * E);
                for (int i = threadIdx.x - 32; i < 3 * E / 2; i += 224) cp_async16(dst + (size_t)i * 16, src + i);
            } else {
                const uint64_t *src = g.cv.tbl + (size_t)g.tid_gate * E;
                for (int i = threadIdx.x - 32; i < 3 * E; i += 224) cp_async8(dst + (size_t)i * 8, src + i);
            }
            cp_async_commit();
        }
        // ---- x of the token, quantized into shared memory
        for (int q0 = warp - 1; q0 < nbx; q0 += 7 * 12) {
            float xv[12];
#pragma unroll
            for (int i = 0; i < 12; ++i) {
                const int q = q0 + i * 7;
                if (q < nbx) xv[i] = __ldg(p.x + (size_t)q * kBlock + lane);
            }
#pragma unroll
            for (int i = 0; i < 12; ++i) {
                const int q = q0 + i * 7;
                if (q < nbx) quantize_block_warp(xv[i], lane, xq_s + (size_t)q * kBlock, xds_s + q);
            }
        }
        cp_async_wait_all();
        bar_arrive_n(2, 256);
        bar_sync_n(1, 224);
        if (blockIdx.x == 0) {
            for (int i = threadIdx.x - 32; i < H; i += 224) g.xq_out[i] = xq_s[i];
            for (int i = threadIdx.x - 32; i < nbx; i += 224) g.xds_out[i] = xds_s[i];
        }
        if (p.pr_w) {
            // the next layer's router on this layer's input: warp w of CTA c
            // takes expert c + (w - 1) * grid
            const int e = (int)blockIdx.x + (warp - 1) * (int)gridDim.x;
            if (e < E) lookahead_predict(p, e, lane);
        }
    }

    // ---- gate/up items: (pick i mod k, row group i / k)
    const int sub = lane % kGULanes, grp = lane / kGULanes;
    const int rloc = warp == 0 ? 28 + grp : (warp - 1) * 4 + grp;
    const size_t scale_off = blob_scales_offset_fmt(FMT, F, nbx);
    const int n_items = k * rgs;
    int m = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++m) {
        const int u = item % k, rg = item / k;
        if (warp != 0 && lane == 0 && u < kr) {
            const long long t0 = clock64();
            while (*v_npick <= u) {
                if (clock64() - t0 > 4000000000ll) {
                    atomicOr(p.error, 4);
                    break;
                }
                __nanosleep(20);
            }
            __threadfence_block();
        }
        __syncwarp();
        const int e = u < kr ? v_e[u] : Er;
        const uint64_t eg = s_tg[e], eu = s_tu[e];
        if (rg == 0 && threadIdx.x == 32) {
            record_read(g.cv, g.tid_gate, e, eg, step_clock);
            record_read(g.cv, g.tid_up, e, eu, step_clock);
        }
        const uint8_t *bg = (const uint8_t *)(uintptr_t)(eg & ~1ull);
        const uint8_t *bu = (const uint8_t *)(uintptr_t)(eu & ~1ull);
        const int r = rg * 32 + rloc;
        const size_t nblk = (size_t)F * nbx, row0 = (size_t)r * nbx;
        constexpr int RND = t1_gu_rounds<FMT>();
        float ag = 0.0f, au = 0.0f;
        for (int bb = 0; bb * kGULanes * RND < nbx; ++bb) {
            WCodes<FMT> wg[RND], wu[RND];
            WScale<FMT> sg[RND], su[RND];
#pragma unroll
            for (int i = 0; i < RND; ++i) {
                const int b = sub + kGULanes * (bb * RND + i);
                if (b < nbx) {
                    wg[i].load(bg, nblk, row0 + b);
                    wu[i].load(bu, nblk, row0 + b);
                    sg[i].load(bg + scale_off, row0 + b);
                    su[i].load(bu + scale_off, row0 + b);
                }
            }
#pragma unroll
            for (int i = 0; i < RND; ++i) {
                const int b = sub + kGULanes * (bb * RND + i);
                if (b < nbx) {
                    const int4 *xa = (const int4 *)(xq_s + (size_t)b * kBlock);
                    const int4 x0 = xa[0], x1 = xa[1];
                    const BlockScale xs = xds_s[b];
                    ag += sg[i].term(wg[i].dot(x0, x1, xs.s), xs);
                    au += su[i].term(wu[i].dot(x0, x1, xs.s), xs);
                }
            }
        }
#pragma unroll
        for (int o = kGULanes / 2; o > 0; o >>= 1) {
            ag += __shfl_xor_sync(0xffffffffu, ag, o);
            au += __shfl_xor_sync(0xffffffffu, au, o);
        }
        float *hrow = sh_h[m & 1];
        if (sub == 0) hrow[rloc] = ag * au / (1.0f + expf(-ag));
        __syncthreads();
        if (warp == 0) {
            // h block rg of assignment u (one token: assignment = pick index)
            quantize_block_warp(hrow[lane], lane, g.hq + (size_t)u * F + (size_t)rg * kBlock, g.hds + (size_t)u * rgs + rg);
            __syncwarp();
            if (lane == 0) red_release_add(&p.done_gu[u], 1u);
        }
    }
    __syncthreads();  // routing results for CTAs without a gate/up item
}

// Row-block mode, 2-8 tokens: the down rows of the cold used experts (read
// zero-copy over the host link) for this CTA's first down item, requested
// only once every cold expert's gate/up items are done.  Every down item
// needs the h of every used expert, so the link first serves the gate/up
// bytes that gate the whole down phase; rows requested as soon as a CTA's
// own gate/up item was done made the last gate/up items wait behind other
// CTAs' down rows (measured on the one-token layer, all-cold: 229 -> 168 us
// with this deferral and the register loads below; that layer now reads
// every down row in its dot loop instead).
__device__ void stage_cold_down(const FusedParams &p, const int *s_uniq, int nu, const uint64_t *s_td, uint8_t *dpre,
                                int rgs) {
    const GemvParams &g = p.g;
    const int H = g.H, nbf = g.F / kBlock, R = p.rb_rows;
    unsigned cold = 0u;  // bit u: pick u is cold
    for (int u = 0; u < nu; ++u) cold |= (unsigned)(s_td[s_uniq[u]] & 1ull) << u;
    if (!cold) return;
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        for (int u = 0; u < nu; ++u) {
            if (!((cold >> u) & 1u)) continue;
            while (ld_acquire(&p.done_gu[u]) < (unsigned)rgs) {
                if (clock64() - t0 > 4000000000ll) {
                    atomicOr(p.error, 2);
                    break;
                }
                __nanosleep(64);
            }
        }
    }
    __syncthreads();
    const int rb = blockIdx.x;
    const int nc = R * nbf, ns = R * nbf / 8, per = nc + ns;
    const size_t soff = blob_scales_offset(H, nbf);
    // the CTA's threads walk the cold picks one after the other (pick-major),
    // so that at any moment the CTAs of the grid read neighbouring rows of
    // the same expert: one sequential stream through each cold blob instead
    // of a few hundred scattered ones, which host memory serves at about
    // twice the rate
    const int n_cold = __popc(cold);
    for (int j = threadIdx.x; j < n_cold * per; j += blockDim.x) {
        const int c = j / per, q = j - c * per;
        int u = 0;  // the c-th cold pick
        for (int left = c; u < nu; ++u)
            if ((cold >> u) & 1u) {
                if (left == 0) break;
                --left;
            }
        const uint8_t *bd = (const uint8_t *)(uintptr_t)(s_td[s_uniq[u]] & ~1ull);
        // register loads, not cp.async: from host memory the asynchronous
        // copies of this pattern ran at half the link rate in this kernel
        if (q < nc)
            *(uint4 *)(dpre + ((size_t)u * nc + q) * 16) = ld_weights((const uint4 *)(bd + ((size_t)rb * nc + q) * 16));
        else
            *(uint4 *)(dpre + (size_t)nu * nc * 16 + ((size_t)u * ns + (q - nc)) * 16) =
                ld_weights((const uint4 *)(bd + soff + (size_t)rb * nc * 2 + (size_t)(q - nc) * 16));
    }
    __syncthreads();
}

// FMT: the weight format.  4-bit codes (Q4) run every mode; the other
// formats run the single-token early-start path only (row-block down items
// then read their rows from global memory instead of a shared-memory stage).
template <int LD, int NT, bool RB, int FMT = kFmtQ4>
__global__ void __launch_bounds__(256, 2) decode_layer_kernel(FusedParams p) {
    __shared__ int s_e[kMaxFusedA], s_uniq[kMaxFusedA], s_off[kMaxFusedA + 1], s_asg[kMaxFusedA],
        s_cnt[kMaxFusedA], s_first[kMaxFusedA];
    __shared__ float s_w[kMaxFusedA];
    __shared__ float s_o[RB ? kMaxRbOut : 1];  // row-block mode: [assignment][row] down outputs
    __shared__ int s_nu, s_last, s_npick;
    __shared__ float sh_h[kMaxChunk][32];
    extern __shared__ __align__(16) uint8_t dsm[];
    const GemvParams &g = p.g;
    const int H = g.H, F = g.F, k = g.k;
    const int nbx = H / kBlock, nbf = F / kBlock, rgs = F / kBlock;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    if (p.pdl) {
        // programmatic dependent launch: the previous kernel's writes are
        // visible after this wait; let the next layer's kernel get scheduled
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }
    // the clock is read after the dependency wait: every input of this
    // launch, the promotion pass's clock included, comes from before it
    const uint32_t step_clock = *g.cv.clock + (uint32_t)g.cv.clock_tokens;
    constexpr int DG = 32 / LD, DROWS = kWarps * DG;
    const int n_rb_all = H / DROWS;
    const int R = p.rb_rows;
    uint8_t *dpre = dsm + (RB ? (size_t)p.pre_off : fused_stage_bytes(H, F));
    const bool t1 = NT == 1 && RB && p.tbl_off > 0;
    if (FMT != kFmtQ4 && !t1) {
        // not a launch this instantiation serves (the host never makes one)
        if (threadIdx.x == 0) atomicOr(p.error, 8);
        return;
    }
    if (t1) {
        if (threadIdx.x == 0) s_npick = 0;
        __syncthreads();
        t1_route_gate_up<FMT>(p, s_e, s_w, s_uniq, s_off, s_asg, &s_nu, &s_npick, sh_h, dsm, step_clock);
    }
    // Prologue.  Routed launches: warps 0..T-1 route the tokens (top-k over
    // the logits) while the remaining warps quantize every token's x (small
    // batches: x does not depend on the routing); both before any weight
    // request.
    const bool xpre = g.n_tokens <= kMaxChunk;
    const int n_route_warps = !p.logits ? 0 : xpre ? max(1, min(g.n_tokens, kWarps / 2)) : kWarps;
    if (t1) {
        // routed and x quantized above
    } else if (p.logits && warp < n_route_warps) {
        const int k_ = g.k;
        for (int t = warp; t < g.n_tokens; t += n_route_warps) {
            int me;
            float mw;
            warp_topk_row(p.logits + (size_t)t * p.n_route, p.n_route, k_, p.renorm, lane, me, mw);
            if (lane < k_) {
                s_e[t * k_ + lane] = me;
                s_w[t * k_ + lane] = mw;
                if (blockIdx.x == 0) {
                    p.idx_out[t * k_ + lane] = me;
                    p.w_out[t * k_ + lane] = mw;
                }
            }
        }
    } else if (xpre) {
        int8_t *xq_s0 = (int8_t *)dsm;
        BlockScale *xds_s0 = (BlockScale *)(dsm + kMaxChunk * H);
        const int nblk = g.n_tokens * nbx;
        const int w0 = warp - n_route_warps, nw = kWarps - n_route_warps;
        for (int q0 = w0; q0 < nblk; q0 += nw * 12) {
            float xv[12];
#pragma unroll
            for (int i = 0; i < 12; ++i) {
                const int q = q0 + i * nw;
                if (q < nblk) xv[i] = __ldg(p.x + (size_t)q * kBlock + lane);
            }
#pragma unroll
            for (int i = 0; i < 12; ++i) {
                const int q = q0 + i * nw;
                if (q < nblk) quantize_block_warp(xv[i], lane, xq_s0 + (size_t)q * kBlock, xds_s0 + q);
            }
        }
    }
    // (the plan's barriers order these shared-memory writes before any use)
    if (!t1) fused_plan(p, s_e, s_uniq, s_off, s_asg, &s_nu, s_cnt, s_first, s_w);
    const int nu = s_nu;
    if (!t1 && xpre && blockIdx.x == 0) {
        // the context's copy of the quantized x (for inspection)
        const int8_t *xq_s0 = (const int8_t *)dsm;
        const BlockScale *xds_s0 = (const BlockScale *)(dsm + kMaxChunk * H);
        for (int i = threadIdx.x; i < g.n_tokens * H; i += blockDim.x) g.xq_out[i] = xq_s0[i];
        for (int i = threadIdx.x; i < g.n_tokens * nbx; i += blockDim.x) g.xds_out[i] = xds_s0[i];
    }

    // This CTA's first down item (codes + scales of its rows) is copied
    // into shared memory with cp.async, issued right behind the CTA's first
    // gate/up weight loads (or at once when the CTA has no gate/up item), so
    // the down weights stream while the gate/up item runs.  Row-block mode:
    // rows [rb R, rb R + R) of every used expert, laid out as codes
    // [expert][row][block] then scales [expert][row][block].
    const int n_dn_items = RB ? H / R : nu * n_rb_all;
    const bool prefetched = (int)blockIdx.x < n_dn_items;
    bool pf_issued = !prefetched || t1;  // (one routed token: staged during routing)
    bool pf_cold = false;                // per-expert mode: the first item's expert is cold (not staged)
    // warp w stages the rows of used experts w, w + 8, ...; a cold expert's
    // rows (host memory) are left to stage_cold_down on the first item
    // (early) and read with register loads on later ones (cp.async from host
    // memory ran at half the link rate)
    auto stage_rb = [&](int rb, bool early) {
        const int nc = R * nbf, ns = R * nbf / 8, per = nc + ns;
        const size_t soff = blob_scales_offset(H, nbf);
        for (int u = warp; u < nu; u += kWarps) {
            const uint64_t ed = g.cv.tbl[(size_t)g.tid_down * g.cv.E + s_uniq[u]];
            const bool cold = ed & 1ull;
            if (cold && early) continue;
            const uint8_t *bd = (const uint8_t *)(uintptr_t)(ed & ~1ull);
            for (int j = lane; j < per; j += 32) {
                uint8_t *dst = j < nc ? dpre + ((size_t)u * nc + j) * 16
                                      : dpre + (size_t)nu * nc * 16 + ((size_t)u * ns + (j - nc)) * 16;
                const uint8_t *src = j < nc ? bd + ((size_t)rb * nc + j) * 16
                                            : bd + soff + (size_t)rb * nc * 2 + (size_t)(j - nc) * 16;
                if (cold)
                    *(uint4 *)dst = ld_weights((const uint4 *)src);
                else
                    cp_async16(dst, src);
            }
        }
        cp_async_commit();
    };
    auto issue_prefetch = [&]() {
        if (pf_issued) return;
        pf_issued = true;
        if (RB) {
            stage_rb(blockIdx.x, true);
            return;
        }
        const int u = blockIdx.x / n_rb_all, rb = blockIdx.x - u * n_rb_all;
        const uint64_t ed = g.cv.tbl[(size_t)g.tid_down * g.cv.E + s_uniq[u]];
        if (ed & 1ull) {
            // cold: the item reads its rows itself (register loads) once the
            // expert's h is out
            pf_cold = true;
            return;
        }
        const uint8_t *bd = (const uint8_t *)(uintptr_t)(ed & ~1ull);
        const uint8_t *codes = bd + (size_t)rb * DROWS * nbf * 16;
        const uint8_t *scales = bd + blob_scales_offset(H, nbf) + (size_t)rb * DROWS * nbf * 2;
        const int nc = DROWS * nbf, ns = DROWS * nbf * 2 / 16;
        for (int i = threadIdx.x; i < nc + ns; i += blockDim.x) {
            if (i < nc)
                cp_async16(dpre + (size_t)i * 16, codes + (size_t)i * 16);
            else
                cp_async16(dpre + (size_t)nc * 16 + (size_t)(i - nc) * 16, scales + (size_t)(i - nc) * 16);
        }
        cp_async_commit();
    };
    if ((int)blockIdx.x >= nu * rgs) issue_prefetch();

    // ---------------- gate/up items
    if (!t1) {
        int8_t *xq_s = (int8_t *)dsm;                                     // [chunk][H]
        BlockScale *xds_s = (BlockScale *)(dsm + kMaxChunk * H);          // [chunk][nbx]
        const int sub = lane % kGULanes, grp = lane / kGULanes;
        const int rloc = warp * (32 / kGULanes) + grp;
        const size_t scale_off = blob_scales_offset(F, nbx);
        const int n_items = nu * rgs;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            const int u = item / rgs, rg = item - u * rgs;
            const int e = s_uniq[u];
            const int a0 = s_off[u], a1 = s_off[u + 1];
            const uint64_t eg = g.cv.tbl[(size_t)g.tid_gate * g.cv.E + e];
            const uint64_t eu = g.cv.tbl[(size_t)g.tid_up * g.cv.E + e];
            if (rg == 0 && threadIdx.x == 0) {
                record_read(g.cv, g.tid_gate, e, eg, step_clock);
                record_read(g.cv, g.tid_up, e, eu, step_clock);
            }
            const uint8_t *bg = (const uint8_t *)(uintptr_t)(eg & ~1ull);
            const uint8_t *bu = (const uint8_t *)(uintptr_t)(eu & ~1ull);
            const int r = rg * 32 + rloc;
            const uint4 *qg = (const uint4 *)bg + (size_t)r * nbx;
            const uint4 *qu = (const uint4 *)bu + (size_t)r * nbx;
            const __half *dg = (const __half *)(bg + scale_off) + (size_t)r * nbx;
            const __half *du = (const __half *)(bu + scale_off) + (size_t)r * nbx;
            for (int c0 = a0; c0 < a1; c0 += NT) {
                const int nt = min(NT, a1 - c0);
                gu_chunk<NT>(p, c0, nt, rg, rloc, sub, lane, warp, qg, qu, dg, du, xq_s, xds_s, sh_h, s_asg,
                             issue_prefetch, xpre, s_e);
            }
            // publish this row block of expert e (the writers fenced h
            // before the chunk's closing barrier)
            if (threadIdx.x == 0) atomicAdd(&p.done_gu[RB ? u : e], 1u);
        }
    }

    issue_prefetch();

    // ---------------- down items
    if (RB && p.pr_w) lookahead_prefetch(p);  // the next layer's predicted experts into L2
    if (RB) {
        // Row-block mode: item rb = rows [rb R, rb R + R) of H for every used
        // expert, (expert, row) pairs spread over the CTA's lanes (LD lanes a
        // pair).  Each warp waits only for the gate/up items of the experts
        // its pairs touch and reads their h from L2, so the down products of
        // early experts overlap the gate/up of late ones; each item then sums
        // y in j order.
        const int n_items = n_dn_items;
        if ((int)blockIdx.x < n_items) {
            constexpr int VP = 256 / LD;  // (expert, row) pairs per pass
            const int sub = threadIdx.x % LD;
            cp_async_wait_all();
            __syncthreads();  // the first item's staged rows
            if (FMT == kFmtQ4 && !t1) stage_cold_down(p, s_uniq, nu, g.cv.tbl + (size_t)g.tid_down * g.cv.E, dpre, rgs);
            for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
                const bool first = item == (int)blockIdx.x;
                if (!first) {
                    __syncthreads();  // the previous item's reads of the staged rows and s_o
                    if (FMT == kFmtQ4 && !t1) stage_rb(item, false);
                    cp_async_wait_all();
                    __syncthreads();
                }
                if (item == 0 && (int)threadIdx.x < nu) {
                    const int e = s_uniq[threadIdx.x];
                    record_read(g.cv, g.tid_down, e, g.cv.tbl[(size_t)g.tid_down * g.cv.E + e], step_clock);
                }
                const uint4 *wc0 = (const uint4 *)dpre;
                const __half *ws0 = (const __half *)(dpre + (size_t)nu * R * nbf * 16);
                for (int v0 = 0; v0 < nu * R; v0 += VP) {
                    const int vr = v0 + (int)threadIdx.x / LD;
                    const bool act = vr < nu * R;
                    const int u = act ? vr / R : 0, r = vr - u * R;
                    if (first) {
                        // bounded wait for the gate/up items of this warp's experts
                        const int ulo = __shfl_sync(0xffffffffu, u, 0);
                        const int uhi = __reduce_max_sync(0xffffffffu, act ? u : 0);
                        if (lane == 0 && v0 + (int)threadIdx.x / LD < nu * R) {
                            const long long t0 = clock64();
                            for (int uu = ulo; uu <= uhi; ++uu) {
                                while (ld_acquire(&p.done_gu[uu]) < (unsigned)rgs) {
                                    if (clock64() - t0 > 4000000000ll) {
                                        atomicOr(p.error, 2);
                                        break;
                                    }
                                    __nanosleep(20);
                                }
                            }
                        }
                        __syncwarp();
                    }
                    const int a0 = act ? s_off[u] : 0, cnt = act ? s_off[u + 1] - a0 : 0;
                    const int mc = __reduce_max_sync(0xffffffffu, cnt);
                    const uint4 *wc = wc0 + (size_t)vr * nbf;
                    const __half *ws = ws0 + (size_t)vr * nbf;
                    // one token (every format): row item R + r of the expert's
                    // down blob, read from global memory when the dot needs it
                    // (staging the rows in shared memory measured slower)
                    const bool staged = FMT == kFmtQ4 && !t1;
                    const uint8_t *bdg = nullptr;
                    size_t drow = 0;
                    if (!staged && act) {
                        const uint64_t *s_td = (const uint64_t *)(dsm + p.tbl_off) + 2 * g.cv.E;
                        bdg = (const uint8_t *)(uintptr_t)(s_td[s_uniq[u]] & ~1ull);
                        drow = ((size_t)item * R + r) * nbf;
                    }
                    for (int sl = 0; sl < mc; ++sl) {
                        float acc = 0.0f;
                        int a = 0;
                        if (sl < cnt) {
                            a = s_asg[a0 + sl];
                            // h of assignment a from L2 (written by other CTAs of this launch)
                            const int4 *ha = reinterpret_cast<const int4 *>(g.hq + (size_t)a * F);
                            const int2 *hs = reinterpret_cast<const int2 *>(g.hds + (size_t)a * nbf);
                            if (staged) {
#pragma unroll 4
                                for (int b = sub; b < nbf; b += LD) {
                                    const int4 h0 = __ldcg(ha + 2 * b), h1 = __ldcg(ha + 2 * b + 1);
                                    const int2 hsc = __ldcg(hs + b);
                                    const uint4 w4 = wc[b];
                                    acc += (float)q4_block_dot(w4, h0, h1, hsc.y) *
                                           (__half2float(ws[b]) * __int_as_float(hsc.x));
                                }
                            } else {
                                const size_t soff = blob_scales_offset_fmt(FMT, H, nbf);
#pragma unroll 4
                                for (int b = sub; b < nbf; b += LD) {
                                    const int4 h0 = __ldcg(ha + 2 * b), h1 = __ldcg(ha + 2 * b + 1);
                                    const int2 hsc = __ldcg(hs + b);
                                    WCodes<FMT> w;
                                    WScale<FMT> sc;
                                    w.load(bdg, (size_t)H * nbf, drow + b);
                                    sc.load(bdg + soff, drow + b);
                                    acc += sc.term(w.dot(h0, h1, hsc.y), BlockScale{__int_as_float(hsc.x), hsc.y});
                                }
                            }
                        }
#pragma unroll
                        for (int o = LD / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                        if (sl < cnt && sub == 0) s_o[a * R + r] = acc;
                    }
                }
                __syncthreads();
                for (int i = threadIdx.x; i < g.n_tokens * R; i += blockDim.x) {
                    const int t = i / R, r = i - t * R;
                    float y = 0.0f;
                    for (int j = 0; j < k; ++j)
                        if (s_e[t * k + j] >= 0) y += s_w[t * k + j] * s_o[(t * k + j) * R + r];
                    g.y[(size_t)t * H + (size_t)item * R + r] = y;
                }
            }
        }
    } else {
        constexpr int G = 32 / LD, ROWS = kWarps * G;
        int8_t *hq_s = (int8_t *)dsm;                                   // [chunk][F]
        BlockScale *hds_s = (BlockScale *)(dsm + kMaxChunk * F);        // [chunk][nbf]
        const int sub = lane % LD, grp = lane / LD;
        const int rloc = warp * G + grp;
        const int n_rb = H / ROWS;
        const size_t scale_off = blob_scales_offset(H, nbf);
        const int n_items = nu * n_rb;
        if (nu == 0) {
            // no assignment of this shard: y = 0
            for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)g.n_tokens * H;
                 i += (size_t)gridDim.x * blockDim.x)
                g.y[i] = 0.0f;
        }
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            const int u = item / n_rb, rb = item - u * n_rb;
            const int e = s_uniq[u];
            const int a0 = s_off[u], a1 = s_off[u + 1];
            const uint64_t ed = g.cv.tbl[(size_t)g.tid_down * g.cv.E + e];
            if (rb == 0 && threadIdx.x == 0) record_read(g.cv, g.tid_down, e, ed, step_clock);
            const uint8_t *bd = (const uint8_t *)(uintptr_t)(ed & ~1ull);
            const int r = rb * ROWS + rloc;
            const uint4 *qd = (const uint4 *)bd + (size_t)r * nbf;
            const __half *dd = (const __half *)(bd + scale_off) + (size_t)r * nbf;
            bool waited = false;
            const bool from_smem = prefetched && !pf_cold && item == (int)blockIdx.x;
            for (int c0 = a0; c0 < a1; c0 += NT) {
                const int nt = min(NT, a1 - c0);
                dn_chunk<NT, LD>(p, c0, nt, e, r, rloc, sub, qd, dd, hq_s, hds_s, dpre, from_smem, waited, s_asg);
                waited = true;
            }
            // arrival count of this row block; the last item combines
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                const unsigned prev = atomicAdd(&g.counters[rb], 1u);
                s_last = (prev == (unsigned)(nu - 1));
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                const int n_out = g.n_tokens * ROWS;
                for (int i = threadIdx.x; i < n_out; i += blockDim.x) {
                    const int t = i / ROWS, rr = rb * ROWS + (i - t * ROWS);
                    float y = 0.0f;
                    for (int j = 0; j < k; ++j) {
                        const size_t a = (size_t)t * k + j;
                        if (s_e[a] >= 0) y += s_w[a] * __ldcg(g.o + a * H + rr);
                    }
                    g.y[(size_t)t * H + rr] = y;
                }
                if (threadIdx.x == 0) g.counters[rb] = 0u;
            }
            __syncthreads();
        }
    }

    // ---------------- the last CTA to leave resets the per-expert counters
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(p.exit_count, 1u);
        if (prev == gridDim.x - 1) {
            for (int u = 0; u < nu; ++u) p.done_gu[RB ? u : s_uniq[u]] = 0u;
            *p.exit_count = 0u;
            if (p.pr_w) *p.pr_flag = 0u;  // every CTA is past its prefetch
            __threadfence();
        }
    }
}

size_t fused_smem_bytes(int H, int F) {
    const int LD = F / kBlock <= 40 ? 4 : 8;
    const size_t rows = (size_t)kWarps * (32 / LD);
    return fused_stage_bytes(H, F) + rows * (F / kBlock) * kBlockBytes;
}

int fused_down_lanes(int F) { return F / kBlock <= 40 ? 4 : 8; }

static int fused_nt(int T) { return T <= 1 ? 1 : T == 2 ? 2 : T <= 4 ? 4 : 8; }

template <bool RB>
static const void *fused_fn_t(int F, int T) {
    const int ld = fused_down_lanes(F), nt = fused_nt(T);
    if (ld == 4) {
        if (nt == 1) return (const void *)decode_layer_kernel<4, 1, RB>;
        if (nt == 2) return (const void *)decode_layer_kernel<4, 2, RB>;
        if (nt == 4) return (const void *)decode_layer_kernel<4, 4, RB>;
        return (const void *)decode_layer_kernel<4, 8, RB>;
    }
    if (nt == 1) return (const void *)decode_layer_kernel<8, 1, RB>;
    if (nt == 2) return (const void *)decode_layer_kernel<8, 2, RB>;
    if (nt == 4) return (const void *)decode_layer_kernel<8, 4, RB>;
    return (const void *)decode_layer_kernel<8, 8, RB>;
}

static const void *fused_fn(int F, int T, bool rb) { return rb ? fused_fn_t<true>(F, T) : fused_fn_t<false>(F, T); }

// The single-token row-block kernel of a non-Q4 weight format.
template <int FMT>
static const void *fused_fn_fmt_t(int F) {
    return fused_down_lanes(F) == 4 ? (const void *)decode_layer_kernel<4, 1, true, FMT>
                                    : (const void *)decode_layer_kernel<8, 1, true, FMT>;
}
static const void *fused_fn_fmt(int F, int fmt) {
    switch (fmt) {
        case kFmtQ8: return fused_fn_fmt_t<kFmtQ8>(F);
        case kFmtQ5: return fused_fn_fmt_t<kFmtQ5>(F);
        case kFmtQ4K: return fused_fn_fmt_t<kFmtQ4K>(F);
        case kFmtQ6K: return fused_fn_fmt_t<kFmtQ6K>(F);
        case kFmtQ5K: return fused_fn_fmt_t<kFmtQ5K>(F);
        default: return fused_fn(F, 1, true);
    }
}

// Shared-memory opt-in for every token-count variant of one mode (only ever
// raised, so contexts of different shapes coexist); *blocks_per_sm gets the
// smallest resident-CTA count over the variants (a safe cooperative grid).
static int configure_mode(int F, size_t smem, bool rb, int *blocks_per_sm) {
    // the shared-memory opt-in is a per-device function attribute
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> opted;
    std::lock_guard<std::mutex> lk(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
    int best = 1 << 30;
    for (int T : {1, 2, 4, 8}) {
        const void *fn = fused_fn(F, T, rb);
        size_t &cur = opted[{dev, fn}];
        if (smem > cur) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
            cur = smem;
        }
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, 256, smem);
        if (e != cudaSuccess) return (int)e;
        best = b < best ? b : best;
    }
    *blocks_per_sm = best;
    return 0;
}

int fused_configure(int F, size_t smem, int *blocks_per_sm) { return configure_mode(F, smem, false, blocks_per_sm); }
int fused_configure_rb(int F, size_t smem, int *blocks_per_sm) { return configure_mode(F, smem, true, blocks_per_sm); }

int fused_configure_t1_fmt(int F, int fmt, size_t smem, int *blocks_per_sm) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> opted;
    std::lock_guard<std::mutex> lk(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
    const void *fn = fused_fn_fmt(F, fmt);
    size_t &cur = opted[{dev, fn}];
    if (smem > cur) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        cur = smem;
    }
    return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, 256, smem);
}

// Row-block down mode: rows of H per down item for a launch of T tokens, or
// 0 when the mode does not apply (more than kMaxRbA assignments or 8 tokens,
// h of all assignments above kRbStageBudget, or no row count whose staged
// rows fit kRbPrefetchBudget in one pass of (expert, row) pairs).
constexpr size_t kRbStageBudget = 40u << 10;
constexpr size_t kRbPrefetchBudget = 52u << 10;

int fused_rb_rows(int H, int F, int T, int k, int E) {
    const int A = T * k, U = A < E ? A : E, nbf = F / kBlock, LD = fused_down_lanes(F);
    if (T < 1 || T > kMaxChunk || A > kMaxRbA) return 0;
    if ((size_t)A * F + (size_t)A * nbf * sizeof(BlockScale) + 16 > kRbStageBudget) return 0;
    // (expert, row) pairs of an item: one pass of the CTA's lanes, or two for
    // one token (nine experts with a shared one keep 8 rows per item, so the
    // items still fit one grid)
    const int max_pairs = (T == 1 ? 2 : 1) * (256 / LD);
    for (int R = kMaxRbRows; R >= 2; R >>= 1) {
        if (H % R || (R * nbf * 2) % 16) continue;
        if (U * R > max_pairs) continue;
        if ((size_t)U * R * nbf * kBlockBytes > kRbPrefetchBudget) continue;
        return R;
    }
    return 0;
}

// Dynamic shared memory of a row-block launch: x staging or h staging
// (aliased; x is dead once the CTA's gate/up items are done), then the
// staged down rows.
size_t fused_rb_smem(int H, int F, int T, int k, int E, int rows, int *pre_off) {
    const int A = T * k, U = A < E ? A : E, nbf = F / kBlock, nbx = H / kBlock;
    const size_t xs = (size_t)kMaxChunk * H + (size_t)kMaxChunk * nbx * sizeof(BlockScale);
    const size_t hs = (((size_t)A * F + 15) & ~(size_t)15) + (size_t)A * nbf * sizeof(BlockScale);
    const size_t r0 = ((xs > hs ? xs : hs) + 15) / 16 * 16;
    if (pre_off) *pre_off = (int)r0;
    return r0 + (size_t)U * rows * nbf * kBlockBytes;
}

// The early-start path for one routed token keeps the logits in registers
// (16 per lane) and copies the gate and up table rows with 16-byte copies.
bool fused_t1_ok(int E, int k) { return E <= 32 * 16 && E % 2 == 0 && k <= 32; }


int launch_fused(const FusedParams &p, int grid, size_t smem, cudaStream_t st, cudaEvent_t const *ev) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    if (ev) record(ev[0], st);
    void *args[] = {(void *)&p};
    const void *fn = p.g.fmt != kFmtQ4 ? fused_fn_fmt(p.g.F, p.g.fmt) : fused_fn(p.g.F, p.g.n_tokens, p.rb_rows > 0);
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (ev) {
        record(ev[1], st);
        record(ev[2], st);
        record(ev[3], st);
    }
    return (int)e;
}

// --------------------------------------------------------------- hooks
// Block dots of rows row0.. of one expert through the pointer table, with
// the same routine the mat-vec kernels use.  One warp per (row, 32 blocks).
template <int FMT>
__global__ void block_dots_kernel(const uint8_t *blob, int rows, int nb, int row0, int n_rows,
                                  const int8_t *__restrict__ qa, int32_t *__restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_rows * nb) return;
    const int r = row0 + i / nb, b = i % nb;
    WCodes<FMT> w;
    w.load(blob, (size_t)rows * nb, (size_t)r * nb + b);
    const int4 *xa = (const int4 *)(qa + (size_t)b * kBlock);
    int4 x0 = xa[0], x1 = xa[1];
    int s = 0;
    const int8_t *q8 = qa + (size_t)b * kBlock;
    for (int j = 0; j < kBlock; ++j) s += q8[j];
    out[i] = w.dot(x0, x1, s);
}

int launch_block_dots(const uint8_t *blob, int fmt, int rows, int nb, int row0, int n_rows, const int8_t *qa,
                      int32_t *out, cudaStream_t st) {
    int n = n_rows * nb;
    if (n <= 0) return 0;
    if (fmt == kFmtQ8)
        block_dots_kernel<kFmtQ8><<<(n + 255) / 256, 256, 0, st>>>(blob, rows, nb, row0, n_rows, qa, out);
    else if (fmt == kFmtQ5)
        block_dots_kernel<kFmtQ5><<<(n + 255) / 256, 256, 0, st>>>(blob, rows, nb, row0, n_rows, qa, out);
    else if (fmt == kFmtQ4K)
        block_dots_kernel<kFmtQ4K><<<(n + 255) / 256, 256, 0, st>>>(blob, rows, nb, row0, n_rows, qa, out);
    else if (fmt == kFmtQ6K)
        block_dots_kernel<kFmtQ6K><<<(n + 255) / 256, 256, 0, st>>>(blob, rows, nb, row0, n_rows, qa, out);
    else if (fmt == kFmtQ5K)
        block_dots_kernel<kFmtQ5K><<<(n + 255) / 256, 256, 0, st>>>(blob, rows, nb, row0, n_rows, qa, out);
    else
        block_dots_kernel<kFmtQ4><<<(n + 255) / 256, 256, 0, st>>>(blob, rows, nb, row0, n_rows, qa, out);
    return (int)cudaGetLastError();
}

// Streams `n16` 16-byte words with 128-bit loads; the xor of everything read
// goes to *sink so the loads cannot be dropped.
__global__ void __launch_bounds__(256) stream_read_kernel(const uint4 *__restrict__ src, size_t n16, uint32_t *sink) {
    uint32_t acc = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 a = ld_weights(src + i), b = ld_weights(src + i + stride), c = ld_weights(src + i + 2 * stride),
              d = ld_weights(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
        uint4 a = ld_weights(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (acc == 0x9e3779b9u) *sink = acc;
}

int launch_stream_read(const void *src, size_t bytes, uint32_t *sink, int n_sm, cudaStream_t st) {
    stream_read_kernel<<<n_sm * 8, 256, 0, st>>>((const uint4 *)src, bytes / 16, sink);
    return (int)cudaGetLastError();
}

// Table / stamp updates published by the promotion pass.
// Between-step state update: the promotion pass's table / slot / stamp
// writes (read straight from the host's pinned list), the new clock, and the
// per-step records cleared (hit bitmap + miss count, miss bitmap).
__global__ void step_finish_kernel(const Update *__restrict__ u, int n, uint64_t *tbl, int32_t *slot,
                                   uint32_t *stamps, uint32_t *clock, uint32_t new_clock, uint32_t *clear_a, int n_a,
                                   uint32_t *clear_b, int n_b) {
    const int stride = gridDim.x * blockDim.x;
    const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
    if (i0 == 0) *clock = new_clock;
    for (int i = i0; i < n; i += stride) {
        const Update x = u[i];
        if (x.what == 0)
            tbl[x.index] = x.value;
        else if (x.what == 1)
            slot[x.index] = (int32_t)(int64_t)x.value;
        else
            stamps[x.index] = (uint32_t)x.value;
    }
    for (int i = i0; i < n_a; i += stride) clear_a[i] = 0u;
    for (int i = i0; i < n_b; i += stride) clear_b[i] = 0u;
}

int launch_step_finish(const Update *u, int n, uint64_t *tbl, int32_t *slot, uint32_t *stamps, uint32_t *clock,
                       uint32_t new_clock, uint32_t *clear_a, int n_a, uint32_t *clear_b, int n_b, cudaStream_t st) {
    const int work = n > n_a ? (n > n_b ? n : n_b) : (n_a > n_b ? n_a : n_b);
    int grid = (work + 255) / 256;
    grid = grid < 1 ? 1 : grid > 64 ? 64 : grid;
    step_finish_kernel<<<grid, 256, 0, st>>>(u, n, tbl, slot, stamps, clock, new_clock, clear_a, n_a, clear_b, n_b);
    return (int)cudaGetLastError();
}

// Prefill preheat: the (token, expert) assignments of one layer added to the
// layer's use counts, through a per-block histogram in shared memory.
__global__ void count_assign_kernel(const int32_t *__restrict__ idx, int n, int E, int e_base, uint32_t *cnt) {
    extern __shared__ uint32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0u;
    __syncthreads();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int e = idx[i] - e_base;  // this shard's experts only
        if ((unsigned)e < (unsigned)E) atomicAdd(&hist[e], 1u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (hist[e]) atomicAdd(&cnt[e], hist[e]);
}

int launch_count_assign(const int32_t *idx, int n, int E, int e_base, uint32_t *cnt, cudaStream_t st) {
    if (n <= 0) return 0;
    int grid = (n + 1023) / 1024;
    grid = grid > 152 ? 152 : grid;
    count_assign_kernel<<<grid, 256, sizeof(uint32_t) * (size_t)E, st>>>(idx, n, E, e_base, cnt);
    return (int)cudaGetLastError();
}

// Shared expert: the routed assignments of every token followed by one more,
// expert e_shared with weight 1 (routed ids outside [0, e_shared) set error
// bit 0 and are replaced by e_shared, which the plan then reads as valid).
__global__ void shared_assign_kernel(const int32_t *__restrict__ idx, const float *__restrict__ w, int T, int k,
                                     int e_shared, int32_t *idx_a, float *w_a, int *error) {
    pdl_enter();
    const int ka = k + 1;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * ka; i += gridDim.x * blockDim.x) {
        const int t = i / ka, j = i - t * ka;
        if (j == k) {
            idx_a[i] = e_shared;
            w_a[i] = 1.0f;
        } else {
            int e = idx[(size_t)t * k + j];
            if (e < 0 || e >= e_shared) {
                atomicOr(error, 1);
                e = e_shared;
            }
            idx_a[i] = e;
            w_a[i] = w[(size_t)t * k + j];
        }
    }
}

int launch_shared_assign(const int32_t *idx, const float *w, int T, int k, int e_shared, int32_t *idx_a, float *w_a,
                         int *error, cudaStream_t st) {
    const int n = T * (k + 1);
    if (n <= 0) return 0;
    const int grid = (n + 255) / 256 < 152 ? (n + 255) / 256 : 152;
    return (int)launch_pdl(shared_assign_kernel, dim3(grid), dim3(256), 0, st, idx, w, T, k, e_shared, idx_a, w_a,
                           error);
}

// Debug: keep one thread of the stream busy for a bounded time (global
// timer), so that a host-side poll limit can run out without any fault or
// hang; the wait ends by itself after min(ns, 2 s).
__global__ void busy_kernel(unsigned long long ns) {
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    if (ns > 2000000000ull) ns = 2000000000ull;
    const long long c0 = clock64();
    do {
        __nanosleep(1000);
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < ns && clock64() - c0 < 6000000000ll);  // the SM clock bounds it too (~3 s)
}

int launch_busy(unsigned long long ns, cudaStream_t st) {
    busy_kernel<<<1, 1, 0, st>>>(ns);
    return (int)cudaGetLastError();
}

}  // namespace moe
