// Internal interface between the C-ABI runtime (moe_cache.cu) and the
// kernels.  Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {

struct PlanParams {
    const float *x;       // [T][H] (quantized when quantize_x)
    int8_t *xq;           // [T][H]
    BlockScale *xds;      // [T][H/32]
    const int32_t *idx;   // [T][k]
    int32_t *n_uniq;      // [1]
    int32_t *uniq_e;      // [min(T*k, E)]
    int32_t *uniq_off;    // [min(T*k, E) + 1]
    int32_t *assign;      // [T*k]: assignment ids grouped by expert
    int *error;           // [1]: bit 0 = expert id out of range
    int T, k, E, H, quantize_x;
    // expert shard: ids are global in [0, E_route); this context holds
    // [e_base, e_base + E) (local id = id - e_base); assignments to other
    // experts are left out of every used-expert list (placed after them in
    // assign) and contribute nothing
    int e_base, E_route;
};

struct GemvParams {
    CacheView cv;
    int tid_gate, tid_up, tid_down;
    int n_tokens, k, H, F;
    const int8_t *xq;
    const BlockScale *xds;
    const int32_t *n_uniq, *uniq_e, *uniq_off, *assign;
    int8_t *hq;           // [T*k][F]
    BlockScale *hds;      // [T*k][F/32]
    float *o;             // [T*k][H]
    unsigned *counters;   // [H / rows per down item], zero between launches
    const float *w;       // [T][k]
    float *y;             // [T][H]
    int8_t *xq_out;       // fused path: [T][H] copy of the quantized x
    BlockScale *xds_out;  // fused path: [T][H/32]
    int fmt;              // weight format of the mat-vec kernels (kFmtQ4 / kFmtQ8)
    const int32_t *idx;   // [T][k] global expert ids (the combine skips experts of other shards)
    int e_base;           // first expert of this shard (local id = global id - e_base)
};

// Fused small-batch layer (cooperative launch).
struct FusedParams {
    GemvParams g;
    const float *x;          // [T][H]
    const int32_t *idx;      // [T][k] (when logits is null)
    const float *logits;     // [T][n_route]: route in-kernel (top-k + softmax) when not null
    int n_route;             // experts of the whole layer (logit columns; global id range)
    int32_t *idx_out;        // routed: [T][k] written by CTA 0
    float *w_out;            // routed: [T][k] written by CTA 0
    int renorm;
    int pdl;                 // launched with programmatic stream serialization
    unsigned *done_gu;       // [E]: published gate/up row blocks per expert (row-block mode: per
                             // used-expert index), zero between launches
    unsigned *exit_count;    // [1]
    int *error;
    // Row-block down mode (rb_rows > 0): a down item is rb_rows rows of H for
    // every used expert, so it sums y itself; done_gu is then indexed by the
    // used-expert index.  pre_off: shared-memory offset of the down prefetch
    // area.
    int rb_rows;
    int pre_off;
    // One routed token in row-block mode (fused_t1_ok): shared-memory offset
    // of the layer's gate, up and down table rows (0: the general prologue).
    int tbl_off;
    // 1: the last assignment of the token is the layer's shared expert (table
    // column E - 1 of the launch's rows, weight 1), which the single-token
    // path starts at kernel entry; 0: routed experts only
    int n_shared;
    // Lookahead (one routed token, early-start path): predict the next
    // layer's picks as the top-k of pr_b + pr_w . x and prefetch their
    // pool-resident weights into L2 (pr_w null: off).
    const __nv_bfloat16 *pr_w;    // [E][H] router of the next layer
    const float *pr_b;            // [E] its bias
    const uint64_t *pr_tbl;       // [3][E] the next layer's gate, up and down table rows
    float *pr_z;                  // [E] scratch: predicted logits
    unsigned *pr_count;           // [1] predicted logits written (zero between launches)
    unsigned *pr_flag;            // [1] the prediction is out (zero between launches)
    int32_t *pr_set;              // [k] this launch's prediction for the next layer
    const int32_t *pr_mine;       // [k] the previous layer's prediction for this one (or null)
    unsigned long long *pr_stats; // [2] predicted picks, of them actually picked
    size_t pr_blob;               // bytes of one expert tensor blob
};

// One grouped GEMM launch (gate/up with SwiGLU + h quantization, or down).
struct GemmParams {
    const int32_t *n_uniq, *uniq_e, *uniq_off, *tile_off, *assign;
    const uint2 *tile_rec;      // per tile: (u | row tile << 16, token tile | valid columns << 16)
    const uint64_t *tbl[2];     // expert tables of the A operands (gate, up) or (down, -)
    const float *a_scaleT;      // [K/32][A_pad]: block scales of the sorted activation rows
    int rows, K;                // weight rows (output features) and reduction length
    int A, A_pad, k, F_out;
    __half *hq16;               // gate/up: [A_pad][F] sorted h codes as fp16
    float *hdT;                 // gate/up: [F/32][A_pad] sorted h scales
    int8_t *hq;                 // gate/up: [A][F] h codes by assignment
    BlockScale *hds;            // gate/up: [A][F/32] by assignment
    float *o;                   // down: [A][H] by assignment
    int *error;                 // bit set when a bounded wait expires
};

struct TilingParams {
    CacheView cv;
    const int32_t *n_uniq, *uniq_e, *uniq_off;
    int32_t *tile_off_gu, *tile_off_dn;
    uint2 *rec_gu, *rec_dn;
    int cap_gu, cap_dn;
    int tid0, n_tokens, rt_gu, bn_gu, rt_dn, bn_dn;
};

struct PrefillLaunch {
    TilingParams tiling;
    GemmParams gu, dn;
    CUtensorMap tm_x, tm_h;     // sorted fp16 activations / h codes, 128-B swizzle
    const int8_t *xq;
    const BlockScale *xds;
    __half *xs16;
    float *xdT;
    const float *w;
    float *y;
    int T, k, H, n_sm;
    const int32_t *idx;         // [T][k] global expert ids (the combine skips other shards' experts)
    int e_base, E;              // this shard's experts: global ids [e_base, e_base + E)
};

// Staging of a prefill layer's cold expert tensors into lent pool slots.
struct StageParams {
    const uint64_t *tbl;      // [n_tensors][E]
    uint64_t *etbl;           // [3][E]: effective table rows of the layer
    const int32_t *n_uniq, *uniq_e;
    uint64_t *jobs;           // [2 * n_slots]: (source, destination) per staged blob
    int *n_jobs;
    uint64_t slot_base, slot_stride;
    int n_slots, tid0, E;
};

// One table / slot / stamp write of the promotion pass.
struct Update {
    uint32_t what;   // 0: tbl[index] = value; 1: slot[index] = value; 2: stamps[index] = value
    uint32_t index;
    uint64_t value;
};

int launch_topk(const float *logits, int T, int E, int k, int renorm, int32_t *idx, float *w, cudaStream_t st);
int launch_quantize(const float *x, int n_blocks, int8_t *q, BlockScale *ds, int n_sm, cudaStream_t st);
int launch_plan(const PlanParams &p, cudaStream_t st);
int launch_gemv(const GemvParams &p, int grid_gu, int grid_dn, cudaStream_t st, cudaEvent_t const *ev = nullptr);
int down_rows_per_item(int F);
int launch_block_dots(const uint8_t *blob, int fmt, int rows, int nb, int row0, int n_rows, const int8_t *qa,
                      int32_t *out, cudaStream_t st);
int launch_stream_read(const void *src, size_t bytes, uint32_t *sink, int n_sm, cudaStream_t st);
size_t fused_smem_bytes(int H, int F);
int fused_configure(int F, size_t smem, int *blocks_per_sm);
int fused_rb_rows(int H, int F, int T, int k, int E);
size_t fused_rb_smem(int H, int F, int T, int k, int E, int rows, int *pre_off);
bool fused_t1_ok(int E, int k);
int fused_configure_rb(int F, size_t smem, int *blocks_per_sm);
int fused_configure_t1_fmt(int F, int fmt, size_t smem, int *blocks_per_sm);
int launch_fused(const FusedParams &p, int grid, size_t smem, cudaStream_t st, cudaEvent_t const *ev);
int launch_prefill(const PrefillLaunch &L, cudaStream_t st, cudaEvent_t const *ev = nullptr);
int launch_stage(const StageParams &p, size_t blob_bytes, int n_sm, cudaStream_t st);
int launch_prefetch_table(const uint64_t *tbl_rows, const int32_t *map, const void *buf, int cap, size_t stride,
                          int E, uint64_t *etbl, cudaStream_t st);
int gemm_configure();
int gemm_bn(bool dual);
int gemm_rows_per_tile(bool dual);
int launch_step_finish(const Update *u, int n, uint64_t *tbl, int32_t *slot, uint32_t *stamps, uint32_t *clock,
                       uint32_t new_clock, uint32_t *clear_a, int n_a, uint32_t *clear_b, int n_b, cudaStream_t st);
int launch_count_assign(const int32_t *idx, int n, int E, int e_base, uint32_t *cnt, cudaStream_t st);
int launch_busy(unsigned long long ns, cudaStream_t st);
int launch_shared_assign(const int32_t *idx, const float *w, int T, int k, int e_shared, int32_t *idx_a, float *w_a,
                         int *error, cudaStream_t st);

}  // namespace moe
