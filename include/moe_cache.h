/*
 * moe_cache.h -- C ABI of the GB300 routed-expert MoE feed-forward with a
 * quantized HBM expert cache.
 *
 * Every entry point returns an int status (MOE_OK = 0, negative = error;
 * moe_last_error() gives a message) unless stated otherwise.  No C++
 * exception crosses this boundary.  A context is not thread-safe: calls on
 * one context must not overlap.  Device pointers are CUDA device addresses
 * (or unified addresses) on the context's device; host pointers are plain
 * process memory.  Streams are cudaStream_t passed as void*; in route_topk
 * and moe_ffn_forward NULL means the context's stream.
 *
 * Data formats
 *   Q4 block (canonical, 18 bytes): binary16 scale d (little endian), then
 *   16 code bytes; byte j holds element j (low nibble) and element j+16
 *   (high nibble); weight = d * (q - 8), q in 0..15.
 *   Expert tensor (canonical): [n_experts][rows][cols/32] Q4 blocks,
 *   expert-major.  gate and up have rows = ffn, cols = hidden; down has
 *   rows = hidden, cols = ffn.  Tensor id = layer * 3 + kind.
 *   Miss key: (tensor_id << 12) | expert (uint32).
 *
 * Sources (page titles and sections): Zapdev-labs/a6000-custom-kernels (the
 * pointer-table GEMV diagram and the paragraphs after it: per-tensor d_tbl
 * with an LSB tag, the HBM pool, zero-copy reads of pinned host memory, the
 * miss recorder, stamps and the promotion pass between graphs);
 * neurall/llama.cpp, "How it works" (an expert is admitted after a second
 * miss inside a 64-token window; expert blocks borrowed by the prompt pass and returned);
 * mx-llama.cpp FEATURES.md (q8_1 activation quantization reused across the
 * matmuls of one input; planes of quants and scales); mihailescu2m/llama.cpp
 * (MUL_MAT_ID over used tiles only; top-k of 512 scores).
 */
#ifndef MOE_CACHE_H
#define MOE_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_ARG (-1)        /* an argument is out of range or inconsistent */
#define MOE_ERR_OOM (-2)        /* a device or pinned host allocation failed */
#define MOE_ERR_CUDA (-3)       /* a CUDA runtime call failed */
#define MOE_ERR_NOT_PINNED (-4) /* host memory that must be pinned is not */
#define MOE_ERR_TIMEOUT (-5)    /* a host-side poll limit was exceeded */
#define MOE_ERR_CAPACITY (-6)   /* an output buffer is too small */
#define MOE_ERR_STATE (-7)      /* call not valid in the current state */
#define MOE_ERR_FAULT (-8)      /* a kernel reported a fault (expert id out of range, expired bounded
                                   wait), or an injected (test) upload failure */

#define MOE_KIND_GATE 0
#define MOE_KIND_UP 1
#define MOE_KIND_DOWN 2

typedef struct moe_ctx moe_ctx;

/* Configuration of one context (one model's routed-expert FFN stack). */
typedef struct moe_cfg {
    int32_t hidden;             /* H: model width, multiple of 32 */
    int32_t ffn;                /* F: expert FFN width, multiple of 32 */
    int32_t n_experts;          /* E: experts per layer, 1..4096 (12-bit key) */
    int32_t top_k;              /* k: experts per token, 1..32, <= E */
    int32_t n_layers;           /* L: MoE layers; 3*L expert tensors */
    int32_t slots_per_tensor;   /* HBM pool slots reserved per expert tensor */
    int32_t max_tokens;         /* largest n_tokens of one forward */
    int32_t window_tokens;      /* admission window (tokens), e.g. 64 */
    int32_t max_swaps_per_step; /* admissions per cache_step, 0 = no limit */
    int32_t renorm_topk;        /* 1: weights = softmax over the k selected */
    int32_t poll_timeout_ms;    /* host poll limit in cache_step (0 = 10 s) */
    int32_t device;             /* CUDA device ordinal */
    int32_t weight_format;      /* MOE_FMT_Q4_0 (0), _Q8_0 (1), _Q5_0 (2), _Q4_K (3), _Q6_K (4) or _Q5_K (5) */
    int32_t shared_experts;     /* 1: every layer has one shared expert (register_shared_expert), E <= 4095 */
} moe_cfg;

/* Expert weight formats (blocks of 32 weights, one binary16 scale d each).
 * Q4_0: 18-byte blocks, d then 16 code bytes (byte j = element j in the low
 *   nibble, element j+16 in the high nibble), w = d * (q - 8).
 * Q8_0: 34-byte blocks, d then 32 signed code bytes in element order,
 *   w = d * q (one of the other block formats the dot kernels of
 *   Zapdev-labs/a6000-custom-kernels accept; the byte layout is the plain
 *   reading: scale, then codes in element order).
 * Q5_0: 22-byte blocks, d, then 4 bytes whose little-endian word holds bit 4
 *   of element j in bit j, then 16 nibble bytes in the Q4 order;
 *   w = d * (q - 16) with q in 0..31 (another of those formats; same reading
 *   of the layout).
 * Q4_K: super-blocks of 256 weights (8 sub-blocks of 32), 144 bytes: d, dmin
 *   (binary16), 12 bytes of 6-bit sub-block scales sc_j and mins m_j (j < 4:
 *   sc = b[j] & 63, m = b[j+4] & 63; j >= 4: sc = (b[j+4] & 15) |
 *   (b[j-4] >> 6) << 4, m = (b[j+4] >> 4) | (b[j] >> 6) << 4), 128 code bytes
 *   (chunk c of 32: sub-block 2c in the low nibbles, 2c+1 in the high);
 *   w = d * sc_j * q - dmin * m_j (a K-quant format of those kernels; same
 *   reading of the layout).  Needs hidden and ffn multiples of 256.
 * Q6_K: super-blocks of 256 weights (16 sub-blocks of 16), 210 bytes in the
 *   layout the format is published with: 128 bytes ql, 64 bytes qh, 16
 *   signed 8-bit scales sc_j, binary16 d; in 128-weight half n, element
 *   32m + l (m = 0..3) has its low 4 bits in ql[64n + 32(m & 1) + l] (low
 *   nibble for m < 2, high for m >= 2) and its high 2 bits in bits 2m..2m+1
 *   of qh[32n + l]; w = d * sc_j * (q - 32), j = element / 16 (another
 *   K-quant of those kernels; the pages print no layout).  Needs hidden and
 *   ffn multiples of 256.
 * Q5_K: super-blocks of 256 weights (8 sub-blocks of 32), 176 bytes in the
 *   published layout: d, dmin (binary16), the 12 packed 6-bit scale/min
 *   bytes as in Q4_K, 32 bytes qh (bit j of qh[l] = bit 4 of element l of
 *   sub-block j), then 128 code bytes in the Q4_K order (low four bits);
 *   w = d * sc_j * q - dmin * m_j, q in 0..31.  Needs hidden and ffn
 *   multiples of 256.
 * Q8_0, Q5_0, Q4_K, Q6_K and Q5_K contexts run batch-1 routed forwards
 * through the single-launch layer and every other forward through the
 * mat-vec kernels (no tensor-core prompt path, no lookahead). */
#define MOE_FMT_Q4_0 0
#define MOE_FMT_Q8_0 1
#define MOE_FMT_Q5_0 2
#define MOE_FMT_Q4_K 3
#define MOE_FMT_Q6_K 4
#define MOE_FMT_Q5_K 5

typedef struct moe_stats_t {
    uint64_t steps;        /* cache_step calls */
    uint64_t hits;         /* (tensor, expert) reads served by the pool */
    uint64_t misses;       /* (tensor, expert) reads served from host memory */
    uint64_t admissions;   /* experts uploaded into the pool */
    uint64_t evictions;    /* experts removed from the pool */
    uint64_t upload_bytes; /* bytes copied host -> pool by cache_step / return */
    uint64_t cold_bytes;   /* weight bytes the kernels read zero-copy */
    uint64_t clock;        /* token clock */
    uint64_t lookahead_predicted; /* decode lookahead: picks predicted a layer ahead */
    uint64_t lookahead_hits;      /* ... of them actually picked by that layer */
} moe_stats_t;

/*
 * Create a context on cfg->device (the per-tensor tables, HBM pools, stamps
 * and miss buffer of Zapdev-labs/a6000-custom-kernels, after the
 * pointer-table diagram, sized by the caller).  cuda_stream (cudaStream_t; NULL is the
 * legacy default stream, as everywhere in CUDA) is the stream every forward
 * of this context runs on; the caller keeps owning it.  The library allocates and owns: the HBM
 * expert pool (3*L*slots_per_tensor slots of one expert tensor's plane blob:
 * 18, 34, 22, 24, 26.25 or 28 bytes per 32 weights for Q4_0, Q8_0, Q5_0,
 * Q4_K, Q6_K or Q5_K, rounded up to 256 bytes), the
 * pointer tables, stamps, miss log, workspaces, an upload stream and the
 * pinned host copies of registered tensors.  *out receives the context.
 * Errors: MOE_ERR_ARG (sizes), MOE_ERR_OOM, MOE_ERR_CUDA.
 */
int moe_layer_init(const moe_cfg *cfg, void *cuda_stream, moe_ctx **out);

/*
 * Register one expert tensor (layer, kind) and seed its pool
 * (Zapdev-labs/a6000-custom-kernels, after the pointer-table diagram: every
 * expert tensor has its own table, pool and stamps, and pools are seeded at
 * registration from a routing-frequency table).
 * host_q4: canonical tensor [n_experts][rows][cols/32][18 B] (Q4_0),
 *   [...][34 B] (Q8_0), [...][22 B] (Q5_0), or [n_experts][rows][cols/256]
 *   super-blocks of 144 B (Q4_K), 210 B (Q6_K) or 176 B (Q5_K), per
 *   cfg.weight_format, any host
 *   memory; the library copies it into its own pinned, device-mapped host
 *   memory in plane layout (all codes, then all scales) and never reads
 *   host_q4 again, so the caller may free it on return.
 * capacity: pool slots of this tensor (<= slots_per_tensor).
 * seed_order: n_experts distinct expert ids, most frequently routed first
 *   (a routing-frequency table); the first n_seed (<= capacity) are
 *   uploaded to slots 0..n_seed-1 (stamp 0).  NULL means 0,1,2,...
 * Every other expert's table entry points at its pinned host copy with the
 * low bit set.  *tensor_id (may be NULL) receives layer*3 + kind.
 * Blocking (returns after the seed uploads finished).
 * Errors: MOE_ERR_ARG (shape, cols % 32, ids out of range or repeated,
 * already registered), MOE_ERR_OOM, MOE_ERR_CUDA.
 */
int register_expert_tensor(moe_ctx *ctx, int layer, int kind, const void *host_q4, int rows, int cols,
                           int capacity, const int32_t *seed_order, int n_seed, int *tensor_id);

/*
 * Register the shared expert of (layer, kind) (the shared-expert block among
 * the fusion arguments of the dot kernels, Zapdev-labs/a6000-custom-kernels):
 * one expert that every token runs next to its routed ones, with weight 1:
 * y[t] = sum_j w[t,j] o[t,j] + o_shared[t].  Needs cfg.shared_experts = 1;
 * then every layer needs its three shared tensors before its first forward.
 * host_w: one canonical expert [rows][cols/32][block bytes] in the context's
 * weight format, copied (the caller may free it).  The shared expert lives
 * in its own HBM allocation, never cold and never in the pool: its table
 * entry is column E of the tensor's row, so it runs inside the same gate/up,
 * down (and, for prompts, grouped GEMM) launches as the routed experts, as
 * assignment k of every token.  Shared-expert contexts run batch-1 routed
 * forwards through the single-launch layer (the shared expert is its last
 * pick, started at kernel entry) and other small batches through the
 * mat-vec kernels.  Synchronous.
 * Errors: MOE_ERR_STATE (no shared experts in cfg), MOE_ERR_ARG (shape,
 * already registered), MOE_ERR_OOM, MOE_ERR_CUDA.
 */
int register_shared_expert(moe_ctx *ctx, int layer, int kind, const void *host_w, int rows, int cols);

/*
 * Router top-k (mihailescu2m/llama.cpp, "the graph-shape problem": only the
 * top entries of the 512 scores are needed).  d_logits: fp32 [n_tokens][E]
 * device, row-major.  d_idx: int32 [n_tokens][k] device, the k largest
 * logits per token ordered by (logit desc, expert asc): ties go to the
 * lower index.  d_w: fp32 [n_tokens][k] device, the routing weights
 * (softmax over the k selected logits if cfg.renorm_topk, else softmax over
 * all E, read at the selected experts).  NaN logits give unspecified
 * choices.  Asynchronous on `stream`; caller-owned buffers.
 * Errors: MOE_ERR_ARG.
 */
int route_topk(moe_ctx *ctx, const float *d_logits, int n_tokens, int n_experts, int k, int32_t *d_idx,
               float *d_w, void *stream);

/*
 * One routed-expert FFN layer (Zapdev-labs/a6000-custom-kernels: the
 * pointer-table mat-vec, MUL_MAT_ID): for each token t and each j < k,
 * expert e = d_idx[t][j] computes h = silu(gate_e . x_t) * (up_e . x_t)
 * from int8-quantized x (blocks of 32, binary16 scale), quantizes h the
 * same way, computes o = down_e . h, and y[t] = sum_j d_w[t][j] * o.
 * Block dots are exact int32 sums of (q_w - 8) * q_a (Q4_0; the other
 * formats' codes and offsets as defined above); each block is scaled by
 * d_w * d_a in fp32 (K-quants: by their sub-block scales and mins).  Each expert's weights are read through the
 * tensor's pointer table: pool slot (tag 0, HBM) or pinned host memory
 * (tag 1, read zero-copy).  Cold reads are logged once per (tensor,
 * expert) in the miss log; pool hits write the step's clock into the
 * slot's stamp.  n_tokens <= 32 runs the mat-vec kernels; larger batches
 * run the grouped per-expert GEMM over tokens sorted by expert (Q4_0
 * contexts with hidden and ffn multiples of 64; other contexts run the
 * mat-vec kernels at every size).
 * d_x: fp32 [n_tokens][H] device; d_idx/d_w as produced by route_topk;
 * d_y: fp32 [n_tokens][H] device, written.  `stream` must be the
 * context's stream (or NULL).  Asynchronous; capturable in a CUDA graph
 * for a fixed n_tokens.  Errors: MOE_ERR_ARG, MOE_ERR_STATE (tensors of
 * the layer not registered).
 */
int moe_ffn_forward(moe_ctx *ctx, int layer, const float *d_x, int n_tokens, const int32_t *d_idx,
                    const float *d_w, float *d_y, void *stream);

/*
 * route_topk followed by moe_ffn_forward, as one call (the top-k of
 * mihailescu2m/llama.cpp and the pointer-table mat-vec of
 * Zapdev-labs/a6000-custom-kernels, as in those two calls): same results (d_idx
 * and d_w are written as route_topk writes them), and for small batches
 * (n_tokens <= 32, n_tokens*k <= 256) one kernel launch in which every CTA
 * routes the tokens itself.  d_logits: fp32 [n_tokens][E] device.
 * Asynchronous; `stream` as in moe_ffn_forward.  Errors: as the two calls.
 */
int moe_ffn_forward_routed(moe_ctx *ctx, int layer, const float *d_x, const float *d_logits, int n_tokens,
                           int32_t *d_idx, float *d_w, float *d_y, void *stream);

/*
 * Expert shard (neurall/llama.cpp README, "More GPUs": every GPU keeps its
 * own expert cache in its own memory; the pages do not say how experts are
 * split, and this library's reading is expert parallelism: GPU r holds a
 * contiguous range of every layer's experts, so the GPUs cache disjoint
 * experts).  After this call the context holds experts
 * [expert_base, expert_base + n_experts) of layers with n_route experts:
 * its tensors are registered with those n_experts experts only (local id =
 * global id - expert_base, which is also the expert field of its miss keys
 * and the index of its tables and seed orders); route_topk and the routed
 * forward take n_route logits per token and write global ids; every forward
 * takes global ids in [0, n_route) and leaves out the assignments whose
 * expert is outside the range: it reads, logs, stamps and counts nothing for
 * them, and y[t] = sum over this range's j of d_w[t][j] * o (0 when none),
 * the rank's partial sum; the sum over every shard is the layer's output.
 * (0, n_experts) is the unsharded default.  Not with shared_experts.
 * Errors: MOE_ERR_ARG (range), MOE_ERR_STATE (shared experts).
 */
int moe_set_expert_shard(moe_ctx *ctx, int expert_base, int n_route);

/*
 * Dispatched rows of an expert shard (neurall/llama.cpp README, "More GPUs";
 * see moe_set_expert_shard): moe_ffn_forward over n_rows token rows that are part of a step of
 * step_tokens tokens (step_tokens >= n_rows): an expert-parallel rank that
 * receives only the rows routed to its experts stamps its pool hits with the
 * clock of the whole step (clock + step_tokens), as a rank that saw every
 * token would, and the caller passes step_tokens to cache_step.  Otherwise
 * as moe_ffn_forward.  Errors: as moe_ffn_forward, and MOE_ERR_ARG when
 * n_rows < 0 or step_tokens < max(n_rows, 1).
 */
int moe_ffn_forward_rows(moe_ctx *ctx, int layer, const float *d_x, int n_rows, const int32_t *d_idx,
                         const float *d_w, float *d_y, int step_tokens, void *stream);

/*
 * Promotion pass between steps (Zapdev-labs/a6000-custom-kernels:
 * ggml_cuda_moe_cache_step between graphs, never captured; neurall/llama.cpp:
 * admission on a second miss inside a 64-token window).  Waits (host
 * poll, bounded by cfg.poll_timeout_ms) for the forwards issued so far,
 * advances the clock by n_tokens, reads the miss log and the stamps, and
 * for each miss in ascending key order: admits the expert when its previous
 * sighting is less than window_tokens old, into the lowest free slot or
 * else the slot with the smallest stamp older than this step (ties: lowest
 * slot), otherwise records the sighting.  Per-tensor pools (the default)
 * search the missing tensor's own slots; a shared pool (moe_set_global_pool)
 * searches every pool slot of the arena, whichever layer's expert it holds.
 * Uploads run on the context's
 * upload stream; the context stream waits for them before its next forward.
 * While pool slots are borrowed, nothing is admitted.  The miss log is
 * cleared.  Errors: MOE_ERR_TIMEOUT (nothing changed; retry), MOE_ERR_CUDA,
 * MOE_ERR_FAULT: an injected upload failure (moe_debug_fail_upload), or a
 * kernel reported a device error since the last step or drain (bit 0: an
 * expert id outside [0, n_experts) was read as expert 0; other bits: a
 * bounded wait expired and its work item was skipped) -- the step's cache
 * update is done, the affected forwards' outputs are not valid, and the
 * error word is cleared (moe_last_error names the bits).
 */
int cache_step(moe_ctx *ctx, int n_tokens);

/*
 * Copy the miss keys logged since the last cache_step (or drain) to
 * host_out, sorted ascending, unique, and clear the log (the miss recorder
 * of Zapdev-labs/a6000-custom-kernels, after the pointer-table diagram:
 * (tensor_id << 12 | expert) keys in a device buffer).  *n_out gets the
 * count even when cap is too small (then MOE_ERR_CAPACITY and the log is
 * kept).  Synchronizes with the context stream.  MOE_ERR_FAULT (after the
 * keys are out and the log is cleared): a device error was reported, as for
 * cache_step.  n_out may be NULL.  Errors: MOE_ERR_ARG (NULL host_out when
 * there are keys to copy), MOE_ERR_CAPACITY, MOE_ERR_FAULT, MOE_ERR_CUDA.
 */
int miss_drain(moe_ctx *ctx, uint32_t *host_out, size_t cap, size_t *n_out);

/*
 * Lend n_slots pool slots to a prefill pass (neurall/llama.cpp, "How it
 * works": the large micro-batch workspace exists only during a prompt pass).
 * Global slot g is local slot g / (3L) of tensor g % (3L); the n highest
 * global slots are taken, their experts evicted (table entries back to
 * host).  *d_ws gets the device address of the contiguous lent region and
 * *bytes its size.  Synchronous.  Errors: MOE_ERR_ARG, MOE_ERR_STATE
 * (already borrowed).
 */
int moe_pool_borrow(moe_ctx *ctx, int n_slots, void **d_ws, size_t *bytes);

/*
 * Give the lent slots back (neurall/llama.cpp, "How it works": when the
 * prompt pass ends its space goes back to the expert cache, refilled with
 * the hot experts and, with prefill preheat, the ones the pass used): each
 * returned pool slot, in ascending global
 * order, is refilled (stamp = clock) with the best non-resident expert, by
 * (use count of the prompt pass, descending; rank in its tensor's seed
 * order, ascending; tensor id, ascending).  Per-tensor pools take the slot's
 * own tensor's experts, a shared pool every tensor's.  Without preheat every
 * use count is 0: the refill follows seed order (the learned hot experts).
 * Synchronous.  Errors: MOE_ERR_STATE.
 */
int moe_pool_return(moe_ctx *ctx);

/*
 * Upload overlap (eager forwards; no counterpart on the source pages, an
 * ordering refinement of the promotion pass's uploads).  By default the promotion pass makes the
 * context stream wait for all of its pool uploads before the next forward.
 * With enable = 1 it records one event per layer after that layer's uploads
 * instead, and a layer's next forward waits only for its own layer's event,
 * so the first layers of the next step run while later layers' experts are
 * still being uploaded.  Results, cache state and statistics are the same
 * (a layer's kernels read only its own tables; an evicted expert's entry
 * already points at its host copy).  Forwards must then be issued outside
 * stream capture (a captured graph could not wait on the per-step events):
 * a pending wait inside a capture fails with MOE_ERR_STATE, and a graph
 * captured earlier must not be replayed while the overlap is on (its
 * launches would not wait for the uploads).  Off by default.  Synchronous.
 * Errors: MOE_ERR_CUDA.
 */
int moe_set_upload_overlap(moe_ctx *ctx, int enable);

/*
 * One pool of expert blocks for all layers (neurall/llama.cpp, "How it
 * works", Expert cache: the per-layer reserve gave way to one pool that every
 * layer draws on; features table, global expert pool row).  With enable = 1
 * the arena's slots of every registered tensor (its capacity's worth, at
 * global slots s * 3L + tensor_id, s < capacity) form one pool: seeding is
 * unchanged, but an admission takes the lowest free pool slot of the whole
 * arena, else the pool slot with the oldest stamp below the clock (ties:
 * lowest global slot), evicting whichever layer's expert holds it.  Tensors
 * registered with capacity 0 still receive slots.  The promotion pass then
 * reads all 3L x slots_per_tensor stamps when it admits.  Call before the
 * first register_expert_tensor.  Errors: MOE_ERR_STATE (a tensor is already
 * registered).
 */
int moe_set_global_pool(moe_ctx *ctx, int enable);

/*
 * Prefill preheat (neurall/llama.cpp, "How it works": blocks lent to a
 * prompt pass come back holding the model's hot experts and the experts the
 * pass itself needed; features table, prefill preheat row).  With
 * enable = 1, every forward issued while slots are lent also adds its
 * (token, expert) assignments to per-(layer, expert) use counts (one small
 * kernel after the layer, on the context stream); moe_pool_return ranks the
 * refill by them and clears them.  Allocates 4 x L x E bytes of device
 * memory on first use.  Errors: MOE_ERR_STATE (slots are lent), MOE_ERR_CUDA.
 */
int moe_set_preheat(moe_ctx *ctx, int enable);

/*
 * Put the cache back in its registered state (no counterpart on the source
 * pages: lets measurements start from the same seeded state), with a pool mode chosen anew
 * (global_pool = 1: one pool for all layers, as moe_set_global_pool; 0: a
 * pool per tensor).  Every tensor holds its seeded experts again (seed order
 * in local slots 0..n_seed-1; slots already holding their seed expert are
 * not uploaded again), stamps, sightings, clock, miss log and preheat counts
 * are cleared, statistics restart from zero (upload_bytes keeps counting),
 * and lookahead buffers are marked empty.  Lets runs that must start from
 * the same state (a per-tensor and a shared pool, say) share one
 * registration and its pinned host copies.  Synchronous.  Errors:
 * MOE_ERR_STATE (slots are lent), MOE_ERR_CUDA.
 */
int moe_cache_reset(moe_ctx *ctx, int global_pool);

/*
 * Owner and stamp of every arena slot (inspection, for tests of the shared
 * pool of neurall/llama.cpp, "How it works"; 3L x slots_per_tensor entries,
 * global slot g = local slot g / 3L of tensor g % 3L), either pool mode;
 * synchronizes with all streams.  owner_key: (tensor_id << 12 | expert), or
 * -1 for a free, lent or unused slot; stamps: the device stamp of the slot.
 * Either output may be NULL; host arrays of 3L x slots_per_tensor entries.
 * Errors: MOE_ERR_ARG (NULL context), MOE_ERR_CUDA.
 */
int moe_pool_snapshot(moe_ctx *ctx, int32_t *owner_key, uint32_t *stamps);

/*
 * Lookahead prefetch (mihailescu2m/llama.cpp, Metal streaming notes: expert
 * reads for the next layer start a layer early).  Decode: see moe_set_router
 * (needs the routers; enabling succeeds without a prompt-pass path then).
 * Prompt passes: with enable = 1, every forward of more than 32 tokens for layer l also
 * enqueues, on the context's upload stream, copy-engine uploads of the
 * expert tensors of layer (l + 1) mod L that are cold at that moment into
 * one of two device prefetch buffers; the prompt forward of that layer then
 * reads those experts from the buffer instead of zero-copy host memory.  A
 * prompt micro-batch of thousands of tokens uses every expert of a layer, so
 * the predicted set is the layer's whole cold set.  The effective table is
 * rebuilt from the live table when the layer runs: an expert admitted in the
 * meantime is read from its pool slot, one evicted in the meantime from host
 * memory.  Cache state, miss log, stamps and results are the same as without
 * prefetch.  Enable after every tensor is registered: the buffers (2 x 3 x
 * (the largest cold count of a tensor) x tensor slot bytes of device memory)
 * are sized then.  enable = 0 stops issuing prefetches (buffers are kept).
 * Errors: MOE_ERR_STATE (a layer not registered), MOE_ERR_CUDA (allocation).
 */
int moe_set_lookahead(moe_ctx *ctx, int enable);

/*
 * Router of one layer, for decode lookahead (mihailescu2m/llama.cpp, MoE
 * expert streaming, lookahead prefetch: layer L+1's router predicts its
 * experts from layer L's input, so their reads start a layer early).
 * host_w: fp32 [n_experts][hidden] (stored as bf16), host_b: fp32
 * [n_experts] or NULL (zeros); the layer's logits are modelled as
 * b + W x.  With lookahead on (moe_set_lookahead) and the router of layer
 * l + 1 set, every batch-1 routed forward of layer l (the single-launch
 * layer kernel, Q4 weights, no shared expert) also computes b + W x_l for
 * layer l + 1 from its own input x_l, takes the top-k as the prediction and
 * prefetches the predicted experts' pool-resident gate, up and down blobs
 * into L2 (host-resident experts are not prefetched).  Outputs, cache state
 * and statistics other than the two lookahead counters of moe_stats are the
 * same as without it.  Allocates (on the first call) L x E x H x 2 bytes for
 * the routers plus small buffers.  Synchronous.  Errors: MOE_ERR_ARG,
 * MOE_ERR_OOM, MOE_ERR_CUDA.
 */
int moe_set_router(moe_ctx *ctx, int layer, const float *host_w, const float *host_b);

/*
 * Snapshot of one tensor's cache state (inspection for tests: the table,
 * slots and stamps of Zapdev-labs/a6000-custom-kernels' pointer-table cache;
 * synchronizes with all streams).
 * Any output may be NULL.  tbl: uint64 [E], the device pointer table as the
 * kernels read it; slot_of: int32 [E] (-1 = cold; the local slot, or the
 * global slot with a shared pool); last_seen: int32 [E] (-1 = no sighting);
 * owner: int32 [slots_per_tensor] (-1 = free or lent; with a shared pool,
 * the expert of this tensor held in its home slot s * 3L + tensor_id, -1 if
 * another tensor's or free); stamps: uint32 [slots_per_tensor] (device stamp
 * of each of those slots).  All host arrays.  Errors: MOE_ERR_ARG (NULL
 * context, tensor_id out of range or not registered), MOE_ERR_CUDA.
 */
int moe_cache_snapshot(moe_ctx *ctx, int tensor_id, uint64_t *tbl, int32_t *slot_of, int32_t *last_seen,
                       int32_t *owner, uint32_t *stamps);

/* Base addresses used by table entries (inspection for tests; the pool and
 * host copies the pointer tables of Zapdev-labs/a6000-custom-kernels point
 * into): the pool and the pinned host copy of one tensor (expert e of the
 * tensor lives at host_base + e * slot_bytes, once the tensor is
 * registered); *n_tensors = 3L.  Any output may be NULL.  Errors:
 * MOE_ERR_ARG (NULL context, tensor_id out of range). */
int moe_cache_layout(moe_ctx *ctx, int tensor_id, uint64_t *pool_base, uint64_t *host_base,
                     uint64_t *slot_bytes, int32_t *n_tensors);

/* Counters since init (moe_cache_reset restarts all but upload_bytes; the
 * pages report cache hit rates: neurall/llama.cpp, features table): see
 * moe_stats_t.  Synchronizes with the context stream when decode lookahead
 * is set up (its two counters live on the device).  Errors: MOE_ERR_ARG
 * (NULL context or out), MOE_ERR_CUDA. */
int moe_stats(moe_ctx *ctx, moe_stats_t *out);

/* (No counterpart on the source pages.)  Message of the last error on ctx
 * (or, when ctx is NULL, of the last failed
 * call that takes no context or was given a NULL one: moe_layer_init,
 * moe_probe_host_read, moe_expert_ffn_noalloc[_status]; kept per host
 * thread).  Valid until the next such call.  Never fails; "" when there was
 * none. */
const char *moe_last_error(moe_ctx *ctx);

/* Release everything the context owns (no counterpart on the source
 * pages).  Synchronizes first.  NULL is a no-op.  Returns nothing. */
void moe_destroy(moe_ctx *ctx);

/* ---- inspection and measurement hooks (tests, benchmark; no counterpart
 * on the source pages) ---------------------------------------------------- */

/*
 * Integer block dots of the mat-vec kernels' block-dot routine: out[r][b] =
 * sum_i (q_w,i - 8) * qa[b*32 + i] for rows row0..row0+n_rows-1 of expert
 * `expert` of tensor_id, read through the pointer table (pool or host).
 * d_qa: int8 [cols] device; d_out: int32 [n_rows][cols/32] device.
 * Synchronous.  Errors: MOE_ERR_ARG.
 */
int moe_debug_block_dots(moe_ctx *ctx, int tensor_id, int expert, int row0, int n_rows, const int8_t *d_qa,
                         int32_t *d_out);

/*
 * Copy a workspace of the most recent forward to host memory (synchronizes):
 * what = 0: quantized x codes int8 [n_tokens][H]; 1: x scales binary16
 * [n_tokens][H/32]; 2: quantized h codes int8 [n_tokens*k][F] (row
 * a = t*k + j); 3: h scales binary16 [n_tokens*k][F/32].  bytes must
 * equal the workspace size.  Errors: MOE_ERR_ARG, MOE_ERR_STATE.
 */
int moe_debug_read(moe_ctx *ctx, int what, void *host_out, size_t bytes);

/*
 * Zero-copy read bandwidth of pinned host memory: a kernel streams `bytes`
 * from host_pinned (device-mapped) with 128-bit loads, `iters` times; *gbs
 * receives the best GB/s.  Also measures cudaMemcpyAsync H2D into *copy_gbs
 * when non-NULL.  Synchronous.  host_pinned must come from cudaHostAlloc
 * (mapped) or be registered; else MOE_ERR_NOT_PINNED.
 */
int moe_probe_host_read(const void *host_pinned, size_t bytes, int iters, double *gbs, double *copy_gbs);

/*
 * Test hook: make the n-th following pool upload (1-based; 0 = off) report
 * failure; the step rolls that admission back (the expert stays cold, the
 * victim stays evicted) and returns MOE_ERR_FAULT after finishing the
 * step consistently.  Errors: MOE_ERR_ARG (NULL context, nth < 0).
 */
int moe_debug_fail_upload(moe_ctx *ctx, int nth);

/*
 * Failure-detection hook: enqueue on the context stream one kernel that
 * stays busy for `microseconds` (<= 2 s, measured on the device's global
 * timer) and then ends by itself.  A cache_step issued behind it with a
 * shorter cfg.poll_timeout_ms returns MOE_ERR_TIMEOUT without changing any
 * cache state; the context stays usable and the step can be retried.
 * Errors: MOE_ERR_ARG, MOE_ERR_CUDA.
 */
int moe_debug_busy(moe_ctx *ctx, int microseconds);

/*
 * Kernel timing (benchmark hook): when enabled, every forward records CUDA
 * events on the context stream around its gate/up and its down launches:
 * the mat-vec kernels (or the single-launch layer kernel, whose time is then
 * the gate/up figure) for small batches, the two grouped GEMM kernels for
 * prompt batches (also inside a captured graph).  moe_debug_timing_read
 * synchronizes and writes, per layer, the device time in ms of the most
 * recent gate/up and down launch of that layer since the last read (0 when
 * the layer ran no forward); both arrays hold n_layers doubles (host;
 * either may be NULL).  Errors: MOE_ERR_ARG (NULL context), MOE_ERR_CUDA.
 */
int moe_debug_timing(moe_ctx *ctx, int enable);
int moe_debug_timing_read(moe_ctx *ctx, double *gate_up_ms, double *down_ms);

/*
 * One routed-expert FFN layer that allocates nothing (no counterpart on the
 * source pages: this entry point exists for callers that cannot allocate
 * device memory when they run a layer, such as processes whose device memory
 * is entirely reserved by another allocator, or hosts that forbid device
 * allocation after start-up).  It computes what
 * moe_ffn_forward computes for a small batch, with the caller's expert tables
 * instead of a context: d_tbl holds 3 rows of n_experts uint64 entries
 * (gate, up, down), each the device address of one Q4_0 expert blob in the
 * plane layout the library uses (tag bit 0 clear), or of a device-mapped pinned
 * host copy with bit 0 set, as moe_cache_snapshot reports them.  d_x, d_idx,
 * d_w, d_y as in moe_ffn_forward; `stream` is any stream (NULL = legacy
 * default stream).  No miss log, stamp or clock is kept.
 * Every intermediate lives in one file-scope device array of 8 MiB held by
 * every GPU that loads the library until the process exits; a call needs
 * about T*k*(4*H + F + F/4) + T*(H + H/4) bytes plus small tables and is
 * rejected with MOE_ERR_CAPACITY (message in moe_last_error(NULL)) when that
 * exceeds 8 MiB.  Limits: n_tokens <= 32, n_tokens*top_k <= 256, hidden a
 * multiple of the down row block (64 for ffn/32 <= 40, else 32).  The first
 * call on a device looks up the array's device address and configures the
 * kernel; later calls on that device
 * (and shape) only clear the parts of the array that must start at zero and
 * launch one kernel.  All calls share the array and each leaves its contents
 * behind, so calls that overlap on the GPU (other streams, other host
 * threads) race.  The call returns before the kernel has run, so faults the
 * kernel detects (an expert id outside [0, n_experts), which it reads as
 * expert 0; a bounded wait that expired) are not in its return value: they
 * are left in the array's error word, which moe_expert_ffn_noalloc_status
 * reads.  Errors: MOE_ERR_ARG, MOE_ERR_CAPACITY, MOE_ERR_CUDA.
 */
int moe_expert_ffn_noalloc(const float *d_x, int n_tokens, const int32_t *d_idx, const float *d_w,
                           const uint64_t *d_tbl, int hidden, int ffn, int n_experts, int top_k, float *d_y,
                           void *stream);

/*
 * Device-side status of the most recent moe_expert_ffn_noalloc call on the
 * current device (no counterpart on the source pages; the companion of the
 * allocation-free entry point).  Waits for `stream` (the stream that call
 * used, NULL = legacy default stream), reads the kernel's error word from the
 * first bytes of the entry point's device array and returns MOE_OK when it is
 * zero, else MOE_ERR_FAULT with moe_last_error(NULL) naming the bits (1: an
 * expert id outside [0, n_experts) was read as expert 0; 2, 4: a bounded wait
 * expired and its work item was skipped; that call's output is then not
 * valid).  The word stays until the next call on the device clears it.
 * Allocates nothing.  MOE_OK when no call has run on the device yet.
 * Errors: MOE_ERR_FAULT, MOE_ERR_CUDA.
 */
int moe_expert_ffn_noalloc_status(void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_CACHE_H */
