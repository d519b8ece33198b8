// C-ABI runtime of the GB300 routed-expert FFN with a quantized HBM expert
// cache: context lifetime, registration (plane repack into pinned, device-
// mapped host memory and pool seeding), forward dispatch, the promotion pass
// between steps, the miss log, pool borrowing around a prefill pass, and the
// inspection hooks.  See moe_cache.h for the contract of each entry point.
//
// Sources: Zapdev-labs/a6000-custom-kernels (per-tensor d_tbl / pool / stamp
// array, LSB-tagged host entries, miss buffer, promotion pass between
// graphs, seeding from a routing-frequency file); neurall/llama.cpp, "How it
// works" (an expert is admitted once it has been missed twice inside a 64-token window; the prompt
// pass borrows expert blocks and gives them back refilled with hot experts).
#include "../../include/moe_cache.h"
#include "kernels.h"
#include "repack.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

using moe::BlockScale;
using moe::Update;

namespace {

thread_local std::string g_init_error;

struct TensorState {
    bool registered = false;
    int capacity = 0, n_seed = 0;
    uint8_t *home = nullptr;  // pinned, device-mapped: n_experts blobs of slot_stride bytes
    uint64_t home_dev = 0;
    std::vector<int32_t> seed_order, rank, slot_of, owner, last_seen;  // slot_of: global slot in a shared pool
    std::vector<uint64_t> tbl;  // host mirror of the device table row
    std::vector<uint8_t> lent;
};

}  // namespace

struct moe_ctx {
    moe_cfg cfg{};
    int dev = 0, n_sm = 0;
    int n_tensors = 0, E = 0, spt = 0, H = 0, F = 0, k = 0, M = 0;
    // shared expert (cfg.shared_experts): table rows hold E + 1 entries (the
    // last = the layer's shared expert, always in HBM) and every token gets
    // k + 1 assignments (the last = the shared expert, weight 1)
    bool shared = false;
    int Et = 0, ka = 0;                    // table row length, assignments per token
    // expert shard (moe_set_expert_shard): this context holds experts
    // [e_base, e_base + E) of a layer of E_route experts; forwards take
    // global ids and skip the other shards' assignments
    int e_base = 0, E_route = 0;
    // tokens of the step a forward belongs to (moe_ffn_forward_rows); 0: its
    // own token count
    int clock_tokens = 0;
    // a non-Q4 format with the single-launch layer for one routed token
    bool fused_t1_fmt = false;
    std::vector<uint8_t *> sh_blob;        // [n_tensors]: device blob of the shared expert
    int32_t *idx_a = nullptr;              // [M][ka]: routed ids + E
    float *w_a = nullptr;                  // [M][ka]: routed weights + 1
    size_t blob = 0, stride = 0;
    int fmt = 0;  // moe::kFmtQ4, kFmtQ8, kFmtQ5 or kFmtQ4K
    cudaStream_t stream = nullptr, up = nullptr;
    cudaEvent_t ev_fwd = nullptr, ev_up = nullptr;

    uint8_t *arena = nullptr;
    size_t arena_bytes = 0;
    uint64_t *d_tbl = nullptr;
    int32_t *d_slot = nullptr;
    uint32_t *d_stamps = nullptr, *d_bitmap = nullptr, *d_misslog = nullptr, *d_clock = nullptr;
    unsigned long long *d_cold = nullptr;
    int miss_cap = 0, bitmap_words = 0;

    int8_t *xq = nullptr, *hq = nullptr;
    BlockScale *xds = nullptr, *hds = nullptr;
    int32_t *plan_i = nullptr;  // n_uniq | uniq_e | uniq_off | assign
    int *d_error = nullptr;
    float *o = nullptr;
    unsigned *counters = nullptr;
    int n_counters = 0;
    // prefill (grouped GEMM) workspaces
    bool gemm_ok = false;
    int A_pad = 0;
    __half *xs16 = nullptr, *hq16 = nullptr;
    float *xdT = nullptr, *hdT = nullptr;
    int32_t *tile_off = nullptr;  // [2][U + 1]
    uint2 *tile_rec = nullptr;    // per-tile records: [cap_gu] gate/up, then [cap_dn] down
    int cap_gu = 0, cap_dn = 0;
    CUtensorMap tm_x{}, tm_h{};
    // prefill staging of cold experts into lent slots
    uint64_t *etbl = nullptr;     // [3][Et]
    uint64_t *stage_jobs = nullptr;
    int *stage_n = nullptr;
    int stage_cap = 0;
    // lookahead prefetch of the next layer's cold experts (prompt passes)
    bool lookahead = false;
    int pf_cap = 0;                         // expert blobs per tensor per buffer
    uint8_t *pf_buf[2] = {nullptr, nullptr};  // [3][pf_cap] blobs of `stride` bytes
    int32_t *d_pfmap[2] = {nullptr, nullptr}, *h_pfmap[2] = {nullptr, nullptr};  // [3][Et]: buffer index or -1
    cudaEvent_t ev_pf[2] = {nullptr, nullptr}, ev_pf_free[2] = {nullptr, nullptr};
    int pf_layer[2] = {-1, -1};
    bool pf_map_pending[2] = {false, false};
    // decode lookahead (batch-1 routed forwards): the routers of the layers;
    // layer l's kernel applies layer l + 1's router to its input and
    // prefetches the predicted experts' pool-resident weights into L2
    bool la_decode = false;
    __nv_bfloat16 *d_router = nullptr;        // [L][E][H]
    float *d_rbias = nullptr;                 // [L][E]
    std::vector<uint8_t> has_router;          // [L]
    float *d_prz = nullptr;                   // [E] predicted logits (scratch)
    unsigned *d_prcount = nullptr;            // [2]: logits written, prediction out
    int32_t *d_prset = nullptr;               // [L][k]: the prediction for layer l
    unsigned long long *d_prstats = nullptr;  // [2]: predicted picks, of them picked
    // fused small-batch layer kernel
    unsigned *done_gu = nullptr, *exit_count = nullptr;
    size_t fused_smem = 0, fused_smem_rb = 0;
    int fused_blocks = 0, fused_blocks_rb = 0;
    int pdl = 1;  // fused layer kernels use programmatic dependent launch

    uint32_t *h_stamps = nullptr;    // pinned mirror, refreshed per tensor when a victim is chosen
    uint32_t *d_stepbuf = nullptr;   // [hit bitmap: hit_words][miss count][miss keys]
    uint32_t *h_step = nullptr;      // pinned: hit bitmap, miss count and the first kStepKeys keys
    int *h_err = nullptr;            // pinned: the device error word, read with every step record
    int hit_words = 0;               // words of the hit bitmap: one bit per stamp index
    Update *h_upd = nullptr, *d_upd = nullptr;  // pinned, mapped (d_upd: its device address)
    int upd_cap = 0, n_upd = 0;

    std::vector<TensorState> t;
    uint64_t clock = 0;
    int n_lent = 0;
    // a single pool that every layer draws on (instead of a reserve
    // per tensor): owner and membership of every arena slot
    bool global_pool = false;
    std::vector<int32_t> g_owner;  // (tid << 12 | e) or -1
    std::vector<uint8_t> g_pool, g_lent;
    // upload overlap: a layer's next forward waits only for its own layer's
    // uploads (one event per layer) instead of the whole promotion pass's
    bool overlap = false;
    std::vector<cudaEvent_t> ev_layer_up;
    std::vector<uint8_t> layer_pending;
    int cur_up_layer = -1;                 // layer of the last upload issued in this pass
    // prefill preheat: assignments per (layer, expert) routed while slots are lent
    bool preheat = false;
    uint32_t *d_use = nullptr;
    moe_stats_t stats{};
    int last_T = -1;
    int fail_nth = 0;
    int grid_gu = 0, grid_dn = 0;
    // kernel timing hook: 4 events per layer, recorded by each forward
    bool timing = false;
    std::vector<cudaEvent_t> tev;
    std::vector<uint8_t> tev_used;
    std::string err;
};

namespace {

int fail(moe_ctx *c, int code, const std::string &msg) {
    if (c)
        c->err = msg;
    else
        g_init_error = msg;
    return code;
}

#define CK(call)                                                                                   \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess)                                                                     \
            return fail(ctx, e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA,         \
                        std::string(#call) + ": " + cudaGetErrorString(e_));                       \
    } while (0)

inline int32_t *p_n_uniq(moe_ctx *c) { return c->plan_i; }
inline int32_t *p_uniq_e(moe_ctx *c) { return c->plan_i + 1; }
inline int32_t *p_uniq_off(moe_ctx *c) { return c->plan_i + 1 + std::min(c->M * c->ka, c->Et); }
inline int32_t *p_assign(moe_ctx *c) { return c->plan_i + 2 + 2 * std::min(c->M * c->ka, c->Et); }

inline uint64_t pool_addr(moe_ctx *c, int tid, int local) {
    size_t g = (size_t)local * c->n_tensors + tid;
    return (uint64_t)(uintptr_t)(c->arena + g * c->stride);
}
inline uint64_t slot_addr(moe_ctx *c, size_t g) { return (uint64_t)(uintptr_t)(c->arena + g * c->stride); }
// Stamp index of a pool slot (the device's stamp and hit-bit position):
// tensor-major for per-tensor pools, the arena slot for a shared pool.
inline int32_t stamp_index(moe_ctx *c, int tid, int slot) {
    if (slot < 0) return -1;
    return c->global_pool ? slot : tid * std::max(1, c->spt) + slot;
}
inline uint64_t home_entry(moe_ctx *c, int tid, int e) {
    return (c->t[tid].home_dev + (uint64_t)e * c->stride) | 1ull;
}

void push_upd(moe_ctx *c, uint32_t what, size_t index, uint64_t value) {
    if (c->n_upd < c->upd_cap) c->h_upd[c->n_upd++] = Update{what, (uint32_t)index, value};
}

void set_entry(moe_ctx *c, int tid, int e, uint64_t entry, int32_t slot) {
    TensorState &ts = c->t[tid];
    ts.tbl[e] = entry;
    ts.slot_of[e] = slot;
    push_upd(c, 0, (size_t)tid * c->Et + e, entry);
    push_upd(c, 1, (size_t)tid * c->Et + e, (uint64_t)(int64_t)stamp_index(c, tid, slot));
}

constexpr size_t kStepKeys = 256;  // miss keys read back with the hit bitmap

// Publish the queued updates on `st` (table, slots, stamps, clock) in one
// kernel that reads them from the pinned list; with clear_step, the step's
// hit bitmap, miss count and miss bitmap are zeroed too.
int publish(moe_ctx *ctx, cudaStream_t st, bool clear_step = false) {
    const int na = clear_step ? ctx->hit_words + 1 : 0;
    const int nb = clear_step ? ctx->n_tensors * ctx->bitmap_words : 0;
    int rc = moe::launch_step_finish(ctx->d_upd, ctx->n_upd, ctx->d_tbl, ctx->d_slot, ctx->d_stamps, ctx->d_clock,
                                     (uint32_t)ctx->clock, ctx->d_stepbuf, na, ctx->d_bitmap, nb, st);
    if (rc) return fail(ctx, MOE_ERR_CUDA, std::string("step finish: ") + cudaGetErrorString((cudaError_t)rc));
    ctx->n_upd = 0;
    return MOE_OK;
}

// A kernel reported a device error since the last check (bit 0: an expert id
// outside [0, E), read as expert 0; other bits: a bounded wait expired and its
// work item was skipped): clear the word and report it once.
int device_fault(moe_ctx *ctx) {
    const int bits = *ctx->h_err;
    *ctx->h_err = 0;
    CK(cudaMemsetAsync(ctx->d_error, 0, sizeof(int), ctx->stream));
    char msg[160];
    snprintf(msg, sizeof msg, "device error bits 0x%x: %s", bits,
             (bits & 1) ? "an expert id outside [0, n_experts) (read as expert 0)" : "a bounded wait expired");
    return fail(ctx, MOE_ERR_FAULT, msg);
}

int wait_event(moe_ctx *ctx, cudaEvent_t ev) {
    int limit = ctx->cfg.poll_timeout_ms > 0 ? ctx->cfg.poll_timeout_ms : 10000;
    auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t q = cudaEventQuery(ev);
        if (q == cudaSuccess) return MOE_OK;
        if (q != cudaErrorNotReady) return fail(ctx, MOE_ERR_CUDA, std::string("event: ") + cudaGetErrorString(q));
        double ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
        if (ms > limit) return fail(ctx, MOE_ERR_TIMEOUT, "timed out waiting for the device");
        std::this_thread::yield();
    }
}

int sync_all(moe_ctx *ctx) {
    CK(cudaStreamSynchronize(ctx->stream));
    CK(cudaStreamSynchronize(ctx->up));
    return MOE_OK;
}

// Registration-time repack of canonical blocks into plane blobs (host code
// of its own header, so that it can also be compiled for tests on the host).
using moe::repack;

// 2-D fp16 tensor map [rows][cols] (row-major), box {64 elements, box_rows},
// 128-B swizzle, zero fill out of bounds.
int make_tmap(moe_ctx *ctx, CUtensorMap *tm, void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return fail(ctx, MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
        enc = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ctx, MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    return MOE_OK;
}

// Lookahead prefetch: copy-engine uploads of layer l's currently cold expert
// tensors into prefetch buffer l % 2 on the upload stream, after the last
// prompt forward that read that buffer.  A run of consecutive cold experts is
// one copy.  The buffer's map (expert -> copy index or -1) goes along.
int prefetch_layer(moe_ctx *ctx, int l) {
    const int b = l & 1, E = ctx->E, Et = ctx->Et;
    for (int kd = 0; kd < 3; ++kd)
        if (!ctx->t[l * 3 + kd].registered) return MOE_OK;
    // the previous prefetch into this buffer copied the host map: it has to
    // be done before the map is rewritten
    if (ctx->pf_map_pending[b]) CK(cudaEventSynchronize(ctx->ev_pf[b]));
    ctx->pf_map_pending[b] = false;
    CK(cudaStreamWaitEvent(ctx->up, ctx->ev_pf_free[b], 0));
    int32_t *map = ctx->h_pfmap[b];
    for (int kd = 0; kd < 3; ++kd) {
        const TensorState &ts = ctx->t[l * 3 + kd];
        uint8_t *dst0 = ctx->pf_buf[b] + (size_t)kd * ctx->pf_cap * ctx->stride;
        int n = 0, run_e = 0, run_m = 0, run_len = 0;
        for (int e = 0; e <= E; ++e) {
            const bool cold = e < E && ts.slot_of[e] < 0 && n < ctx->pf_cap;
            if (run_len && (!cold || run_e + run_len != e)) {
                CK(cudaMemcpyAsync(dst0 + (size_t)run_m * ctx->stride, ts.home + (size_t)run_e * ctx->stride,
                                   (size_t)run_len * ctx->stride, cudaMemcpyHostToDevice, ctx->up));
                run_len = 0;
            }
            if (e == E) break;
            map[kd * Et + e] = cold ? n : -1;
            if (cold) {
                if (!run_len) {
                    run_e = e;
                    run_m = n;
                }
                ++run_len;
                ++n;
            }
        }
    }
    if (Et > E)
        for (int kd = 0; kd < 3; ++kd) map[kd * Et + E] = -1;  // the shared expert stays where it is
    CK(cudaMemcpyAsync(ctx->d_pfmap[b], map, sizeof(int32_t) * 3 * Et, cudaMemcpyHostToDevice, ctx->up));
    CK(cudaEventRecord(ctx->ev_pf[b], ctx->up));
    ctx->pf_map_pending[b] = true;
    ctx->pf_layer[b] = l;
    return MOE_OK;
}

// Upload overlap: called before each pool upload of the promotion pass (they
// come in ascending layer order); closes the previous layer's uploads with its
// event.  finish = true closes the last one.
int note_upload(moe_ctx *ctx, int layer, bool finish = false) {
    if (!ctx->overlap) return MOE_OK;
    const int prev = ctx->cur_up_layer;
    if (prev >= 0 && (finish || prev != layer)) {
        CK(cudaEventRecord(ctx->ev_layer_up[prev], ctx->up));
        ctx->layer_pending[prev] = 1;
    }
    ctx->cur_up_layer = finish ? -1 : layer;
    return MOE_OK;
}

// Victim search of the shared pool for one promotion pass: the free pool
// slots in arena order first, then the occupied slots stamped before this
// step, by (stamp, slot) (both built at the step's first admission).  Slots filled
// in this pass carry the new clock, so they never become victims, and a
// candidate changes hands only by being taken: one sorted list serves every
// admission of the step.
struct GlobalPick {
    bool stamps_read = false, free_built = false;
    std::vector<int> free_slots;
    size_t fpos = 0;
    std::vector<std::pair<uint32_t, int>> victims;
    size_t vpos = 0;
    int took = 0;
    int n_qualified = 0;  // misses of the step that qualify for admission
};

// One admission of (tid, e) into the shared pool: lowest free slot, else the
// oldest stamp below the clock (ties: lowest slot), whichever layer holds it.
int admit_global(moe_ctx *ctx, GlobalPick &gs, int tid, int e, uint64_t clk, int &fault, int &uploads) {
    const int G = ctx->n_tensors * std::max(1, ctx->spt);
    gs.took = 0;
    if (!gs.stamps_read) {
        // the device stamps (the stream is idle here), before this step's
        // first admission edits the mirror
        CK(cudaMemcpy(ctx->h_stamps, ctx->d_stamps, sizeof(uint32_t) * G, cudaMemcpyDeviceToHost));
        gs.stamps_read = true;
    }
    if (!gs.free_built) {
        // one pass over the arena: the free pool slots in order, and the
        // n_qualified smallest (stamp, slot) pairs among the occupied slots
        // stamped before this step (a bounded max-heap; no step can take
        // more victims than it has qualifying misses)
        const size_t need = (size_t)std::max(0, gs.n_qualified);
        auto &h = gs.victims;
        for (int v = 0; v < G; ++v) {
            if (!ctx->g_pool[v] || ctx->g_lent[v]) continue;
            if (ctx->g_owner[v] < 0) {
                gs.free_slots.push_back(v);
                continue;
            }
            const uint32_t st = ctx->h_stamps[v];
            if ((uint64_t)st >= clk || need == 0) continue;
            const std::pair<uint32_t, int> c(st, v);
            if (h.size() < need) {
                h.push_back(c);
                std::push_heap(h.begin(), h.end());
            } else if (c < h.front()) {
                std::pop_heap(h.begin(), h.end());
                h.back() = c;
                std::push_heap(h.begin(), h.end());
            }
        }
        std::sort_heap(h.begin(), h.end());
        gs.free_built = true;
    }
    int g = -1;
    if (gs.fpos < gs.free_slots.size()) {
        g = gs.free_slots[gs.fpos++];
    } else if (gs.vpos < gs.victims.size()) {
        g = gs.victims[gs.vpos++].second;
    }
    if (g < 0) return MOE_OK;  // every pool slot was used this step: skipped, the sighting stays
    const int vkey = ctx->g_owner[g];
    if (vkey >= 0) {
        const int vt = vkey >> 12, ve = vkey & 0xfff;
        set_entry(ctx, vt, ve, home_entry(ctx, vt, ve), -1);
        ctx->t[vt].last_seen[ve] = -1;
        ctx->g_owner[g] = -1;
        ctx->stats.evictions++;
    }
    gs.took = 1;
    if (ctx->fail_nth > 0 && --ctx->fail_nth == 0) {
        // injected upload failure: rolled back; the slot is the next
        // admission's lowest free slot
        fault = 1;
        gs.free_slots.insert(std::lower_bound(gs.free_slots.begin() + (long)gs.fpos, gs.free_slots.end(), g), g);
        return MOE_OK;
    }
    TensorState &ts = ctx->t[tid];
    const uint64_t dst = slot_addr(ctx, (size_t)g);
    int rcu = note_upload(ctx, tid / 3);
    if (rcu) return rcu;
    CK(cudaMemcpyAsync((void *)(uintptr_t)dst, ts.home + (size_t)e * ctx->stride, ctx->blob, cudaMemcpyHostToDevice,
                       ctx->up));
    uploads++;
    set_entry(ctx, tid, e, dst, g);
    ctx->g_owner[g] = (tid << 12) | e;
    ts.last_seen[e] = -1;
    ctx->h_stamps[g] = (uint32_t)clk;
    push_upd(ctx, 2, (size_t)g, (uint32_t)clk);
    ctx->stats.admissions++;
    ctx->stats.upload_bytes += ctx->blob;
    return MOE_OK;
}

uint16_t f32_to_half_bits(float v) {
    __half h = __float2half_rn(v);
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

}  // namespace

namespace moe {
void set_context_free_error(const std::string &msg) { g_init_error = msg; }
}  // namespace moe

extern "C" {

int moe_layer_init(const moe_cfg *cfg, void *cuda_stream, moe_ctx **out) {
    moe_ctx *ctx = nullptr;
    if (!cfg || !out) return fail(nullptr, MOE_ERR_ARG, "null argument");
    *out = nullptr;
    const moe_cfg &c = *cfg;
    if (c.hidden <= 0 || c.hidden % 32 || c.ffn <= 0 || c.ffn % 32 || c.n_experts < 1 || c.n_experts > 4096 ||
        c.top_k < 1 || c.top_k > 32 || c.top_k > c.n_experts || c.n_layers < 1 || c.n_layers * 3 > (1 << 20) ||
        c.slots_per_tensor < 0 || c.slots_per_tensor > c.n_experts || c.max_tokens < 1 || c.window_tokens < 1 ||
        c.max_swaps_per_step < 0 || (c.shared_experts != 0 && (c.shared_experts != 1 || c.n_experts > 4095)) ||
        (c.weight_format != MOE_FMT_Q4_0 && c.weight_format != MOE_FMT_Q8_0 && c.weight_format != MOE_FMT_Q5_0 &&
         c.weight_format != MOE_FMT_Q4_K && c.weight_format != MOE_FMT_Q6_K && c.weight_format != MOE_FMT_Q5_K) ||
        ((c.weight_format == MOE_FMT_Q4_K || c.weight_format == MOE_FMT_Q6_K || c.weight_format == MOE_FMT_Q5_K) &&
         (c.hidden % 256 || c.ffn % 256)))
        return fail(nullptr, MOE_ERR_ARG,
                    "bad cfg: hidden%32, ffn%32, 1<=E<=4096, 1<=k<=min(32,E), layers>=1, 0<=slots<=E, max_tokens>=1, "
                    "weight_format Q4_0, Q8_0, Q5_0, Q4_K, Q6_K or Q5_K (hidden, ffn % 256), shared_experts 0 or 1 "
                    "(then E <= 4095)");
    int down_rows = moe::down_rows_per_item(c.ffn);
    if (c.hidden % down_rows) return fail(nullptr, MOE_ERR_ARG, "hidden must be a multiple of the down row block");
    ctx = new moe_ctx();
    ctx->cfg = c;
    ctx->dev = c.device;
    ctx->E = c.n_experts;
    ctx->H = c.hidden;
    ctx->F = c.ffn;
    ctx->k = c.top_k;
    ctx->shared = c.shared_experts != 0;
    ctx->Et = c.n_experts + (ctx->shared ? 1 : 0);
    ctx->E_route = c.n_experts;
    ctx->ka = c.top_k + (ctx->shared ? 1 : 0);
    ctx->M = c.max_tokens;
    ctx->n_tensors = 3 * c.n_layers;
    ctx->spt = c.slots_per_tensor;
    ctx->fmt = c.weight_format == MOE_FMT_Q8_0   ? moe::kFmtQ8
               : c.weight_format == MOE_FMT_Q5_0 ? moe::kFmtQ5
               : c.weight_format == MOE_FMT_Q4_K ? moe::kFmtQ4K
               : c.weight_format == MOE_FMT_Q6_K ? moe::kFmtQ6K
               : c.weight_format == MOE_FMT_Q5_K ? moe::kFmtQ5K
                                                 : moe::kFmtQ4;
    ctx->blob = moe::blob_bytes_fmt(ctx->fmt, c.ffn, c.hidden / 32);
    ctx->stride = (ctx->blob + 255) / 256 * 256;
    auto cleanup_fail = [&](int rc) {
        std::string m = ctx->err;
        moe_destroy(ctx);
        g_init_error = m;
        return rc;
    };
#define CKI(call)                                                                                  \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess) {                                                                   \
            ctx->err = std::string(#call) + ": " + cudaGetErrorString(e_);                         \
            return cleanup_fail(e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA);     \
        }                                                                                          \
    } while (0)
    CKI(cudaSetDevice(ctx->dev));
    CKI(cudaDeviceGetAttribute(&ctx->n_sm, cudaDevAttrMultiProcessorCount, ctx->dev));
    ctx->stream = (cudaStream_t)cuda_stream;  // NULL: the legacy default stream
    CKI(cudaStreamCreateWithFlags(&ctx->up, cudaStreamNonBlocking));
    CKI(cudaEventCreateWithFlags(&ctx->ev_fwd, cudaEventDisableTiming));
    CKI(cudaEventCreateWithFlags(&ctx->ev_up, cudaEventDisableTiming));

    const int nt = ctx->n_tensors, E = ctx->E, Et = ctx->Et;
    ctx->arena_bytes = (size_t)nt * ctx->spt * ctx->stride;
    if (ctx->arena_bytes) CKI(cudaMalloc(&ctx->arena, ctx->arena_bytes));
    ctx->bitmap_words = (Et + 31) / 32;
    ctx->miss_cap = nt * E;
    CKI(cudaMalloc(&ctx->d_tbl, sizeof(uint64_t) * nt * Et));
    CKI(cudaMalloc(&ctx->d_slot, sizeof(int32_t) * nt * Et));
    CKI(cudaMemset(ctx->d_slot, 0xff, sizeof(int32_t) * nt * Et));
    CKI(cudaMemset(ctx->d_tbl, 0, sizeof(uint64_t) * nt * Et));
    ctx->sh_blob.assign(nt, nullptr);
    CKI(cudaMalloc(&ctx->d_stamps, sizeof(uint32_t) * (size_t)nt * std::max(1, ctx->spt)));
    CKI(cudaMemset(ctx->d_stamps, 0, sizeof(uint32_t) * (size_t)nt * std::max(1, ctx->spt)));
    CKI(cudaMalloc(&ctx->d_bitmap, sizeof(uint32_t) * (size_t)nt * ctx->bitmap_words));
    CKI(cudaMemset(ctx->d_bitmap, 0, sizeof(uint32_t) * (size_t)nt * ctx->bitmap_words));
    ctx->hit_words = (int)(((size_t)nt * std::max(1, ctx->spt) + 31) / 32);
    {
        const size_t hb = (size_t)ctx->hit_words;
        CKI(cudaMalloc(&ctx->d_stepbuf, sizeof(uint32_t) * (hb + 1 + (size_t)ctx->miss_cap)));
        CKI(cudaMemset(ctx->d_stepbuf, 0, sizeof(uint32_t) * (hb + 1)));
        ctx->d_misslog = ctx->d_stepbuf + hb;
    }
    CKI(cudaMalloc(&ctx->d_clock, sizeof(uint32_t)));
    CKI(cudaMemset(ctx->d_clock, 0, sizeof(uint32_t)));
    CKI(cudaMalloc(&ctx->d_cold, sizeof(unsigned long long)));
    CKI(cudaMemset(ctx->d_cold, 0, sizeof(unsigned long long)));

    const size_t M = ctx->M, A = M * ctx->ka, U = std::min<size_t>(A, Et);
    if (ctx->shared) {
        CKI(cudaMalloc(&ctx->idx_a, sizeof(int32_t) * A));
        CKI(cudaMalloc(&ctx->w_a, sizeof(float) * A));
    }
    CKI(cudaMalloc(&ctx->xq, M * ctx->H));
    CKI(cudaMalloc(&ctx->xds, sizeof(BlockScale) * M * (ctx->H / 32)));
    CKI(cudaMalloc(&ctx->plan_i, sizeof(int32_t) * (2 + 2 * U + A)));
    CKI(cudaMalloc(&ctx->d_error, sizeof(int)));
    CKI(cudaMemset(ctx->d_error, 0, sizeof(int)));
    CKI(cudaMalloc(&ctx->hq, A * ctx->F));
    CKI(cudaMalloc(&ctx->hds, sizeof(BlockScale) * A * (ctx->F / 32)));
    CKI(cudaMalloc(&ctx->o, sizeof(float) * A * ctx->H));
    ctx->n_counters = ctx->H / down_rows;
    CKI(cudaMalloc(&ctx->counters, sizeof(unsigned) * ctx->n_counters));
    CKI(cudaMemset(ctx->counters, 0, sizeof(unsigned) * ctx->n_counters));

    // prefill workspaces: sorted fp16 operands of the grouped GEMM
    // (Q4 only: the GEMM's converters expand 4-bit codes)
    if (ctx->M > 32 && ctx->H % 64 == 0 && ctx->F % 64 == 0 && ctx->fmt == moe::kFmtQ4) {
        ctx->A_pad = (int)((A + 127) / 128 * 128 + 128);
        const size_t AP = ctx->A_pad;
        CKI(cudaMalloc(&ctx->xs16, sizeof(__half) * AP * ctx->H));
        CKI(cudaMemset(ctx->xs16, 0, sizeof(__half) * AP * ctx->H));
        CKI(cudaMalloc(&ctx->xdT, sizeof(float) * AP * (ctx->H / 32)));
        CKI(cudaMemset(ctx->xdT, 0, sizeof(float) * AP * (ctx->H / 32)));
        CKI(cudaMalloc(&ctx->hq16, sizeof(__half) * AP * ctx->F));
        CKI(cudaMemset(ctx->hq16, 0, sizeof(__half) * AP * ctx->F));
        CKI(cudaMalloc(&ctx->hdT, sizeof(float) * AP * (ctx->F / 32)));
        CKI(cudaMemset(ctx->hdT, 0, sizeof(float) * AP * (ctx->F / 32)));
        CKI(cudaMalloc(&ctx->tile_off, sizeof(int32_t) * 2 * (U + 1)));
        // tiles per GEMM <= row tiles x (assignments / tile width + used experts)
        const int rg = moe::gemm_rows_per_tile(true), rd = moe::gemm_rows_per_tile(false);
        ctx->cap_gu = ((ctx->F + rg - 1) / rg) * (int)((A + moe::gemm_bn(true) - 1) / moe::gemm_bn(true) + U);
        ctx->cap_dn = ((ctx->H + rd - 1) / rd) * (int)((A + moe::gemm_bn(false) - 1) / moe::gemm_bn(false) + U);
        CKI(cudaMalloc(&ctx->tile_rec, sizeof(uint2) * ((size_t)ctx->cap_gu + ctx->cap_dn)));
        CKI(cudaMalloc(&ctx->etbl, sizeof(uint64_t) * 3 * Et));
        ctx->stage_cap = 3 * E;
        CKI(cudaMalloc(&ctx->stage_jobs, sizeof(uint64_t) * 2 * ctx->stage_cap));
        CKI(cudaMalloc(&ctx->stage_n, sizeof(int)));
        if (make_tmap(ctx, &ctx->tm_x, ctx->xs16, AP, ctx->H, (uint32_t)moe::gemm_bn(true)) ||
            make_tmap(ctx, &ctx->tm_h, ctx->hq16, AP, ctx->F, (uint32_t)moe::gemm_bn(false)))
            return cleanup_fail(MOE_ERR_CUDA);
        CKI((cudaError_t)moe::gemm_configure());
        ctx->gemm_ok = true;
    }

    CKI(cudaMalloc(&ctx->done_gu, sizeof(unsigned) * (E + 1)));
    CKI(cudaMemset(ctx->done_gu, 0, sizeof(unsigned) * (E + 1)));
    ctx->exit_count = ctx->done_gu + E;
    ctx->fused_smem = moe::fused_smem_bytes(ctx->H, ctx->F);
    {
        int bps = 0;
        CKI((cudaError_t)moe::fused_configure(ctx->F, ctx->fused_smem, &bps));
        ctx->fused_blocks = bps * ctx->n_sm;
        // row-block down mode: the largest launch of up to 8 tokens that uses it
        for (int T = 1; T <= std::min(ctx->M, 8); ++T) {
            const int rows = moe::fused_rb_rows(ctx->H, ctx->F, T, ctx->k, E);
            if (rows > 0) {
                size_t sm = moe::fused_rb_smem(ctx->H, ctx->F, T, ctx->k, E, rows, nullptr);
                if (T == 1 && moe::fused_t1_ok(E, ctx->k)) sm = (sm + 15) / 16 * 16 + (size_t)24 * E;
                ctx->fused_smem_rb = std::max(ctx->fused_smem_rb, sm);
            }
        }
        if (ctx->fused_smem_rb > 0) {
            CKI((cudaError_t)moe::fused_configure_rb(ctx->F, ctx->fused_smem_rb, &bps));
            ctx->fused_blocks_rb = bps * ctx->n_sm;
        }
        if (ctx->shared || ctx->fmt != moe::kFmtQ4) {
            // other formats and shared experts: the single-launch layer for
            // one routed token only (the shared expert is its last pick, its
            // weights requested at kernel entry), the mat-vec kernels for
            // the rest
            ctx->fused_blocks = 0;
            ctx->fused_blocks_rb = 0;
            const int rows = moe::fused_rb_rows(ctx->H, ctx->F, 1, ctx->ka, Et);
            if (rows > 0 && moe::fused_t1_ok(E, ctx->ka)) {
                size_t sm = moe::fused_rb_smem(ctx->H, ctx->F, 1, ctx->ka, Et, rows, nullptr);
                sm = (sm + 15) / 16 * 16 + (size_t)24 * Et;
                CKI((cudaError_t)moe::fused_configure_t1_fmt(ctx->F, ctx->fmt, sm, &bps));
                if (bps > 0) {
                    ctx->fused_smem_rb = sm;
                    ctx->fused_blocks_rb = bps * ctx->n_sm;
                    ctx->fused_t1_fmt = true;
                }
            }
        }
    }

    CKI(cudaHostAlloc(&ctx->h_stamps, sizeof(uint32_t) * (size_t)nt * std::max(1, ctx->spt), cudaHostAllocDefault));
    ctx->upd_cap = 6 * nt * E + 64;
    CKI(cudaHostAlloc(&ctx->h_upd, sizeof(Update) * (size_t)ctx->upd_cap, cudaHostAllocMapped));
    CKI(cudaHostGetDevicePointer((void **)&ctx->d_upd, ctx->h_upd, 0));
    CKI(cudaHostAlloc(&ctx->h_step, sizeof(uint32_t) * ((size_t)ctx->hit_words + 1 + kStepKeys),
                      cudaHostAllocDefault));
    CKI(cudaHostAlloc(&ctx->h_err, sizeof(int), cudaHostAllocDefault));
    *ctx->h_err = 0;
    CKI(cudaDeviceSynchronize());
#undef CKI
    ctx->t.resize(nt);
    ctx->grid_gu = ctx->n_sm * 4;
    ctx->grid_dn = ctx->n_sm * 4;
    *out = ctx;
    return MOE_OK;
}

int register_expert_tensor(moe_ctx *ctx, int layer, int kind, const void *host_q4, int rows, int cols, int capacity,
                           const int32_t *seed_order, int n_seed, int *tensor_id) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (layer < 0 || layer >= ctx->cfg.n_layers || kind < 0 || kind > 2 || !host_q4)
        return fail(ctx, MOE_ERR_ARG, "bad layer/kind/pointer");
    const int er = kind == MOE_KIND_DOWN ? ctx->H : ctx->F, ec = kind == MOE_KIND_DOWN ? ctx->F : ctx->H;
    if (rows != er || cols != ec || cols % 32) return fail(ctx, MOE_ERR_ARG, "tensor shape does not match cfg");
    if (capacity < 0 || capacity > ctx->spt || n_seed < 0 || n_seed > capacity)
        return fail(ctx, MOE_ERR_ARG, "need 0 <= n_seed <= capacity <= slots_per_tensor");
    const int tid = layer * 3 + kind, E = ctx->E;
    TensorState &ts = ctx->t[tid];
    if (ts.registered) return fail(ctx, MOE_ERR_ARG, "tensor already registered");
    std::vector<int32_t> order(E);
    if (seed_order) {
        std::vector<uint8_t> seen(E, 0);
        for (int i = 0; i < E; ++i) {
            int e = seed_order[i];
            if (e < 0 || e >= E || seen[e]) return fail(ctx, MOE_ERR_ARG, "seed_order must be a permutation of 0..E-1");
            seen[e] = 1;
            order[i] = e;
        }
    } else {
        for (int i = 0; i < E; ++i) order[i] = i;
    }
    CK(cudaSetDevice(ctx->dev));
    void *home = nullptr;
    CK(cudaHostAlloc(&home, ctx->stride * E, cudaHostAllocMapped | cudaHostAllocPortable));
    void *home_dev = nullptr;
    cudaError_t ge = cudaHostGetDevicePointer(&home_dev, home, 0);
    if (ge != cudaSuccess) {
        cudaFreeHost(home);
        return fail(ctx, MOE_ERR_CUDA, std::string("cudaHostGetDevicePointer: ") + cudaGetErrorString(ge));
    }
    ts.home = (uint8_t *)home;
    ts.home_dev = (uint64_t)(uintptr_t)home_dev;
    repack((const uint8_t *)host_q4, ts.home, ctx->fmt, E, rows, cols / 32, ctx->stride);
    ts.capacity = capacity;
    ts.n_seed = n_seed;
    ts.seed_order = order;
    ts.rank.assign(E, 0);
    for (int i = 0; i < E; ++i) ts.rank[order[i]] = i;
    ts.slot_of.assign(E, -1);
    ts.owner.assign(ctx->spt, -1);
    ts.last_seen.assign(E, -1);
    ts.lent.assign(ctx->spt, 0);
    ts.tbl.resize(E);
    for (int e = 0; e < E; ++e) ts.tbl[e] = home_entry(ctx, tid, e);
    if (ctx->global_pool)
        for (int s = 0; s < capacity; ++s) ctx->g_pool[(size_t)s * ctx->n_tensors + tid] = 1;
    for (int s = 0; s < n_seed; ++s) {
        int e = order[s];
        uint64_t dst = pool_addr(ctx, tid, s);
        CK(cudaMemcpyAsync((void *)(uintptr_t)dst, ts.home + (size_t)e * ctx->stride, ctx->blob,
                           cudaMemcpyHostToDevice, ctx->up));
        ts.tbl[e] = dst;
        if (ctx->global_pool) {
            const int g = s * ctx->n_tensors + tid;
            ts.slot_of[e] = g;
            ctx->g_owner[g] = (tid << 12) | e;
        } else {
            ts.slot_of[e] = s;
            ts.owner[s] = e;
        }
    }
    std::vector<int32_t> dslot(E);
    for (int e = 0; e < E; ++e) dslot[e] = stamp_index(ctx, tid, ts.slot_of[e]);
    CK(cudaMemcpyAsync(ctx->d_tbl + (size_t)tid * ctx->Et, ts.tbl.data(), sizeof(uint64_t) * E,
                       cudaMemcpyHostToDevice, ctx->up));
    CK(cudaMemcpyAsync(ctx->d_slot + (size_t)tid * ctx->Et, dslot.data(), sizeof(int32_t) * E, cudaMemcpyHostToDevice,
                       ctx->up));
    CK(cudaStreamSynchronize(ctx->up));
    ts.registered = true;
    ctx->stats.upload_bytes += (uint64_t)n_seed * ctx->blob;
    if (tensor_id) *tensor_id = tid;
    return MOE_OK;
}

int register_shared_expert(moe_ctx *ctx, int layer, int kind, const void *host_w, int rows, int cols) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (!ctx->shared) return fail(ctx, MOE_ERR_STATE, "shared expert: the context was made without shared_experts");
    if (layer < 0 || layer >= ctx->cfg.n_layers || kind < 0 || kind > 2 || !host_w)
        return fail(ctx, MOE_ERR_ARG, "bad layer/kind/pointer");
    const int er = kind == MOE_KIND_DOWN ? ctx->H : ctx->F, ec = kind == MOE_KIND_DOWN ? ctx->F : ctx->H;
    if (rows != er || cols != ec) return fail(ctx, MOE_ERR_ARG, "shared expert shape does not match cfg");
    const int tid = layer * 3 + kind;
    if (ctx->sh_blob[tid]) return fail(ctx, MOE_ERR_ARG, "shared expert already registered");
    CK(cudaSetDevice(ctx->dev));
    std::vector<uint8_t> blob(ctx->blob);
    repack((const uint8_t *)host_w, blob.data(), ctx->fmt, 1, rows, cols / 32, ctx->blob);
    uint8_t *d = nullptr;
    CK(cudaMalloc(&d, ctx->stride));
    cudaError_t e = cudaMemcpy(d, blob.data(), ctx->blob, cudaMemcpyHostToDevice);
    const uint64_t entry = (uint64_t)(uintptr_t)d;
    if (e == cudaSuccess)
        e = cudaMemcpy(ctx->d_tbl + (size_t)tid * ctx->Et + ctx->E, &entry, sizeof(entry), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(d);
        return fail(ctx, MOE_ERR_CUDA, std::string("shared expert upload: ") + cudaGetErrorString(e));
    }
    ctx->sh_blob[tid] = d;
    ctx->stats.upload_bytes += ctx->blob;
    return MOE_OK;
}

int route_topk(moe_ctx *ctx, const float *d_logits, int n_tokens, int n_experts, int k, int32_t *d_idx, float *d_w,
               void *stream) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (n_tokens < 0 || n_experts != ctx->E_route || k != ctx->k || (n_tokens > 0 && (!d_logits || !d_idx || !d_w)))
        return fail(ctx, MOE_ERR_ARG, "route_topk: bad sizes or pointers");
    cudaStream_t st = stream ? (cudaStream_t)stream : ctx->stream;
    int rc = moe::launch_topk(d_logits, n_tokens, n_experts, k, ctx->cfg.renorm_topk, d_idx, d_w, st);
    if (rc) return fail(ctx, MOE_ERR_CUDA, std::string("topk launch: ") + cudaGetErrorString((cudaError_t)rc));
    return MOE_OK;
}

static int ffn_forward_impl(moe_ctx *ctx, int layer, const float *d_x, int n_tokens, const int32_t *d_idx,
                            const float *d_w, float *d_y, void *stream, const float *d_logits, int32_t *idx_out,
                            float *w_out);

int moe_ffn_forward(moe_ctx *ctx, int layer, const float *d_x, int n_tokens, const int32_t *d_idx, const float *d_w,
                    float *d_y, void *stream) {
    return ffn_forward_impl(ctx, layer, d_x, n_tokens, d_idx, d_w, d_y, stream, nullptr, nullptr, nullptr);
}

int moe_ffn_forward_routed(moe_ctx *ctx, int layer, const float *d_x, const float *d_logits, int n_tokens,
                           int32_t *d_idx, float *d_w, float *d_y, void *stream) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (n_tokens > 0 && (!d_logits || !d_idx || !d_w)) return fail(ctx, MOE_ERR_ARG, "routed forward: null pointer");
    if (n_tokens > 0 && n_tokens <= 32 && n_tokens * ctx->ka <= 256 &&
        (ctx->fused_blocks > 0 || (n_tokens == 1 && ctx->fused_t1_fmt && ctx->e_base == 0 && ctx->E_route == ctx->E)))
        return ffn_forward_impl(ctx, layer, d_x, n_tokens, d_idx, d_w, d_y, stream, d_logits, d_idx, d_w);
    int rc = route_topk(ctx, d_logits, n_tokens, ctx->E_route, ctx->k, d_idx, d_w, stream);
    if (rc) return rc;
    return ffn_forward_impl(ctx, layer, d_x, n_tokens, d_idx, d_w, d_y, stream, nullptr, nullptr, nullptr);
}

int moe_set_expert_shard(moe_ctx *ctx, int expert_base, int n_route) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (ctx->shared) return fail(ctx, MOE_ERR_STATE, "expert shard: not with shared experts");
    if (expert_base < 0 || n_route < ctx->E || n_route > 4096 || expert_base > n_route - ctx->E)
        return fail(ctx, MOE_ERR_ARG, "expert shard: need 0 <= expert_base <= n_route - n_experts, n_route <= 4096");
    ctx->e_base = expert_base;
    ctx->E_route = n_route;
    return MOE_OK;
}

int moe_ffn_forward_rows(moe_ctx *ctx, int layer, const float *d_x, int n_rows, const int32_t *d_idx,
                         const float *d_w, float *d_y, int step_tokens, void *stream) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (n_rows < 0 || step_tokens < n_rows || step_tokens < 1)
        return fail(ctx, MOE_ERR_ARG, "forward_rows: need 0 <= n_rows <= step_tokens, step_tokens >= 1");
    ctx->clock_tokens = step_tokens;
    const int rc = ffn_forward_impl(ctx, layer, d_x, n_rows, d_idx, d_w, d_y, stream, nullptr, nullptr, nullptr);
    ctx->clock_tokens = 0;
    return rc;
}

static int ffn_forward_body(moe_ctx *ctx, int layer, const float *d_x, int n_tokens, const int32_t *d_idx,
                            const float *d_w, float *d_y, void *stream, const float *d_logits, int32_t *idx_out,
                            float *w_out);

// One layer, then (prefill preheat, while pool slots are lent to a prompt
// pass) the layer's (token, expert) assignments added to its use counts.
static int ffn_forward_impl(moe_ctx *ctx, int layer, const float *d_x, int n_tokens, const int32_t *d_idx,
                            const float *d_w, float *d_y, void *stream, const float *d_logits, int32_t *idx_out,
                            float *w_out) {
    int rc = ffn_forward_body(ctx, layer, d_x, n_tokens, d_idx, d_w, d_y, stream, d_logits, idx_out, w_out);
    if (rc || !ctx->preheat || !ctx->n_lent || n_tokens <= 0 || !ctx->d_use) return rc;
    rc = moe::launch_count_assign(d_idx, n_tokens * ctx->k, ctx->E, ctx->e_base, ctx->d_use + (size_t)layer * ctx->E,
                                  ctx->stream);
    if (rc) return fail(ctx, MOE_ERR_CUDA, std::string("use counts: ") + cudaGetErrorString((cudaError_t)rc));
    return MOE_OK;
}

static int ffn_forward_body(moe_ctx *ctx, int layer, const float *d_x, int n_tokens, const int32_t *d_idx,
                            const float *d_w, float *d_y, void *stream, const float *d_logits, int32_t *idx_out,
                            float *w_out) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (layer < 0 || layer >= ctx->cfg.n_layers || n_tokens < 0 || n_tokens > ctx->M)
        return fail(ctx, MOE_ERR_ARG, "forward: bad layer or n_tokens (> max_tokens?)");
    if (stream && (cudaStream_t)stream != ctx->stream)
        return fail(ctx, MOE_ERR_ARG, "forward: stream must be the context stream");
    for (int kd = 0; kd < 3; ++kd)
        if (!ctx->t[layer * 3 + kd].registered) return fail(ctx, MOE_ERR_STATE, "forward: layer not registered");
    if (n_tokens == 0) return MOE_OK;
    if (!d_x || !d_idx || !d_w || !d_y) return fail(ctx, MOE_ERR_ARG, "forward: null pointer");
    cudaStream_t st = ctx->stream;
    if (ctx->overlap && ctx->layer_pending[layer]) {
        // this layer's admissions of the last promotion pass must be in
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        CK(cudaStreamIsCapturing(st, &cs));
        if (cs != cudaStreamCaptureStatusNone)
            return fail(ctx, MOE_ERR_STATE, "forward: upload overlap needs forwards issued outside stream capture");
        CK(cudaStreamWaitEvent(st, ctx->ev_layer_up[layer], 0));
        ctx->layer_pending[layer] = 0;
    }
    const bool sharded = ctx->e_base != 0 || ctx->E_route != ctx->E;
    // one routed token through the single-launch layer of a format or
    // shared-expert context (which routes and adds the shared expert itself)
    const bool t1_only = ctx->fused_t1_fmt && n_tokens == 1 && d_logits && !sharded;
    if (ctx->shared) {
        for (int kd = 0; kd < 3; ++kd)
            if (!ctx->sh_blob[layer * 3 + kd])
                return fail(ctx, MOE_ERR_STATE, "forward: shared expert of this layer not registered");
    }
    if (ctx->shared && !t1_only) {
        // the layer's shared expert joins every token as assignment k (id E,
        // weight 1); the routed ids are checked against E here
        int rc0 = moe::launch_shared_assign(d_idx, d_w, n_tokens, ctx->k, ctx->E, ctx->idx_a, ctx->w_a, ctx->d_error,
                                            st);
        if (rc0) return fail(ctx, MOE_ERR_CUDA, "shared-expert assignment launch failed");
        d_idx = ctx->idx_a;
        d_w = ctx->w_a;
    }
    const int T = n_tokens, H = ctx->H;
    const bool small = T <= 32;
    int rc = 0;
    moe::GemvParams gp{};
    gp.cv.tbl = ctx->d_tbl;
    gp.cv.slot = ctx->d_slot;
    gp.cv.stamps = ctx->d_stamps;
    gp.cv.miss_bitmap = ctx->d_bitmap;
    gp.cv.miss_list = ctx->d_misslog + 1;
    gp.cv.miss_count = ctx->d_misslog;
    gp.cv.clock = ctx->d_clock;
    gp.cv.cold_reads = ctx->d_cold;
    gp.cv.E = ctx->Et;
    gp.cv.slots_per_tensor = std::max(1, ctx->spt);
    gp.cv.bitmap_words = ctx->bitmap_words;
    gp.cv.miss_cap = ctx->miss_cap;
    gp.cv.hit_bitmap = ctx->d_stepbuf;
    gp.cv.hit_words = ctx->hit_words;
    gp.cv.clock_tokens = ctx->clock_tokens > 0 ? ctx->clock_tokens : n_tokens;
    gp.tid_gate = layer * 3 + 0;
    gp.tid_up = layer * 3 + 1;
    gp.tid_down = layer * 3 + 2;
    gp.n_tokens = T;
    gp.k = ctx->ka;
    gp.H = H;
    gp.F = ctx->F;
    gp.xq = ctx->xq;
    gp.xds = ctx->xds;
    gp.n_uniq = p_n_uniq(ctx);
    gp.uniq_e = p_uniq_e(ctx);
    gp.uniq_off = p_uniq_off(ctx);
    gp.assign = p_assign(ctx);
    gp.hq = ctx->hq;
    gp.hds = ctx->hds;
    gp.o = ctx->o;
    gp.counters = ctx->counters;
    gp.w = d_w;
    gp.y = d_y;
    const int A = T * ctx->ka, U = std::min(A, ctx->Et);
    gp.xq_out = ctx->xq;
    gp.xds_out = ctx->xds;
    gp.fmt = ctx->fmt;
    gp.idx = d_idx;
    gp.e_base = ctx->e_base;
    if (small && A <= 256 && (ctx->fused_blocks > 0 || t1_only)) {
        moe::FusedParams fp{};
        fp.g = gp;
        fp.x = d_x;
        fp.idx = d_idx;
        fp.done_gu = ctx->done_gu;
        fp.exit_count = ctx->exit_count;
        fp.error = ctx->d_error;
        fp.logits = d_logits;
        fp.n_route = sharded ? ctx->E_route : ctx->Et;
        fp.idx_out = idx_out;
        fp.w_out = w_out;
        fp.renorm = ctx->cfg.renorm_topk;
        fp.pdl = ctx->pdl;
        int items = U * std::max(ctx->F / 32, ctx->n_counters);
        int grid = std::min(items, ctx->fused_blocks);
        size_t smem = ctx->fused_smem;
        const int rows = ctx->fused_blocks_rb > 0 ? moe::fused_rb_rows(H, ctx->F, T, ctx->ka, ctx->Et) : 0;
        if (rows > 0) {
            // row-block down mode: each down item sums y for its rows
            fp.rb_rows = rows;
            smem = moe::fused_rb_smem(H, ctx->F, T, ctx->ka, ctx->Et, rows, &fp.pre_off);
            if (T == 1 && d_logits && moe::fused_t1_ok(ctx->E, ctx->ka) && !sharded) {
                // one routed token: the gate, up and down table rows follow
                // (with the shared expert's column last)
                fp.tbl_off = (int)((smem + 15) / 16 * 16);
                smem = (size_t)fp.tbl_off + (size_t)24 * ctx->Et;
                fp.n_shared = ctx->shared ? 1 : 0;
                if (ctx->la_decode && !ctx->shared) {
                    const int L = ctx->cfg.n_layers, E = ctx->E;
                    if (layer + 1 < L && ctx->has_router[layer + 1]) {
                        fp.pr_w = ctx->d_router + (size_t)(layer + 1) * E * H;
                        fp.pr_b = ctx->d_rbias + (size_t)(layer + 1) * E;
                        fp.pr_tbl = ctx->d_tbl + (size_t)(layer + 1) * 3 * ctx->Et;
                        fp.pr_z = ctx->d_prz;
                        fp.pr_count = ctx->d_prcount;
                        fp.pr_flag = ctx->d_prcount + 1;
                        fp.pr_set = ctx->d_prset + (size_t)(layer + 1) * ctx->k;
                        fp.pr_stats = ctx->d_prstats;
                        fp.pr_blob = ctx->blob;
                    }
                    if (layer > 0 && ctx->has_router[layer]) {
                        fp.pr_mine = ctx->d_prset + (size_t)layer * ctx->k;
                        fp.pr_stats = ctx->d_prstats;
                    }
                }
            }
            items = std::max(U * (ctx->F / 32), H / rows);
            grid = std::min(items, ctx->fused_blocks_rb);
            // the lookahead predictor takes up to 7 experts per CTA (warps 1..7)
            if (fp.pr_w && 7 * grid < ctx->E) fp.pr_w = nullptr;
        }
        const cudaEvent_t *ev = nullptr;
        if (ctx->timing) {
            ev = ctx->tev.data() + 4 * (size_t)layer;
            ctx->tev_used[layer] = 1;
        }
        rc = moe::launch_fused(fp, grid, smem, st, ev);
        if (rc) return fail(ctx, MOE_ERR_CUDA, std::string("fused launch: ") + cudaGetErrorString((cudaError_t)rc));
        ctx->last_T = T;
        return MOE_OK;
    }
    if (!small) rc = moe::launch_quantize(d_x, T * (H / 32), ctx->xq, ctx->xds, ctx->n_sm, st);
    if (rc) return fail(ctx, MOE_ERR_CUDA, "quantize launch failed");
    moe::PlanParams pp{};
    pp.x = d_x;
    pp.xq = ctx->xq;
    pp.xds = ctx->xds;
    pp.idx = d_idx;
    pp.n_uniq = p_n_uniq(ctx);
    pp.uniq_e = p_uniq_e(ctx);
    pp.uniq_off = p_uniq_off(ctx);
    pp.assign = p_assign(ctx);
    pp.error = ctx->d_error;
    pp.T = T;
    pp.k = ctx->ka;
    pp.E = ctx->Et;
    pp.e_base = ctx->e_base;
    pp.E_route = sharded ? ctx->E_route : ctx->Et;
    pp.H = H;
    pp.quantize_x = small ? 1 : 0;
    rc = moe::launch_plan(pp, st);
    if (rc) return fail(ctx, MOE_ERR_CUDA, std::string("plan launch: ") + cudaGetErrorString((cudaError_t)rc));

    if (!small && ctx->gemm_ok) {
        // prefill: grouped tensor-core GEMM over tokens sorted by expert
        const int Umax = std::min(ctx->M * ctx->ka, ctx->Et);
        moe::PrefillLaunch L{};
        L.tiling.cv = gp.cv;
        L.tiling.n_uniq = gp.n_uniq;
        L.tiling.uniq_e = gp.uniq_e;
        L.tiling.uniq_off = gp.uniq_off;
        L.tiling.tile_off_gu = ctx->tile_off;
        L.tiling.tile_off_dn = ctx->tile_off + Umax + 1;
        L.tiling.rec_gu = ctx->tile_rec;
        L.tiling.rec_dn = ctx->tile_rec + ctx->cap_gu;
        L.tiling.cap_gu = ctx->cap_gu;
        L.tiling.cap_dn = ctx->cap_dn;
        L.tiling.tid0 = layer * 3;
        L.tiling.n_tokens = T;
        L.tiling.rt_gu = (ctx->F + moe::gemm_rows_per_tile(true) - 1) / moe::gemm_rows_per_tile(true);
        L.tiling.bn_gu = moe::gemm_bn(true);
        L.tiling.rt_dn = (ctx->H + moe::gemm_rows_per_tile(false) - 1) / moe::gemm_rows_per_tile(false);
        L.tiling.bn_dn = moe::gemm_bn(false);
        moe::GemmParams g{};
        g.n_uniq = gp.n_uniq;
        g.uniq_e = gp.uniq_e;
        g.uniq_off = gp.uniq_off;
        g.assign = gp.assign;
        g.A = A;
        g.A_pad = ctx->A_pad;
        g.k = ctx->ka;
        g.F_out = ctx->F;
        g.error = ctx->d_error;
        L.gu = g;
        L.gu.tile_off = L.tiling.tile_off_gu;
        L.gu.tile_rec = L.tiling.rec_gu;
        // with pool slots lent to this prompt pass, the layer's cold expert
        // tensors are staged there once and read from HBM by the GEMMs
        const uint64_t *rows = ctx->d_tbl + (size_t)(layer * 3) * ctx->Et;
        const int pb = layer & 1;
        const bool prefetched = ctx->lookahead && ctx->pf_layer[pb] == layer;
        if (prefetched) {
            // this layer's cold experts were uploaded a layer ahead: read them
            // from the prefetch buffer (entries rebuilt from the live table)
            CK(cudaStreamWaitEvent(st, ctx->ev_pf[pb], 0));
            rc = moe::launch_prefetch_table(rows, ctx->d_pfmap[pb], ctx->pf_buf[pb], ctx->pf_cap, ctx->stride, ctx->Et,
                                            ctx->etbl, st);
            if (rc) return fail(ctx, MOE_ERR_CUDA, "prefetch table launch failed");
            rows = ctx->etbl;
        } else if (ctx->n_lent > 0) {
            const int nt = ctx->n_tensors, G = nt * ctx->spt;
            moe::StageParams sp{};
            sp.tbl = ctx->d_tbl;
            sp.etbl = ctx->etbl;
            sp.n_uniq = gp.n_uniq;
            sp.uniq_e = gp.uniq_e;
            sp.jobs = ctx->stage_jobs;
            sp.n_jobs = ctx->stage_n;
            sp.slot_base = (uint64_t)(uintptr_t)(ctx->arena + (size_t)(G - ctx->n_lent) * ctx->stride);
            sp.slot_stride = ctx->stride;
            sp.n_slots = std::min(ctx->n_lent, ctx->stage_cap);
            sp.tid0 = layer * 3;
            sp.E = ctx->Et;
            rc = moe::launch_stage(sp, ctx->blob, ctx->n_sm, st);
            if (rc) return fail(ctx, MOE_ERR_CUDA, "stage launch failed");
            rows = ctx->etbl;
        }
        L.gu.tbl[0] = rows + 0 * (size_t)ctx->Et;
        L.gu.tbl[1] = rows + 1 * (size_t)ctx->Et;
        L.gu.a_scaleT = ctx->xdT;
        L.gu.rows = ctx->F;
        L.gu.K = H;
        L.gu.hq16 = ctx->hq16;
        L.gu.hdT = ctx->hdT;
        L.gu.hq = ctx->hq;
        L.gu.hds = ctx->hds;
        L.dn = g;
        L.dn.tile_off = L.tiling.tile_off_dn;
        L.dn.tile_rec = L.tiling.rec_dn;
        L.dn.tbl[0] = rows + 2 * (size_t)ctx->Et;
        L.dn.tbl[1] = nullptr;
        L.dn.a_scaleT = ctx->hdT;
        L.dn.rows = H;
        L.dn.K = ctx->F;
        L.dn.o = ctx->o;
        L.tm_x = ctx->tm_x;
        L.tm_h = ctx->tm_h;
        L.xq = ctx->xq;
        L.xds = ctx->xds;
        L.xs16 = ctx->xs16;
        L.xdT = ctx->xdT;
        L.w = d_w;
        L.y = d_y;
        L.T = T;
        L.idx = d_idx;
        L.e_base = ctx->e_base;
        L.E = ctx->Et;
        L.k = ctx->ka;
        L.H = H;
        L.n_sm = ctx->n_sm;
        const cudaEvent_t *pev = nullptr;
        if (ctx->timing) {
            pev = ctx->tev.data() + 4 * (size_t)layer;
            ctx->tev_used[layer] = 1;
        }
        rc = moe::launch_prefill(L, st, pev);
        if (rc) return fail(ctx, MOE_ERR_CUDA, std::string("prefill launch: ") + cudaGetErrorString((cudaError_t)rc));
        ctx->last_T = T;
        if (prefetched) {
            CK(cudaEventRecord(ctx->ev_pf_free[pb], st));  // the buffer may be refilled after this layer
            ctx->pf_layer[pb] = -1;
        }
        if (ctx->lookahead) {
            // the next layer's cold experts, uploaded while this layer computes
            rc = prefetch_layer(ctx, (layer + 1) % ctx->cfg.n_layers);
            if (rc) return rc;
        }
        return MOE_OK;
    }
    int max_gu = U * (ctx->F / 32), max_dn = U * ctx->n_counters;
    const cudaEvent_t *ev = nullptr;
    if (ctx->timing) {
        ev = ctx->tev.data() + 4 * (size_t)layer;
        ctx->tev_used[layer] = 1;
    }
    rc = moe::launch_gemv(gp, std::min(max_gu, ctx->grid_gu), std::min(max_dn, ctx->grid_dn), st, ev);
    if (rc) return fail(ctx, MOE_ERR_CUDA, std::string("gemv launch: ") + cudaGetErrorString((cudaError_t)rc));
    ctx->last_T = T;
    return MOE_OK;
}

int cache_step(moe_ctx *ctx, int n_tokens) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (n_tokens < 0) return fail(ctx, MOE_ERR_ARG, "cache_step: n_tokens < 0");
    CK(cudaSetDevice(ctx->dev));
    const int nt = ctx->n_tensors, spt = std::max(1, ctx->spt);
    const size_t hb = (size_t)ctx->hit_words;
    const size_t fast = std::min<size_t>(ctx->miss_cap, kStepKeys);
    // one read-back after the forwards issued so far: hit bitmap, miss count
    // and the first keys (the stamps are read only for tensors that admit)
    CK(cudaMemcpyAsync(ctx->h_step, ctx->d_stepbuf, sizeof(uint32_t) * (hb + 1 + fast), cudaMemcpyDeviceToHost,
                       ctx->stream));
    CK(cudaMemcpyAsync(ctx->h_err, ctx->d_error, sizeof(int), cudaMemcpyDeviceToHost, ctx->stream));
    CK(cudaEventRecord(ctx->ev_fwd, ctx->stream));
    int rc = wait_event(ctx, ctx->ev_fwd);
    if (rc) return rc;
    const uint32_t *hits = ctx->h_step;
    const size_t n_miss = std::min<size_t>(ctx->h_step[hb], ctx->miss_cap);
    std::vector<uint32_t> keys(n_miss);
    std::copy(ctx->h_step + hb + 1, ctx->h_step + hb + 1 + std::min(n_miss, fast), keys.begin());
    if (n_miss > fast)
        CK(cudaMemcpy(keys.data() + fast, ctx->d_misslog + 1 + fast, sizeof(uint32_t) * (n_miss - fast),
                      cudaMemcpyDeviceToHost));
    std::sort(keys.begin(), keys.end());
    keys.erase(std::unique(keys.begin(), keys.end()), keys.end());

    ctx->clock += (uint64_t)n_tokens;
    const uint64_t clk = ctx->clock;
    const uint32_t clk32 = (uint32_t)clk;
    // hits of the step: pool slots (with an owner) whose bit is set
    for (int w = 0; w < ctx->hit_words; ++w) {
        uint32_t m = hits[w];
        while (m) {
            const int b = w * 32 + __builtin_ctz(m);
            m &= m - 1;
            if (ctx->global_pool) {
                if (b < nt * spt && ctx->g_owner[b] >= 0) ctx->stats.hits++;
                continue;
            }
            const int tid = b / spt, sl = b % spt;
            if (tid >= nt || !ctx->t[tid].registered) continue;
            const TensorState &ts = ctx->t[tid];
            if (sl < ts.capacity && ts.owner[sl] >= 0) ctx->stats.hits++;
        }
    }
    ctx->stats.misses += keys.size();
    ctx->stats.steps++;
    for (uint32_t key : keys) {
        int tid = (int)(key >> 12);
        if (tid < nt && ctx->t[tid].registered) ctx->stats.cold_bytes += ctx->blob;
    }

    ctx->n_upd = 0;
    int fault = 0, swaps = 0, uploads = 0;
    std::vector<char> fresh;  // tensors whose stamp mirror was read back this step
    GlobalPick gs;            // shared pool: free slots and victims of this step
    if (ctx->n_lent == 0) {
        // the misses that qualify for admission (second sighting inside the
        // window; each key is unique and cold, so nothing below changes this)
        std::vector<int> q_tid;
        for (uint32_t key : keys) {
            const int tid = (int)(key >> 12), e = (int)(key & 0xfff);
            if (tid >= nt || e >= ctx->E || !ctx->t[tid].registered) continue;
            const int64_t ls = ctx->t[tid].last_seen[e];
            if (ls >= 0 && (int64_t)clk - ls < (int64_t)ctx->cfg.window_tokens) q_tid.push_back(tid);
        }
        gs.n_qualified = (int)q_tid.size();
        if (!ctx->global_pool && !q_tid.empty()) {
            // many admitting tensors: one read of every stamp beats one
            // round trip per tensor
            const size_t n_q = (size_t)(std::unique(q_tid.begin(), q_tid.end()) - q_tid.begin());
            if ((size_t)nt * spt * sizeof(uint32_t) <= n_q * 16384) {
                CK(cudaMemcpy(ctx->h_stamps, ctx->d_stamps, sizeof(uint32_t) * (size_t)nt * spt,
                              cudaMemcpyDeviceToHost));
                fresh.assign(nt, 1);
            }
        }
        for (uint32_t key : keys) {
            const int tid = (int)(key >> 12), e = (int)(key & 0xfff);
            if (tid >= nt || e >= ctx->E || !ctx->t[tid].registered) continue;
            TensorState &ts = ctx->t[tid];
            const int64_t ls = ts.last_seen[e];
            if (!(ls >= 0 && (int64_t)clk - ls < (int64_t)ctx->cfg.window_tokens)) {
                ts.last_seen[e] = (int32_t)clk;
                continue;
            }
            if (ctx->cfg.max_swaps_per_step && swaps >= ctx->cfg.max_swaps_per_step) continue;
            if (ctx->global_pool) {
                int rc2 = admit_global(ctx, gs, tid, e, clk, fault, uploads);
                if (rc2) return rc2;
                swaps += gs.took;
                continue;
            }
            if (fresh.empty()) fresh.assign(nt, 0);
            if (!fresh[tid]) {
                // the device stamps of this tensor (the stream is idle here),
                // before this step's first admission into it edits the mirror
                CK(cudaMemcpy(ctx->h_stamps + (size_t)tid * spt, ctx->d_stamps + (size_t)tid * spt,
                              sizeof(uint32_t) * spt, cudaMemcpyDeviceToHost));
                fresh[tid] = 1;
            }
            int slot = -1;
            for (int s = 0; s < ts.capacity; ++s)
                if (!ts.lent[s] && ts.owner[s] < 0) {
                    slot = s;
                    break;
                }
            if (slot < 0) {
                uint32_t best = 0;
                for (int s = 0; s < ts.capacity; ++s) {
                    if (ts.lent[s]) continue;
                    uint32_t st = ctx->h_stamps[(size_t)tid * spt + s];
                    if ((uint64_t)st < clk && (slot < 0 || st < best)) {
                        slot = s;
                        best = st;
                    }
                }
            }
            if (slot < 0) continue;
            const int victim = ts.owner[slot];
            if (victim >= 0) {
                set_entry(ctx, tid, victim, home_entry(ctx, tid, victim), -1);
                ts.last_seen[victim] = -1;
                ts.owner[slot] = -1;
                ctx->stats.evictions++;
            }
            swaps++;
            if (ctx->fail_nth > 0 && --ctx->fail_nth == 0) {
                // injected upload failure: the admission is rolled back, the
                // slot stays free and the expert stays cold with its sighting
                fault = 1;
                continue;
            }
            const uint64_t dst = pool_addr(ctx, tid, slot);
            rc = note_upload(ctx, tid / 3);
            if (rc) return rc;
            CK(cudaMemcpyAsync((void *)(uintptr_t)dst, ts.home + (size_t)e * ctx->stride, ctx->blob,
                               cudaMemcpyHostToDevice, ctx->up));
            uploads++;
            set_entry(ctx, tid, e, dst, slot);
            ts.owner[slot] = e;
            ts.last_seen[e] = -1;
            ctx->h_stamps[(size_t)tid * spt + slot] = clk32;
            push_upd(ctx, 2, (size_t)tid * spt + slot, clk32);
            ctx->stats.admissions++;
            ctx->stats.upload_bytes += ctx->blob;
        }
    }
    if (uploads && ctx->overlap) {
        // each layer's next forward waits for its own uploads
        rc = note_upload(ctx, -1, true);
        if (rc) return rc;
    } else if (uploads) {
        // the table entries of this step's admissions flip once their uploads
        // (side stream) are in
        CK(cudaEventRecord(ctx->ev_up, ctx->up));
        CK(cudaStreamWaitEvent(ctx->stream, ctx->ev_up, 0));
    }
    rc = publish(ctx, ctx->stream, true);
    if (rc) return rc;
    ctx->stats.clock = clk;
    if (fault) return fail(ctx, MOE_ERR_FAULT, "injected upload failure (admission rolled back)");
    if (*ctx->h_err) return device_fault(ctx);
    return MOE_OK;
}

int miss_drain(moe_ctx *ctx, uint32_t *host_out, size_t cap, size_t *n_out) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    CK(cudaSetDevice(ctx->dev));
    CK(cudaStreamSynchronize(ctx->stream));
    uint32_t cnt = 0;
    CK(cudaMemcpy(&cnt, ctx->d_misslog, sizeof(uint32_t), cudaMemcpyDeviceToHost));
    size_t n = std::min<size_t>(cnt, ctx->miss_cap);
    std::vector<uint32_t> keys(n);
    if (n) CK(cudaMemcpy(keys.data(), ctx->d_misslog + 1, sizeof(uint32_t) * n, cudaMemcpyDeviceToHost));
    std::sort(keys.begin(), keys.end());
    keys.erase(std::unique(keys.begin(), keys.end()), keys.end());
    if (n_out) *n_out = keys.size();
    if (keys.size() > cap) return fail(ctx, MOE_ERR_CAPACITY, "miss_drain: output too small");
    if (!keys.empty()) {
        if (!host_out) return fail(ctx, MOE_ERR_ARG, "miss_drain: null output");
        memcpy(host_out, keys.data(), sizeof(uint32_t) * keys.size());
    }
    CK(cudaMemsetAsync(ctx->d_bitmap, 0, sizeof(uint32_t) * (size_t)ctx->n_tensors * ctx->bitmap_words, ctx->stream));
    CK(cudaMemsetAsync(ctx->d_stepbuf, 0, sizeof(uint32_t) * ((size_t)ctx->hit_words + 1),
                       ctx->stream));
    CK(cudaMemcpyAsync(ctx->h_err, ctx->d_error, sizeof(int), cudaMemcpyDeviceToHost, ctx->stream));
    CK(cudaStreamSynchronize(ctx->stream));
    if (*ctx->h_err) return device_fault(ctx);
    return MOE_OK;
}

int moe_pool_borrow(moe_ctx *ctx, int n_slots, void **d_ws, size_t *bytes) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    const int nt = ctx->n_tensors, G = nt * ctx->spt;
    if (ctx->n_lent) return fail(ctx, MOE_ERR_STATE, "borrow: slots already lent");
    if (n_slots < 1 || n_slots > G) return fail(ctx, MOE_ERR_ARG, "borrow: n_slots out of range");
    CK(cudaSetDevice(ctx->dev));
    int rc = sync_all(ctx);
    if (rc) return rc;
    ctx->n_upd = 0;
    for (int g = G - n_slots; g < G; ++g) {
        if (ctx->global_pool) {
            const int key = ctx->g_owner[g];
            if (key >= 0) {
                const int vt = key >> 12, ve = key & 0xfff;
                set_entry(ctx, vt, ve, home_entry(ctx, vt, ve), -1);
                ctx->t[vt].last_seen[ve] = -1;
                ctx->g_owner[g] = -1;
                ctx->stats.evictions++;
            }
            ctx->g_lent[g] = 1;
            continue;
        }
        const int tid = g % nt, local = g / nt;
        TensorState &ts = ctx->t[tid];
        if (!ts.registered || local >= ts.capacity) continue;
        const int e = ts.owner[local];
        if (e >= 0) {
            set_entry(ctx, tid, e, home_entry(ctx, tid, e), -1);
            ts.last_seen[e] = -1;
            ts.owner[local] = -1;
            ctx->stats.evictions++;
        }
        ts.lent[local] = 1;
    }
    rc = publish(ctx, ctx->stream);
    if (rc) return rc;
    CK(cudaStreamSynchronize(ctx->stream));
    ctx->n_lent = n_slots;
    if (d_ws) *d_ws = ctx->arena + (size_t)(G - n_slots) * ctx->stride;
    if (bytes) *bytes = (size_t)n_slots * ctx->stride;
    return MOE_OK;
}

int moe_pool_return(moe_ctx *ctx) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (!ctx->n_lent) return fail(ctx, MOE_ERR_STATE, "return: nothing lent");
    CK(cudaSetDevice(ctx->dev));
    int rc = sync_all(ctx);
    if (rc) return rc;
    const int nt = ctx->n_tensors, G = nt * ctx->spt, E = ctx->E;
    const uint32_t clk32 = (uint32_t)ctx->clock;
    // prefill preheat: the prompt pass's assignments per (layer, expert)
    std::vector<uint32_t> use;
    if (ctx->preheat && ctx->d_use) {
        use.resize((size_t)ctx->cfg.n_layers * E);
        CK(cudaMemcpy(use.data(), ctx->d_use, sizeof(uint32_t) * use.size(), cudaMemcpyDeviceToHost));
        CK(cudaMemset(ctx->d_use, 0, sizeof(uint32_t) * use.size()));
    }
    // candidate order: prompt use count (desc), seed rank (asc), tensor (asc)
    auto better = [&](int ta, int ea, int tb, int eb) {
        const uint32_t ca = use.empty() ? 0 : use[(size_t)(ta / 3) * E + ea];
        const uint32_t cb = use.empty() ? 0 : use[(size_t)(tb / 3) * E + eb];
        if (ca != cb) return ca > cb;
        const int ra = ctx->t[ta].rank[ea], rb = ctx->t[tb].rank[eb];
        if (ra != rb) return ra < rb;
        return ta < tb;
    };
    auto fill = [&](int tid, int e, int slot, uint64_t dst) -> int {
        TensorState &ts = ctx->t[tid];
        CK(cudaMemcpyAsync((void *)(uintptr_t)dst, ts.home + (size_t)e * ctx->stride, ctx->blob,
                           cudaMemcpyHostToDevice, ctx->stream));
        set_entry(ctx, tid, e, dst, slot);
        ts.last_seen[e] = -1;
        push_upd(ctx, 2, (size_t)stamp_index(ctx, tid, slot), clk32);
        ctx->stats.upload_bytes += ctx->blob;
        return MOE_OK;
    };
    ctx->n_upd = 0;
    if (ctx->global_pool) {
        std::vector<std::pair<int, int>> cands;
        for (int tid = 0; tid < nt; ++tid) {
            if (!ctx->t[tid].registered) continue;
            for (int e = 0; e < E; ++e)
                if (ctx->t[tid].slot_of[e] < 0) cands.emplace_back(tid, e);
        }
        std::sort(cands.begin(), cands.end(), [&](const std::pair<int, int> &a, const std::pair<int, int> &b) {
            return better(a.first, a.second, b.first, b.second);
        });
        size_t pos = 0;
        for (int g = G - ctx->n_lent; g < G; ++g) {
            ctx->g_lent[g] = 0;
            if (!ctx->g_pool[g] || pos == cands.size()) continue;
            const int tid = cands[pos].first, e = cands[pos].second;
            ++pos;
            rc = fill(tid, e, g, slot_addr(ctx, (size_t)g));
            if (rc) return rc;
            ctx->g_owner[g] = (tid << 12) | e;
        }
    } else {
        for (int g = G - ctx->n_lent; g < G; ++g) {
            const int tid = g % nt, local = g / nt;
            TensorState &ts = ctx->t[tid];
            if (!ts.registered || local >= ts.capacity) continue;
            ts.lent[local] = 0;
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (ts.slot_of[e] < 0 && (best < 0 || better(tid, e, tid, best))) best = e;
            if (best < 0) continue;
            rc = fill(tid, best, local, pool_addr(ctx, tid, local));
            if (rc) return rc;
            ts.owner[local] = best;
        }
    }
    rc = publish(ctx, ctx->stream);
    if (rc) return rc;
    CK(cudaStreamSynchronize(ctx->stream));
    ctx->n_lent = 0;
    return MOE_OK;
}

int moe_set_upload_overlap(moe_ctx *ctx, int enable) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    CK(cudaSetDevice(ctx->dev));
    int rc = sync_all(ctx);
    if (rc) return rc;
    if (enable && ctx->ev_layer_up.empty()) {
        ctx->ev_layer_up.assign(ctx->cfg.n_layers, nullptr);
        for (cudaEvent_t &e : ctx->ev_layer_up) CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    }
    ctx->layer_pending.assign(ctx->cfg.n_layers, 0);
    ctx->cur_up_layer = -1;
    ctx->overlap = enable != 0;
    return MOE_OK;
}

int moe_set_global_pool(moe_ctx *ctx, int enable) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    for (const TensorState &ts : ctx->t)
        if (ts.registered) return fail(ctx, MOE_ERR_STATE, "global pool: choose the pool mode before registering");
    ctx->global_pool = enable != 0;
    const size_t G = (size_t)ctx->n_tensors * ctx->spt;
    ctx->g_owner.assign(ctx->global_pool ? G : 0, -1);
    ctx->g_pool.assign(ctx->global_pool ? G : 0, 0);
    ctx->g_lent.assign(ctx->global_pool ? G : 0, 0);
    return MOE_OK;
}

int moe_set_preheat(moe_ctx *ctx, int enable) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (ctx->n_lent) return fail(ctx, MOE_ERR_STATE, "preheat: switch it while no slot is lent");
    CK(cudaSetDevice(ctx->dev));
    if (enable && !ctx->d_use) {
        const size_t n = (size_t)ctx->cfg.n_layers * ctx->E;
        CK(cudaMalloc(&ctx->d_use, sizeof(uint32_t) * n));
        CK(cudaMemset(ctx->d_use, 0, sizeof(uint32_t) * n));
        CK(cudaDeviceSynchronize());
    }
    ctx->preheat = enable != 0;
    return MOE_OK;
}

int moe_cache_reset(moe_ctx *ctx, int global_pool) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (ctx->n_lent) return fail(ctx, MOE_ERR_STATE, "reset: slots are lent");
    CK(cudaSetDevice(ctx->dev));
    int rc = sync_all(ctx);
    if (rc) return rc;
    const int nt = ctx->n_tensors, E = ctx->E, spt = ctx->spt;
    const size_t G = (size_t)nt * spt;
    // what every arena slot holds now: slots that already hold their seed
    // expert are not uploaded again
    std::vector<int32_t> held(G, -1);
    for (int tid = 0; tid < nt; ++tid) {
        const TensorState &ts = ctx->t[tid];
        if (!ts.registered) continue;
        for (int e = 0; e < E; ++e) {
            const int s = ts.slot_of[e];
            if (s >= 0) held[ctx->global_pool ? (size_t)s : (size_t)s * nt + tid] = (tid << 12) | e;
        }
    }
    ctx->global_pool = global_pool != 0;
    ctx->g_owner.assign(ctx->global_pool ? G : 0, -1);
    ctx->g_pool.assign(ctx->global_pool ? G : 0, 0);
    ctx->g_lent.assign(ctx->global_pool ? G : 0, 0);
    const int Et = ctx->Et;
    std::vector<uint64_t> tbl((size_t)nt * Et, 0);
    std::vector<int32_t> dslot((size_t)nt * Et, -1);
    for (int tid = 0; tid < nt; ++tid)
        if (ctx->sh_blob[tid]) tbl[(size_t)tid * Et + E] = (uint64_t)(uintptr_t)ctx->sh_blob[tid];
    for (int tid = 0; tid < nt; ++tid) {
        TensorState &ts = ctx->t[tid];
        if (!ts.registered) continue;
        ts.slot_of.assign(E, -1);
        ts.owner.assign(spt, -1);
        ts.last_seen.assign(E, -1);
        ts.lent.assign(spt, 0);
        for (int e = 0; e < E; ++e) ts.tbl[e] = home_entry(ctx, tid, e);
        if (ctx->global_pool)
            for (int s = 0; s < ts.capacity; ++s) ctx->g_pool[(size_t)s * nt + tid] = 1;
        for (int s = 0; s < ts.n_seed; ++s) {
            const int e = ts.seed_order[s];
            const size_t g = (size_t)s * nt + tid;
            const uint64_t dst = slot_addr(ctx, g);
            if (held[g] != ((tid << 12) | e)) {
                CK(cudaMemcpyAsync((void *)(uintptr_t)dst, ts.home + (size_t)e * ctx->stride, ctx->blob,
                                   cudaMemcpyHostToDevice, ctx->stream));
                ctx->stats.upload_bytes += ctx->blob;
            }
            ts.tbl[e] = dst;
            if (ctx->global_pool) {
                ts.slot_of[e] = (int32_t)g;
                ctx->g_owner[g] = (tid << 12) | e;
            } else {
                ts.slot_of[e] = s;
                ts.owner[s] = e;
            }
        }
        for (int e = 0; e < E; ++e) {
            tbl[(size_t)tid * Et + e] = ts.tbl[e];
            dslot[(size_t)tid * Et + e] = stamp_index(ctx, tid, ts.slot_of[e]);
        }
    }
    CK(cudaMemcpyAsync(ctx->d_tbl, tbl.data(), sizeof(uint64_t) * tbl.size(), cudaMemcpyHostToDevice, ctx->stream));
    CK(cudaMemcpyAsync(ctx->d_slot, dslot.data(), sizeof(int32_t) * dslot.size(), cudaMemcpyHostToDevice,
                       ctx->stream));
    CK(cudaMemsetAsync(ctx->d_stamps, 0, sizeof(uint32_t) * (size_t)nt * std::max(1, spt), ctx->stream));
    CK(cudaMemsetAsync(ctx->d_bitmap, 0, sizeof(uint32_t) * (size_t)nt * ctx->bitmap_words, ctx->stream));
    CK(cudaMemsetAsync(ctx->d_stepbuf, 0, sizeof(uint32_t) * ((size_t)ctx->hit_words + 1), ctx->stream));
    CK(cudaMemsetAsync(ctx->d_clock, 0, sizeof(uint32_t), ctx->stream));
    CK(cudaMemsetAsync(ctx->d_cold, 0, sizeof(unsigned long long), ctx->stream));
    if (ctx->d_use)
        CK(cudaMemsetAsync(ctx->d_use, 0, sizeof(uint32_t) * (size_t)ctx->cfg.n_layers * E, ctx->stream));
    if (ctx->d_prstats) {
        CK(cudaMemsetAsync(ctx->d_prstats, 0, sizeof(unsigned long long) * 2, ctx->stream));
        CK(cudaMemsetAsync(ctx->d_prset, 0xff, sizeof(int32_t) * (size_t)ctx->cfg.n_layers * ctx->k, ctx->stream));
    }
    CK(cudaStreamSynchronize(ctx->stream));
    for (int b = 0; b < 2; ++b) {
        ctx->pf_layer[b] = -1;
        ctx->pf_map_pending[b] = false;
    }
    ctx->n_upd = 0;
    ctx->clock = 0;
    const uint64_t up = ctx->stats.upload_bytes;
    ctx->stats = moe_stats_t{};
    ctx->stats.upload_bytes = up;
    return MOE_OK;
}

int moe_pool_snapshot(moe_ctx *ctx, int32_t *owner_key, uint32_t *stamps) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    CK(cudaSetDevice(ctx->dev));
    int rc = sync_all(ctx);
    if (rc) return rc;
    const int nt = ctx->n_tensors, spt = ctx->spt, G = nt * spt;
    if (!G) return MOE_OK;
    std::vector<uint32_t> st((size_t)nt * std::max(1, spt));
    if (stamps) CK(cudaMemcpy(st.data(), ctx->d_stamps, sizeof(uint32_t) * st.size(), cudaMemcpyDeviceToHost));
    for (int g = 0; g < G; ++g) {
        const int tid = g % nt, local = g / nt;
        int key = -1;
        if (ctx->global_pool) {
            key = ctx->g_owner[g];
        } else {
            const TensorState &ts = ctx->t[tid];
            if (ts.registered && local < ts.capacity && !ts.lent[local] && ts.owner[local] >= 0)
                key = (tid << 12) | ts.owner[local];
        }
        if (owner_key) owner_key[g] = key;
        if (stamps) stamps[g] = st[ctx->global_pool ? (size_t)g : (size_t)tid * spt + local];
    }
    return MOE_OK;
}

int moe_set_lookahead(moe_ctx *ctx, int enable) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    CK(cudaSetDevice(ctx->dev));
    if (!enable) {
        ctx->lookahead = false;
        ctx->la_decode = false;
        return MOE_OK;
    }
    // decode: the layers whose routers are set are predicted a layer ahead
    ctx->la_decode = ctx->d_router != nullptr;
    if (!ctx->gemm_ok) {
        if (ctx->la_decode) return MOE_OK;  // no prompt-pass path: decode lookahead only
        return fail(ctx, MOE_ERR_STATE, "lookahead: no prompt-pass path and no router set");
    }
    int cap = 0;
    for (int tid = 0; tid < ctx->n_tensors; ++tid) {
        const TensorState &ts = ctx->t[tid];
        if (!ts.registered) return fail(ctx, MOE_ERR_STATE, "lookahead: register every tensor first");
        cap = std::max(cap, ctx->E - ts.capacity);
    }
    if (cap > ctx->pf_cap) {
        int rc = sync_all(ctx);
        if (rc) return rc;
        for (int b = 0; b < 2; ++b) {
            cudaFree(ctx->pf_buf[b]);
            ctx->pf_buf[b] = nullptr;
            CK(cudaMalloc(&ctx->pf_buf[b], (size_t)3 * cap * ctx->stride));
            ctx->pf_layer[b] = -1;
        }
        ctx->pf_cap = cap;
    }
    for (int b = 0; b < 2; ++b) {
        if (!ctx->d_pfmap[b]) CK(cudaMalloc(&ctx->d_pfmap[b], sizeof(int32_t) * 3 * ctx->Et));
        if (!ctx->h_pfmap[b]) CK(cudaHostAlloc(&ctx->h_pfmap[b], sizeof(int32_t) * 3 * ctx->Et, cudaHostAllocDefault));
        if (!ctx->ev_pf[b]) CK(cudaEventCreateWithFlags(&ctx->ev_pf[b], cudaEventDisableTiming));
        if (!ctx->ev_pf_free[b]) CK(cudaEventCreateWithFlags(&ctx->ev_pf_free[b], cudaEventDisableTiming));
    }
    ctx->lookahead = cap > 0;
    return MOE_OK;
}

int moe_set_router(moe_ctx *ctx, int layer, const float *host_w, const float *host_b) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (layer < 0 || layer >= ctx->cfg.n_layers || !host_w)
        return fail(ctx, MOE_ERR_ARG, "set_router: bad layer or null router");
    if (ctx->H % 8) return fail(ctx, MOE_ERR_ARG, "set_router: hidden must be a multiple of 8");
    CK(cudaSetDevice(ctx->dev));
    const int L = ctx->cfg.n_layers, E = ctx->E, H = ctx->H;
    if (!ctx->d_router) {
        int rc = sync_all(ctx);
        if (rc) return rc;
        if (cudaMalloc(&ctx->d_router, sizeof(__nv_bfloat16) * (size_t)L * E * H) != cudaSuccess ||
            cudaMalloc(&ctx->d_rbias, sizeof(float) * (size_t)L * E) != cudaSuccess ||
            cudaMalloc(&ctx->d_prz, sizeof(float) * E) != cudaSuccess ||
            cudaMalloc(&ctx->d_prcount, sizeof(unsigned) * 2) != cudaSuccess ||
            cudaMalloc(&ctx->d_prset, sizeof(int32_t) * (size_t)L * ctx->k) != cudaSuccess ||
            cudaMalloc(&ctx->d_prstats, sizeof(unsigned long long) * 2) != cudaSuccess) {
            cudaFree(ctx->d_router);
            cudaFree(ctx->d_rbias);
            cudaFree(ctx->d_prz);
            cudaFree(ctx->d_prcount);
            cudaFree(ctx->d_prset);
            cudaFree(ctx->d_prstats);
            ctx->d_router = nullptr;
            ctx->d_rbias = ctx->d_prz = nullptr;
            ctx->d_prcount = nullptr;
            ctx->d_prset = nullptr;
            ctx->d_prstats = nullptr;
            return fail(ctx, MOE_ERR_OOM, "set_router: device allocation failed");
        }
        CK(cudaMemset(ctx->d_prcount, 0, sizeof(unsigned) * 2));
        CK(cudaMemset(ctx->d_prset, 0xff, sizeof(int32_t) * (size_t)L * ctx->k));
        CK(cudaMemset(ctx->d_prstats, 0, sizeof(unsigned long long) * 2));
        ctx->has_router.assign(L, 0);
    }
    std::vector<__nv_bfloat16> w((size_t)E * H);
    for (size_t i = 0; i < w.size(); ++i) w[i] = __float2bfloat16_rn(host_w[i]);
    std::vector<float> b(E, 0.0f);
    if (host_b) memcpy(b.data(), host_b, sizeof(float) * E);
    CK(cudaStreamSynchronize(ctx->stream));
    CK(cudaMemcpy(ctx->d_router + (size_t)layer * E * H, w.data(), sizeof(__nv_bfloat16) * w.size(),
                  cudaMemcpyHostToDevice));
    CK(cudaMemcpy(ctx->d_rbias + (size_t)layer * E, b.data(), sizeof(float) * E, cudaMemcpyHostToDevice));
    ctx->has_router[layer] = 1;
    return MOE_OK;
}

int moe_cache_snapshot(moe_ctx *ctx, int tensor_id, uint64_t *tbl, int32_t *slot_of, int32_t *last_seen,
                       int32_t *owner, uint32_t *stamps) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (tensor_id < 0 || tensor_id >= ctx->n_tensors || !ctx->t[tensor_id].registered)
        return fail(ctx, MOE_ERR_ARG, "snapshot: bad tensor id");
    CK(cudaSetDevice(ctx->dev));
    int rc = sync_all(ctx);
    if (rc) return rc;
    const TensorState &ts = ctx->t[tensor_id];
    const int E = ctx->E;
    if (tbl)
        CK(cudaMemcpy(tbl, ctx->d_tbl + (size_t)tensor_id * ctx->Et, sizeof(uint64_t) * E, cudaMemcpyDeviceToHost));
    if (slot_of) memcpy(slot_of, ts.slot_of.data(), sizeof(int32_t) * E);
    if (last_seen) memcpy(last_seen, ts.last_seen.data(), sizeof(int32_t) * E);
    if (ctx->global_pool) {
        // the tensor's home slots g = s * n_tensors + tensor_id of the shared pool
        const int nt = ctx->n_tensors;
        std::vector<uint32_t> st;
        if (stamps && ctx->spt) {
            st.resize((size_t)nt * ctx->spt);
            CK(cudaMemcpy(st.data(), ctx->d_stamps, sizeof(uint32_t) * st.size(), cudaMemcpyDeviceToHost));
        }
        for (int s = 0; s < ctx->spt; ++s) {
            const size_t g = (size_t)s * nt + tensor_id;
            const int key = ctx->g_owner[g];
            if (owner) owner[s] = (key >= 0 && (key >> 12) == tensor_id) ? (key & 0xfff) : -1;
            if (stamps) stamps[s] = st[g];
        }
        return MOE_OK;
    }
    if (owner)
        for (int s = 0; s < ctx->spt; ++s) owner[s] = ts.lent[s] ? -1 : ts.owner[s];
    if (stamps && ctx->spt)
        CK(cudaMemcpy(stamps, ctx->d_stamps + (size_t)tensor_id * ctx->spt, sizeof(uint32_t) * ctx->spt,
                      cudaMemcpyDeviceToHost));
    return MOE_OK;
}

int moe_cache_layout(moe_ctx *ctx, int tensor_id, uint64_t *pool_base, uint64_t *host_base, uint64_t *slot_bytes,
                     int32_t *n_tensors) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (tensor_id < 0 || tensor_id >= ctx->n_tensors) return fail(ctx, MOE_ERR_ARG, "layout: bad tensor id");
    if (pool_base) *pool_base = (uint64_t)(uintptr_t)ctx->arena;
    if (host_base) *host_base = ctx->t[tensor_id].home_dev;
    if (slot_bytes) *slot_bytes = ctx->stride;
    if (n_tensors) *n_tensors = ctx->n_tensors;
    return MOE_OK;
}

int moe_stats(moe_ctx *ctx, moe_stats_t *out) {
    if (!ctx || !out) return fail(ctx, MOE_ERR_ARG, "null argument");
    *out = ctx->stats;
    out->clock = ctx->clock;
    out->lookahead_predicted = out->lookahead_hits = 0;
    if (ctx->d_prstats) {
        CK(cudaSetDevice(ctx->dev));
        CK(cudaStreamSynchronize(ctx->stream));
        unsigned long long h[2] = {0, 0};
        CK(cudaMemcpy(h, ctx->d_prstats, sizeof(h), cudaMemcpyDeviceToHost));
        out->lookahead_predicted = h[0];
        out->lookahead_hits = h[1];
    }
    return MOE_OK;
}

const char *moe_last_error(moe_ctx *ctx) { return ctx ? ctx->err.c_str() : g_init_error.c_str(); }

void moe_destroy(moe_ctx *ctx) {
    if (!ctx) return;
    cudaSetDevice(ctx->dev);
    cudaStreamSynchronize(ctx->stream);
    if (ctx->up) cudaStreamSynchronize(ctx->up);
    for (auto &ts : ctx->t)
        if (ts.home) cudaFreeHost(ts.home);
    cudaFree(ctx->arena);
    cudaFree(ctx->d_tbl);
    cudaFree(ctx->d_slot);
    cudaFree(ctx->d_stamps);
    cudaFree(ctx->d_use);
    cudaFree(ctx->idx_a);
    cudaFree(ctx->w_a);
    for (uint8_t *b : ctx->sh_blob) cudaFree(b);
    cudaFree(ctx->d_bitmap);
    cudaFree(ctx->d_stepbuf);
    cudaFree(ctx->d_clock);
    cudaFree(ctx->d_cold);
    cudaFree(ctx->xq);
    cudaFree(ctx->xds);
    cudaFree(ctx->plan_i);
    cudaFree(ctx->d_error);
    cudaFree(ctx->hq);
    cudaFree(ctx->hds);
    cudaFree(ctx->o);
    cudaFree(ctx->counters);
    cudaFree(ctx->xs16);
    cudaFree(ctx->xdT);
    cudaFree(ctx->hq16);
    cudaFree(ctx->hdT);
    cudaFree(ctx->tile_off);
    cudaFree(ctx->tile_rec);
    cudaFree(ctx->done_gu);
    cudaFree(ctx->etbl);
    cudaFree(ctx->d_router);
    cudaFree(ctx->d_rbias);
    cudaFree(ctx->d_prz);
    cudaFree(ctx->d_prcount);
    cudaFree(ctx->d_prset);
    cudaFree(ctx->d_prstats);
    cudaFree(ctx->stage_jobs);
    cudaFree(ctx->stage_n);
    for (int b = 0; b < 2; ++b) {
        cudaFree(ctx->pf_buf[b]);
        cudaFree(ctx->d_pfmap[b]);
        if (ctx->h_pfmap[b]) cudaFreeHost(ctx->h_pfmap[b]);
        if (ctx->ev_pf[b]) cudaEventDestroy(ctx->ev_pf[b]);
        if (ctx->ev_pf_free[b]) cudaEventDestroy(ctx->ev_pf_free[b]);
    }
    if (ctx->h_stamps) cudaFreeHost(ctx->h_stamps);
    if (ctx->h_upd) cudaFreeHost(ctx->h_upd);
    if (ctx->h_step) cudaFreeHost(ctx->h_step);
    if (ctx->h_err) cudaFreeHost(ctx->h_err);
    for (cudaEvent_t e : ctx->tev) cudaEventDestroy(e);
    if (ctx->ev_fwd) cudaEventDestroy(ctx->ev_fwd);
    if (ctx->ev_up) cudaEventDestroy(ctx->ev_up);
    if (ctx->up) cudaStreamDestroy(ctx->up);
    for (cudaEvent_t e : ctx->ev_layer_up) cudaEventDestroy(e);
    delete ctx;
}

int moe_debug_block_dots(moe_ctx *ctx, int tensor_id, int expert, int row0, int n_rows, const int8_t *d_qa,
                         int32_t *d_out) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (tensor_id < 0 || tensor_id >= ctx->n_tensors || !ctx->t[tensor_id].registered || expert < 0 ||
        expert > ctx->E || (expert == ctx->E && !ctx->sh_blob[tensor_id]) || !d_qa || !d_out)
        return fail(ctx, MOE_ERR_ARG, "block_dots: bad arguments");
    const int kind = tensor_id % 3;
    const int rows = kind == 2 ? ctx->H : ctx->F, cols = kind == 2 ? ctx->F : ctx->H;
    if (row0 < 0 || n_rows < 0 || row0 + n_rows > rows) return fail(ctx, MOE_ERR_ARG, "block_dots: bad rows");
    CK(cudaSetDevice(ctx->dev));
    int rc = sync_all(ctx);
    if (rc) return rc;
    const uint8_t *blob = expert == ctx->E ? ctx->sh_blob[tensor_id]
                                           : (const uint8_t *)(uintptr_t)(ctx->t[tensor_id].tbl[expert] & ~1ull);
    rc = moe::launch_block_dots(blob, ctx->fmt, rows, cols / 32, row0, n_rows, d_qa, d_out, ctx->stream);
    if (rc) return fail(ctx, MOE_ERR_CUDA, "block_dots launch failed");
    CK(cudaStreamSynchronize(ctx->stream));
    return MOE_OK;
}

int moe_debug_read(moe_ctx *ctx, int what, void *host_out, size_t bytes) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    if (ctx->last_T < 0) return fail(ctx, MOE_ERR_STATE, "debug_read: no forward yet");
    CK(cudaSetDevice(ctx->dev));
    CK(cudaStreamSynchronize(ctx->stream));
    const size_t T = ctx->last_T, A = T * ctx->ka;
    size_t need = 0;
    switch (what) {
        case 0: need = T * ctx->H; break;
        case 1: need = T * (ctx->H / 32) * 2; break;
        case 2: need = A * ctx->F; break;
        case 3: need = A * (ctx->F / 32) * 2; break;
        default: return fail(ctx, MOE_ERR_ARG, "debug_read: bad what");
    }
    if (bytes != need || !host_out) return fail(ctx, MOE_ERR_ARG, "debug_read: wrong size");
    if (what == 0 || what == 2) {
        CK(cudaMemcpy(host_out, what == 0 ? (void *)ctx->xq : (void *)ctx->hq, need, cudaMemcpyDeviceToHost));
        return MOE_OK;
    }
    const size_t n = need / 2;
    std::vector<BlockScale> tmp(n);
    CK(cudaMemcpy(tmp.data(), what == 1 ? ctx->xds : ctx->hds, sizeof(BlockScale) * n, cudaMemcpyDeviceToHost));
    uint16_t *o = (uint16_t *)host_out;
    for (size_t i = 0; i < n; ++i) o[i] = f32_to_half_bits(tmp[i].d);  // exact: d is a binary16 value
    return MOE_OK;
}

int moe_probe_host_read(const void *host_pinned, size_t bytes, int iters, double *gbs, double *copy_gbs) {
    moe_ctx *ctx = nullptr;
    if (!host_pinned || bytes < 16 || iters < 1 || !gbs) return fail(nullptr, MOE_ERR_ARG, "probe: bad arguments");
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, host_pinned) != cudaSuccess || at.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return fail(nullptr, MOE_ERR_NOT_PINNED, "probe: memory is not pinned host memory");
    }
    void *dptr = nullptr;
    CK(cudaHostGetDevicePointer(&dptr, (void *)host_pinned, 0));
    int dev = 0, n_sm = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
    uint32_t *sink = nullptr;
    CK(cudaMalloc(&sink, 4));
    cudaStream_t st;
    CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
    cudaEvent_t a, b;
    CK(cudaEventCreate(&a));
    CK(cudaEventCreate(&b));
    bytes &= ~(size_t)15;
    double best = 0;
    for (int i = 0; i < iters + 1; ++i) {
        CK(cudaEventRecord(a, st));
        moe::launch_stream_read(dptr, bytes, sink, n_sm, st);
        CK(cudaEventRecord(b, st));
        CK(cudaEventSynchronize(b));
        float ms = 0;
        CK(cudaEventElapsedTime(&ms, a, b));
        if (i > 0) best = std::max(best, bytes / (ms * 1e-3) / 1e9);
    }
    *gbs = best;
    if (copy_gbs) {
        size_t cb = std::min<size_t>(bytes, (size_t)1 << 30);
        void *dbuf = nullptr;
        CK(cudaMalloc(&dbuf, cb));
        double bc = 0;
        for (int i = 0; i < iters + 1; ++i) {
            CK(cudaEventRecord(a, st));
            CK(cudaMemcpyAsync(dbuf, host_pinned, cb, cudaMemcpyHostToDevice, st));
            CK(cudaEventRecord(b, st));
            CK(cudaEventSynchronize(b));
            float ms = 0;
            CK(cudaEventElapsedTime(&ms, a, b));
            if (i > 0) bc = std::max(bc, cb / (ms * 1e-3) / 1e9);
        }
        cudaFree(dbuf);
        *copy_gbs = bc;
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaStreamDestroy(st);
    cudaFree(sink);
    return MOE_OK;
}

int moe_debug_timing(moe_ctx *ctx, int enable) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    CK(cudaSetDevice(ctx->dev));
    if (enable && ctx->tev.empty()) {
        ctx->tev.resize(4 * (size_t)ctx->cfg.n_layers);
        for (auto &e : ctx->tev) CK(cudaEventCreate(&e));
        ctx->tev_used.assign(ctx->cfg.n_layers, 0);
    }
    ctx->timing = enable != 0;
    return MOE_OK;
}

int moe_debug_timing_read(moe_ctx *ctx, double *gate_up_ms, double *down_ms) {
    if (!ctx) return fail(nullptr, MOE_ERR_ARG, "null ctx");
    CK(cudaSetDevice(ctx->dev));
    CK(cudaStreamSynchronize(ctx->stream));
    for (int l = 0; l < ctx->cfg.n_layers; ++l) {
        float a = 0, b = 0;
        if (l < (int)ctx->tev_used.size() && ctx->tev_used[l]) {
            CK(cudaEventElapsedTime(&a, ctx->tev[4 * l], ctx->tev[4 * l + 1]));
            CK(cudaEventElapsedTime(&b, ctx->tev[4 * l + 2], ctx->tev[4 * l + 3]));
            ctx->tev_used[l] = 0;
        }
        if (gate_up_ms) gate_up_ms[l] = a;
        if (down_ms) down_ms[l] = b;
    }
    return MOE_OK;
}

int moe_debug_fail_upload(moe_ctx *ctx, int nth) {
    if (!ctx || nth < 0) return fail(ctx, MOE_ERR_ARG, "bad argument");
    ctx->fail_nth = nth;
    return MOE_OK;
}

int moe_debug_busy(moe_ctx *ctx, int microseconds) {
    if (!ctx || microseconds < 0 || microseconds > 2000000) return fail(ctx, MOE_ERR_ARG, "bad argument");
    CK(cudaSetDevice(ctx->dev));
    int rc = moe::launch_busy((unsigned long long)microseconds * 1000ull, ctx->stream);
    if (rc) return fail(ctx, MOE_ERR_CUDA, "busy launch failed");
    return MOE_OK;
}

}  // extern "C"
