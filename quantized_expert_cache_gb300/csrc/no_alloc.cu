// An allocation-free entry point for one routed-expert FFN layer.
//
// Some callers cannot allocate device memory at the point where they run a
// layer: processes whose device memory is fully reserved by an outside
// allocator, or embedded hosts that forbid cudaMalloc after start-up.
// moe_expert_ffn_noalloc serves them: it takes the caller's inputs, outputs
// and expert tables, and keeps every intermediate (quantized x and h, per-
// assignment outputs, arrival counters, a private miss log) in one file-scope
// device array of fixed size, so the call itself allocates nothing.
//
// The array lives as long as the library is loaded, once on every device
// that loads it (kNoAllocScratchBytes each).  Host code cannot use its name as
// a device address: the first call on a device looks its address up with
// cudaGetSymbolAddress (with that device current) and every later call on that
// device reuses it.  All calls share the array, so calls that overlap on the
// GPU (different streams, or different host threads) race on it.
//
// The kernel's error word sits at a fixed place, the first bytes of the
// array, so that moe_expert_ffn_noalloc_status can read what the most recent
// call left there without knowing that call's sizes.
#include "../../include/moe_cache.h"
#include "kernels.h"

#include <cstdio>
#include <mutex>
#include <string>

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace

namespace moe {
void set_context_free_error(const std::string &msg);  // shared with moe_last_error(NULL)
}

namespace {

constexpr size_t kErrWordBytes = 256;  // [0, 256): the error word of the most recent call

struct DevSetup {
    bool done = false;
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch
    int n_sm = 0;
    // kernel configuration of the last (hidden, ffn) seen on this device
    int cfg_h = 0, cfg_f = 0, bps = 0;
};
DevSetup g_dev[kMaxDevices];
std::mutex g_mu;

int fail(int code, const std::string &m) {
    moe::set_context_free_error(m);
    return code;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Carve the scratch array for one call; returns the bytes needed.
struct Carve {
    size_t off = 0;
    unsigned char *base = nullptr;
    template <class T>
    T *take(size_t count) {
        T *p = reinterpret_cast<T *>(base ? base + off : nullptr);
        off = align256(off + count * sizeof(T));
        return p;
    }
};

}  // namespace

extern "C" {

int moe_expert_ffn_noalloc(const float *d_x, int n_tokens, const int32_t *d_idx, const float *d_w,
                           const uint64_t *d_tbl, int hidden, int ffn, int n_experts, int top_k, float *d_y,
                           void *stream) {
    if (n_tokens < 0 || hidden <= 0 || hidden % 32 || ffn <= 0 || ffn % 32 || n_experts < 1 || n_experts > 4096 ||
        top_k < 1 || top_k > n_experts)
        return fail(MOE_ERR_ARG, "noalloc: bad sizes");
    if (n_tokens == 0) return MOE_OK;
    if (!d_x || !d_idx || !d_w || !d_tbl || !d_y) return fail(MOE_ERR_ARG, "noalloc: null pointer");
    const int A = n_tokens * top_k;
    const int down_rows = moe::down_rows_per_item(ffn);
    if (n_tokens > 32 || A > 256 || hidden % down_rows)
        return fail(MOE_ERR_ARG, "noalloc: needs n_tokens <= 32, n_tokens*top_k <= 256 and hidden a multiple of " +
                                     std::to_string(down_rows));
    const int E = n_experts, H = hidden, F = ffn, n_rb = H / down_rows;
    // scratch layout (sizes only first); the error word comes first
    Carve c;
    c.off = kErrWordBytes;
    auto layout = [&](Carve &cv, moe::FusedParams *fp) {
        uint32_t *bitmap = cv.take<uint32_t>((size_t)3 * ((E + 31) / 32));
        uint32_t *misslog = cv.take<uint32_t>(1 + (size_t)3 * E);
        uint32_t *clock = cv.take<uint32_t>(1);
        int32_t *slot = cv.take<int32_t>((size_t)3 * E);
        uint32_t *stamps = cv.take<uint32_t>(1);
        unsigned *done = cv.take<unsigned>((size_t)E + 1);
        unsigned *counters = cv.take<unsigned>((size_t)n_rb);
        int8_t *xq = cv.take<int8_t>((size_t)n_tokens * H);
        moe::BlockScale *xds = cv.take<moe::BlockScale>((size_t)n_tokens * (H / 32));
        int8_t *hq = cv.take<int8_t>((size_t)A * F);
        moe::BlockScale *hds = cv.take<moe::BlockScale>((size_t)A * (F / 32));
        float *o = cv.take<float>((size_t)A * H);
        if (fp) {
            moe::GemvParams &g = fp->g;
            g.cv.tbl = d_tbl;
            g.cv.slot = slot;
            g.cv.stamps = stamps;
            g.cv.miss_bitmap = bitmap;
            g.cv.miss_list = misslog + 1;
            g.cv.miss_count = misslog;
            g.cv.clock = clock;
            g.cv.cold_reads = nullptr;
            g.cv.E = E;
            g.cv.slots_per_tensor = 1;
            g.cv.bitmap_words = (E + 31) / 32;
            g.cv.miss_cap = 3 * E;
            g.cv.clock_tokens = n_tokens;
            g.tid_gate = 0;
            g.tid_up = 1;
            g.tid_down = 2;
            g.n_tokens = n_tokens;
            g.k = top_k;
            g.H = H;
            g.F = F;
            g.hq = hq;
            g.hds = hds;
            g.o = o;
            g.counters = counters;
            g.w = d_w;
            g.y = d_y;
            g.xq_out = xq;
            g.xds_out = xds;
            g.idx = d_idx;
            g.e_base = 0;
            fp->n_route = E;
            fp->x = d_x;
            fp->idx = d_idx;
            fp->done_gu = done;
            fp->exit_count = done + E;
            fp->error = reinterpret_cast<int *>(cv.base);
        }
        // [array start, xq) holds the error word and the small tables (zeroed
        // per call); slot is set to -1
        return std::make_pair(cv.base ? (size_t)((unsigned char *)slot - cv.base) : (size_t)0,
                              cv.base ? (size_t)((unsigned char *)xq - cv.base) : (size_t)0);
    };
    layout(c, nullptr);
    const size_t need = c.off;
    if (need > kNoAllocScratchBytes)
        return fail(MOE_ERR_CAPACITY, "noalloc: this call needs " + std::to_string(need) + " scratch bytes, above the " +
                                          std::to_string(kNoAllocScratchBytes) + "-byte maximum");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_CUDA, "noalloc: no current device");
    const size_t smem = moe::fused_smem_bytes(H, F);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        DevSetup &d = g_dev[dev];
        if (!d.done) {
            // once per device, with the device current: the array's address
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p)
                return fail(MOE_ERR_CUDA, std::string("noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
            e = cudaDeviceGetAttribute(&d.n_sm, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "noalloc: device attribute query failed");
            d.scratch = (unsigned char *)p;
            d.done = true;
        }
    }
    DevSetup &d = g_dev[dev];
    int bps = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (d.cfg_h != H || d.cfg_f != F) {
            e = (cudaError_t)moe::fused_configure(F, smem, &d.bps);
            if (e != cudaSuccess || d.bps < 1) {
                d.cfg_h = d.cfg_f = 0;
                return fail(MOE_ERR_CUDA, "noalloc: kernel configuration failed");
            }
            d.cfg_h = H;
            d.cfg_f = F;
        }
        bps = d.bps;
    }
    moe::FusedParams fp{};
    Carve cv;
    cv.base = d.scratch;
    cv.off = kErrWordBytes;
    const auto offs = layout(cv, &fp);
    cudaStream_t st = (cudaStream_t)stream;
    // the error word, the counters, the miss log and the clock must start
    // at zero, the slot table at -1 (so no stamp is written); the large
    // buffers are written before they are read
    e = cudaMemsetAsync(d.scratch, 0, offs.second, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(d.scratch + offs.first, 0xff, (size_t)3 * E * sizeof(int32_t), st);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, std::string("noalloc: memset: ") + cudaGetErrorString(e));
    const int U = A < E ? A : E;
    const int items = U * ((F / 32) > n_rb ? (F / 32) : n_rb);
    const int grid = items < bps * d.n_sm ? items : bps * d.n_sm;
    int rc = moe::launch_fused(fp, grid, smem, st, nullptr);
    if (rc) return fail(MOE_ERR_CUDA, std::string("noalloc: launch: ") + cudaGetErrorString((cudaError_t)rc));
    return MOE_OK;
}

int moe_expert_ffn_noalloc_status(void *stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_CUDA, "noalloc status: no current device");
    unsigned char *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev[dev].done) scratch = g_dev[dev].scratch;
    }
    if (!scratch) return MOE_OK;  // no call has run on this device
    cudaStream_t st = (cudaStream_t)stream;
    int word = 0;
    e = cudaMemcpyAsync(&word, scratch, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, std::string("noalloc status: ") + cudaGetErrorString(e));
    if (word == 0) return MOE_OK;
    std::string m = "noalloc: the kernel reported error bits " + std::to_string(word) + ":";
    if (word & 1) m += " an expert id outside [0, n_experts) was read as expert 0;";
    if (word & 6) m += " a bounded wait expired and its work item was skipped;";
    return fail(MOE_ERR_FAULT, m + " the output of that call is not valid");
}

}  // extern "C"
