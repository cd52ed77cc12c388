// verkv_api.cu -- the C ABI of libverkv: argument checks, workspace carve-up, stream and event
// orchestration, and the host side of the fetch ("Verify Before You Fetch": the abstract page's
// GPU-resident pivotal tokens and sketch with the complete cache in CPU memory; summary page,
// KVFETCH steps 1-5).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <condition_variable>
#include <functional>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "verkv_internal.h"

using namespace verkv;

namespace {

// An NVTX range for the lifetime of the object: each stage of the hot path shows up by name on a
// profiler's timeline (the calls cost nothing without a tool attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Alignment the kernels rely on: bf16 rows and queries are read in 16-byte vectors or bulk
// copies; every other array is read and written in 4-byte words.  A null pointer passes (the
// null checks are separate).
bool bad16(const void *p) { return ((uintptr_t)p & 15u) != 0; }
bool bad4(const void *p) { return ((uintptr_t)p & 3u) != 0; }

struct Layout {
    size_t err, flc, nacc, rmask, rnext, scores, qstats, F, slb, fids, fcounts, staging, part_piv, part_fet, total;
    int W, units_layer, qh_layer, max_piv, max_fet, dense_chunks;
};

// MEMCPY-mode staging (page-locked on the host and its device copy): a header of the layer
// units' first staged rows (int64, 256-byte aligned), then the fetched rows of every unit,
// contiguous and unit by unit, so that one copy moves a whole fetch.
size_t staging_header(int units_layer) { return align256((size_t)units_layer * 8); }
size_t staging_bytes(int units_layer, size_t n, size_t d) {
    return staging_header(units_layer) + (size_t)units_layer * n * 4 * d;
}

bool valid_shape(const verkv_shape *s) {
    if (!s) return false;
    const int G = s->q_per_kv;
    return s->batch >= 1 && s->layers >= 1 && s->kv_heads >= 1 &&
           (G == 1 || G == 2 || G == 4 || G == 8) && (s->head_dim == 64 || s->head_dim == 128) &&
           s->n >= 1 && s->n <= 131072 && s->cap >= 1 && s->cap <= s->n &&
           (int64_t)s->batch * s->layers * s->kv_heads <= (1 << 24);
}

bool make_layout(const verkv_shape *s, Layout &L) {
    if (!valid_shape(s)) return false;
    const size_t n = (size_t)s->n, d = (size_t)s->head_dim, G = (size_t)s->q_per_kv;
    L.W = (s->n + 31) / 32;
    L.units_layer = s->batch * s->kv_heads;
    L.qh_layer = L.units_layer * s->q_per_kv;
    L.max_piv = (s->cap + PIV_ITEM_ROWS - 1) / PIV_ITEM_ROWS;
    L.max_fet = (s->n + FET_RANGE - 1) / FET_RANGE;
    L.dense_chunks = (s->n + PART_ROWS - 1) / PART_ROWS;  // >= max_fet: sizes the shared buffer
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    L.err = take(256);
    L.flc = take((size_t)L.units_layer * 4);
    L.nacc = take((size_t)L.qh_layer * 4);
    L.rmask = take((size_t)L.units_layer * RMASK_W * 4);
    L.rnext = take(4);
    L.scores = take((size_t)L.qh_layer * n * 4);
    L.qstats = take((size_t)L.qh_layer * sizeof(verkv_head_stats));
    L.F = take((size_t)L.qh_layer * L.W * 4);
    L.slb = take((size_t)L.units_layer * L.W * 4);
    L.fids = take((size_t)L.units_layer * n * 4);
    L.fcounts = take((size_t)L.units_layer * 4);
    L.staging = take(staging_bytes(L.units_layer, n, d));
    L.part_piv = take((size_t)L.units_layer * L.max_piv * G * (d + 2) * 4);
    L.part_fet = take((size_t)L.units_layer * L.dense_chunks * G * (d + 2) * 4);
    L.total = off;
    return true;
}

// A small fixed pool of host threads for the MEMCPY-mode gather.
class Pool {
  public:
    explicit Pool(int nthreads) {
        for (int i = 0; i < nthreads; ++i) workers_.emplace_back([this, i] { loop(i); });
    }
    ~Pool() {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto &t : workers_) t.join();
    }
    int size() const { return (int)workers_.size(); }
    // Runs fn(worker_index) on every worker and waits for all of them.
    void run(const std::function<void(int)> &fn) {
        std::unique_lock<std::mutex> lk(mu_);
        job_ = &fn;
        pending_ = (int)workers_.size();
        ++generation_;
        cv_.notify_all();
        done_cv_.wait(lk, [this] { return pending_ == 0; });
        job_ = nullptr;
    }

  private:
    void loop(int idx) {
        uint64_t seen = 0;
        for (;;) {
            const std::function<void(int)> *job;
            {
                std::unique_lock<std::mutex> lk(mu_);
                cv_.wait(lk, [&] { return stop_ || generation_ != seen; });
                if (stop_) return;
                seen = generation_;
                job = job_;
            }
            (*job)(idx);
            {
                std::lock_guard<std::mutex> g(mu_);
                if (--pending_ == 0) done_cv_.notify_all();
            }
        }
    }
    std::vector<std::thread> workers_;
    std::mutex mu_;
    std::condition_variable cv_, done_cv_;
    const std::function<void(int)> *job_ = nullptr;
    int pending_ = 0;
    uint64_t generation_ = 0;
    bool stop_ = false;
};

}  // namespace

namespace verkv {

cudaError_t ensure_smem(const void *func, size_t bytes) {
    struct Entry {
        int device;
        const void *func;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(mu);
    for (Entry &x : done) {
        if (x.device == dev && x.func == func) {
            if (x.bytes >= bytes) return cudaSuccess;
            e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e == cudaSuccess) x.bytes = bytes;
            return e;
        }
    }
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done.push_back({dev, func, bytes});
    return e;
}

}  // namespace verkv

struct verkv_ctx {
    int device = 0;
    int sms = 0;
    cudaStream_t main = nullptr, side = nullptr;
    cudaEvent_t e_sel = nullptr, e_fetch = nullptr;
    verkv_shape sh{};
    Layout L{};
    unsigned char *ws = nullptr;
    uint32_t *err = nullptr;
    float *scores = nullptr;
    verkv_head_stats *qstats = nullptr;
    uint32_t *F = nullptr;
    int32_t *fids = nullptr, *fcounts = nullptr;
    int32_t *flc = nullptr;  // per-KV-head completion counters of the certify kernel's fetch list
    int32_t *nacc = nullptr; // per-query-head n_fetch accumulators of the zero-copy refine
    uint32_t *rmask = nullptr; // per-KV-head masks of fetched-row ranges holding rows
    int32_t *rnext = nullptr;  // the zero-copy refine's item counter
    uint32_t *slb = nullptr; // per-KV-head shortlist bitmaps
    int shortlist = 0;       // shortlist size per KV head; 0: every token of L may be fetched
    bool shortlisted = false;  // the last attend built shortlists
    uint16_t *staging = nullptr;
    float *part_piv = nullptr, *part_fet = nullptr;
    int fetch_mode = VERKV_FETCH_ZEROCOPY;
    bool fetch_keys = false;  // move K rows too, although the exact sketch holds every key
    // MEMCPY mode
    unsigned char *host_staging = nullptr;
    int32_t *host_ids = nullptr, *host_counts = nullptr;     // mapped page-locked
    int32_t *host_ids_dev = nullptr, *host_counts_dev = nullptr;
    Pool *pool = nullptr;
    // The preceding attend
    bool pending = false;
    bool attended = false;
    int layer = 0;
    verkv_pivotal piv{};
    const int32_t *user_ids = nullptr, *user_counts = nullptr;
    const void *q = nullptr;
    const void *sketch = nullptr;
    bool sketch_exact = true;  // format of the preceding attend's sketch
    std::string last_error;
    // Failure injection (verkv_test_inject)
    int64_t inject_copy_fail = 0;    // fetch copies still to fail on the host
    int beta_maxit = 0;              // 0: the kernel's default cap
    int sel_gather = 1;              // the select's gathered finish (clusters of 1 and 4)
    int seq0 = 0;                    // Philox sequence index of this context's first sequence
    int64_t score_stall_ns = 0;      // > 0: the next attend's scoring kernel stalls one stage
    // Measurement
    int64_t launches[VERKV_K_COUNT] = {};
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_pool;
    size_t prof_used = 0;
    struct Rec {
        int kernel;
        cudaEvent_t a, b;
    };
    std::vector<Rec> prof_recs;
};

namespace {

verkv_status fail(verkv_ctx *c, verkv_status st, const std::string &msg) {
    if (c) c->last_error = msg;
    return st;
}

verkv_status cuda_fail(verkv_ctx *c, cudaError_t e, const char *where) {
    return fail(c, VERKV_ECUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

#define VERKV_CUDA(call, where)                              \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, where); \
    } while (0)

cudaEvent_t prof_event(verkv_ctx *ctx) {
    if (ctx->prof_used == ctx->prof_pool.size()) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        ctx->prof_pool.push_back(e);
    }
    return ctx->prof_pool[ctx->prof_used++];
}

// Launch with accounting: counts the launch and, when profiling, brackets it with events.
template <typename F>
cudaError_t tracked(verkv_ctx *ctx, int kernel, cudaStream_t s, F &&launch) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (ctx->prof_on && (a = prof_event(ctx)) != nullptr) cudaEventRecord(a, s);
    const cudaError_t e = launch();
    if (e != cudaSuccess) return e;
    ctx->launches[kernel]++;
    if (a && (b = prof_event(ctx)) != nullptr) {
        cudaEventRecord(b, s);
        ctx->prof_recs.push_back({kernel, a, b});
    }
    return cudaSuccess;
}

LayerIdx layer_idx(const verkv_ctx *ctx, int layer) {
    LayerIdx li;
    li.layers = ctx->sh.layers;
    li.layer = layer;
    li.kv_heads = ctx->sh.kv_heads;
    li.G = ctx->sh.q_per_kv;
    return li;
}

// Arguments of the pivotal partial sums of one layer call.
PartialArgs pivotal_args(const verkv_ctx *ctx, const verkv_pivotal &piv, const void *q,
                         const LayerIdx &li, bool sketch_exact) {
    const int d = ctx->sh.head_dim;
    PartialArgs pa{};
    pa.rows = (const uint16_t *)piv.kv;
    pa.ids = piv.ids;
    pa.pr = piv.r;
    pa.count = piv.count;
    pa.q = (const uint16_t *)q;
    pa.F = ctx->F;
    pa.qstats = ctx->qstats;
    pa.scores = ctx->scores;
    pa.part = ctx->part_piv;
    pa.err = ctx->err;
    pa.row_stride = ctx->sh.cap;
    pa.units_total = ctx->sh.batch * ctx->sh.layers * ctx->sh.kv_heads;
    pa.max_chunks = ctx->L.max_piv;
    pa.n = ctx->sh.n;
    pa.W = ctx->L.W;
    pa.d = d;
    pa.mode = ROWS_PIVOTAL;
    pa.keys = nullptr;
    pa.row16 = d / 4;
    pa.voff16 = d / 8;
    pa.scale = (float)(1.0 / sqrt((double)d));
    pa.li = li;
    pa.sketch_logits = sketch_exact ? 0 : 1;
    return pa;
}

// One host-to-device copy of the MEMCPY-mode fetch, on the side stream (or an injected failure).
cudaError_t copy_rows(verkv_ctx *ctx, void *dst, const void *src, size_t bytes) {
    if (ctx->inject_copy_fail > 0) {
        --ctx->inject_copy_fail;
        return cudaErrorInvalidValue;
    }
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, ctx->side);
}

}  // namespace

extern "C" {

const char *verkv_status_string(int st) {
    switch (st) {
        case VERKV_OK: return "VERKV_OK";
        case VERKV_EINVAL: return "VERKV_EINVAL";
        case VERKV_EBUDGET: return "VERKV_EBUDGET";
        case VERKV_ECAPACITY: return "VERKV_ECAPACITY";
        case VERKV_ENOCONVERGE: return "VERKV_ENOCONVERGE";
        case VERKV_ECUDA: return "VERKV_ECUDA";
        case VERKV_ECOPY: return "VERKV_ECOPY";
        case VERKV_ETIMEOUT: return "VERKV_ETIMEOUT";
        case VERKV_ESTATE: return "VERKV_ESTATE";
        case VERKV_ETOOLARGE: return "VERKV_ETOOLARGE";
        default: return "VERKV_UNKNOWN";
    }
}

size_t verkv_sketch_bytes(const verkv_shape *shape, int32_t format) {
    if (!valid_shape(shape)) return 0;
    const size_t rows = (size_t)shape->batch * shape->layers * shape->kv_heads * shape->n;
    if (format == VERKV_SKETCH_EXACT) return rows * 2 * shape->head_dim;
    if (format == VERKV_SKETCH_Q2) return rows * q2_row_bytes(shape->head_dim);
    return 0;
}

size_t verkv_workspace_size(const verkv_shape *shape) {
    Layout L;
    return make_layout(shape, L) ? L.total : 0;
}

verkv_status verkv_create(verkv_ctx **out, int device, void *stream, const verkv_shape *shape,
                          void *workspace, size_t workspace_bytes) {
    if (!out) return VERKV_EINVAL;
    *out = nullptr;
    Layout L;
    if (!make_layout(shape, L)) return VERKV_EINVAL;
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u)) return VERKV_EINVAL;
    verkv_ctx *ctx = new verkv_ctx();
    ctx->device = device;
    ctx->sh = *shape;
    ctx->L = L;
    ctx->main = (cudaStream_t)stream;
    ctx->ws = (unsigned char *)workspace;
    cudaError_t e = cudaSetDevice(device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ctx->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->e_sel, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->e_fetch, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        verkv_destroy(ctx);
        return VERKV_ECUDA;
    }
    unsigned char *w = ctx->ws;
    ctx->err = (uint32_t *)(w + L.err);
    ctx->scores = (float *)(w + L.scores);
    ctx->qstats = (verkv_head_stats *)(w + L.qstats);
    ctx->F = (uint32_t *)(w + L.F);
    ctx->fids = (int32_t *)(w + L.fids);
    ctx->fcounts = (int32_t *)(w + L.fcounts);
    ctx->flc = (int32_t *)(w + L.flc);
    ctx->nacc = (int32_t *)(w + L.nacc);
    ctx->rmask = (uint32_t *)(w + L.rmask);
    ctx->rnext = (int32_t *)(w + L.rnext);
    ctx->slb = (uint32_t *)(w + L.slb);
    ctx->staging = (uint16_t *)(w + L.staging);
    ctx->part_piv = (float *)(w + L.part_piv);
    ctx->part_fet = (float *)(w + L.part_fet);
    e = cudaMemsetAsync(ctx->err, 0, 256, ctx->main);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->fcounts, 0, (size_t)L.units_layer * 4, ctx->main);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->flc, 0, (size_t)L.units_layer * 4, ctx->main);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->nacc, 0, (size_t)L.qh_layer * 4, ctx->main);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->rmask, 0, (size_t)L.units_layer * RMASK_W * 4, ctx->main);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->rnext, 0, 4, ctx->main);
    if (e != cudaSuccess) {
        verkv_destroy(ctx);
        return VERKV_ECUDA;
    }
    *out = ctx;
    return VERKV_OK;
}

void verkv_destroy(verkv_ctx *ctx) {
    if (!ctx) return;
    if (ctx->main || ctx->side) {
        if (ctx->main) cudaStreamSynchronize(ctx->main);
        if (ctx->side) cudaStreamSynchronize(ctx->side);
    }
    delete ctx->pool;
    if (ctx->host_staging) cudaFreeHost(ctx->host_staging);
    if (ctx->host_ids) cudaFreeHost(ctx->host_ids);
    if (ctx->host_counts) cudaFreeHost(ctx->host_counts);
    for (cudaEvent_t e : ctx->prof_pool) cudaEventDestroy(e);
    if (ctx->e_sel) cudaEventDestroy(ctx->e_sel);
    if (ctx->e_fetch) cudaEventDestroy(ctx->e_fetch);
    if (ctx->side) cudaStreamDestroy(ctx->side);
    delete ctx;
}

verkv_status verkv_set_sequence_offset(verkv_ctx *ctx, int32_t seq0) {
    if (!ctx) return VERKV_EINVAL;
    if (seq0 < 0) return fail(ctx, VERKV_EINVAL, "sequence offset: must be >= 0");
    ctx->seq0 = seq0;
    return VERKV_OK;
}

verkv_status verkv_set_fetch_mode(verkv_ctx *ctx, int mode_flags) {
    if (!ctx) return VERKV_EINVAL;
    const int mode = mode_flags & ~VERKV_FETCH_KEYS;
    if (mode != VERKV_FETCH_ZEROCOPY && mode != VERKV_FETCH_MEMCPY)
        return fail(ctx, VERKV_EINVAL, "unknown fetch mode");
    ctx->fetch_keys = (mode_flags & VERKV_FETCH_KEYS) != 0;
    if (mode == VERKV_FETCH_MEMCPY && !ctx->host_staging) {
        const size_t rows = (size_t)ctx->L.units_layer * ctx->sh.n;
        VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
        VERKV_CUDA(cudaHostAlloc((void **)&ctx->host_staging,
                                 staging_bytes(ctx->L.units_layer, ctx->sh.n, ctx->sh.head_dim),
                                 cudaHostAllocDefault), "cudaHostAlloc(staging)");
        VERKV_CUDA(cudaHostAlloc((void **)&ctx->host_ids, rows * 4, cudaHostAllocMapped),
                   "cudaHostAlloc(ids)");
        VERKV_CUDA(cudaHostAlloc((void **)&ctx->host_counts, (size_t)ctx->L.units_layer * 4,
                                 cudaHostAllocMapped), "cudaHostAlloc(counts)");
        VERKV_CUDA(cudaHostGetDevicePointer((void **)&ctx->host_ids_dev, ctx->host_ids, 0),
                   "cudaHostGetDevicePointer(ids)");
        VERKV_CUDA(cudaHostGetDevicePointer((void **)&ctx->host_counts_dev, ctx->host_counts, 0),
                   "cudaHostGetDevicePointer(counts)");
        unsigned hw = std::thread::hardware_concurrency();
        ctx->pool = new Pool((int)std::max(1u, std::min(hw, 16u)));
    }
    ctx->fetch_mode = mode;
    return VERKV_OK;
}

verkv_status verkv_poissoncomp(verkv_ctx *ctx, const float *tau, double eta, verkv_hset H,
                               uint64_t seed, const void *kv_full, float *r_full,
                               const verkv_pivotal *out) {
    if (!ctx) return VERKV_EINVAL;
    if (!tau || !kv_full || !r_full || !out || !out->ids || !out->r || !out->kv || !out->count ||
        !out->resident || !out->c)
        return fail(ctx, VERKV_EINVAL, "poissoncomp: null pointer");
    if (!(eta > 0.0) || eta > 1.0 || H.n_sink < 0 || H.n_local < 0)
        return fail(ctx, VERKV_EINVAL, "poissoncomp: eta must be in (0, 1], H sizes >= 0");
    const int n = ctx->sh.n;
    const int64_t forced = std::min<int64_t>(n, (int64_t)H.n_sink + H.n_local);
    const int n_rest = (int)(n - forced);
    const double eta_n = eta * (double)n;
    const double b_rest = eta_n - (double)forced;
    if (n_rest > 0 && !(b_rest > 0.0))
        return fail(ctx, VERKV_EBUDGET, "poissoncomp: eta * n must exceed the forced H set");
    const NvtxRange nvtx("verkv_poissoncomp");
    if (bad16(kv_full) || bad16(out->kv) || bad4(tau) || bad4(r_full) || bad4(out->ids) ||
        bad4(out->r) || bad4(out->count) || bad4(out->resident) || bad4(out->c))
        return fail(ctx, VERKV_EINVAL, "poissoncomp: kv rows need 16-byte, other arrays 4-byte alignment");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    const int units = ctx->sh.batch * ctx->sh.layers * ctx->sh.kv_heads;
    PcArgs a{};
    a.tau = tau;
    a.r_full = r_full;
    a.ids = out->ids;
    a.pr = out->r;
    a.count = out->count;
    a.resident = out->resident;
    a.c_out = out->c;
    a.err = ctx->err;
    a.b_rest = b_rest;
    a.eta_n = eta_n;
    a.n = n;
    a.W = ctx->L.W;
    a.cap = ctx->sh.cap;
    a.n_sink = H.n_sink;
    a.n_local = H.n_local;
    a.layers = ctx->sh.layers;
    a.kv_heads = ctx->sh.kv_heads;
    a.n_rest = n_rest;
    int cl = (n + 32767) / 32768;
    cl = std::max(1, std::min(cl, 8));
    int chunk = (n + cl - 1) / cl;
    chunk = (chunk + 1023) / 1024 * 1024;
    a.cl = cl;
    a.chunk = chunk;
    a.seed_lo = (uint32_t)seed;
    a.seed_hi = (uint32_t)(seed >> 32);
    a.seq0 = ctx->seq0;
    VERKV_CUDA(tracked(ctx, VERKV_K_PC_SOLVE, ctx->main, [&] { return launch_pc_solve(a, units, ctx->main); }), "k_pc_solve");
    VERKV_CUDA(tracked(ctx, VERKV_K_PC_GATHER, ctx->main, [&] {
                   return launch_pc_gather((const uint16_t *)kv_full, out->ids, out->count,
                                           (uint16_t *)out->kv, units, ctx->sh.cap, n,
                                           ctx->sh.head_dim, ctx->main);
               }), "k_pc_gather");
    return VERKV_OK;
}

verkv_status verkv_sketch_build(verkv_ctx *ctx, const void *kv_full, int32_t format,
                                void *sketch_out) {
    if (!ctx) return VERKV_EINVAL;
    if (!kv_full || !sketch_out) return fail(ctx, VERKV_EINVAL, "sketch_build: null pointer");
    if (format != VERKV_SKETCH_EXACT && format != VERKV_SKETCH_Q2)
        return fail(ctx, VERKV_EINVAL, "sketch_build: unknown format");
    if (bad16(kv_full) || bad16(sketch_out))
        return fail(ctx, VERKV_EINVAL, "sketch_build: kv_full and the sketch need 16-byte alignment");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    const int64_t rows = (int64_t)ctx->sh.batch * ctx->sh.layers * ctx->sh.kv_heads * ctx->sh.n;
    if (format == VERKV_SKETCH_Q2) {
        VERKV_CUDA(tracked(ctx, VERKV_K_SKETCH, ctx->main, [&] {
                       return launch_sketch_q2((const uint16_t *)kv_full, (uint8_t *)sketch_out,
                                               rows, ctx->sh.head_dim, ctx->main);
                   }), "k_sketch_q2");
        return VERKV_OK;
    }
    VERKV_CUDA(tracked(ctx, VERKV_K_SKETCH, ctx->main, [&] {
                   return launch_sketch_exact((const uint16_t *)kv_full, (uint16_t *)sketch_out,
                                              rows, ctx->sh.head_dim, ctx->main);
               }), "k_sketch_exact");
    return VERKV_OK;
}

verkv_status verkv_attend_verified(verkv_ctx *ctx, int32_t layer, const void *q,
                                   const verkv_pivotal *pivotal, const float *r_full,
                                   const verkv_sketch *sketch, float eps, float delta,
                                   int32_t *fetch_ids_out, int32_t *fetch_counts_out) {
    if (!ctx) return VERKV_EINVAL;
    if (layer < 0 || layer >= ctx->sh.layers) return fail(ctx, VERKV_EINVAL, "attend: bad layer");
    if (!q || !pivotal || !r_full || !sketch || !sketch->data || !pivotal->ids || !pivotal->r ||
        !pivotal->kv || !pivotal->count || !pivotal->resident)
        return fail(ctx, VERKV_EINVAL, "attend: null pointer");
    if (sketch->format != VERKV_SKETCH_EXACT && sketch->format != VERKV_SKETCH_Q2)
        return fail(ctx, VERKV_EINVAL, "attend: unknown sketch format");
    if (!(eps > 0.0f) || !(delta > 0.0f) || !(delta < 1.0f) || !isfinite(eps))
        return fail(ctx, VERKV_EINVAL, "attend: need eps > 0 and 0 < delta < 1");
    if (bad16(q) || bad16(sketch->data) || bad16(pivotal->kv))
        return fail(ctx, VERKV_EINVAL, "attend: q, the sketch and the pivotal rows need 16-byte alignment");
    if (bad4(r_full) || bad4(pivotal->ids) || bad4(pivotal->r) || bad4(pivotal->count) ||
        bad4(pivotal->resident) || bad4(fetch_ids_out) || bad4(fetch_counts_out))
        return fail(ctx, VERKV_EINVAL, "attend: int32 / float arrays need 4-byte alignment");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    const NvtxRange nvtx("verkv_attend_verified: score, certificate, selection");
    const LayerIdx li = layer_idx(ctx, layer);
    const int n = ctx->sh.n, d = ctx->sh.head_dim;

    ScoreArgs sa{};
    sa.sketch = (const uint16_t *)sketch->data;
    sa.q = (const uint16_t *)q;
    sa.scores = ctx->scores;
    sa.err = ctx->err;
    sa.n = n;
    sa.d = d;
    sa.scale = (float)(1.0 / sqrt((double)d));
    sa.li = li;
    if (ctx->score_stall_ns > 0) {  // injected: one stalled stage, a short wait limit
        sa.wait_ns = (unsigned long long)ctx->score_stall_ns;
        sa.stall_first = 1;
        ctx->score_stall_ns = 0;
    }
    if (sketch->format == VERKV_SKETCH_Q2) {
        VERKV_CUDA(tracked(ctx, VERKV_K_SCORE, ctx->main, [&] { return launch_score_q2(sa, ctx->L.units_layer, ctx->main, true); }), "k_score_q2");
    } else {
        VERKV_CUDA(tracked(ctx, VERKV_K_SCORE, ctx->main, [&] { return launch_score(sa, ctx->L.units_layer, ctx->main, true); }), "k_score");
    }

    if (ctx->shortlist > 0) {
        ShortlistArgs sla{};
        sla.scores = ctx->scores;
        sla.r_full = r_full;
        sla.out = ctx->slb;
        sla.n = n;
        sla.W = ctx->L.W;
        sla.size = ctx->shortlist;
        sla.li = li;
        VERKV_CUDA(tracked(ctx, VERKV_K_SHORTLIST, ctx->main, [&] { return launch_shortlist(sla, ctx->L.units_layer, ctx->main); }), "k_shortlist");
    }

    CertifyArgs ca{};
    ca.scores = ctx->scores;
    ca.shortlist = ctx->shortlist > 0 ? ctx->slb : nullptr;
    ctx->shortlisted = ctx->shortlist > 0;
    ca.r_full = r_full;
    ca.resident = pivotal->resident;
    ca.F = ctx->F;
    ca.qstats = ctx->qstats;
    ca.err = ctx->err;
    ca.n = n;
    ca.W = ctx->L.W;
    ca.cl = certify_cluster_size(n, ctx->L.qh_layer, ctx->sms);
    ca.chunk = certify_chunk(n, ca.cl);
    ca.eps = eps;
    ca.ldelta = (float)log(2.0 / (double)delta);
    ca.li = li;
    ca.beta_maxit = ctx->beta_maxit;
    ca.sel_gather = ctx->sel_gather;
    // The per-KV-head fetch list is built only for those who read it: the MEMCPY gather, or a
    // caller asking for ids or counts.  The zero-copy refine reads the selection bitmaps.
    const bool need_list = ctx->fetch_mode != VERKV_FETCH_ZEROCOPY || fetch_ids_out || fetch_counts_out;
    ca.fl_counter = need_list ? ctx->flc : nullptr;
    ca.rmask = ctx->rmask;
    ca.refine_next = ctx->rnext;
    ca.ids = ctx->fids;
    ca.counts = ctx->fcounts;
    ca.ids_user = fetch_ids_out;
    ca.counts_user = fetch_counts_out;
    if (ctx->fetch_mode == VERKV_FETCH_MEMCPY) {
        ca.ids_host = ctx->host_ids_dev;
        ca.counts_host = ctx->host_counts_dev;
    }
    VERKV_CUDA(tracked(ctx, VERKV_K_CERTIFY, ctx->main, [&] {
                   return launch_certify(ca, ctx->L.qh_layer, certify_smem_bytes(ca.chunk), ctx->main);
               }), "k_certify");
    // MEMCPY mode: verkv_fetch_refine waits on the host for the selection
    if (ctx->fetch_mode != VERKV_FETCH_ZEROCOPY)
        VERKV_CUDA(cudaEventRecord(ctx->e_sel, ctx->main), "cudaEventRecord");

    // The pivotal partial sums need only the selection: in MEMCPY mode they run here, during the
    // host gather; the zero-copy refine kernel of verkv_fetch_refine does them itself.
    if (ctx->fetch_mode != VERKV_FETCH_ZEROCOPY) {
        const PartialArgs pa = pivotal_args(ctx, *pivotal, q, li, sketch->format == VERKV_SKETCH_EXACT);
        int grid = std::min(ctx->L.units_layer * ctx->L.max_piv, ctx->sms * 8);
        VERKV_CUDA(tracked(ctx, VERKV_K_PARTIAL_PIVOTAL, ctx->main, [&] { return launch_partial(pa, ctx->L.units_layer, std::max(grid, 1), ctx->main); }), "k_partial");
    }

    ctx->pending = true;
    ctx->attended = true;
    ctx->layer = layer;
    ctx->piv = *pivotal;
    ctx->user_ids = fetch_ids_out;
    ctx->user_counts = fetch_counts_out;
    ctx->q = q;
    ctx->sketch = sketch->data;
    ctx->sketch_exact = sketch->format == VERKV_SKETCH_EXACT;
    return VERKV_OK;
}

verkv_status verkv_fetch_refine(verkv_ctx *ctx, const int32_t *ids, const int32_t *counts,
                                const void *host_kv, float *o_out, float *lse_out,
                                verkv_head_stats *stats_out) {
    if (!ctx) return VERKV_EINVAL;
    if (!ctx->pending) return fail(ctx, VERKV_ESTATE, "fetch_refine: no preceding attend_verified");
    if ((ids && ids != ctx->user_ids) || (counts && counts != ctx->user_counts))
        return fail(ctx, VERKV_EINVAL, "fetch_refine: ids/counts must be the attend outputs or NULL");
    if (!host_kv || !o_out) return fail(ctx, VERKV_EINVAL, "fetch_refine: null pointer");
    if (bad16(host_kv) || bad4(o_out) || bad4(lse_out) || bad4(stats_out))
        return fail(ctx, VERKV_EINVAL, "fetch_refine: host_kv needs 16-byte, outputs 4-byte alignment");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    const NvtxRange nvtx("verkv_fetch_refine: fetch, refine, merge");
    const LayerIdx li = layer_idx(ctx, ctx->layer);
    const int n = ctx->sh.n, d = ctx->sh.head_dim;
    // With the exact sketch every key is already on the GPU: only V rows move, unless asked.
    // A 2-bit sketch holds no exact key, so fetched rows bring their K row too.
    const bool v_only = !ctx->fetch_keys && ctx->sketch_exact;
    const size_t row_bytes = (size_t)4 * d;                 // a K|V row of the host cache
    const size_t move_bytes = v_only ? (size_t)2 * d : row_bytes;
    const size_t move_off = v_only ? (size_t)2 * d : 0;     // V follows K inside a row

    PartialArgs pa{};
    pa.q = (const uint16_t *)ctx->q;
    pa.F = ctx->F;
    pa.qstats = ctx->qstats;
    pa.part = ctx->part_fet;
    pa.err = ctx->err;
    pa.rmask = ctx->rmask;
    pa.ids = ctx->fids;
    pa.pr = nullptr;
    pa.count = ctx->fcounts;
    pa.row_stride = n;
    pa.max_chunks = ctx->L.max_fet;
    pa.n = n;
    pa.W = ctx->L.W;
    pa.d = d;
    pa.scale = (float)(1.0 / sqrt((double)d));
    pa.li = li;
    pa.keys = v_only ? (const uint16_t *)ctx->sketch : nullptr;
    int grid = std::max(1, std::min(ctx->L.units_layer * ctx->L.max_fet, ctx->sms * 8));

    MergeArgs ma{};
    ma.part_piv = ctx->part_piv;
    ma.part_fet = ctx->part_fet;
    ma.rmask = ctx->rmask;
    ma.pcount = ctx->piv.count;
    ma.fcount = ctx->fcounts;
    ma.qstats = ctx->qstats;
    ma.o = o_out;
    ma.lse = lse_out;
    ma.stats = stats_out;
    ma.max_piv = ctx->L.max_piv;
    ma.max_fet = ctx->L.max_fet;
    ma.cap = ctx->sh.cap;
    ma.d = d;
    ma.li = li;

    if (ctx->fetch_mode == VERKV_FETCH_ZEROCOPY) {
        // One kernel on the context's stream for the pivotal partial sums and the fetched rows,
        // read straight from page-locked host memory; the merge follows.
        cudaPointerAttributes attr;
        cudaError_t e = cudaPointerGetAttributes(&attr, host_kv);
        if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
            cudaGetLastError();
            return fail(ctx, VERKV_EINVAL, "fetch_refine: host_kv is not page-locked host memory");
        }
        pa.rows = (const uint16_t *)attr.devicePointer;
        pa.mode = ROWS_HOST;
        pa.row16 = d / 4;
        pa.voff16 = d / 8;
        pa.resident = ctx->piv.resident;
        pa.nacc = ctx->nacc;
        pa.refine_next = ctx->rnext;
        ma.nacc = ctx->nacc;
        const PartialArgs piv = pivotal_args(ctx, ctx->piv, ctx->q, li, ctx->sketch_exact);
        const int items = ctx->L.units_layer * (ctx->L.max_fet + ctx->L.max_piv);
        grid = std::max(1, std::min(items, ctx->sms * 8));
        VERKV_CUDA(tracked(ctx, VERKV_K_FETCH_HOST, ctx->main, [&] {
                       return launch_refine(piv, pa, ctx->L.units_layer, grid, ctx->main);
                   }), "k_refine");
    } else {
        VERKV_CUDA(cudaEventSynchronize(ctx->e_sel), "cudaEventSynchronize");
        // When profiling, two events on the (idle) side stream bracket the host gather.
        cudaEvent_t g0 = ctx->prof_on ? prof_event(ctx) : nullptr;
        if (g0) VERKV_CUDA(cudaEventRecord(g0, ctx->side), "cudaEventRecord");
        const int U = ctx->L.units_layer;
        const unsigned char *src_base = (const unsigned char *)host_kv;
        // Flatten (unit, row) into one index space and split it evenly over the pool.
        std::vector<int64_t> start(U + 1, 0);
        for (int ul = 0; ul < U; ++ul) start[ul + 1] = start[ul] + ctx->host_counts[ul];
        const int64_t total = start[U];
        const int P = ctx->pool->size();
        const size_t head = staging_header(U);
        int64_t *offs = reinterpret_cast<int64_t *>(ctx->host_staging);
        for (int ul = 0; ul < U; ++ul) offs[ul] = start[ul];
        unsigned char *rows_h = ctx->host_staging + head;
        nvtxRangePushA("fetch: host gather");
        ctx->pool->run([&](int w) {
            const int64_t lo = total * w / P, hi = total * (w + 1) / P;
            int ul = (int)(std::upper_bound(start.begin(), start.end(), lo) - start.begin()) - 1;
            for (int64_t x = lo; x < hi; ++x) {
                while (x >= start[ul + 1]) ++ul;
                const int64_t j = x - start[ul];
                const int ug = li.unit_global(ul);
                const int id = ctx->host_ids[(size_t)ul * n + j];
                memcpy(rows_h + (size_t)x * move_bytes,
                       src_base + ((size_t)ug * n + id) * row_bytes + move_off, move_bytes);
            }
        });
        nvtxRangePop();
        if (g0) {
            cudaEvent_t g1 = prof_event(ctx);
            if (g1) {
                VERKV_CUDA(cudaEventRecord(g1, ctx->side), "cudaEventRecord");
                ctx->prof_recs.push_back({VERKV_K_FETCH_GATHER, g0, g1});
            }
        }
        // One copy: the header and every unit's rows.
        const cudaError_t ce = tracked(ctx, VERKV_K_FETCH_COPY, ctx->side, [&]() -> cudaError_t {
            return copy_rows(ctx, ctx->staging, ctx->host_staging, head + (size_t)total * move_bytes);
        });
        if (ce != cudaSuccess)
            return fail(ctx, VERKV_ECOPY, std::string("fetch copy: ") + cudaGetErrorString(ce));
        VERKV_CUDA(cudaEventRecord(ctx->e_fetch, ctx->side), "cudaEventRecord");
        VERKV_CUDA(cudaStreamWaitEvent(ctx->main, ctx->e_fetch, 0), "cudaStreamWaitEvent");
        pa.staged_off = reinterpret_cast<const int64_t *>(ctx->staging);
        pa.rows = reinterpret_cast<const uint16_t *>(reinterpret_cast<const unsigned char *>(ctx->staging) + head);
        pa.mode = ROWS_STAGED;
        pa.row16 = (int)(move_bytes / 16);
        pa.voff16 = v_only ? 0 : d / 8;
        VERKV_CUDA(tracked(ctx, VERKV_K_PARTIAL_STAGED, ctx->main, [&] { return launch_partial(pa, ctx->L.units_layer, grid, ctx->main); }), "k_partial(staged)");
    }

    VERKV_CUDA(tracked(ctx, VERKV_K_MERGE, ctx->main, [&] { return launch_merge(ma, ctx->L.qh_layer, ctx->main); }), "k_merge");
    ctx->pending = false;
    return VERKV_OK;
}

verkv_status verkv_measure_sketch_stream(verkv_ctx *ctx, int32_t layer, const verkv_sketch *sketch) {
    if (!ctx) return VERKV_EINVAL;
    if (layer < 0 || layer >= ctx->sh.layers) return fail(ctx, VERKV_EINVAL, "sketch stream: bad layer");
    if (!sketch || !sketch->data || sketch->format != VERKV_SKETCH_EXACT)
        return fail(ctx, VERKV_EINVAL, "sketch stream: an exact sketch is required");
    if (bad16(sketch->data)) return fail(ctx, VERKV_EINVAL, "sketch stream: 16-byte alignment required");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    ScoreArgs sa{};
    sa.sketch = (const uint16_t *)sketch->data;
    sa.err = ctx->err;
    sa.n = ctx->sh.n;
    sa.d = ctx->sh.head_dim;
    sa.li = layer_idx(ctx, layer);
    VERKV_CUDA(launch_sketch_stream(sa, ctx->L.units_layer, ctx->main), "k_sketch_stream");
    return VERKV_OK;
}

verkv_status verkv_sync(verkv_ctx *ctx) {
    if (!ctx) return VERKV_EINVAL;
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    VERKV_CUDA(cudaStreamSynchronize(ctx->side), "cudaStreamSynchronize(side)");
    VERKV_CUDA(cudaStreamSynchronize(ctx->main), "cudaStreamSynchronize(main)");
    uint32_t word = 0;
    VERKV_CUDA(cudaMemcpy(&word, ctx->err, sizeof(word), cudaMemcpyDeviceToHost), "read error word");
    if (word == 0) return VERKV_OK;
    VERKV_CUDA(cudaMemset(ctx->err, 0, sizeof(word)), "clear error word");
    if (word & ERR_TAU) return fail(ctx, VERKV_EINVAL, "tau outside (0, 1] or not finite");
    if (word & ERR_CAPACITY) return fail(ctx, VERKV_ECAPACITY, "pivotal set exceeded cap (truncated)");
    if (word & ERR_TIMEOUT) return fail(ctx, VERKV_ETIMEOUT, "a bounded wait on a copy barrier expired");
    if (word & ERR_BADID) return fail(ctx, VERKV_EINVAL, "a pivotal or fetch row id outside [0, n) (skipped)");
    if (word & ERR_BUDGET_SUM) return fail(ctx, VERKV_ENOCONVERGE, "|sum r - eta n| >= 1e-6 n");
    return fail(ctx, VERKV_ENOCONVERGE, "a solve hit its iteration cap");
}

verkv_status verkv_set_shortlist(verkv_ctx *ctx, int32_t size) {
    if (!ctx) return VERKV_EINVAL;
    if (size < 0 || size > SHORTLIST_MAX)
        return fail(ctx, VERKV_EINVAL, "set_shortlist: size must be 0 (off) or 1 .. 256");
    ctx->shortlist = size;
    return VERKV_OK;
}

verkv_status verkv_shortlist_bitmap(verkv_ctx *ctx, uint32_t *out) {
    if (!ctx) return VERKV_EINVAL;
    if (!ctx->shortlisted) return fail(ctx, VERKV_ESTATE, "shortlist_bitmap: no attend with a shortlist");
    if (!out) return fail(ctx, VERKV_EINVAL, "shortlist_bitmap: null pointer");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    VERKV_CUDA(cudaMemcpyAsync(out, ctx->slb, (size_t)ctx->L.units_layer * ctx->L.W * 4,
                               cudaMemcpyDefault, ctx->main), "copy shortlist");
    return VERKV_OK;
}

verkv_status verkv_attend_dense_host(verkv_ctx *ctx, int32_t layer, const void *q,
                                    const void *host_kv, float *o_out, float *lse_out) {
    if (!ctx) return VERKV_EINVAL;
    if (layer < 0 || layer >= ctx->sh.layers) return fail(ctx, VERKV_EINVAL, "dense: bad layer");
    if (!q || !host_kv || !o_out) return fail(ctx, VERKV_EINVAL, "dense: null pointer");
    if (bad16(q) || bad16(host_kv) || bad4(o_out) || bad4(lse_out))
        return fail(ctx, VERKV_EINVAL, "dense: q and host_kv need 16-byte, outputs 4-byte alignment");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, host_kv);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
        cudaGetLastError();
        return fail(ctx, VERKV_EINVAL, "dense: host_kv is not page-locked host memory");
    }
    DenseArgs da{};
    da.rows = (const uint16_t *)attr.devicePointer;
    da.q = (const uint16_t *)q;
    da.part = ctx->part_fet;  // [units_layer][dense_chunks][G][d + 2]
    da.n = ctx->sh.n;
    da.chunks = ctx->L.dense_chunks;
    da.d = ctx->sh.head_dim;
    da.scale = (float)(1.0 / sqrt((double)da.d));
    da.li = layer_idx(ctx, layer);
    const int grid = std::max(1, std::min(ctx->L.units_layer * da.chunks, ctx->sms * 4));
    VERKV_CUDA(tracked(ctx, VERKV_K_DENSE_HOST, ctx->main, [&] {
                   return launch_dense_host(da, ctx->L.units_layer, grid, ctx->main);
               }), "k_dense_host");
    VERKV_CUDA(tracked(ctx, VERKV_K_DENSE_MERGE, ctx->main, [&] {
                   return launch_dense_merge(da, ctx->L.qh_layer, o_out, lse_out, ctx->main);
               }), "k_dense_merge");
    return VERKV_OK;
}

verkv_status verkv_selection_bitmap(verkv_ctx *ctx, uint32_t *out) {
    if (!ctx) return VERKV_EINVAL;
    if (!ctx->attended) return fail(ctx, VERKV_ESTATE, "selection_bitmap: no attend has run");
    if (!out) return fail(ctx, VERKV_EINVAL, "selection_bitmap: null pointer");
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    VERKV_CUDA(cudaMemcpyAsync(out, ctx->F, (size_t)ctx->L.qh_layer * ctx->L.W * 4,
                               cudaMemcpyDefault, ctx->main), "copy F");
    return VERKV_OK;
}

verkv_status verkv_test_inject(verkv_ctx *ctx, int what, int64_t value) {
    if (!ctx) return VERKV_EINVAL;
    switch (what) {
        case VERKV_INJECT_COPY_FAIL:
            if (value < 0) break;
            ctx->inject_copy_fail = value;
            return VERKV_OK;
        case VERKV_INJECT_BETA_MAXIT:
            if (value < 0 || value > 64) break;
            ctx->beta_maxit = (int)value;
            return VERKV_OK;
        case VERKV_INJECT_SCORE_STALL:
            if (value < 1000 || value > 1000000000LL) break;
            ctx->score_stall_ns = value;
            return VERKV_OK;
        case VERKV_INJECT_SELECT_GATHER:
            if (value < 0 || value > 1) break;
            ctx->sel_gather = (int)value;
            return VERKV_OK;
        default:
            break;
    }
    return fail(ctx, VERKV_EINVAL, "test_inject: unknown injection or value out of range");
}

verkv_status verkv_profile_enable(verkv_ctx *ctx, int on) {
    if (!ctx) return VERKV_EINVAL;
    ctx->prof_on = on != 0;
    return VERKV_OK;
}

verkv_status verkv_profile_read(verkv_ctx *ctx, int64_t *launches, double *total_ms) {
    if (!ctx || !launches || !total_ms) return VERKV_EINVAL;
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    VERKV_CUDA(cudaStreamSynchronize(ctx->side), "cudaStreamSynchronize(side)");
    VERKV_CUDA(cudaStreamSynchronize(ctx->main), "cudaStreamSynchronize(main)");
    for (const auto &r : ctx->prof_recs) {
        float ms = 0.0f;
        VERKV_CUDA(cudaEventElapsedTime(&ms, r.a, r.b), "cudaEventElapsedTime");
        launches[r.kernel] += 1;
        total_ms[r.kernel] += ms;
    }
    ctx->prof_recs.clear();
    ctx->prof_used = 0;
    return VERKV_OK;
}

verkv_status verkv_profile_timeline(verkv_ctx *ctx, int64_t max_records, int32_t *kernel,
                                    double *start_ms, double *end_ms, int64_t *n_out) {
    if (!ctx || !kernel || !start_ms || !end_ms || !n_out || max_records < 0) return VERKV_EINVAL;
    VERKV_CUDA(cudaSetDevice(ctx->device), "cudaSetDevice");
    VERKV_CUDA(cudaStreamSynchronize(ctx->side), "cudaStreamSynchronize(side)");
    VERKV_CUDA(cudaStreamSynchronize(ctx->main), "cudaStreamSynchronize(main)");
    int64_t k = 0;
    for (const auto &r : ctx->prof_recs) {
        if (k >= max_records) break;
        float a = 0.0f, b = 0.0f;
        VERKV_CUDA(cudaEventElapsedTime(&a, ctx->prof_recs[0].a, r.a), "cudaEventElapsedTime");
        VERKV_CUDA(cudaEventElapsedTime(&b, ctx->prof_recs[0].a, r.b), "cudaEventElapsedTime");
        kernel[k] = r.kernel;
        start_ms[k] = a;
        end_ms[k] = b;
        ++k;
    }
    *n_out = k;
    return VERKV_OK;
}

verkv_status verkv_launch_counts(verkv_ctx *ctx, int64_t *out) {
    if (!ctx || !out) return VERKV_EINVAL;
    for (int k = 0; k < VERKV_K_COUNT; ++k) out[k] = ctx->launches[k];
    return VERKV_OK;
}

const char *verkv_kernel_name(int k) {
    static const char *names[VERKV_K_COUNT] = {
        "k_pc_solve", "k_pc_gather", "k_sketch", "k_score", "k_certify",
        "k_partial(pivotal)", "k_refine", "k_partial(staged)", "k_merge",
        "k_dense_host", "k_dense_merge", "k_shortlist", "fetch_copy", "fetch_gather"};
    return (k >= 0 && k < VERKV_K_COUNT) ? names[k] : "";
}

const char *verkv_last_error(verkv_ctx *ctx) { return ctx ? ctx->last_error.c_str() : ""; }

}  // extern "C"
