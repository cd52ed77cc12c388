// verkv_internal.h -- kernel argument blocks and launchers shared by libverkv's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/verkv.h"

namespace verkv {

// Device error word bits (latched with atomicOr, read and cleared by verkv_sync).
enum : uint32_t {
    ERR_TAU = 1u << 0,         // tau outside (0, 1] or not finite
    ERR_CAPACITY = 1u << 1,    // pivotal set larger than cap
    ERR_NOCONVERGE = 1u << 2,  // a solve hit its iteration cap
    ERR_BUDGET_SUM = 1u << 3,  // |sum r - eta n| >= 1e-6 n after the c solve
    ERR_TIMEOUT = 1u << 4,     // a bounded wait on a copy barrier expired
    ERR_BADID = 1u << 5,       // a pivotal or fetch row id outside [0, n) (the row was skipped)
};

// ---------------------------------------------------------------------------------------------
// PoissonComp: c solve, r, Philox sample, compaction (one cluster per unit).
struct PcArgs {
    const float *tau;        // [units][n]
    float *r_full;           // [units][n]
    int32_t *ids;            // [units][cap]
    float *pr;               // [units][cap]
    int32_t *count;          // [units]
    uint32_t *resident;      // [units][W]
    float *c_out;            // [units]
    uint32_t *err;
    double b_rest;           // eta n - |forced|
    double eta_n;            // eta n
    int n, W, cap, n_sink, n_local, layers, kv_heads;
    int n_rest;              // n - |forced|
    int cl, chunk;           // CTAs per cluster, tokens per CTA (multiple of 1024)
    uint32_t seed_lo, seed_hi;
    int seq0;                // the first sequence's index in the Philox counter
};
cudaError_t launch_pc_solve(const PcArgs &a, int units, cudaStream_t s);

// Pivotal row gather: pkv[u][slot] = kv_full[u][ids[u][slot]].
cudaError_t launch_pc_gather(const uint16_t *kv_full, const int32_t *ids, const int32_t *count,
                             uint16_t *pkv, int units, int cap, int n, int d, cudaStream_t s);

// Exact sketch: sketch[u][i] = K row of kv_full[u][i].
cudaError_t launch_sketch_exact(const uint16_t *kv_full, uint16_t *sketch, int64_t rows, int d,
                                cudaStream_t s);

// The 2-bit sketch: rows of q2_row_bytes(d) bytes per token (codes, per-group floor and step).
int q2_row_bytes(int d);
cudaError_t launch_sketch_q2(const uint16_t *kv_full, uint8_t *sketch, int64_t rows, int d,
                             cudaStream_t s);

// Raise `func`'s dynamic shared-memory limit to at least `bytes` on the current device.  The
// attribute is per device, so the limit set is remembered per (device, kernel) under a lock;
// host threads and devices may call it concurrently.
cudaError_t ensure_smem(const void *func, size_t bytes);

// Launch `kernel` on stream s with programmatic stream serialisation: it may start before the
// previous kernel on s has finished, and must call pdl_wait() before reading what the stream
// produced (the decode path's kernels do so first thing).
// With pdl false the launch is an ordinary stream-ordered one (pdl_wait() then returns at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_opt_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    return launch_opt_pdl(true, kernel, grid, block, smem, s, static_cast<Args &&>(args)...);
}

// ---------------------------------------------------------------------------------------------
// Layer-local indexing of a decode call: u' = b * kv_heads + h (units of the layer), query head
// qh = u' * G + g, global unit u = (b * layers + layer) * kv_heads + h.
struct LayerIdx {
    int layers, layer, kv_heads, G;
    __host__ __device__ __forceinline__ int unit_global(int ul) const {
        const int b = ul / kv_heads, h = ul - b * kv_heads;
        return (b * layers + layer) * kv_heads + h;
    }
};

// Sketch scores s[qh][i] = q_qh . sketch_i / sqrt(d).
struct ScoreArgs {
    const uint16_t *sketch;  // [units][n][d]
    const uint16_t *q;       // [B][hq][d]
    float *scores;           // [B*hq][n]
    uint32_t *err;
    int n, d;
    float scale;
    LayerIdx li;
    // Failure injection for tests (0 in normal use): the bounded copy waits give up after
    // wait_ns (0: one second), and with stall_first set the first CTA arms its first stage's
    // barrier for a copy it never issues, so that wait runs out.
    unsigned long long wait_ns;
    int stall_first;
};
// `pdl`: launch with programmatic stream serialisation.  Safe for the first kernel of a library
// call because the scoring kernels read the caller's q and sketch only after pdl_wait(), which
// returns once the preceding kernel has finished and its writes are visible.
cudaError_t launch_score(const ScoreArgs &a, int units_layer, cudaStream_t s, bool pdl);
// The same from the 2-bit sketch (a.sketch points at its rows).
cudaError_t launch_score_q2(const ScoreArgs &a, int units_layer, cudaStream_t s, bool pdl);
// The exact sketch's rows of one layer through k_score's copy ring, with no arithmetic.
cudaError_t launch_sketch_stream(const ScoreArgs &a, int units_layer, cudaStream_t s);

// Certificate and selection per query head (one cluster per query head).  When fl_counter is
// set, the last of the G clusters of a KV head to finish also builds that head's fetch list:
// the ascending ids of (OR_g F_g) & ~resident, and n_fetch of its G query heads.
struct CertifyArgs {
    const float *scores;          // [qh][n]
    const float *r_full;          // [units][n]
    const uint32_t *resident;     // [units][W]
    uint32_t *F;                  // [qh][W]
    verkv_head_stats *qstats;     // [qh]
    uint32_t *err;
    int32_t *fl_counter;          // [units_layer], zero between calls; null: no fetch list
    int32_t *ids;                 // [units_layer][n]  (device, used by the fetch)
    int32_t *counts;              // [units_layer]
    int32_t *ids_user;            // optional copy (device or mapped host)
    int32_t *counts_user;
    int32_t *ids_host;            // optional copy into mapped host memory (MEMCPY mode)
    int32_t *counts_host;
    const uint32_t *shortlist;    // [units_layer][W] fetch candidates, or null: all of L
    uint32_t *rmask;              // [units_layer][RMASK_W] cleared here for the refine, or null
    int32_t *refine_next;         // the refine's item counter, set to 0 here, or null
    int n, W, cl, chunk;
    float eps, ldelta;
    LayerIdx li;
    int beta_maxit;               // iteration cap of the beta solve (0: the default, 64)
    int sel_gather;               // 1: clusters of 1 and 4 may end the select by gathering its
                                  // last candidates into rank 0; 0: histogram passes only (tests)
};
cudaError_t launch_certify(const CertifyArgs &a, int qheads, size_t smem, cudaStream_t s);

// The per-KV-head shortlist: the `size` tokens of L with the largest sketch logit over the KV
// head's query heads (ties to the lower id), as a bitmap [units_layer][W].
constexpr int SHORTLIST_MAX = 256;
struct ShortlistArgs {
    const float *scores;   // [qh][n]
    const float *r_full;   // [units][n]
    uint32_t *out;         // [units_layer][W]
    int n, W, size;
    LayerIdx li;
};
cudaError_t launch_shortlist(const ShortlistArgs &a, int units_layer, cudaStream_t s);
int certify_cluster_size(int n, int qheads, int sms);
int certify_chunk(int n, int cl);
size_t certify_smem_bytes(int chunk);


// ---------------------------------------------------------------------------------------------
// Shrinkage-weighted partial sums over a row set: the pivotal rows in HBM, fetched rows staged in
// HBM, or fetched rows read by token id straight from page-locked host memory.
constexpr int PART_ROWS = 64;                      // fetched rows a CTA has in flight
constexpr int PIV_STAGE_ROWS = 64;                 // pivotal rows staged in shared memory at once
constexpr int PIV_ITEM_ROWS = 256;                 // pivotal list positions per partial
// Token ids per partial of fetched rows: a multiple of 32 (whole bitmap words).  (512- and
// 768-token ranges measured slower: more items and partials for the same rows.)
constexpr int FET_RANGE = 1024;
constexpr int RMASK_RANGES = (131072 + FET_RANGE - 1) / FET_RANGE;  // ranges of the largest unit
constexpr int RMASK_W = (RMASK_RANGES + 31) / 32;                 // words of a unit's range mask
                                                   // (n <= 131072)
enum { ROWS_PIVOTAL = 0, ROWS_STAGED = 1, ROWS_HOST = 2 };
struct PartialArgs {
    const uint16_t *rows;     // [src units][row_stride][row16 vectors]; ROWS_HOST: [units][n][2][d]
    const uint16_t *keys;     // if set, K rows come from here by token id ([units][n][d], the
                              // exact sketch) and `rows` supply only V
    int row16;                // 16-byte vectors per row of `rows`
    int voff16;               // offset of the V row inside a row of `rows`, in 16-byte vectors
    const int32_t *ids;       // [src units][row_stride]
    const float *pr;          // pivotal r [src units][row_stride], or null for fetched rows
    const int32_t *count;     // [src units]
    const uint16_t *q;        // [B][hq][d]
    const uint32_t *F;        // [qh][W]
    const verkv_head_stats *qstats;
    const float *scores;      // sketch logits [qh][n]: lambda of Definition 2 uses w-hat
    float *part;              // [units_layer][max_chunks][G][d + 2]
    uint32_t *err;            // ERR_BADID for a row id outside [0, n)
    const uint32_t *resident; // ROWS_HOST in k_refine: the resident bitmaps [units][W]
    int32_t *nacc;            // ROWS_HOST in k_refine: per query head n_fetch accumulators
                              // [qh], zero on entry (k_merge resets them)
    int32_t *refine_next;     // k_refine: the next item to take, 0 on entry (the certify kernel
                              // of the same call resets it)
    uint32_t *rmask;          // fetched-row ranges: bit k of [units_layer][RMASK_W] set when
                              // range k holds rows (only those get a partial); zero on entry
    const int64_t *staged_off; // ROWS_STAGED: first staged row of each layer unit (the staged
                               // rows of all units are contiguous, unit by unit)
    int row_stride;           // cap (pivotal) or n (fetched)
    int units_total;          // pivotal: units of the whole shape (rows of `rows` = units_total * cap)
    int max_chunks;
    int n, W, d;
    int mode;                 // ROWS_PIVOTAL (global units) / ROWS_STAGED / ROWS_HOST (layer units)
    int sketch_logits;        // pivotal rows: lambda's w-hat from `scores` (a 2-bit sketch); 0: the
                              // row's own weight (the exact sketch holds the same key)
    float scale;
    LayerIdx li;
};
cudaError_t launch_partial(const PartialArgs &a, int units_layer, int grid, cudaStream_t s);

// Dense attention over every token of a KV head with the rows read from page-locked host memory
// (the offloaded-dense baseline): per chunk of PART_ROWS rows a partial (N[d], D, m) with the
// chunk's own max logit m, merged with running-max rescaling.
struct DenseArgs {
    const uint16_t *rows;   // host-mapped [units][n][2][d]
    const uint16_t *q;      // [B][hq][d]
    float *part;            // [units_layer][chunks][G][d + 2]
    int n, chunks, d;
    float scale;
    LayerIdx li;
};
cudaError_t launch_dense_host(const DenseArgs &a, int units_layer, int grid, cudaStream_t s);
cudaError_t launch_dense_merge(const DenseArgs &a, int qheads, float *o, float *lse, cudaStream_t s);

// Merge partials into o, lse and the per-head stats.
struct MergeArgs {
    const float *part_piv;
    const float *part_fet;
    const int32_t *pcount;       // pivotal count [units]
    const int32_t *fcount;       // fetch count [units_layer]
    const verkv_head_stats *qstats;
    float *o;                    // [qh][d]
    float *lse;                  // [qh] or null
    verkv_head_stats *stats;     // [qh] or null
    int32_t *nacc;               // per query head n_fetch counted by k_refine (read and reset),
                                 // or null: qstats carries it (the certify kernel's fetch list)
    const uint32_t *rmask;       // [units_layer][RMASK_W]: the fetched-row ranges with a partial
    int max_piv, max_fet, cap, d;
    LayerIdx li;
};
cudaError_t launch_merge(const MergeArgs &a, int qheads, cudaStream_t s);

// The zero-copy path's partial sums in one launch: the ROWS_HOST blocks (fet) and the
// ROWS_PIVOTAL blocks (piv) of every layer unit; launch_merge follows.
cudaError_t launch_refine(const PartialArgs &piv, const PartialArgs &fet, int units_layer, int grid,
                          cudaStream_t s);

}  // namespace verkv
