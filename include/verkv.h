/*
 * verkv.h -- C ABI of libverkv, VerKV's decode-time hot path on one GPU (sm_103a).
 *
 * Method: "Verify Before You Fetch: Reliable KV Cache Compression for LLM Inference" (arXiv
 * abstract page; Markdown summary page of the same title, whose section, equation, definition,
 * lemma and theorem names are cited below).  The abstract states the problem this interface
 * follows: a compact set of pivotal tokens and a token-level sketch of the full KV cache live on
 * the GPU, the complete cache lives in CPU memory, and each decode query either certifies its
 * attention against a user (epsilon, delta) tolerance or fetches extra tokens from the CPU and
 * refines.
 *
 * Conventions for every call:
 *  - The caller owns every tensor.  Device pointers are plain CUDA device addresses; "host"
 *    pointers must be page-locked (cudaHostAlloc / cudaHostRegister or torch pin_memory) because
 *    the GPU reads or writes them directly.  Nothing is allocated on the hot path: the context
 *    allocates its side stream, events and (only in VERKV_FETCH_MEMCPY mode) page-locked staging
 *    in verkv_create / verkv_set_fetch_mode, and all device scratch lives in the caller's
 *    workspace of verkv_workspace_size() bytes.
 *  - Calls are asynchronous and stream-ordered on the stream given to verkv_create, except that
 *    verkv_fetch_refine in VERKV_FETCH_MEMCPY mode waits on the host for the selection of the
 *    preceding verkv_attend_verified.  Errors detected on the device (invalid tau, pivotal
 *    capacity overflow, a solve that hit its iteration cap, a pivotal or fetch row id outside
 *    [0, n), whose row is then skipped) are latched in a device error word
 *    and returned by the next verkv_sync.  No call throws; a call that returns an error has not
 *    launched work unless stated.
 *  - Layouts.  A "unit" is one (sequence b, layer l, KV head h) of a verkv_shape; units are
 *    numbered u = (b * layers + l) * kv_heads + h.  Query head j of sequence b belongs to KV head
 *    j / q_per_kv (grouped-query attention).  bf16 is IEEE bfloat16 (uint16 bit patterns).
 *  - Alignment.  bf16 rows and queries (q, the sketch, the pivotal kv, kv_full, host_kv) are
 *    read in 16-byte vectors or bulk copies and must start on 16-byte boundaries; every other
 *    array must be 4-byte aligned.  A misaligned pointer is VERKV_EINVAL, returned before any
 *    launch.
 *  - One context per host thread; calls on one context must not overlap.
 */
#ifndef VERKV_H
#define VERKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VERKV_OK = 0,
    VERKV_EINVAL = 1,      /* bad argument, or tau outside (0, 1] / not finite (device) */
    VERKV_EBUDGET = 2,     /* eta * n does not exceed the forced H set */
    VERKV_ECAPACITY = 3,   /* a pivotal set larger than shape.cap (device; truncated) */
    VERKV_ENOCONVERGE = 4, /* a solve hit its iteration cap (device; result still written) */
    VERKV_ECUDA = 5,       /* CUDA runtime error (see verkv_last_error) */
    VERKV_ECOPY = 6,       /* host-to-device fetch failed */
    VERKV_ETIMEOUT = 7,    /* a bounded device wait expired */
    VERKV_ESTATE = 8,      /* calls out of order, e.g. fetch_refine without attend */
    VERKV_ETOOLARGE = 9    /* verkv_certify_noalloc: more logits than its fixed scratch holds */
} verkv_status;

typedef struct verkv_ctx verkv_ctx;

/* Sizes of one cache.  n is the context length per unit; cap the pivotal capacity per unit. */
typedef struct {
    int32_t batch;     /* B sequences                                    >= 1        */
    int32_t layers;    /* L                                              >= 1        */
    int32_t kv_heads;  /* h_kv                                           >= 1        */
    int32_t q_per_kv;  /* G query heads per KV head                      1, 2, 4, 8  */
    int32_t head_dim;  /* d                                              64 or 128   */
    int32_t n;         /* tokens per unit                                1 .. 131072 */
    int32_t cap;       /* pivotal capacity per unit                      1 .. n      */
} verkv_shape;

/* Tokens forced into H (summary page, PoissonComp: H includes the sink and local tokens):
 * the first n_sink and the last n_local tokens of every unit. */
typedef struct {
    int32_t n_sink;
    int32_t n_local;
} verkv_hset;

/* The GPU-resident pivotal set H u S of every unit (caller-owned device memory).
 *   ids       int32  [units][cap]        token ids of H u S, ascending
 *   r         float  [units][cap]        r_i of each pivotal token (1 for H)
 *   kv        bf16   [units][cap][2][d]  K row then V row of each pivotal token
 *   count     int32  [units]             |H u S|
 *   resident  uint32 [units][ceil(n/32)] bit i%32 of word i/32 set iff token i is in H u S
 *   c         float  [units]             the PoissonComp constant c (float32; +inf if eta n >= n)
 * When cap is a multiple of 4 and ids, r and kv start on 16-byte boundaries, the MEMCPY path
 * bulk-copies each block of 64 pivotal rows (with its ids and r) into shared memory; otherwise it
 * reads them from global memory.  Both give the same bits. */
typedef struct {
    int32_t *ids;
    float *r;
    void *kv;
    int32_t *count;
    uint32_t *resident;
    float *c;
} verkv_pivotal;

/* Token-level sketch of the full cache (abstract page; summary page, KVFETCH step 1).
 * VERKV_SKETCH_EXACT: a bf16 copy of every key, [units][n][d] -- the "perfect sketch" of the
 * summary page's Figure 5 and the setting of Theorem 2.
 * VERKV_SKETCH_Q2: the "2-bit sketch" of the same figure, in a layout of ours (the pages give
 *   none): per token a row of R = 16 * ceil((d/4 + d/8) / 16) bytes (48 for d = 128, 32 for
 *   d = 64), [units][n][R].  Per group of 32 channels, floor = the largest binary16 at or below
 *   the group's minimum key value and step = the smallest binary16 at or above
 *   float32((max - floor) / 3) (both clamped to +-65504); code = rint(float32((x - floor) /
 *   step)) clamped to 0..3 (0 when step is 0).  Bytes: d/4 of codes (channel c in bits
 *   2 (c mod 4) of byte c/4), then per group floor and step as little-endian binary16, then zero
 *   padding.  The certificate scores the keys floor + code * step; fetched tokens then move
 *   their K and V rows, since the GPU holds no exact key. */
enum { VERKV_SKETCH_EXACT = 0, VERKV_SKETCH_Q2 = 1 };
typedef struct {
    int32_t format;
    const void *data;
} verkv_sketch;

/* How verkv_fetch_refine moves the selected rows from the host-resident full cache.
 * ZEROCOPY: one kernel on the context's stream reads the selected rows straight from
 *           page-locked host memory and accumulates them into the refined estimator together
 *           with the sums over the resident tokens; the merge follows (no host round trip, no
 *           staging; default).
 * MEMCPY:   the host waits for the selection, gathers the rows into page-locked staging with a
 *           thread pool, and cudaMemcpyAsync moves them on the side stream while the sums over
 *           the resident tokens run.
 * With the exact sketch the GPU already holds every key, so by default only the V row of a
 * fetched token crosses the host link and its K row is read from the sketch; or-ing in
 * VERKV_FETCH_KEYS moves the full K|V row instead (same results, twice the link bytes). */
enum { VERKV_FETCH_ZEROCOPY = 0, VERKV_FETCH_MEMCPY = 1, VERKV_FETCH_KEYS = 4 };

/* Per query head results of one attend + fetch_refine, written by verkv_fetch_refine.
 *   m          max sketch logit q.k/sqrt(d) (the shift of every weight below)
 *   D          sum of sketch weights over all tokens (the certificate's D)
 *   beta       beta(L) of the fixed point of Definition 2
 *   V, b       V(L) and b(L) of Lemma 1
 *   eps_hat    eps-hat(L) of Eq. (7)
 *   eps_final  eps-hat(L_g[k*:]) of Eq. (10) (equals eps_hat when certified)
 *   D_hat      the returned estimator of D (shift m)
 *   M2         sum over sampled, unfetched tokens of (lambda w / r)^2 (1 - r), an unbiased
 *              estimate of V(L_g[k*:])
 *   lse        m + log(D_hat)
 *   certified  1 iff eps_hat < eps (no fetch needed)
 *   k_star     k* of Eq. (10)
 *   n_L        |L|
 *   n_fetch    |F \ S| for this head (rows not already resident)
 *   iters      iterations of the beta solve
 *   flags      or of: 1 the beta solve hit its cap; 2 the select ran out of passes;
 *              4 (shortlist variant only) the whole shortlist left eps-hat >= eps;
 *              8 the select ended by ranking its last candidates in one CTA (information only) */
typedef struct {
    float m, D, beta, V, b, eps_hat, eps_final, D_hat, M2, lse;
    int32_t certified, k_star, n_L, n_fetch, iters, flags;
} verkv_head_stats;

/* Bytes of a sketch of `format` for every unit of `shape` (0 if the shape or format is invalid). */
size_t verkv_sketch_bytes(const verkv_shape *shape, int32_t format);

/* Bytes of device workspace a context for `shape` needs (0 if the shape is invalid). */
size_t verkv_workspace_size(const verkv_shape *shape);

/* Create a context on `device` that issues work on `stream` (a cudaStream_t; NULL = legacy
 * default stream).  `workspace` is caller-owned device memory of at least
 * verkv_workspace_size(shape) bytes, 256-byte aligned; it must outlive the context and must not
 * be shared by two contexts.  Returns VERKV_EINVAL for a bad shape or workspace, VERKV_ECUDA if
 * the side stream or events cannot be created. */
verkv_status verkv_create(verkv_ctx **ctx, int device, void *stream, const verkv_shape *shape,
                          void *workspace, size_t workspace_bytes);

/* Release the side stream, events, staging and thread pool (after synchronising). */
void verkv_destroy(verkv_ctx *ctx);

/* Select VERKV_FETCH_ZEROCOPY or VERKV_FETCH_MEMCPY, optionally or-ed with VERKV_FETCH_KEYS.
 * MEMCPY allocates page-locked staging of units_per_layer * n * 4d bytes on first use. */
verkv_status verkv_set_fetch_mode(verkv_ctx *ctx, int mode_flags);

/* Sequence b of this context draws its Poisson sample as sequence seq0 + b (the fourth word of
 * the Philox counter in verkv_poissoncomp), so that a batch split over several contexts, each
 * holding the sequences seq0 .. seq0 + batch - 1 of it, draws exactly the sample that one context
 * for the whole batch would.  seq0 >= 0 (VERKV_EINVAL otherwise); 0 by default.  Takes effect at
 * the next verkv_poissoncomp. */
verkv_status verkv_set_sequence_offset(verkv_ctx *ctx, int32_t seq0);

/* PoissonComp (summary page, Methodology, POISSONCOMP: Eq. (3), the H / L partition and the
 * Poisson sample S), for every unit of the shape.
 *   tau     device float [units][n]: normalised importance scores; must be finite and in (0, 1]
 *           outside the forced H set (VERKV_EINVAL on the device otherwise)
 *   eta     budget fraction in (0, 1]; requires eta * n > n_sink + n_local when tokens remain
 *           outside the forced set (VERKV_EBUDGET, checked on the host before any launch)
 *   H       the forced H set
 *   seed    Philox4x32-10 key; token i of unit (b, l, h) draws word i%4 of the block at counter
 *           (i/4, h, l, seq0 + b) (seq0 from verkv_set_sequence_offset, 0 by default),
 *           u_i = (word >> 8) * 2^-24, and is kept iff u_i < r_i
 *   kv_full device bf16 [units][n][2][d]: the full cache, read to fill out->kv
 *   r_full  device float [units][n] out: r_i = min(1, c tau_i) for every token (1 in H)
 *   out     the pivotal set (every member must point to caller device memory of the sizes above)
 * c is the exact root of sum_i min(1, c tau_i) = eta n, located by bisection and finished
 * exactly on its linear piece, then published as float32; r_i is the float32 product. */
verkv_status verkv_poissoncomp(verkv_ctx *ctx, const float *tau, double eta, verkv_hset H,
                               uint64_t seed, const void *kv_full, float *r_full,
                               const verkv_pivotal *out);

/* Build the sketch from the full device cache kv_full bf16 [units][n][2][d] into sketch_out
 * (device, verkv_sketch_bytes(shape, format) bytes).  VERKV_SKETCH_EXACT copies every key row
 * (bf16 [units][n][d]); VERKV_SKETCH_Q2 quantises every key row to 2 bits (layout above). */
verkv_status verkv_sketch_build(verkv_ctx *ctx, const void *kv_full, int32_t format,
                                void *sketch_out);

/* KVFetch steps 1-4 for one layer (summary page, KVFETCH: Verification and Adaptive Fetching;
 * Definition 2, Lemma 1, Eqs. (5), (7), (9), (10)) plus the estimator over the resident tokens.
 *   layer          which layer of the shape
 *   q              device bf16 [batch][kv_heads * q_per_kv][d]: one decode query per sequence
 *   pivotal        the PoissonComp output (all layers; this call reads layer `layer`)
 *   r_full         device float [units][n] from verkv_poissoncomp
 *   sketch         the sketch (all layers)
 *   eps, delta     the tolerance: certified iff eps-hat(L) < eps; 0 < delta < 1; eps > 0
 *   fetch_ids_out  optional (NULL) device or page-locked host int32 [batch*kv_heads][n]: for each
 *                  KV head of this layer, the ascending ids of the union over its query heads of
 *                  F \ S (the rows that must move)
 *   fetch_counts_out optional int32 [batch*kv_heads]: the number of ids per KV head (either
 *                  output may be given without the other).  The list is built at the end of the
 *                  certificate kernel only when one of the two is given or the fetch mode is
 *                  MEMCPY; in ZEROCOPY mode verkv_fetch_refine reads the selection bitmaps
 *                  directly, so a caller that needs neither output saves that step.
 * Per query head: sketch logits for all n tokens, w-hat = exp(logit - max), the beta fixed point,
 * the certificate, and when it fails the order of Eq. (9) (ties to the lower token id) and the
 * minimal k* of Eq. (10).  In MEMCPY mode the shrinkage-weighted partial sums over the pivotal
 * set follow here; in ZEROCOPY mode verkv_fetch_refine computes them.
 * Asynchronous; results are completed by verkv_fetch_refine, which reads q, the pivotal set and
 * the sketch again: keep them unchanged until it has been issued. */
verkv_status verkv_attend_verified(verkv_ctx *ctx, int32_t layer, const void *q,
                                   const verkv_pivotal *pivotal, const float *r_full,
                                   const verkv_sketch *sketch, float eps, float delta,
                                   int32_t *fetch_ids_out, int32_t *fetch_counts_out);

/* KVFetch step 5 and the refined attention (summary page, KVFETCH step 5 and Theorem 2;
 * abstract page: fetch additional tokens from the CPU and refine).
 *   ids, counts  NULL, or exactly the fetch_ids_out / fetch_counts_out pointers given to the
 *                preceding verkv_attend_verified (VERKV_EINVAL otherwise)
 *   host_kv      page-locked host bf16 [units][n][2][d]: the complete cache
 *   o_out        device float [batch][kv_heads * q_per_kv][d]: N-hat / D-hat
 *   lse_out      optional device float [batch][kv_heads * q_per_kv]: m + log D-hat
 *   stats_out    optional device verkv_head_stats [batch][kv_heads * q_per_kv]
 * Returns VERKV_ESTATE without a preceding attend on this context. */
verkv_status verkv_fetch_refine(verkv_ctx *ctx, const int32_t *ids, const int32_t *counts,
                                const void *host_kv, float *o_out, float *lse_out,
                                verkv_head_stats *stats_out);

/* Shortlist variant (summary page, Experimental Setup: "128-token shortlist per KV head"; the
 * pages give it no further role, so this is our reading).  With size S in 1 .. 256, each later
 * verkv_attend_verified first picks, per KV head, the S tokens of L with the largest sketch
 * logit over the KV head's query heads (ties to the lower token id), and a query head whose
 * certificate fails may fetch only those: the order of Eq. (10) runs over the shortlist while
 * every other token of L stays in the remaining set.  If the whole shortlist still leaves
 * eps-hat >= eps, all of it is fetched and the head's stats flags include 4 (the returned
 * estimator is then not certified).  S = 0 (the default) turns it off.  VERKV_EINVAL otherwise. */
verkv_status verkv_set_shortlist(verkv_ctx *ctx, int32_t size);

/* Copy the shortlists of the preceding verkv_attend_verified into `out`, device or page-locked
 * host uint32 [batch * kv_heads][ceil(n/32)] (bit i%32 of word i/32 set iff token i is listed).
 * Stream-ordered; VERKV_ESTATE if no attend with the shortlist on has run on this context. */
verkv_status verkv_shortlist_bitmap(verkv_ctx *ctx, uint32_t *out);

/* The offloaded-dense baseline (summary page, System Performance: the "Dense (offload)" system
 * VerKV is compared with): exact attention for every query head of `layer` over all n tokens,
 * every K|V row read from the page-locked host cache -- nothing of the cache is resident.
 *   q        device bf16 [batch][kv_heads * q_per_kv][d]
 *   host_kv  page-locked host bf16 [units][n][2][d]
 *   o_out    device float [batch][kv_heads * q_per_kv][d]: softmax(q K^T / sqrt(d)) V
 *   lse_out  optional device float [batch][kv_heads * q_per_kv]: log sum_i exp(q.k_i / sqrt(d))
 * Uses the context's workspace; independent of verkv_attend_verified (its state is untouched). */
verkv_status verkv_attend_dense_host(verkv_ctx *ctx, int32_t layer, const void *q,
                                    const void *host_kv, float *o_out, float *lse_out);

/* Copy the per-query-head fetch sets F of the preceding verkv_attend_verified (Eq. (10):
 * F = L \ L_g[k*:]) into `out`, device or page-locked host uint32
 * [batch * kv_heads * q_per_kv][ceil(n/32)] (bit i%32 of word i/32 set iff token i is in F).
 * Stream-ordered; VERKV_ESTATE if no attend has run on this context. */
verkv_status verkv_selection_bitmap(verkv_ctx *ctx, uint32_t *out);

/* Allocation-free certificate.  The paper has no counterpart: this is a convenience of the
 * library.  Some callers cannot call cudaMalloc -- for instance code inside a serving runtime that
 * has already reserved the GPU's memory for its own KV pools, or a plugin interface that hands an
 * operator only its input and output buffers -- and so cannot provide the workspace a context
 * needs.  This call runs the same sketch-logit and certificate/selection kernels as
 * verkv_attend_verified (the certificate, beta, k* and F of every query head) without a context
 * and without allocating: the logits live in one array of VERKV_NOALLOC_MAX_LOGITS floats
 * (16 MiB) that the library keeps on every GPU that loads it, until the process exits.
 *   device     the GPU to run on; made current for the call, and the caller's current device
 *              is restored before the call returns
 *   stream     cudaStream_t the kernels are issued on (NULL = legacy default stream)
 *   units      KV heads in this call (consecutive in every array below)   >= 1
 *   q_per_kv   query heads per KV head                                    1, 2, 4, 8
 *   head_dim   d                                                          64 or 128
 *   n          tokens per unit                                            1 .. 131072
 *   q          device bf16 [units * q_per_kv][d], 16-byte aligned
 *   sketch     device bf16 [units][n][d] exact sketch, 16-byte aligned
 *   r_full     device float [units][n] from verkv_poissoncomp (r_i < 1 marks L); r_full,
 *              stats_out, F_out and err_out must be 4-byte aligned
 *   eps, delta the tolerance, as in verkv_attend_verified
 *   stats_out  device verkv_head_stats [units * q_per_kv]: the certificate fields (m, D, beta,
 *              V, b, eps_hat, eps_final, certified, k_star, n_L, iters, flags); D_hat, M2, lse
 *              and n_fetch are written as 0
 *   F_out      device uint32 [units * q_per_kv][ceil(n/32)]: the fetch set F of each query head,
 *              laid out as in verkv_selection_bitmap
 *   err_out    device uint32, one word: set to 0 by the call, then or-ed on the device with 4
 *              if a beta solve hit its iteration cap, 16 if a bounded copy wait expired (the
 *              outputs of that call are then not valid)
 * Returns VERKV_ETOOLARGE, launching nothing, when units * q_per_kv * n exceeds
 * VERKV_NOALLOC_MAX_LOGITS; VERKV_EINVAL for another bad argument (a misaligned pointer
 * included), checked before any CUDA call; VERKV_ECUDA if a CUDA call fails.  The first call on a device also looks up the device address of the array (set-up that
 * runs once per device); make that first call before any stream capture.  All calls on a GPU
 * share the array, which keeps the last call's logits: nothing in it has to start at zero, as
 * every call writes each logit before reading it, but calls that overlap on the GPU (other
 * streams, other host threads) race on it and must be ordered by the caller. */
enum { VERKV_NOALLOC_MAX_LOGITS = 1 << 22 };
verkv_status verkv_certify_noalloc(int device, void *stream, int32_t units, int32_t q_per_kv,
                                   int32_t head_dim, int32_t n, const void *q, const void *sketch,
                                   const float *r_full, float eps, float delta,
                                   verkv_head_stats *stats_out, uint32_t *F_out,
                                   uint32_t *err_out);

/* Failure injection, for tests of the error paths (each affects only this context; nothing
 * faults, traps or hangs the GPU):
 *   VERKV_INJECT_COPY_FAIL   value > 0: the next `value` MEMCPY-mode fetch copies fail on the host
 *                            without reaching CUDA, and verkv_fetch_refine returns VERKV_ECOPY
 *   VERKV_INJECT_BETA_MAXIT  value >= 1: the beta solve stops after `value` passes (a head that
 *                            needs more is flagged and verkv_sync returns VERKV_ENOCONVERGE);
 *                            0 restores the default cap
 *   VERKV_INJECT_SCORE_STALL value >= 1000: in the next verkv_attend_verified the first CTA of the
 *                            sketch-scoring kernel arms its first copy barrier for a copy it never
 *                            issues, and its bounded copy waits give up after `value` ns; the
 *                            kernel latches VERKV_ETIMEOUT (returned by verkv_sync) and returns,
 *                            and the context stays usable.  One call only.
 *   VERKV_INJECT_SELECT_GATHER value 0: the selection never ends by gathering its last candidates
 *                            into one CTA (clusters of 1 and 4 do by default, when at most 512
 *                            remain) but runs its histogram passes to the end, for a bitwise
 *                            comparison of the two; 1 restores the default.
 * Returns VERKV_EINVAL for an unknown `what` or a value out of range. */
enum { VERKV_INJECT_COPY_FAIL = 1, VERKV_INJECT_BETA_MAXIT = 2, VERKV_INJECT_SCORE_STALL = 3,
       VERKV_INJECT_SELECT_GATHER = 4 };
verkv_status verkv_test_inject(verkv_ctx *ctx, int what, int64_t value);

/* Measurement.  Every kernel launch is counted per kernel; with profiling enabled each launch is
 * also bracketed by two CUDA events on the stream it runs on (host cost ~2 event records).
 * Kernel ids, in launch order: */
enum {
    VERKV_K_PC_SOLVE = 0,      /* PoissonComp c solve, r, sample, compaction     */
    VERKV_K_PC_GATHER,         /* pivotal K/V row gather                          */
    VERKV_K_SKETCH,            /* sketch build (exact or 2-bit)                   */
    VERKV_K_SCORE,             /* sketch logits for every token and query head    */
    VERKV_K_CERTIFY,           /* beta solve, certificate, selection (Eq. 7-10),
                                  and the per-KV-head fetch id list               */
    VERKV_K_PARTIAL_PIVOTAL,   /* shrinkage-weighted sums over the pivotal set
                                  (MEMCPY mode)                                   */
    VERKV_K_FETCH_HOST,        /* "k_refine": zero-copy fetch, exact sums over the
                                  fetched rows and the pivotal sums               */
    VERKV_K_PARTIAL_STAGED,    /* exact sums over rows staged by cudaMemcpyAsync  */
    VERKV_K_MERGE,             /* merge partials into o, lse and statistics       */
    VERKV_K_DENSE_HOST,        /* offloaded-dense baseline: all rows from host    */
    VERKV_K_DENSE_MERGE,       /* its running-max merge                           */
    VERKV_K_SHORTLIST,         /* per-KV-head fetch shortlist (when enabled)      */
    VERKV_K_FETCH_COPY,        /* MEMCPY mode: the side stream's host-to-device
                                  copies of one fetch (not a kernel; timed with
                                  events on the side stream when profiling)       */
    VERKV_K_FETCH_GATHER,      /* MEMCPY mode: the host threads' gather of the
                                  fetched rows into page-locked staging (events on
                                  the idle side stream mark its start and end)    */
    VERKV_K_COUNT
};

/* Start (on != 0) or stop recording per-launch events.  Do not enable during stream capture. */
verkv_status verkv_profile_enable(verkv_ctx *ctx, int on);

/* Wait for the context's streams, then add the recorded launches and their event-timed
 * milliseconds per kernel id into launches[VERKV_K_COUNT] and total_ms[VERKV_K_COUNT]
 * (caller-zeroed host arrays) and discard the records. */
verkv_status verkv_profile_read(verkv_ctx *ctx, int64_t *launches, double *total_ms);

/* The recorded launches since the last verkv_profile_read, in record order, without discarding
 * them: kernel id and start / end in milliseconds from the first record's start event (host
 * arrays of max_records entries; *n_out the number written, at most max_records).  Waits for the
 * context's streams.  With MEMCPY mode this shows the side stream's copies (VERKV_K_FETCH_COPY)
 * against the pivotal sums on the main stream (VERKV_K_PARTIAL_PIVOTAL). */
verkv_status verkv_profile_timeline(verkv_ctx *ctx, int64_t max_records, int32_t *kernel,
                                    double *start_ms, double *end_ms, int64_t *n_out);

/* Measurement: stream the exact sketch rows that verkv_attend_verified would score for `layer`
 * (every KV head of the layer, d * 2 bytes a token) through the scoring kernel's copy grid and
 * ring, without any arithmetic, on the context's stream (asynchronous).  Its time is that of a
 * bare one-launch read of the same bytes, the reference the scoring kernel's time is set
 * against.  The sketch must be VERKV_SKETCH_EXACT with a 16-byte aligned data pointer, else
 * VERKV_EINVAL; bad layer: VERKV_EINVAL.  Not counted in verkv_launch_counts. */
verkv_status verkv_measure_sketch_stream(verkv_ctx *ctx, int32_t layer, const verkv_sketch *sketch);

/* Kernel launches issued by this context since it was created, per kernel id
 * (out[VERKV_K_COUNT], host).  Counts launches made during stream capture once. */
verkv_status verkv_launch_counts(verkv_ctx *ctx, int64_t *out);

/* Name of a kernel id ("" if out of range). */
const char *verkv_kernel_name(int kernel);

/* Wait for all work on the context's streams, then return (and clear) the first error latched
 * by the device since the previous verkv_sync, or a pending CUDA error. */
verkv_status verkv_sync(verkv_ctx *ctx);

/* Text of the last error on this context ("" if none). */
const char *verkv_last_error(verkv_ctx *ctx);

/* Name of a status code. */
const char *verkv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* VERKV_H */
