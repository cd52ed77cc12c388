// k_attend.cu -- the bounded shrinkage estimator over the GPU-resident pivotal tokens, the
// refine over fetched tokens, and the merge ("Verify Before You Fetch", summary page,
// Definition 2 / Eq. (5), KVFETCH step 5; abstract page: fetch additional tokens from the CPU and
// refine the attention computation).
//
// k_partial   split-K over a row set: each CTA item is a block of PIV_ITEM_ROWS pivotal rows, or
//             the fetched rows of one FET_RANGE token-id range, of one KV head, taken 64 at a
//             time; each row a contiguous 4d-byte K|V pair read with 16-byte coalesced loads,
//             four row groups in flight per warp (all of them for host rows), accumulated into
//             one partial.  It computes the G logits, w = exp(logit - m), the
//             weight of Eq. (5) -- 1 for H and for tokens of F, lambda / r for sampled, unfetched
//             tokens, with the certificate's lambda = clip(beta r / (w-hat (1 - r)), r, 1) from
//             the sketch weight w-hat, taken as lambda / r = clip(beta / (w-hat (1 - r)), 1, 1 / r)
//             -- and accumulates D-hat, N-hat and the sample second moment.  All CTAs of a query head share its shift m, so partials add without
//             rescaling.  Three row sources:
//               ROWS_PIVOTAL   the pivotal buffer in HBM;
//               ROWS_STAGED    fetched rows already copied to HBM (the cudaMemcpyAsync fetch);
//               ROWS_HOST      fetched rows read straight from page-locked host memory by token
//                              id -- the zero-copy fetch and the refine in one pass, no staging.
//             When the sketch is exact the GPU already holds every key, so K comes from the sketch
//             by token id and only the V rows cross the host link.
// k_pivotal   the pivotal set's pass of the MEMCPY path (during the host gather): a producer warp
//             streams 64-row stages of K|V rows (TMA tensor copies, 128-byte swizzle), ids and r
//             into a two-stage shared-memory ring; four consumer warps sum them on the tensor cores
//             with the stage code of pivotal_mma.cuh, which every pivotal path shares (the same
//             bits); each CTA takes a run of 256-row chunks holding about an equal share of rows.
// k_refine    the zero-copy path's partial sums in one launch: the ROWS_HOST items of every KV
//             head, each deriving its rows from the selection bitmaps of one token-id range (no
//             fetch list needed), and the pivotal items (the same stage code).
// k_merge     sums the partials in a fixed order and writes o = N-hat / D-hat, m + log D-hat and
//             the per-head statistics.
// k_dense_host, k_dense_merge   the offloaded-dense baseline: exact attention over every token with
//             the K|V rows read from page-locked host memory, online-softmax partials per chunk.
#include <math.h>

#include <cuda.h>

#include <algorithm>

#include "pivotal_mma.cuh"
#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

template <int G, int LPR>
__device__ __forceinline__ float reduce_heads_a(float (&p)[G], int lane) {
    int hc = G;
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
        if (hc > 1) {
            const int half = hc / 2;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int j = 0; j < G / 2; ++j) {
                if (j < half) {
                    const float send = upper ? p[j] : p[half + j];
                    const float keep = upper ? p[half + j] : p[j];
                    p[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
                }
            }
            hc = half;
        } else {
            p[0] += __shfl_xor_sync(0xFFFFFFFFu, p[0], off);
        }
    }
    return p[0];
}

// The head a lane holds after reduce_heads_a (a function of its lane bits only).
template <int G, int LPR>
__device__ __forceinline__ int head_of_lane(int lane) {
    int head = 0, hc = G;
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
        if (hc > 1) {
            const int half = hc / 2;
            if (lane & off) head += half;
            hc = half;
        }
    }
    return head;
}

// Row-group lane (0..LPR-1) holding head g after reduce_heads_a.
template <int G, int LPR>
__device__ __forceinline__ int lane_of_head(int g) {
    int lanebits = 0, hc = G, off = LPR / 2;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (hc > 1) {
            const int half = hc / 2;
            if (g >= half) {
                lanebits |= off;
                g -= half;
            }
            hc = half;
            off >>= 1;
        }
    }
    return lanebits;
}

template <int G>
__device__ __forceinline__ float pick(const float (&v)[G], int i) {
    float r = v[0];
#pragma unroll
    for (int g = 1; g < G; ++g) r = (i == g) ? v[g] : r;
    return r;
}

__device__ __forceinline__ uint4 ld_host(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// One item of the split-K sums over fetched rows: positions [lo, hi) of a row list of layer unit
// `ul` (ids[p] is the token id at position p), taken PART_ROWS at a time, into partial
// `part_idx`.  Row data is addressed by token id (ROWS_HOST: the unit's host cache) or by list
// position (ROWS_STAGED: rows copied to the device).  A fetched row is exact: weight 1 for the
// query heads whose F holds it, 0 for the others.  An empty item writes nothing unless
// write_empty (then a zero partial).  lo and hi are uniform over the CTA.
template <int D, int G, int MODE>
__device__ __forceinline__ void partial_rows(const PartialArgs &a, int ul, int part_idx, int lo,
                                             int hi, const int32_t *ids, bool write_empty) {
    static_assert(MODE == ROWS_HOST || MODE == ROWS_STAGED, "fetched rows only");
    constexpr int LPR = D / 8, RPW = 32 / LPR, NW = 4;
    constexpr int ITER = (PART_ROWS / NW) / RPW;  // row groups per warp
    // Row groups in flight per warp: all of them for host rows (link latency), else four.
    constexpr int U = MODE == ROWS_HOST ? ITER : (ITER < 4 ? ITER : 4);
    constexpr int SUBMASK = LPR / G - 1;
    __shared__ float sN[NW][G][D];
    __shared__ float sD[NW][RPW][G];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cgp = lane % LPR, rg = lane / LPR;
    const int myhead = head_of_lane<G, LPR>(lane);
    const int hq = a.li.kv_heads * G;
    if (lo >= hi && !write_empty) return;

    const int b = ul / a.li.kv_heads, h = ul - b * a.li.kv_heads;
    const int ug = a.li.unit_global(ul);
    float qv[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 v = *reinterpret_cast<const uint4 *>(a.q + ((size_t)b * hq + h * G + g) * D + cgp * 8);
        unpack8(v, qv[g]);
    }
    const float mh_ = a.qstats[ul * G + myhead].m;
    const uint32_t *Fh = a.F + (size_t)(ul * G + myhead) * a.W;
    float acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[g][c] = 0.0f;
    float dacc = 0.0f;

    // ROWS_HOST indexes the full host cache of the unit by token id; ROWS_STAGED by position
    // from the unit's first staged row.
    const uint4 *rows = reinterpret_cast<const uint4 *>(a.rows) +
                        (MODE == ROWS_HOST ? (size_t)ug * a.n : (size_t)a.staged_off[ul]) * a.row16;
    const uint4 *keys = a.keys ? reinterpret_cast<const uint4 *>(a.keys) + (size_t)ug * a.n * (D / 8)
                               : nullptr;
#pragma unroll 1
    for (int cbase = lo; cbase < hi; cbase += PART_ROWS) {
        const int rbase = cbase + warp * (PART_ROWS / NW);
#pragma unroll 1
        for (int it0 = 0; it0 < ITER; it0 += U) {
            int id[U];
            bool valid[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int row = rbase + (it0 + u) * RPW + rg;
                valid[u] = row < hi;
                id[u] = valid[u] ? ids[row] : 0;
                if ((unsigned)id[u] >= (unsigned)a.n) {  // not a token of the unit: skip the row
                    raise_error(a.err, ERR_BADID);
                    valid[u] = false;
                    id[u] = 0;
                }
            }
            uint4 kq[U], vq[U];
            uint32_t fw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                kq[u] = make_uint4(0, 0, 0, 0);
                vq[u] = make_uint4(0, 0, 0, 0);
                fw[u] = 0u;
                if (valid[u]) {
                    const size_t rr = MODE == ROWS_HOST ? (size_t)id[u] : (size_t)(rbase + (it0 + u) * RPW + rg);
                    if (keys) {
                        kq[u] = ldg_stream(keys + (size_t)id[u] * (D / 8) + cgp);
                    } else if (MODE == ROWS_HOST) {
                        kq[u] = ld_host(rows + rr * a.row16 + cgp);
                    } else {
                        kq[u] = ldg_stream(rows + rr * a.row16 + cgp);
                    }
                    if (MODE == ROWS_HOST) {
                        vq[u] = ld_host(rows + rr * a.row16 + a.voff16 + cgp);
                    } else {
                        vq[u] = ldg_stream(rows + rr * a.row16 + a.voff16 + cgp);
                    }
                    fw[u] = Fh[id[u] >> 5];
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float k[8], v[8];
                unpack8(kq[u], k);
                unpack8(vq[u], v);
                float p[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float s = 0.0f;
#pragma unroll
                    for (int c = 0; c < 8; ++c) s = fmaf(qv[g][c], k[c], s);
                    p[g] = s;
                }
                const float dot = reduce_heads_a<G, LPR>(p, lane);
                // Weight of this row for the lane's head: exact w if the head's F holds it.
                float cw = 0.0f;
                if (valid[u] && ((fw[u] >> (id[u] & 31)) & 1u)) {
                    // Weights to a few 1e-6 relative (the exp2-based exponential): the sums need 1e-3.
                    cw = __expf(dot * a.scale - mh_);
                    if ((cgp & SUBMASK) == 0) dacc += cw;
                }
                // Every lane of the row needs the weight of every head.
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float cwg = __shfl_sync(0xFFFFFFFFu, cw, rg * LPR + lane_of_head<G, LPR>(g));
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[g][c] = fmaf(cwg, v[c], acc[g][c]);
                }
            }
        }
    }
    // Reduce over the row groups of the warp, then over warps (fixed order).
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[g][c] += __shfl_xor_sync(0xFFFFFFFFu, acc[g][c], off);
    if (rg == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < 8; ++c) sN[warp][g][cgp * 8 + c] = acc[g][c];
    }
    if ((cgp & SUBMASK) == 0) sD[warp][rg][myhead] = dacc;
    __syncthreads();
    float *out = a.part + ((size_t)ul * a.max_chunks + part_idx) * G * (D + 2);
    for (int e = tid; e < G * (D + 2); e += 128) {
        const int g = e / (D + 2), c = e - g * (D + 2);
        float s = 0.0f;
        if (c < D) {
#pragma unroll
            for (int w = 0; w < NW; ++w) s += sN[w][g][c];
        } else if (c == D) {
#pragma unroll
            for (int w = 0; w < NW; ++w)
#pragma unroll
                for (int j = 0; j < RPW; ++j) s += sD[w][j][g];
        }  // c == D + 1: a fetched row adds nothing to the second moment
        out[e] = s;
    }
    __syncthreads();
}

// 16-byte asynchronous copy global -> shared (L2 only), and the wait for all of this thread's.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The pivotal rows [ch PIV_ITEM_ROWS, ...) of layer unit `ul` into partial `ch`, staged by the
// CTA's 128 threads with 16-byte asynchronous copies into the swizzled stage layout (stage rows
// beyond the unit's count are zeros), PIV_STAGE_ROWS at a time in `buf` (PivLayout<D>::BYTES of
// shared memory, 16-byte aligned).
template <int D, int G, bool SKL>
__device__ __forceinline__ void pivotal_chunk_plain(const PartialArgs &a, int ul, int ch,
                                                    unsigned char *buf) {
    using LY = PivLayout<D>;
    static_assert(piv_red_bytes<D, G>() <= LY::BYTES, "the reduction reuses the stage");
    const int ug = a.li.unit_global(ul);
    const int count = min(a.count[ug], a.row_stride);
    const int lo = ch * PIV_ITEM_ROWS;
    if (lo >= count) return;  // uniform over the CTA
    const int hi = min(lo + PIV_ITEM_ROWS, count);
    PivChunk<D, G, SKL> pc;
    pc.init(a, ul);
    const int tid = threadIdx.x;
    constexpr int VPR = LY::ROWB / 16;  // 16-byte vectors per row
    const uint4 *src = reinterpret_cast<const uint4 *>(a.rows) + (size_t)ug * a.row_stride * VPR;
    for (int s0 = lo; s0 < hi; s0 += LY::ROWS) {
        const int rows = min(LY::ROWS, hi - s0);
        for (int v = tid; v < LY::ROWS * VPR; v += 128) {
            const int r = v / VPR, c = v - r * VPR;  // c: 16-byte chunk of the K|V row
            constexpr int KC = D / 8;                // chunks of a K (or V) row
            unsigned char *dst = buf + LY::off(c / KC, r, (c % KC) * 8);
            if (r < rows) cp_async16(dst, src + (size_t)(s0 + r) * VPR + c);
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (tid < LY::ROWS) {
            const size_t at = (size_t)ug * a.row_stride + s0 + tid;
            reinterpret_cast<int32_t *>(buf + LY::IDS)[tid] = tid < rows ? a.ids[at] : 0;
            reinterpret_cast<float *>(buf + LY::RS)[tid] = tid < rows ? a.pr[at] : 1.0f;
        }
        cp_async_wait_all();
        __syncthreads();
        pc.stage(a, buf, rows);
        __syncthreads();
    }
    pc.finish(reinterpret_cast<float *>(buf), a.part + ((size_t)ul * a.max_chunks + ch) * G * (D + 2),
              true, [] { __syncthreads(); });
}

// The fetched rows of layer unit `ul` with token ids in [k * FET_RANGE, (k + 1) * FET_RANGE):
// positions [lo, hi) of the unit's ascending fetch list (binary search, one thread).
__device__ __forceinline__ void range_bounds(const int32_t *list, int count, int k, int &lo, int &hi) {
    __shared__ int s_b[2];
    if (threadIdx.x == 0) {
        for (int e = 0; e < 2; ++e) {
            const int key = (k + e) * FET_RANGE;
            int l = 0, r = count;  // first position whose id >= key
            while (l < r) {
                const int m = (l + r) >> 1;
                if (list[m] < key) l = m + 1;
                else r = m;
            }
            s_b[e] = l;
        }
    }
    __syncthreads();
    lo = s_b[0];
    hi = s_b[1];
    __syncthreads();
}

// Pivotal rows in chunks of PIV_ITEM_ROWS list positions (staged by the CTA itself: the fallback
// when a pivotal buffer cannot be bulk-copied); staged fetched rows by token-id range (FET_RANGE
// ids per partial, a zero partial for an empty range), as k_refine reads them from host memory,
// so that both fetch modes produce the same partials.
template <int D, int G, int MODE, bool SKL>
__global__ void __launch_bounds__(128) k_partial(PartialArgs a, int units_layer) {
    extern __shared__ __align__(128) unsigned char kp_stage[];  // pivotal: PivLayout<D>::BYTES
    pdl_wait();
    pdl_trigger();
    const int total_items = units_layer * a.max_chunks;
    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int ul = item / a.max_chunks, ch = item - ul * a.max_chunks;
        if (MODE == ROWS_PIVOTAL) {
            pivotal_chunk_plain<D, G, SKL>(a, ul, ch, kp_stage);
        } else {
            const int32_t *list = a.ids + (size_t)ul * a.row_stride;
            int lo, hi;
            range_bounds(list, min(a.count[ul], a.row_stride), ch, lo, hi);
            if (threadIdx.x == 0 && lo < hi) atomicOr(&a.rmask[ul * RMASK_W + (ch >> 5)], 1u << (ch & 31));
            partial_rows<D, G, ROWS_STAGED>(a, ul, ch, lo, hi, list, false);
        }
    }
}

// The CTA's run of pivotal items (item = unit * max_chunks + chunk, in unit order).  A chunk's first
// row, counted over the layer's units, is nondecreasing in the item index (a chunk past its unit's
// count starts at the unit's end), so cutting the rows into gridDim.x equal ranges and giving each
// chunk to the range that holds its first row splits the items into contiguous runs of about
// equal rows: at most one chunk more than an equal share.  Every thread of the CTA calls it and
// gets the same run.
template <int NT>
__device__ void pivotal_run(const PartialArgs &a, int units_layer, int &item0, int &item1) {
    __shared__ int s_wsum[NT / 32];
    __shared__ int s_cut[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total_items = units_layer * a.max_chunks;
    const int per_t = (units_layer + NT - 1) / NT;  // units per thread
    const int u0 = min(units_layer, tid * per_t), u1 = min(units_layer, u0 + per_t);
    int mine = 0;
    for (int u = u0; u < u1; ++u) mine += min(a.count[a.li.unit_global(u)], a.row_stride);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    if (tid == 0) s_cut[0] = s_cut[1] = total_items;
    __syncthreads();
    int base = incl - mine, rows = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        if (w < warp) base += s_wsum[w];
        rows += s_wsum[w];
    }
    const long long share = ((long long)rows + gridDim.x - 1) / gridDim.x;
    const long long lo_row = share * blockIdx.x, hi_row = lo_row + share;
    int first_lo = total_items, first_hi = total_items;
    long long p = base;
    for (int u = u0; u < u1; ++u) {
        const int cnt = min(a.count[a.li.unit_global(u)], a.row_stride);
        for (int ch = 0; ch < a.max_chunks; ++ch) {
            const long long start = p + min(ch * PIV_ITEM_ROWS, cnt);
            const int item = u * a.max_chunks + ch;
            if (start >= lo_row) first_lo = min(first_lo, item);
            if (start >= hi_row) first_hi = min(first_hi, item);
        }
        p += cnt;
    }
    if (first_lo < total_items) atomicMin(&s_cut[0], first_lo);
    if (first_hi < total_items) atomicMin(&s_cut[1], first_hi);
    __syncthreads();
    item0 = s_cut[0];
    item1 = max(item0, s_cut[1]);
}

// k_pivotal: the estimator's pass over the pivotal set on its own (MEMCPY mode, where it runs
// during the host gather).  Warps 0-3 consume, warp 4 produces: for every stage of PIV_STAGE_ROWS
// rows of the CTA's chunks (a contiguous run of them) the producer waits for the
// ring slot to be released, then issues one tensor copy per 64-channel box (the tensor map
// describes the pivotal rows as [rows][K|V][d] bf16 with the 128-byte swizzle) and two bulk copies
// for the ids and r, all completing on the slot's mbarrier; the consumers run the stage on the
// tensor cores and release the slot.  Box rows past the unit's count hold other rows (or the
// zero fill past the buffer); the consumer that owns them zeroes them before use.  Waits are
// bounded: on expiry (or once another thread has given up) the kernel keeps its control flow but
// skips the work, latches ERR_TIMEOUT, waits (bounded) for the copies it issued and returns.
constexpr int PV_NS = 2;         // ring slots per CTA
constexpr int PV_CONS = 4;       // consumer warps
constexpr int PV_NT = 32 * (PV_CONS + 1);
constexpr int PV_CTAS_PER_SM = 3;
template <int D, int G>
__host__ __device__ constexpr size_t pv_smem_bytes() {
    // 1024 bytes of slack: the ring starts at the first 1024-byte boundary (the swizzle's unit).
    // The chunk-end reduction runs in the ring slot of the chunk's last stage.
    static_assert(piv_red_bytes<D, G>() <= PivLayout<D>::BYTES, "the reduction fits a slot");
    return 1024 + (size_t)PV_NS * PivLayout<D>::BYTES;
}

template <int D, int G, bool SKL>
__global__ void __launch_bounds__(PV_NT, PV_CTAS_PER_SM) k_pivotal(PartialArgs a, int units_layer,
                                                                  const __grid_constant__ CUtensorMap rows_map) {
    using LY = PivLayout<D>;
    extern __shared__ __align__(1024) unsigned char pv_raw[];
    __shared__ __align__(8) uint64_t full[PV_NS], empty[PV_NS];
    __shared__ int s_abort;
    __shared__ int s_last[PV_NS];  // the last stage issued into each slot (-1: none)
    unsigned char *pv_smem = pv_raw + ((1024u - (smem_addr(pv_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < PV_NS * LY::BYTES / 16; i += PV_NT)
        reinterpret_cast<uint4 *>(pv_smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        for (int k = 0; k < PV_NS; ++k) {
            mbar_init(&full[k], 1);
            mbar_init(&empty[k], PV_CONS);
            s_last[k] = -1;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    fence_proxy_async_smem();  // the zeros before any copy into the same memory
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    volatile int *abort = &s_abort;
    // A contiguous run of items per CTA (consecutive chunks of a unit share its queries), with
    // about the same number of rows in every run.
    int item0, item1;
    pivotal_run<PV_NT>(a, units_layer, item0, item1);
    if (warp == PV_CONS) {
        if (lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&rows_map)) : "memory");
        int j = 0, cur = -1, ug = 0, count = 0;
        for (int item = item0; item < item1; ++item) {
            const int ul = item / a.max_chunks, ch = item - ul * a.max_chunks;
            if (ul != cur) {
                cur = ul;
                ug = a.li.unit_global(ul);
                count = min(a.count[ug], a.row_stride);
            }
            const int lo = ch * PIV_ITEM_ROWS;
            if (lo >= count) continue;
            const int hi = min(lo + PIV_ITEM_ROWS, count);
            for (int s0 = lo; s0 < hi; s0 += LY::ROWS, ++j) {
                const int slot = j % PV_NS;
                if (lane != 0) continue;
                bool go = *abort == 0;
                if (go && j >= PV_NS)
                    go = mbar_wait_or_abort(&empty[slot], (uint32_t)(((j / PV_NS) - 1) & 1), abort);
                if (!go) {
                    *abort = 1;
                    continue;
                }
                const int rows = min(LY::ROWS, hi - s0);
                const uint32_t lb = (uint32_t)((rows + 3) & ~3) * 4;  // within the capacity (a multiple of 4)
                unsigned char *st = pv_smem + (size_t)slot * LY::BYTES;
                const int row_g = ug * a.row_stride + s0;  // row of the tensor map
                mbar_expect_tx(&full[slot], (uint32_t)(LY::NB * LY::BOX) + 2 * lb);
                s_last[slot] = j;
#pragma unroll
                for (int b = 0; b < LY::NB; ++b)
                    tma_load_3d(st + b * LY::BOX, &rows_map, (b % LY::HALVES) * 64, b / LY::HALVES,
                                row_g, &full[slot]);
                bulk_g2s(st + LY::IDS, a.ids + row_g, lb, &full[slot]);
                bulk_g2s(st + LY::RS, a.pr + row_g, lb, &full[slot]);
            }
        }
        __syncwarp();
    } else {
        int j = 0, cur = -1, count = 0;
        PivChunk<D, G, SKL> pc;
        for (int item = item0; item < item1; ++item) {
            const int ul = item / a.max_chunks, ch = item - ul * a.max_chunks;
            if (ul != cur) {  // the unit's queries and head values, once per unit
                cur = ul;
                count = min(a.count[a.li.unit_global(ul)], a.row_stride);
                pc.load_unit(a, ul);
            }
            const int lo = ch * PIV_ITEM_ROWS;
            if (lo >= count) continue;
            const int hi = min(lo + PIV_ITEM_ROWS, count);
            pc.reset();
            auto cons_bar = [] { asm volatile("bar.sync 1, %0;" ::"n"(32 * PV_CONS) : "memory"); };
            for (int s0 = lo; s0 < hi; s0 += LY::ROWS, ++j) {
                const int slot = j % PV_NS;
                bool ok = *abort == 0 && mbar_wait_or_abort(&full[slot], (uint32_t)((j / PV_NS) & 1), abort);
                ok = __all_sync(0xFFFFFFFFu, ok);
                unsigned char *st = pv_smem + (size_t)slot * LY::BYTES;
                const int rows = min(LY::ROWS, hi - s0);
                if (ok) {
                    // This warp's rows past the count hold other rows: zero them.
                    for (int r = max(rows, warp * 16); r < warp * 16 + 16; ++r) piv_zero_row<D>(st, r);
                    __syncwarp();
                    pc.stage(a, st, rows);
                } else if (lane == 0) {
                    *abort = 1;
                }
                if (s0 + LY::ROWS >= hi) {
                    // The chunk's last stage: its slot holds the reduction once all four warps
                    // are done with the rows.
                    cons_bar();
                    pc.finish(reinterpret_cast<float *>(st),
                              a.part + ((size_t)ul * a.max_chunks + ch) * G * (D + 2), *abort == 0,
                              cons_bar);
                }
                fence_proxy_async_smem();  // generic accesses before the slot's next copy
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
        }
    }
    __syncthreads();
    if (*abort) {
        // Latch the timeout and let the copies this CTA issued land before it exits: the last
        // stage issued into each slot, at its phase.
        if (tid == 0) {
            raise_error(a.err, ERR_TIMEOUT);
            for (int k = 0; k < PV_NS; ++k)
                if (s_last[k] >= 0) mbar_wait_bounded(&full[k], (uint32_t)((s_last[k] / PV_NS) & 1));
        }
        __syncthreads();
    }
}

// The tensor map of a pivotal buffer: [rows][2][d] bf16 (rows = every unit's capacity), boxes of
// 64 channels x 1 x 64 rows with the 128-byte swizzle.
static cudaError_t pivotal_rows_map(CUtensorMap *map, const void *rows, long long nrows, int d) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)d, 2, (cuuint64_t)nrows};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 4};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)PIV_STAGE_ROWS};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(rows), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_partial(const PartialArgs &a, int units_layer, int grid, cudaStream_t s) {
    const int G = a.li.G;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // Pivotal rows go through the pipelined kernel when every copy it makes is 16-byte aligned
    // and the rows fit the tensor map's 32-bit coordinates, else through k_partial, which stages
    // them with 16-byte asynchronous copies.
    const bool bulk = a.mode == ROWS_PIVOTAL && a.row16 == a.d / 4 && a.voff16 == a.d / 8 &&
                      !a.keys && (a.row_stride & 3) == 0 &&
                      (long long)a.units_total * a.row_stride <= 0x7FFFFFFFLL &&  // map coordinates
                      (reinterpret_cast<uintptr_t>(a.rows) & 15) == 0 &&
                      (reinterpret_cast<uintptr_t>(a.ids) & 15) == 0 &&
                      (reinterpret_cast<uintptr_t>(a.pr) & 15) == 0;
    const bool skl = a.sketch_logits != 0;
    if (bulk) {
        const int total = units_layer * a.max_chunks;
        const int g = std::max(1, std::min(total, sms * PV_CTAS_PER_SM));
        CUtensorMap map;
        const cudaError_t me = pivotal_rows_map(&map, a.rows, (long long)a.units_total * a.row_stride, a.d);
        if (me != cudaSuccess) return me;
#define VERKV_PIVOTAL(DD, GG, SS)                                                               \
        if (a.d == DD && G == GG && skl == SS) {                                                \
            const size_t smem = pv_smem_bytes<DD, GG>();                                        \
            const cudaError_t e = ensure_smem((const void *)k_pivotal<DD, GG, SS>, smem);       \
            if (e != cudaSuccess) return e;                                                     \
            return launch_pdl(k_pivotal<DD, GG, SS>, dim3(g), dim3(PV_NT), smem, s, a, units_layer, map); \
        }
        VERKV_PIVOTAL(128, 1, false) VERKV_PIVOTAL(128, 2, false) VERKV_PIVOTAL(128, 4, false) VERKV_PIVOTAL(128, 8, false)
        VERKV_PIVOTAL(64, 1, false) VERKV_PIVOTAL(64, 2, false) VERKV_PIVOTAL(64, 4, false) VERKV_PIVOTAL(64, 8, false)
        VERKV_PIVOTAL(128, 1, true) VERKV_PIVOTAL(128, 2, true) VERKV_PIVOTAL(128, 4, true) VERKV_PIVOTAL(128, 8, true)
        VERKV_PIVOTAL(64, 1, true) VERKV_PIVOTAL(64, 2, true) VERKV_PIVOTAL(64, 4, true) VERKV_PIVOTAL(64, 8, true)
#undef VERKV_PIVOTAL
        return cudaErrorInvalidValue;
    }
#define VERKV_PART(DD, GG)                                                                      \
    if (a.d == DD && G == GG) {                                                                 \
        if (a.mode == ROWS_PIVOTAL) {                                                           \
            const size_t smem = PivLayout<DD>::BYTES;                                           \
            if (skl) {                                                                          \
                const cudaError_t e = ensure_smem((const void *)k_partial<DD, GG, ROWS_PIVOTAL, true>, smem); \
                if (e != cudaSuccess) return e;                                                 \
                return launch_pdl(k_partial<DD, GG, ROWS_PIVOTAL, true>, dim3(grid), dim3(128), smem, s, a, units_layer); \
            }                                                                                   \
            const cudaError_t e = ensure_smem((const void *)k_partial<DD, GG, ROWS_PIVOTAL, false>, smem); \
            if (e != cudaSuccess) return e;                                                     \
            return launch_pdl(k_partial<DD, GG, ROWS_PIVOTAL, false>, dim3(grid), dim3(128), smem, s, a, units_layer); \
        }                                                                                       \
        return launch_pdl(k_partial<DD, GG, ROWS_STAGED, false>, dim3(grid), dim3(128), 0, s, a, units_layer); \
    }
    VERKV_PART(128, 1) VERKV_PART(128, 2) VERKV_PART(128, 4) VERKV_PART(128, 8)
    VERKV_PART(64, 1) VERKV_PART(64, 2) VERKV_PART(64, 4) VERKV_PART(64, 8)
#undef VERKV_PART
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------------------
// k_merge: per query head, d / MG_COLS CTAs, each over MG_COLS columns of N-hat plus the D-hat
// and second-moment columns: 8 groups of MG_COLS + 2 threads, one column each, sum every eighth
// chunk (pivotal chunks, then the per-range fetched ones that hold rows), then the groups are
// added in a fixed order.
constexpr int MG_GROUPS = 8;
constexpr int MG_COLS = 64;
constexpr int MG_TASKS = MG_GROUPS * (MG_COLS + 2);
constexpr int MG_NT = (MG_TASKS + 31) / 32 * 32;
static_assert(MG_GROUPS == 8, "k_merge picks a group's ranges with the byte mask 0x01010101");

__global__ void __launch_bounds__(MG_NT) k_merge(MergeArgs a) {
    __shared__ float red[MG_GROUPS][MG_COLS + 2];
    const int D = a.d, ncol = D + 2, halves = D / MG_COLS;
    const int qh = blockIdx.x / halves, half = blockIdx.x - qh * halves;
    const int G = a.li.G;
    const int ul = qh / G, g = qh - ul * G;
    const int ug = a.li.unit_global(ul);
    // Read before the wait on the refine kernel: the pivotal counts (PoissonComp) and the head's
    // certificate statistics were complete before the refine kernel could start, and this kernel
    // is scheduled only after that start.
    int pc = a.pcount[ug];
    verkv_head_stats st;
    if (half == 0 && threadIdx.x == 0) st = a.qstats[qh];
    pdl_wait();
    pdl_trigger();
    if (pc > a.cap) pc = a.cap;
    const int npc = (pc + PIV_ITEM_ROWS - 1) / PIV_ITEM_ROWS;
    const int t = threadIdx.x;
    if (t < MG_TASKS) {
        const int grp = t / (MG_COLS + 2), j = t - grp * (MG_COLS + 2);
        const int c = j < MG_COLS ? half * MG_COLS + j : D + (j - MG_COLS);
        const float *pp = a.part_piv + ((size_t)ul * a.max_piv * G + g) * ncol + c;
        const float *pf = a.part_fet + ((size_t)ul * a.max_fet * G + g) * ncol + c;
        const int stride = G * ncol;
        const uint32_t *rm = a.rmask + (size_t)ul * RMASK_W;  // the fetched-row ranges with a partial
        float s = 0.0f;
        // The group's pivotal chunks, eight loads in flight, added in chunk order.
        for (int b0 = grp; b0 < npc; b0 += 8 * MG_GROUPS) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int ch = b0 + k * MG_GROUPS;
                v[k] = ch < npc ? pp[ch * stride] : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (b0 + k * MG_GROUPS < npc) s += v[k];
        }
        // Then its fetched-row ranges (ch = grp mod 8) in ascending order, the empty ones
        // skipped: at most four per mask word, loaded together.
#pragma unroll
        for (int wd = 0; wd < RMASK_W; ++wd) {
            uint32_t bits = rm[wd] & (0x01010101u << grp);
            float v[4];
            bool has[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                has[k] = bits != 0u;
                v[k] = has[k] ? pf[(32 * wd + __ffs(bits) - 1) * stride] : 0.0f;
                bits &= bits - 1u;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (has[k]) s += v[k];
        }
        red[grp][j] = s;
    }
    __syncthreads();
    if (t < MG_COLS + 2) {
        float tt = red[0][t];
#pragma unroll
        for (int k = 1; k < MG_GROUPS; ++k) tt += red[k][t];
        red[0][t] = tt;  // only this thread reads or writes column t of row 0 now
    }
    __syncthreads();
    const float Dh = red[0][MG_COLS];
    if (t < MG_COLS) a.o[(size_t)qh * D + half * MG_COLS + t] = red[0][t] / Dh;
    if (half == 0 && t == 0) {
        st.D_hat = Dh;
        st.M2 = red[0][MG_COLS + 1];
        st.lse = st.m + logf(Dh);
        if (a.nacc) {
            st.n_fetch = a.nacc[qh];
            a.nacc[qh] = 0;  // ready for the next call
        }
        if (a.lse) a.lse[qh] = st.lse;
        if (a.stats) a.stats[qh] = st;
    }
}

cudaError_t launch_merge(const MergeArgs &a, int qheads, cudaStream_t s) {
    if (a.d % MG_COLS) return cudaErrorInvalidValue;
    return launch_pdl(k_merge, dim3(qheads * (a.d / MG_COLS)), dim3(MG_NT), 0, s, a);
}

// ---------------------------------------------------------------------------------------------
// k_refine: the zero-copy path's partial sums in one launch -- the fetched-row ranges of every
// layer unit first (so the host reads start at once), then its pivotal blocks (their HBM reads
// hide behind the host link).  When there are more items than resident CTAs (batch 8, 128K), the
// CTAs take items in that order from a counter (one atomic per item), so a CTA that drew light
// ranges takes more of them and the launch ends within about one item of its last host read.
// Each item writes its own partial, so which CTA took it does not change a bit.  k_merge follows.
template <int D, int G, bool SKL>
__global__ void __launch_bounds__(128, 3) k_refine(PartialArgs piv, PartialArgs fet, int units_layer) {
    extern __shared__ __align__(128) unsigned char kr_stage[];  // PivLayout<D>::BYTES
    pdl_wait();
    pdl_trigger();
    constexpr int WR = FET_RANGE / 32;  // bitmap words per range (one thread each)
    static_assert(WR >= 16 && WR <= 64, "the range's words are scanned by at most two warps");
    __shared__ int32_t s_ids[FET_RANGE];
    __shared__ int s_wsum[2];
    __shared__ int s_item;
    const int per_unit = fet.max_chunks + piv.max_chunks;
    const int total = units_layer * per_unit;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // When every item has a CTA of its own (one wave, as at batch 1) CTA b takes item b and no
    // counter is touched: an atomic round trip per CTA measured slower there.
    const bool one_wave = total <= (int)gridDim.x;
    for (int pass = 0;; ++pass) {
        int item;
        if (one_wave) {
            item = pass == 0 ? (int)blockIdx.x : total;
        } else {
            if (tid == 0) s_item = atomicAdd(fet.refine_next, 1);
            __syncthreads();
            item = s_item;
            __syncthreads();  // every thread has read it before thread 0 takes the next
        }
        if (item >= total) break;
        const int k = item / units_layer, ul = item - k * units_layer;
        const int ug = fet.li.unit_global(ul);
        if (k < fet.max_chunks) {
            // The rows to fetch in this token range: (OR over the unit's query heads of F) minus
            // the resident tokens, compacted in ascending id order; per query head, the count of
            // its own F minus the resident tokens adds into n_fetch.
            const int w = k * WR + tid;
            uint32_t uw = 0u;
            int nf[G];
#pragma unroll
            for (int g = 0; g < G; ++g) nf[g] = 0;
            if (tid < WR && w < fet.W) {
                const uint32_t rw = fet.resident[(size_t)ug * fet.W + w];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint32_t fg = fet.F[(size_t)(ul * G + g) * fet.W + w] & ~rw;
                    uw |= fg;
                    nf[g] = __popc(fg);
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int t = warp_sum(nf[g]);
                if (lane == 0 && warp < (WR + 31) / 32 && t) atomicAdd(&fet.nacc[ul * G + g], t);
            }
            const int c = __popc(uw);
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31 && warp < 2) s_wsum[warp] = incl;
            __syncthreads();
            int pos = incl - c + (warp == 1 ? s_wsum[0] : 0);
            const int cnt = s_wsum[0] + s_wsum[1];
            for (uint32_t x = uw; x; x &= x - 1) s_ids[pos++] = w * 32 + (__ffs(x) - 1);
            if (tid == 0 && cnt > 0) atomicOr(&fet.rmask[ul * RMASK_W + (k >> 5)], 1u << (k & 31));
            __syncthreads();
            partial_rows<D, G, ROWS_HOST>(fet, ul, k, 0, cnt, s_ids, false);
        } else {
            pivotal_chunk_plain<D, G, SKL>(piv, ul, k - fet.max_chunks, kr_stage);
        }
    }
}

cudaError_t launch_refine(const PartialArgs &piv, const PartialArgs &fet, int units_layer, int grid,
                          cudaStream_t s) {
    const int G = piv.li.G;
    const bool skl = piv.sketch_logits != 0;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // The grid: the CTAs that are resident at once (every CTA loops over its items).
#define VERKV_REFINE(DD, GG, SS)                                                                \
    if (piv.d == DD && G == GG && skl == SS) {                                                  \
        const size_t smem = PivLayout<DD>::BYTES;                                               \
        cudaError_t e = ensure_smem((const void *)k_refine<DD, GG, SS>, smem);                  \
        if (e != cudaSuccess) return e;                                                         \
        int per_sm = 0;                                                                         \
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_refine<DD, GG, SS>, 128, smem); \
        if (e != cudaSuccess) return e;                                                         \
        const int g = std::max(1, std::min(grid, sms * std::max(per_sm, 1)));                   \
        return launch_pdl(k_refine<DD, GG, SS>, dim3(g), dim3(128), smem, s, piv, fet, units_layer); \
    }
    VERKV_REFINE(128, 1, false) VERKV_REFINE(128, 2, false) VERKV_REFINE(128, 4, false) VERKV_REFINE(128, 8, false)
    VERKV_REFINE(64, 1, false) VERKV_REFINE(64, 2, false) VERKV_REFINE(64, 4, false) VERKV_REFINE(64, 8, false)
    VERKV_REFINE(128, 1, true) VERKV_REFINE(128, 2, true) VERKV_REFINE(128, 4, true) VERKV_REFINE(128, 8, true)
    VERKV_REFINE(64, 1, true) VERKV_REFINE(64, 2, true) VERKV_REFINE(64, 4, true) VERKV_REFINE(64, 8, true)
#undef VERKV_REFINE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------------------
// k_dense_host: the offloaded-dense baseline.  Each CTA item is PART_ROWS consecutive tokens of
// one KV head; every K|V row (4d bytes, contiguous) is read from page-locked host memory with all
// of the warp's row groups in flight, the G logits land in shared memory, the chunk's max per
// head is taken, and w = exp(logit - max) weights the V rows.  The partial is (N[d], D, max).
template <int D, int G>
__global__ void __launch_bounds__(128) k_dense_host(DenseArgs a, int units_layer) {
    constexpr int LPR = D / 8, RPW = 32 / LPR, NW = 4;
    constexpr int ITER = (PART_ROWS / NW) / RPW;
    constexpr int SUBMASK = LPR / G - 1;
    __shared__ float sS[PART_ROWS][G];
    __shared__ float sMax[G];
    __shared__ float sN[NW][G][D];
    __shared__ float sD[NW][RPW][G];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cgp = lane % LPR, rg = lane / LPR;
    const int myhead = head_of_lane<G, LPR>(lane);
    const int hq = a.li.kv_heads * G;
    const int total_items = units_layer * a.chunks;
    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int ul = item / a.chunks, ch = item - ul * a.chunks;
        const int b = ul / a.li.kv_heads, h = ul - b * a.li.kv_heads;
        const int ug = a.li.unit_global(ul);
        float qv[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 v = *reinterpret_cast<const uint4 *>(a.q + ((size_t)b * hq + h * G + g) * D + cgp * 8);
            unpack8(v, qv[g]);
        }
        const uint4 *rows = reinterpret_cast<const uint4 *>(a.rows) + (size_t)ug * a.n * (D / 4);
        const int rbase = ch * PART_ROWS + warp * (PART_ROWS / NW);
        uint4 kq[ITER], vq[ITER];
#pragma unroll
        for (int u = 0; u < ITER; ++u) {
            const int row = rbase + u * RPW + rg;
            kq[u] = make_uint4(0, 0, 0, 0);
            vq[u] = make_uint4(0, 0, 0, 0);
            if (row < a.n) {
                kq[u] = ld_host(rows + (size_t)row * (D / 4) + cgp);
                vq[u] = ld_host(rows + (size_t)row * (D / 4) + D / 8 + cgp);
            }
        }
        // logits of the chunk
#pragma unroll
        for (int u = 0; u < ITER; ++u) {
            const int rl = warp * (PART_ROWS / NW) + u * RPW + rg;  // row within the chunk
            float k[8];
            unpack8(kq[u], k);
            float p[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float s = 0.0f;
#pragma unroll
                for (int c = 0; c < 8; ++c) s = fmaf(qv[g][c], k[c], s);
                p[g] = s;
            }
            const float dot = reduce_heads_a<G, LPR>(p, lane);
            if ((cgp & SUBMASK) == 0)
                sS[rl][myhead] = ch * PART_ROWS + rl < a.n ? dot * a.scale : -INFINITY;
        }
        __syncthreads();
        if (tid < G) {
            float m = -INFINITY;
            for (int r = 0; r < PART_ROWS; ++r) m = fmaxf(m, sS[r][tid]);
            sMax[tid] = m;
        }
        __syncthreads();
        float acc[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[g][c] = 0.0f;
        float dacc = 0.0f;
        const float mh = sMax[myhead];
#pragma unroll
        for (int u = 0; u < ITER; ++u) {
            const int rl = warp * (PART_ROWS / NW) + u * RPW + rg;
            float v[8];
            unpack8(vq[u], v);
            const float s = sS[rl][myhead];
            const float w = s == -INFINITY ? 0.0f : expf(s - mh);
            if ((cgp & SUBMASK) == 0) dacc += w;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float wg = __shfl_sync(0xFFFFFFFFu, w, rg * LPR + lane_of_head<G, LPR>(g));
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[g][c] = fmaf(wg, v[c], acc[g][c]);
            }
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[g][c] += __shfl_xor_sync(0xFFFFFFFFu, acc[g][c], off);
        if (rg == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int c = 0; c < 8; ++c) sN[warp][g][cgp * 8 + c] = acc[g][c];
        }
        if ((cgp & SUBMASK) == 0) sD[warp][rg][myhead] = dacc;
        __syncthreads();
        float *out = a.part + ((size_t)ul * a.chunks + ch) * G * (D + 2);
        for (int e = tid; e < G * (D + 2); e += 128) {
            const int g = e / (D + 2), c = e - g * (D + 2);
            float t = 0.0f;
            if (c < D) {
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) t += sN[w2][g][c];
            } else if (c == D) {
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2)
#pragma unroll
                    for (int j = 0; j < RPW; ++j) t += sD[w2][j][g];
            } else {
                t = sMax[g];
            }
            out[e] = t;
        }
        __syncthreads();
    }
}

cudaError_t launch_dense_host(const DenseArgs &a, int units_layer, int grid, cudaStream_t s) {
    const int G = a.li.G;
#define VERKV_DENSE(DD, GG)                                                                     \
    if (a.d == DD && G == GG) {                                                                 \
        k_dense_host<DD, GG><<<grid, 128, 0, s>>>(a, units_layer);                              \
        return cudaGetLastError();                                                              \
    }
    VERKV_DENSE(128, 1) VERKV_DENSE(128, 2) VERKV_DENSE(128, 4) VERKV_DENSE(128, 8)
    VERKV_DENSE(64, 1) VERKV_DENSE(64, 2) VERKV_DENSE(64, 4) VERKV_DENSE(64, 8)
#undef VERKV_DENSE
    return cudaErrorInvalidValue;
}

// Threads of a dense-merge CTA: DM_GROUPS groups of 128, each summing every DM_GROUPS-th chunk.
constexpr int DM_NT = 1024;
constexpr int DM_GROUPS = DM_NT / 128;

// One CTA per query head: the global max M over the chunk maxima, then every chunk's (N, D)
// scaled by exp(m_chunk - M), summed by 8 groups over interleaved chunks and the groups in a
// fixed order; o = N / D, lse = M + log D.
__global__ void __launch_bounds__(DM_NT) k_dense_merge(DenseArgs a, float *o, float *lse) {
    extern __shared__ float red[];  // [DM_GROUPS][d + 1]
    __shared__ float sM;
    const int qh = blockIdx.x;
    const int G = a.li.G;
    const int ul = qh / G, g = qh - ul * G;
    const int D = a.d, ncol = D + 2;
    const float *pp = a.part + ((size_t)ul * a.chunks * G + g) * ncol;
    const size_t stride = (size_t)G * ncol;
    if (threadIdx.x < 32) {
        float m = -INFINITY;
        for (int ch = threadIdx.x; ch < a.chunks; ch += 32) m = fmaxf(m, pp[ch * stride + D + 1]);
        m = warp_max(m);
        if (threadIdx.x == 0) sM = m;
    }
    __syncthreads();
    const float M = sM;
    const int grp = threadIdx.x / 128, c0 = threadIdx.x % 128;
    for (int c = c0; c <= D; c += 128) {
        float t = 0.0f;
        for (int ch = grp; ch < a.chunks; ch += DM_GROUPS)
            t += pp[ch * stride + c] * expf(pp[ch * stride + D + 1] - M);
        red[grp * (D + 1) + c] = t;
    }
    __syncthreads();
    if (threadIdx.x <= D) {
        const int c = threadIdx.x;
        float t = red[c];
#pragma unroll
        for (int k = 1; k < DM_GROUPS; ++k) t += red[k * (D + 1) + c];
        red[c] = t;
    }
    __syncthreads();
    const float Dh = red[D];
    for (int c = threadIdx.x; c < D; c += DM_NT) o[(size_t)qh * D + c] = red[c] / Dh;
    if (threadIdx.x == 0 && lse) lse[qh] = M + logf(Dh);
}

cudaError_t launch_dense_merge(const DenseArgs &a, int qheads, float *o, float *lse, cudaStream_t s) {
    k_dense_merge<<<qheads, DM_NT, DM_GROUPS * (a.d + 1) * sizeof(float), s>>>(a, o, lse);
    return cudaGetLastError();
}

}  // namespace verkv
