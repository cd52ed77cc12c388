// k_score.cu -- KVFetch step 1 ("Verify Before You Fetch", summary page, KVFETCH: Verification
// and Adaptive Fetching, step 1).
//
// k_score streams the bf16 sketch once per KV head through a ring of TMA tensor copies in shared
// memory (64-row stages, boxes of 64 channels with the 128-byte swizzle) and scores it against all
// G query heads of the group on the tensor cores: each warp takes 16 rows of a stage as the A
// operand of mma.m16n8k16 (ldmatrix from the swizzled stage) and the group's query heads as the
// B operand (heads padded to 8), so a stage costs a warp D/16 mma instead of a CUDA-core dot
// product per head.  The 2-bit sketch (k_score_q2) keeps the CUDA-core bulk-copy ring.
#include <cuda_fp16.h>
#include <math.h>

#include "pivotal_mma.cuh"
#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

// ---------------------------------------------------------------------------------------------
// Recursive-halving reduce: the G partial dot products of the LPR lanes of one row are summed;
// afterwards lane bits (LPR/2 ... LPR/G) name the head a lane holds, and the remaining low bits
// hold copies of the same total.
template <int G, int LPR>
__device__ __forceinline__ float reduce_heads(float (&p)[G], int lane, int &head) {
    static_assert(G <= LPR, "G must not exceed the lanes per row");
    head = 0;
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
            if (upper) head += half;
            hc = half;
        } else {
            p[0] += __shfl_xor_sync(0xFFFFFFFFu, p[0], off);
        }
    }
    return p[0];
}

// TMA bulk-copy pipeline.  Each CTA streams a contiguous span of sketch rows of one KV head (the
// span is sized so the grid is SC_CTAS_PER_SM CTAs per SM) through a ring of SC_STAGES shared-memory stages of SC_ROWS rows: thread 0 issues one
// cp.async.bulk per stage that completes on the stage's mbarrier; every warp waits on the barrier,
// scores its rows from shared memory (16 lanes per 256-byte row: conflict-free 16-byte loads), and
// after a block barrier the freed stage is refilled.  Waits are bounded by %globaltimer: on expiry
// the kernel latches ERR_TIMEOUT, waits (bounded again) for its own copies in flight and returns.
constexpr int SC_NT = 256;
constexpr int SC_STAGES = 4;
constexpr int SC_ROWS = 64;
constexpr int SC_CTAS_PER_SM = 2;  // resident CTAs per SM the grid is sized for (registers allow two)

// Packed pair arithmetic: two f32 lanes in one 64-bit register (fma.rn.f32x2).
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float sum2(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// The two bf16 of a 32-bit word as an f32 pair (element 0 in the low half).
__device__ __forceinline__ unsigned long long bf16x2_to_f32x2(uint32_t w) {
    return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// A row of the sketch is scored by LPR lanes, each holding CPL channels: 16 (two 16-byte vectors,
// at vector indices cgp and cgp + LPR so the lanes of a row read consecutive 16-byte words) when
// G <= 4, else 8.  Products accumulate as channel pairs with fma.rn.f32x2, one accumulator pair
// per head.
// The exact sketch on the tensor cores.  Each CTA streams a contiguous span of one KV head's rows
// (spans sized for TC_CTAS_PER_SM CTAs per SM) through TC_STAGES stages of 64 rows: thread 0 issues
// the stage's D/64 tensor copies, which complete on the stage's mbarrier; every warp waits on it,
// computes S = K Q^T for its 16 rows (two accumulator chains over the k-steps) and stores the
// logits of the real heads; after a block barrier the freed stage is refilled.  Rows past the
// unit's end arrive as zeros (the copy's out-of-bounds fill) and rows past the span are not
// stored.  Waits are bounded by %globaltimer: on expiry the kernel latches ERR_TIMEOUT, waits
// (bounded again) for its own copies in flight and returns.
constexpr int TC_NT = 128;           // four warps: one 16-row tile of each stage apiece
constexpr int TC_STAGES = 4;
constexpr int TC_ROWS = 64;
constexpr int TC_CTAS_PER_SM = 3;    // shared memory (4 x 16 KB stages) and registers allow three

template <int D>
constexpr size_t tc_smem_bytes() { return 1024 + (size_t)TC_STAGES * (D / 64) * PivLayout<D>::BOX; }

template <int D, int G>
__global__ void __launch_bounds__(TC_NT, TC_CTAS_PER_SM) k_score(ScoreArgs a, int spans_per_unit, int span_rows,
                                                               const __grid_constant__ CUtensorMap map) {
    // The first kernel of a library call may be launched with programmatic serialisation, so it
    // can be resident before the kernel ahead of it on the stream (the caller's q projection, a
    // sketch build, the previous call's merge) has finished: it reads nothing the caller wrote
    // (the sketch, q) before pdl_wait().  The trigger lets the certificate kernel be scheduled
    // early.
    pdl_trigger();
    using LY = PivLayout<D>;
    constexpr int KS = D / 16, HALVES = D / 64, STAGE = HALVES * LY::BOX;
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    __shared__ __align__(8) uint64_t full[TC_STAGES];
    __shared__ int s_abort;
    unsigned char *ring = tc_raw + ((1024u - (smem_addr(tc_raw) & 1023u)) & 1023u);  // swizzle unit

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int ul = blockIdx.x / spans_per_unit;
    const int span = blockIdx.x - ul * spans_per_unit;
    const int b = ul / a.li.kv_heads, h = ul - b * a.li.kv_heads;
    const int ug = a.li.unit_global(ul);
    const int hq = a.li.kv_heads * G;
    const int row0 = span * span_rows;
    const int nrows = min(a.n - row0, span_rows);
    if (nrows <= 0) return;  // uniform over the CTA
    const int nst = (nrows + TC_ROWS - 1) / TC_ROWS;

    if (tid == 0) {
        for (int k = 0; k < TC_STAGES; ++k) mbar_init(&full[k], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    __syncthreads();
    auto issue = [&](int k) {
        uint64_t *bar = &full[k % TC_STAGES];
        mbar_expect_tx(bar, (uint32_t)STAGE);
        if (a.stall_first && blockIdx.x == 0 && k == 0) return;  // test injection: never issued
        unsigned char *st = ring + (size_t)(k % TC_STAGES) * STAGE;
#pragma unroll
        for (int hb = 0; hb < HALVES; ++hb)
            tma_load_3d(st + hb * LY::BOX, &map, hb * 64, row0 + k * TC_ROWS, ug, bar);
    };
    if (tid == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map)) : "memory");
    pdl_wait();
    if (tid == 0)
        for (int k = 0; k < min(TC_STAGES, nst); ++k) issue(k);
    // Q^T as the B operand: query head g of the group (zero for g >= G), channels 2t, 2t + 1 and
    // 2t + 8, 2t + 9 of each k-step, read while the first stages are in flight.
    uint32_t qb[KS][2];
    {
        const uint32_t *qrow =
            reinterpret_cast<const uint32_t *>(a.q + ((size_t)b * hq + h * G + (g < G ? g : 0)) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qb[ks][0] = g < G ? qrow[ks * 8 + t] : 0u;
            qb[ks][1] = g < G ? qrow[ks * 8 + 4 + t] : 0u;
        }
    }

    float *out = a.scores + (size_t)ul * G * a.n + row0;
    const unsigned long long wait_ns = a.wait_ns ? a.wait_ns : TMA_WAIT_NS;
    const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: tile mi, row ri of it
    const int ar = warp * 16 + (mi & 1) * 8 + ri;
    int consumed = 0;
    for (int k = 0; k < nst; ++k) {
        const uint32_t parity = (uint32_t)((k / TC_STAGES) & 1);
        if (!mbar_wait_bounded(&full[k % TC_STAGES], parity, wait_ns)) s_abort = 1;
        __syncthreads();
        if (s_abort) break;
        consumed = k + 1;
        const int rows_k = min(TC_ROWS, nrows - k * TC_ROWS);
        const uint32_t base = smem_addr(ring + (size_t)(k % TC_STAGES) * STAGE);
        float c[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t af[4];
            ldsm_x4(af, base + (uint32_t)LY::off(0, ar, ks * 16 + (mi >> 1) * 8));
            mma_bf16((ks & 1) ? c1 : c, af, qb[ks][0], qb[ks][1]);
        }
        // c[e]: row 16 w + g + 8 (e >> 1) of the stage, head 2t + (e & 1).
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int hd = 2 * t + (e & 1), r = warp * 16 + g + 8 * (e >> 1);
            if (hd < G && r < rows_k) out[(size_t)hd * a.n + k * TC_ROWS + r] = (c[e] + c1[e]) * a.scale;
        }
        __syncthreads();  // every warp is done with the stage: refill it
        if (tid == 0 && k + TC_STAGES < nst) issue(k + TC_STAGES);
    }
    if (s_abort) {
        // Latch the timeout and let the copies this CTA issued land before it exits.
        if (tid == 0) {
            raise_error(a.err, ERR_TIMEOUT);
            const int issued = min(nst, consumed + TC_STAGES);
            for (int k = consumed; k < issued; ++k)
                mbar_wait_bounded(&full[k % TC_STAGES], (uint32_t)((k / TC_STAGES) & 1), wait_ns);
        }
        __syncthreads();
    }
}

// The tensor map of an exact sketch: [units][n][d] bf16 as (channel, row, unit), boxes of 64
// channels x 64 rows x 1 unit with the 128-byte swizzle; rows past a unit's n read as zeros.
static cudaError_t sketch_map(CUtensorMap *map, const void *sketch, int units_total, int n, int d) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)units_total};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n * d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)TC_ROWS, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(sketch), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Spans of rows per unit and rows per span for `ctas_per_sm` CTAs per SM.
static void score_spans(int units_layer, int n, int ctas_per_sm, int rows_per_stage, int &spans,
                        int &span_rows) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)units_layer * n;
    long long sr = (total + (long long)ctas_per_sm * sms - 1) / ((long long)ctas_per_sm * sms);
    sr = (sr + rows_per_stage - 1) / rows_per_stage * rows_per_stage;
    if (sr < rows_per_stage) sr = rows_per_stage;
    span_rows = (int)sr;
    spans = (int)((n + sr - 1) / sr);
}

cudaError_t launch_score(const ScoreArgs &a, int units_layer, cudaStream_t s, bool pdl) {
    int spans = 0, span_rows = 0;
    score_spans(units_layer, a.n, TC_CTAS_PER_SM, TC_ROWS, spans, span_rows);
    CUtensorMap map;
    const cudaError_t me = sketch_map(&map, a.sketch, units_layer * a.li.layers, a.n, a.d);
    if (me != cudaSuccess) return me;
    dim3 grid(spans * units_layer);
    const int G = a.li.G;
#define VERKV_SCORE(DD, GG)                                                                     \
    if (a.d == DD && G == GG) {                                                                 \
        const size_t smem = tc_smem_bytes<DD>();                                                \
        const cudaError_t e = ensure_smem((const void *)k_score<DD, GG>, smem);                \
        if (e != cudaSuccess) return e;                                                         \
        return launch_opt_pdl(pdl, k_score<DD, GG>, grid, dim3(TC_NT), smem, s, a, spans,       \
                              span_rows, map);                                                  \
    }
    VERKV_SCORE(128, 1) VERKV_SCORE(128, 2) VERKV_SCORE(128, 4) VERKV_SCORE(128, 8)
    VERKV_SCORE(64, 1) VERKV_SCORE(64, 2) VERKV_SCORE(64, 4) VERKV_SCORE(64, 8)
#undef VERKV_SCORE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------------------
// k_sketch_stream: the bytes k_score moves, without its arithmetic -- the same grid, spans, stages
// and tensor copies, with thread 0 waiting on each stage and refilling its slot at once.  Its time
// is that of a bare one-launch read of a layer's sketch: the reference k_score's time is set against.
template <int D>
__global__ void __launch_bounds__(TC_NT, TC_CTAS_PER_SM) k_sketch_stream(ScoreArgs a, int spans_per_unit,
                                                                       int span_rows,
                                                                       const __grid_constant__ CUtensorMap map) {
    using LY = PivLayout<D>;
    constexpr int HALVES = D / 64, STAGE = HALVES * LY::BOX;
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    __shared__ __align__(8) uint64_t full[TC_STAGES];
    if (threadIdx.x != 0) return;
    unsigned char *ring = tc_raw + ((1024u - (smem_addr(tc_raw) & 1023u)) & 1023u);
    const int ul = blockIdx.x / spans_per_unit;
    const int span = blockIdx.x - ul * spans_per_unit;
    const int ug = a.li.unit_global(ul);
    const int row0 = span * span_rows;
    const int nrows = min(a.n - row0, span_rows);
    if (nrows <= 0) return;
    const int nst = (nrows + TC_ROWS - 1) / TC_ROWS;
    for (int k = 0; k < TC_STAGES; ++k) mbar_init(&full[k], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    auto issue = [&](int k) {
        uint64_t *bar = &full[k % TC_STAGES];
        mbar_expect_tx(bar, (uint32_t)STAGE);
        unsigned char *st = ring + (size_t)(k % TC_STAGES) * STAGE;
        for (int hb = 0; hb < HALVES; ++hb)
            tma_load_3d(st + hb * LY::BOX, &map, hb * 64, row0 + k * TC_ROWS, ug, bar);
    };
    for (int k = 0; k < min(TC_STAGES, nst); ++k) issue(k);
    for (int k = 0; k < nst; ++k) {
        if (!mbar_wait_bounded(&full[k % TC_STAGES], (uint32_t)((k / TC_STAGES) & 1))) {
            // Latch the timeout and let this CTA's copies in flight land before it exits.
            raise_error(a.err, ERR_TIMEOUT);
            for (int j = k + 1; j < min(nst, k + TC_STAGES); ++j)
                mbar_wait_bounded(&full[j % TC_STAGES], (uint32_t)((j / TC_STAGES) & 1));
            return;
        }
        if (k + TC_STAGES < nst) issue(k + TC_STAGES);
    }
}

cudaError_t launch_sketch_stream(const ScoreArgs &a, int units_layer, cudaStream_t s) {
    int spans = 0, span_rows = 0;
    score_spans(units_layer, a.n, TC_CTAS_PER_SM, TC_ROWS, spans, span_rows);
    CUtensorMap map;
    const cudaError_t me = sketch_map(&map, a.sketch, units_layer * a.li.layers, a.n, a.d);
    if (me != cudaSuccess) return me;
#define VERKV_STREAM(DD)                                                                        \
    if (a.d == DD) {                                                                            \
        const size_t smem = tc_smem_bytes<DD>();                                                \
        const cudaError_t e = ensure_smem((const void *)k_sketch_stream<DD>, smem);            \
        if (e != cudaSuccess) return e;                                                         \
        k_sketch_stream<DD><<<dim3(spans * units_layer), dim3(TC_NT), smem, s>>>(a, spans, span_rows, map); \
        return cudaGetLastError();                                                              \
    }
    VERKV_STREAM(128) VERKV_STREAM(64)
#undef VERKV_STREAM
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------------------
// Scoring from the 2-bit sketch.  Same TMA ring, SQ_ROWS rows a stage.  A lane holds CPL
// consecutive channels of a row (its codes are one 32- or 16-bit field, its group's floor and
// step one 32-bit word) and the matching q values; per head its dot product is
// floor * sum(q) + step * sum(q * code), the codes turned into floats in pairs for fma.f32x2.
constexpr int SQ_ROWS = 256;

__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

template <int D, int G>
__global__ void __launch_bounds__(SC_NT, SC_CTAS_PER_SM) k_score_q2(ScoreArgs a, int spans_per_unit,
                                                                   int span_rows) {
    pdl_trigger();  // launched as k_score is: nothing the caller wrote is read before pdl_wait()
    constexpr int CPL = G <= 4 ? 16 : 8;
    constexpr int LPR = D / CPL, RPW = 32 / LPR, NW = SC_NT / 32;
    constexpr int ROWB = (D / 4 + 4 * (D / 32) + 15) / 16 * 16;  // bytes per sketch row
    constexpr int WROWS = SQ_ROWS / NW;
    constexpr int SUBMASK = LPR / G - 1;
    constexpr float MAGIC = 8388608.0f;  // 2^23: float bits 0x4B000000 | c equal 2^23 + c
    extern __shared__ __align__(128) unsigned char ring[];  // [SC_STAGES][SQ_ROWS][ROWB]
    __shared__ __align__(8) uint64_t full[SC_STAGES];
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cgp = lane % LPR, rg = lane / LPR;
    const int ul = blockIdx.x / spans_per_unit;
    const int span = blockIdx.x - ul * spans_per_unit;
    const int b = ul / a.li.kv_heads, h = ul - b * a.li.kv_heads;
    const int ug = a.li.unit_global(ul);
    const int hq = a.li.kv_heads * G;
    const int row0 = span * span_rows;
    const int nrows = min(a.n - row0, span_rows);
    if (nrows <= 0) return;  // uniform over the CTA
    const int nst = (nrows + SQ_ROWS - 1) / SQ_ROWS;
    const unsigned char *src = reinterpret_cast<const unsigned char *>(a.sketch) +
                               ((size_t)ug * a.n + row0) * ROWB;
    const int code_word = (CPL * cgp) / 16, code_shift = (2 * CPL * cgp) % 32;
    const int par_word = D / 16 + (CPL * cgp) / 32;

    const unsigned long long neg_magic = pack2(-MAGIC, -MAGIC);
    if (tid == 0) {
        for (int k = 0; k < SC_STAGES; ++k) mbar_init(&full[k], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    __syncthreads();
    auto issue = [&](int k) {
        const int rows_k = min(SQ_ROWS, nrows - k * SQ_ROWS);
        const uint32_t bytes = (uint32_t)rows_k * ROWB;
        uint64_t *bar = &full[k % SC_STAGES];
        mbar_expect_tx(bar, bytes);
        if (a.stall_first && blockIdx.x == 0 && k == 0) return;  // test injection: never issued
        bulk_g2s(ring + (size_t)(k % SC_STAGES) * SQ_ROWS * ROWB, src + (size_t)k * SQ_ROWS * ROWB,
                 bytes, bar);
    };
    pdl_wait();
    if (tid == 0)
        for (int k = 0; k < min(SC_STAGES, nst); ++k) issue(k);
    // q is read while the first stages are in flight.
    unsigned long long qp[G][CPL / 2];
    float qs[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        qs[g] = 0.0f;
#pragma unroll
        for (int v = 0; v < CPL / 8; ++v) {
            const uint4 x = *reinterpret_cast<const uint4 *>(a.q + ((size_t)b * hq + h * G + g) * D +
                                                             CPL * cgp + 8 * v);
            float f[8];
            unpack8(x, f);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                qp[g][4 * v + t] = pack2(f[2 * t], f[2 * t + 1]);
                qs[g] += f[2 * t] + f[2 * t + 1];
            }
        }
    }

    float *out = a.scores + (size_t)ul * G * a.n + row0;
    const unsigned long long wait_ns = a.wait_ns ? a.wait_ns : TMA_WAIT_NS;
    int consumed = 0;
    for (int k = 0; k < nst; ++k) {
        const uint32_t parity = (uint32_t)((k / SC_STAGES) & 1);
        if (!mbar_wait_bounded(&full[k % SC_STAGES], parity, wait_ns)) s_abort = 1;
        __syncthreads();
        if (s_abort) break;
        consumed = k + 1;
        const int rows_k = min(SQ_ROWS, nrows - k * SQ_ROWS);
        const uint32_t *stage = reinterpret_cast<const uint32_t *>(ring + (size_t)(k % SC_STAGES) * SQ_ROWS * ROWB);
#pragma unroll 2
        for (int j = 0; j < WROWS / RPW; ++j) {
            const int r = warp * WROWS + j * RPW + rg;  // row within the stage
            uint32_t cw = 0u, pw = 0u;
            if (r < rows_k) {
                cw = stage[r * (ROWB / 4) + code_word] >> code_shift;
                pw = stage[r * (ROWB / 4) + par_word];
            }
            const float lo = __half2float(__ushort_as_half((unsigned short)(pw & 0xFFFFu)));
            const float st = __half2float(__ushort_as_half((unsigned short)(pw >> 16)));
            unsigned long long acc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] = 0ull;
#pragma unroll
            for (int i = 0; i < CPL / 2; ++i) {
                const uint32_t c0 = (cw >> (4 * i)) & 3u, c1 = (cw >> (4 * i + 2)) & 3u;
                const unsigned long long cp =
                    fadd2(pack2(__uint_as_float(0x4B000000u | c0), __uint_as_float(0x4B000000u | c1)),
                          neg_magic);
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = ffma2(qp[g][i], cp, acc[g]);
            }
            float p[G];
#pragma unroll
            for (int g = 0; g < G; ++g) p[g] = fmaf(lo, qs[g], st * sum2(acc[g]));
            int head;
            const float sc = reduce_heads<G, LPR>(p, lane, head);
            if ((cgp & SUBMASK) == 0 && r < rows_k)
                out[(size_t)head * a.n + k * SQ_ROWS + r] = sc * a.scale;
        }
        __syncthreads();  // every warp is done with the stage: refill it
        if (tid == 0 && k + SC_STAGES < nst) issue(k + SC_STAGES);
    }
    if (s_abort) {
        if (tid == 0) {
            raise_error(a.err, ERR_TIMEOUT);
            const int issued = min(nst, consumed + SC_STAGES);
            for (int k = consumed; k < issued; ++k)
                mbar_wait_bounded(&full[k % SC_STAGES], (uint32_t)((k / SC_STAGES) & 1), wait_ns);
        }
        __syncthreads();
    }
}

cudaError_t launch_score_q2(const ScoreArgs &a, int units_layer, cudaStream_t s, bool pdl) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)units_layer * a.n;
    long long span_rows = (total + (long long)SC_CTAS_PER_SM * sms - 1) / ((long long)SC_CTAS_PER_SM * sms);
    span_rows = (span_rows + SQ_ROWS - 1) / SQ_ROWS * SQ_ROWS;
    if (span_rows < SQ_ROWS) span_rows = SQ_ROWS;
    const int spans = (int)((a.n + span_rows - 1) / span_rows);
    dim3 grid(spans * units_layer);
    const int G = a.li.G;
#define VERKV_SCORE_Q2(DD, GG)                                                                  \
    if (a.d == DD && G == GG) {                                                                 \
        constexpr int ROWB = (DD / 4 + 4 * (DD / 32) + 15) / 16 * 16;                           \
        const size_t smem = (size_t)SC_STAGES * SQ_ROWS * ROWB;                                 \
        const cudaError_t e = ensure_smem((const void *)k_score_q2<DD, GG>, smem);             \
        if (e != cudaSuccess) return e;                                                         \
        return launch_opt_pdl(pdl, k_score_q2<DD, GG>, grid, dim3(SC_NT), smem, s, a, spans,    \
                              (int)span_rows);                                                  \
    }
    VERKV_SCORE_Q2(128, 1) VERKV_SCORE_Q2(128, 2) VERKV_SCORE_Q2(128, 4) VERKV_SCORE_Q2(128, 8)
    VERKV_SCORE_Q2(64, 1) VERKV_SCORE_Q2(64, 2) VERKV_SCORE_Q2(64, 4) VERKV_SCORE_Q2(64, 8)
#undef VERKV_SCORE_Q2
    return cudaErrorInvalidValue;
}

}  // namespace verkv
