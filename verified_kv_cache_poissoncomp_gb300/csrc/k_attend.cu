// k_attend.cu -- the bounded shrinkage estimator over the GPU-resident pivotal tokens, the fetch
// of selected rows from host memory, and the refine/merge ("Verify Before You Fetch", summary
// page, Definition 2 / Eq. (5), KVFETCH step 5; abstract page: fetch additional tokens from the
// CPU and refine the attention computation).
//
// k_partial   split-K over a row set: each CTA takes 128 rows of one KV head, each row a
//             contiguous 4d-byte K|V pair read with 16-byte coalesced loads; it computes the G
//             logits, w = exp(logit - m), the weight of Eq. (5) (1 for H and for fetched tokens,
//             lambda / r with lambda = clip(beta r / (w (1 - r)), r, 1) for sampled, unfetched
//             tokens), and accumulates D-hat, N-hat and the sample second moment.  All CTAs share
//             the query head's shift m, so partials add without rescaling.
// k_gather_host  reads the fetched rows straight from page-locked host memory (one warp per row).
// k_merge     sums the partials in a fixed order and writes o = N-hat / D-hat, m + log D-hat and
//             the per-head statistics.
#include <math.h>

#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

template <int G, int LPR>
__device__ __forceinline__ float reduce_heads_a(float (&p)[G], int lane, int &head) {
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

template <int D, int G, bool PIV>
__global__ void __launch_bounds__(128) k_partial(PartialArgs a, int units_layer) {
    constexpr int LPR = D / 8, RPW = 32 / LPR, NW = 4;
    constexpr int ITER = (PART_ROWS / NW) / RPW;
    constexpr int SUBMASK = LPR / G - 1;
    constexpr int ROW16 = D / 4;  // 16-byte vectors per K|V row
    __shared__ float sN[NW][G][D];
    __shared__ float sD[NW][RPW][G], sM[NW][RPW][G];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cgp = lane % LPR, rg = lane / LPR;
    const int hq = a.li.kv_heads * G;
    const int total_items = units_layer * a.max_chunks;

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int ul = item / a.max_chunks;
        const int ch = item - ul * a.max_chunks;
        const int b = ul / a.li.kv_heads, h = ul - b * a.li.kv_heads;
        const int ug = a.li.unit_global(ul);
        const int src = PIV ? ug : ul;
        int rows_u = a.count[src];
        if (rows_u > a.row_stride) rows_u = a.row_stride;
        if (ch * PART_ROWS >= rows_u) continue;  // uniform over the CTA

        float qv[G][8], mg[G], bg[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 v = *reinterpret_cast<const uint4 *>(a.q + ((size_t)b * hq + h * G + g) * D + cgp * 8);
            unpack8(v, qv[g]);
            mg[g] = a.qstats[ul * G + g].m;
            bg[g] = a.qstats[ul * G + g].beta;
        }
        float acc[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[g][c] = 0.0f;
        float dacc = 0.0f, m2acc = 0.0f;

        const uint4 *rows = reinterpret_cast<const uint4 *>(a.rows) + (size_t)src * a.row_stride * ROW16;
        const int32_t *ids = a.ids + (size_t)src * a.row_stride;
        const float *prs = PIV ? a.pr + (size_t)src * a.row_stride : nullptr;
        const int rbase = ch * PART_ROWS + warp * (PART_ROWS / NW);
        int myhead = 0;
#pragma unroll 2
        for (int it = 0; it < ITER; ++it) {
            const int row = rbase + it * RPW + rg;
            const bool valid = row < rows_u;
            uint4 kq = make_uint4(0, 0, 0, 0), vq = make_uint4(0, 0, 0, 0);
            int id = 0;
            float r = 1.0f;
            if (valid) {
                kq = ldg_stream(rows + (size_t)row * ROW16 + cgp);
                vq = ldg_stream(rows + (size_t)row * ROW16 + (D / 8) + cgp);
                id = ids[row];
                if (PIV) r = prs[row];
            }
            float k[8], v[8];
            unpack8(kq, k);
            unpack8(vq, v);
            float p[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float s = 0.0f;
#pragma unroll
                for (int c = 0; c < 8; ++c) s = fmaf(qv[g][c], k[c], s);
                p[g] = s;
            }
            int hh;
            const float dot = reduce_heads_a<G, LPR>(p, lane, hh);
            myhead = hh;
            // Weight of this row for head hh (computed by the lanes that hold hh).
            float cw = 0.0f;
            if (valid) {
                const float w = expf(dot * a.scale - pick<G>(mg, hh));
                const uint32_t fword = a.F[(size_t)(ul * G + hh) * a.W + (id >> 5)];
                const bool inF = (fword >> (id & 31)) & 1u;
                float coef;
                if (PIV) {
                    if (r >= 1.0f || inF) {
                        coef = 1.0f;
                    } else {
                        float lam = 1.0f;
                        if (w > 0.0f)
                            lam = fminf(1.0f, fmaxf(r, __fdiv_rn(pick<G>(bg, hh) * r, w * (1.0f - r))));
                        coef = __fdiv_rn(lam, r);
                    }
                } else {
                    coef = inF ? 1.0f : 0.0f;
                }
                cw = coef * w;
                if ((cgp & SUBMASK) == 0) {
                    dacc += cw;
                    if (PIV && r < 1.0f && !inF) m2acc += cw * cw * (1.0f - r);
                }
            }
            // Every lane of the row needs the weight of every head.
            float cwg[G];
#pragma unroll
            for (int g = 0; g < G; ++g)
                cwg[g] = __shfl_sync(0xFFFFFFFFu, cw, rg * LPR + lane_of_head<G, LPR>(g));
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[g][c] = fmaf(cwg[g], v[c], acc[g][c]);
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
        if ((cgp & SUBMASK) == 0) {
            sD[warp][rg][myhead] = dacc;
            sM[warp][rg][myhead] = m2acc;
        }
        __syncthreads();
        float *out = a.part + ((size_t)ul * a.max_chunks + ch) * G * (D + 2);
        for (int e = tid; e < G * (D + 2); e += 128) {
            const int g = e / (D + 2), c = e - g * (D + 2);
            float s = 0.0f;
            if (c < D) {
                for (int w = 0; w < NW; ++w) s += sN[w][g][c];
            } else if (c == D) {
                for (int w = 0; w < NW; ++w)
                    for (int j = 0; j < RPW; ++j) s += sD[w][j][g];
            } else {
                for (int w = 0; w < NW; ++w)
                    for (int j = 0; j < RPW; ++j) s += sM[w][j][g];
            }
            out[e] = s;
        }
        __syncthreads();
    }
}

cudaError_t launch_partial(const PartialArgs &a, int units_layer, int grid, cudaStream_t s) {
    const int G = a.li.G;
#define VERKV_PART(DD, GG)                                                              \
    if (a.d == DD && G == GG) {                                                         \
        if (a.pivotal) k_partial<DD, GG, true><<<grid, 128, 0, s>>>(a, units_layer);    \
        else k_partial<DD, GG, false><<<grid, 128, 0, s>>>(a, units_layer);             \
        return cudaGetLastError();                                                      \
    }
    VERKV_PART(128, 1) VERKV_PART(128, 2) VERKV_PART(128, 4) VERKV_PART(128, 8)
    VERKV_PART(64, 1) VERKV_PART(64, 2) VERKV_PART(64, 4) VERKV_PART(64, 8)
#undef VERKV_PART
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------------------
// Zero-copy fetch: one warp per row; four rows in flight per warp.
__global__ void __launch_bounds__(256) k_gather_host(GatherArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ul = blockIdx.y;
    const int ug = a.li.unit_global(ul);
    const int row16 = a.d / 4;
    const int cnt = a.counts[ul];
    const uint4 *src = reinterpret_cast<const uint4 *>(a.host_kv) + (size_t)ug * a.n * row16;
    uint4 *dst = reinterpret_cast<uint4 *>(a.staging) + (size_t)ul * a.n * row16;
    const int32_t *ids = a.ids + (size_t)ul * a.n;
    const int stride = gridDim.x * 8 * 4;
    for (int j0 = (blockIdx.x * 8 + warp) * 4; j0 < cnt; j0 += stride) {
        uint4 v[4];
        int id[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = j0 + k;
            id[k] = j < cnt ? ids[j] : 0;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (j0 + k < cnt && lane < row16) v[k] = src[(size_t)id[k] * row16 + lane];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (j0 + k < cnt && lane < row16) dst[(size_t)(j0 + k) * row16 + lane] = v[k];
    }
}

cudaError_t launch_gather_host(const GatherArgs &a, int units_layer, cudaStream_t s) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int bx = (sms * 4 + units_layer - 1) / units_layer;
    if (bx < 1) bx = 1;
    k_gather_host<<<dim3(bx, units_layer), 256, 0, s>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_merge(MergeArgs a) {
    extern __shared__ float tot[];  // [d + 2]
    const int qh = blockIdx.x;
    const int G = a.li.G;
    const int ul = qh / G, g = qh - ul * G;
    const int ug = a.li.unit_global(ul);
    const int D = a.d;
    int pc = a.pcount[ug];
    if (pc > a.cap) pc = a.cap;
    const int npc = (pc + PART_ROWS - 1) / PART_ROWS;
    const int nfc = (a.fcount[ul] + PART_ROWS - 1) / PART_ROWS;
    for (int c = threadIdx.x; c < D + 2; c += blockDim.x) {
        float s = 0.0f;
        for (int ch = 0; ch < npc; ++ch)
            s += a.part_piv[(((size_t)ul * a.max_piv + ch) * G + g) * (D + 2) + c];
        for (int ch = 0; ch < nfc; ++ch)
            s += a.part_fet[(((size_t)ul * a.max_fet + ch) * G + g) * (D + 2) + c];
        tot[c] = s;
    }
    __syncthreads();
    const float Dh = tot[D];
    for (int c = threadIdx.x; c < D; c += blockDim.x) a.o[(size_t)qh * D + c] = tot[c] / Dh;
    if (threadIdx.x == 0) {
        verkv_head_stats st = a.qstats[qh];
        st.D_hat = Dh;
        st.M2 = tot[D + 1];
        st.lse = st.m + logf(Dh);
        if (a.lse) a.lse[qh] = st.lse;
        if (a.stats) a.stats[qh] = st;
    }
}

cudaError_t launch_merge(const MergeArgs &a, int qheads, cudaStream_t s) {
    k_merge<<<qheads, 128, (a.d + 2) * sizeof(float), s>>>(a);
    return cudaGetLastError();
}

}  // namespace verkv
