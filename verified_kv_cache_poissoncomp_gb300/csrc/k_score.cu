// k_score.cu -- KVFetch step 1 and the fetch list ("Verify Before You Fetch", summary page,
// KVFETCH: Verification and Adaptive Fetching, steps 1 and 5).
//
// k_score     streams the bf16 sketch once per KV head with coalesced 16-byte loads and scores it
//             against all G query heads of the group (q slices held in registers; a recursive-
//             halving shuffle reduce leaves each head's logit in a quarter of the row's lanes).
// k_fetchlist ORs the G bitmaps of a KV head, removes resident tokens and writes the ascending
//             id list of rows to fetch.
#include <math.h>

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

template <int D, int G>
__global__ void __launch_bounds__(256) k_score(ScoreArgs a) {
    constexpr int LPR = D / 8, RPW = 32 / LPR, NW = 8, ROWS = 256, U = 4;
    constexpr int ITER = (ROWS / NW) / RPW;  // row groups per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cgp = lane % LPR, rg = lane / LPR;
    const int ul = blockIdx.y;
    const int b = ul / a.li.kv_heads, h = ul - b * a.li.kv_heads;
    const int ug = a.li.unit_global(ul);
    const int hq = a.li.kv_heads * G;
    const uint4 *rows = reinterpret_cast<const uint4 *>(a.sketch) + (size_t)ug * a.n * (D / 8);

    float qv[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 v = *reinterpret_cast<const uint4 *>(a.q + ((size_t)b * hq + h * G + g) * D + cgp * 8);
        unpack8(v, qv[g]);
    }
    const int row0 = blockIdx.x * ROWS + warp * (ROWS / NW);
    float *out = a.scores + (size_t)ul * G * a.n;
    constexpr int SUBMASK = LPR / G - 1;
#pragma unroll 1
    for (int it = 0; it < ITER; it += U) {
        uint4 kv[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int row = row0 + (it + j) * RPW + rg;
            kv[j] = (it + j < ITER && row < a.n) ? ldg_stream(rows + (size_t)row * (D / 8) + cgp)
                                                 : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int row = row0 + (it + j) * RPW + rg;
            float k[8];
            unpack8(kv[j], k);
            float p[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float acc = 0.0f;
#pragma unroll
                for (int c = 0; c < 8; ++c) acc = fmaf(qv[g][c], k[c], acc);
                p[g] = acc;
            }
            int head;
            const float s = reduce_heads<G, LPR>(p, lane, head);
            if ((cgp & SUBMASK) == 0 && it + j < ITER && row < a.n)
                out[(size_t)head * a.n + row] = s * a.scale;
        }
    }
}

cudaError_t launch_score(const ScoreArgs &a, int units_layer, cudaStream_t s) {
    dim3 grid((a.n + 255) / 256, units_layer);
    const int G = a.li.G;
#define VERKV_SCORE(DD, GG) \
    if (a.d == DD && G == GG) { k_score<DD, GG><<<grid, 256, 0, s>>>(a); return cudaGetLastError(); }
    VERKV_SCORE(128, 1) VERKV_SCORE(128, 2) VERKV_SCORE(128, 4) VERKV_SCORE(128, 8)
    VERKV_SCORE(64, 1) VERKV_SCORE(64, 2) VERKV_SCORE(64, 4) VERKV_SCORE(64, 8)
#undef VERKV_SCORE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------------------
constexpr int FL_NT = 1024;

__global__ void __launch_bounds__(FL_NT) k_fetchlist(FetchListArgs a) {
    __shared__ int wsum[FL_NT / 32];
    __shared__ int nfw[FL_NT / 32][8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ul = blockIdx.x;
    const int ug = a.li.unit_global(ul);
    const int G = a.li.G;
    const int W = a.W;
    const uint32_t *res = a.resident + (size_t)ug * W;
    const uint32_t *F0 = a.F + (size_t)ul * G * W;
    const int wpt = (W + FL_NT - 1) / FL_NT;
    const int w0 = tid * wpt, w1 = min(W, w0 + wpt);
    int my = 0;
    int nf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int w = w0; w < w1; ++w) {
        const uint32_t rw = res[w];
        uint32_t f = 0u;
        for (int g = 0; g < G; ++g) {
            const uint32_t fg = F0[(size_t)g * W + w];
            f |= fg;
            nf[g] += __popc(fg & ~rw);
        }
        my += __popc(f & ~rw);
    }
    // block exclusive scan of my
    int incl = my;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    for (int g = 0; g < G; ++g) {
        const int s = warp_sum(nf[g]);
        if (lane == 0) nfw[warp][g] = s;
    }
    __syncthreads();
    if (warp == 0) {
        int v = wsum[lane];
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        wsum[lane] = x - v;  // exclusive
        if (lane == 31) {
            a.counts[ul] = x;
            if (a.counts_user) a.counts_user[ul] = x;
            if (a.counts_host) a.counts_host[ul] = x;
        }
        if (lane < G) {
            int t = 0;
            for (int w = 0; w < FL_NT / 32; ++w) t += nfw[w][lane];
            a.qstats[ul * G + lane].n_fetch = t;
        }
    }
    __syncthreads();
    int pos = wsum[warp] + incl - my;
    int32_t *ids = a.ids + (size_t)ul * a.n;
    int32_t *idsu = a.ids_user ? a.ids_user + (size_t)ul * a.n : nullptr;
    int32_t *idsh = a.ids_host ? a.ids_host + (size_t)ul * a.n : nullptr;
    for (int w = w0; w < w1; ++w) {
        uint32_t f = 0u;
        for (int g = 0; g < G; ++g) f |= F0[(size_t)g * W + w];
        f &= ~res[w];
        while (f) {
            const int bit = __ffs(f) - 1;
            f &= f - 1;
            const int id = 32 * w + bit;
            ids[pos] = id;
            if (idsu) idsu[pos] = id;
            if (idsh) idsh[pos] = id;
            ++pos;
        }
    }
}

cudaError_t launch_fetchlist(const FetchListArgs &a, int units_layer, cudaStream_t s) {
    k_fetchlist<<<units_layer, FL_NT, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace verkv
