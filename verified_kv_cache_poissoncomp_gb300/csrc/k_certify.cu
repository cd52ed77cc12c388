// k_certify.cu -- KVFetch steps 1-4 on the GPU ("Verify Before You Fetch", summary page,
// KVFETCH: Verification and Adaptive Fetching; Definition 2, Lemma 1, Eqs. (5), (7), (9), (10)).
//
// k_score     streams the bf16 sketch once per KV head with coalesced 16-byte loads and scores it
//             against all G query heads of the group (q slices held in registers; a recursive-
//             halving shuffle reduce leaves each head's logit in a quarter of the row's lanes).
// k_certify   one thread-block cluster per query head keeps w-hat and r of its tokens in shared
//             memory and runs every global step as a cluster all-reduce over distributed shared
//             memory: the max shift, D, the beta fixed point (safeguarded piece-wise Newton: on
//             the current linear piece the root is (A + B) / (1 + S), a ratio of positive sums),
//             the certificate terms of Lemma 1, and, when the certificate fails, a most-
//             significant-digit radix select over the key (g bits, ~token id) that finds the
//             minimal k* of Eq. (10) without sorting: per digit a 256-bin histogram of
//             (count, sum beta_i, sum v_i, max b_i), merged across the cluster, scanned to find
//             the bin where eps-hat of the remaining set drops below eps.
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
constexpr int CT_NT = 512;
constexpr int CT_NW = CT_NT / 32;
constexpr int CT_MAX_CL = 8;
constexpr int CT_TOKENS_PER_CTA = 8192;
constexpr int BETA_MAXIT = 64;

struct HistBin {
    uint32_t cnt;
    float sb;     // sum of beta_i
    float sv;     // sum of v_i
    uint32_t bm;  // max b_i (float bits; b_i >= 0)
};

int certify_cluster_size(int n) {
    int cl = (n + CT_TOKENS_PER_CTA - 1) / CT_TOKENS_PER_CTA;
    if (cl < 1) cl = 1;
    if (cl > CT_MAX_CL) cl = CT_MAX_CL;
    return cl;
}
int certify_chunk(int n, int cl) {
    int chunk = (n + cl - 1) / cl;
    return (chunk + 31) / 32 * 32;
}
size_t certify_smem_bytes(int chunk) {
    return (size_t)chunk * 12 + (size_t)(chunk / 32) * 4 + 2 * CT_MAX_CL * CT_NW * 4 * 4 +
           3 * 256 * sizeof(HistBin) + 64;
}

// lambda and the per-token terms of Lemma 1 for one token of L (r < 1), w = w-hat >= 0.
__device__ __forceinline__ void token_terms(float w, float r, float beta, float &bi, float &vi,
                                            float &bb) {
    float lam = 1.0f;
    if (w > 0.0f) {
        const float x = __fdiv_rn(beta * r, w * (1.0f - r));
        lam = fminf(1.0f, fmaxf(r, x));
    }
    const float lw = lam * w;
    bi = w * (1.0f - lam);
    vi = __fdiv_rn(lw * lw * (1.0f - r), r);
    bb = __fdiv_rn(lw * fmaxf(r, 1.0f - r), r);
}

__device__ __forceinline__ float bern(float b, float V, float l) {
    const float A = b * l * (1.0f / 3.0f);
    return A + sqrtf(fmaf(A, A, 2.0f * V * l));
}

__global__ void __launch_bounds__(CT_NT, 1) k_certify(CertifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *slots = reinterpret_cast<float *>(smem_raw);                  // [2][8][16][4]
    HistBin *hist = reinterpret_cast<HistBin *>(slots + 2 * CT_MAX_CL * CT_NW * 4);  // [2][256]
    HistBin *mh = hist + 512;                                                // [256] merged
    float *sw = reinterpret_cast<float *>(mh + 256);                         // [chunk]
    float *sr = sw + a.chunk;                                                // [chunk]
    uint32_t *skey = reinterpret_cast<uint32_t *>(sr + a.chunk);             // [chunk]
    uint32_t *sres = skey + a.chunk;                                         // [chunk / 32]
    __shared__ int bc_j, bc_cnt_above, bc_cnt_j, bc_final;
    __shared__ float bc_b, bc_v, bc_m, bc_eps;

    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.li.G;
    const int qh = blockIdx.x / a.cl;
    const int ul = qh / G;
    const int ug = a.li.unit_global(ul);
    const int n = a.n, chunk = a.chunk;
    const int base = crank * chunk;
    const float *sc = a.scores + (size_t)qh * n;
    const float *rf = a.r_full + (size_t)ug * n;
    const float eps = a.eps, l = a.ldelta;

    ClusterReducer<CT_NW, 4> red{slots, a.cl, 0};

    // Phase 0: logits and r into shared memory (padding: logit -inf, r = 1).
    float lmax = -__int_as_float(0x7F800000);
    for (int i = tid; i < chunk; i += CT_NT) {
        const int t = base + i;
        float s = -__int_as_float(0x7F800000), r = 1.0f;
        if (t < n) {
            s = sc[t];
            r = rf[t];
        }
        sw[i] = s;
        sr[i] = r;
        lmax = fmaxf(lmax, s);
    }
    for (int w = tid; w < chunk / 32; w += CT_NT) {
        const int gw = base / 32 + w;
        sres[w] = (gw < a.W) ? a.resident[(size_t)ug * a.W + gw] : 0u;
    }
    float m;
    {
        float v[4] = {lmax, 0.f, 0.f, 0.f};
        red.run(v, OpMax());
        m = v[0];
    }
    // Phase 1: w-hat = exp(s - m); D over all tokens; upper end of the beta bracket over L.
    float D, C, nL;
    {
        float d = 0.f, c = 0.f, cnt = 0.f;
        for (int i = tid; i < chunk; i += CT_NT) {
            const float w = expf(sw[i] - m);
            sw[i] = w;
            d += w;
            const float r = sr[i];
            if (r < 1.0f) {
                c += w * (1.0f - r);
                cnt += 1.0f;
            }
        }
        float v[4] = {d, c, cnt, 0.f};
        red.run(v, OpSum());
        D = v[0];
        C = v[1];
        nL = v[2];
    }
    // Phase 2: beta = sum_L w (1 - lambda(beta)).  On the linear piece through beta every token
    // is at its floor (A += w (1 - r)), in the middle (B += w, S += r / (1 - r)) or at 1, and the
    // piece's root is (A + B) / (1 + S); a bracket [lo, hi] guards the iteration.
    float beta = 0.0f;
    int iters = 0, flags = 0;
    if (C > 0.0f) {
        float lo = 0.0f, hi = C;
        beta = C;
        for (iters = 1; iters <= BETA_MAXIT; ++iters) {
            float ab = 0.f, S = 0.f;
            for (int i = tid; i < chunk; i += CT_NT) {
                const float r = sr[i], w = sw[i];
                if (r < 1.0f && w > 0.0f) {
                    const float fl = w * (1.0f - r);
                    if (beta <= fl) {
                        ab += fl;
                    } else if (beta * r < fl) {  // beta < w (1 - r) / r
                        ab += w;
                        S += __fdiv_rn(r, 1.0f - r);
                    }
                }
            }
            float v[4] = {ab, S, 0.f, 0.f};
            red.run(v, OpSum());
            ab = v[0];
            S = v[1];
            const float hval = fmaf(beta, 1.0f + S, -ab);
            if (hval == 0.0f) break;
            if (hval < 0.0f) lo = beta; else hi = beta;
            float nb = __fdiv_rn(ab, 1.0f + S);
            if (!(nb > lo && nb < hi)) nb = (lo > 0.0f) ? sqrtf(lo) * sqrtf(hi) : hi * 0.0625f;
            const bool conv = fabsf(nb - beta) <= 1e-7f * beta || (hi - lo) <= 1e-7f * hi;
            beta = nb;
            if (conv) break;
        }
        if (iters > BETA_MAXIT) {
            iters = BETA_MAXIT;
            flags = 1;
        }
    }
    // Phase 3: certificate terms of Lemma 1 with lambda fixed at the solution.
    float betaL, VL;
    Top2 tb{-1.0f, 0x7FFFFFFF, -1.0f};
    {
        float sb = 0.f, sv = 0.f;
        for (int i = tid; i < chunk; i += CT_NT) {
            const float r = sr[i];
            if (r < 1.0f) {
                float bi, vi, bb;
                token_terms(sw[i], r, beta, bi, vi, bb);
                sb += bi;
                sv += vi;
                tb = top2_merge(tb, Top2{bb, base + i, -1.0f});
            }
        }
        float v[4] = {sb, sv, 0.f, 0.f};
        red.run(v, OpSum());
        betaL = v[0];
        VL = v[1];
        tb = warp_top2(tb);
        // Cluster top-2 through the same slots: encode (b1, id1, b2) in a 4-float vector and
        // combine with a max-merge that keeps the lowest id among equal maxima.
        float t[4] = {tb.b1, __int_as_float(tb.id1), tb.b2, 0.f};
        const unsigned me = cluster.block_rank();
        float *bufp = red.buf(red.parity);
        if (lane < a.cl) {
            float *peer = cluster.map_shared_rank(bufp, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k) peer[(me * CT_NW + warp) * 4 + k] = t[k];
        }
        cluster.sync();
        Top2 acc{-1.0f, 0x7FFFFFFF, -1.0f};
        const int total = a.cl * CT_NW;
        for (int e = lane; e < total; e += 32)
            acc = top2_merge(acc, Top2{bufp[e * 4 + 0], __float_as_int(bufp[e * 4 + 1]), bufp[e * 4 + 2]});
        tb = warp_top2(acc);
        red.parity ^= 1;
    }
    const float b1 = fmaxf(tb.b1, 0.0f), b2 = fmaxf(tb.b2, 0.0f);
    const int id1 = tb.id1;
    const float eps_hat = (betaL + bern(b1, VL, l)) / D;
    const bool certified = eps_hat < eps;

    // Phase 4: selection (Eqs. (9)-(10)) by radix select on key56 = (g bits << 24) | (2^24-1-id).
    int kstar = 0, ndig = 0;
    unsigned long long P = 0ull;
    float eps_final = eps_hat;
    if (!certified) {
        const float A = b1 * l * (1.0f / 3.0f);
        const float R = sqrtf(fmaf(A, A, 2.0f * VL * l));
        for (int i = tid; i < chunk; i += CT_NT) {
            const float r = sr[i];
            uint32_t key = 0u;
            if (r < 1.0f) {
                float bi, vi, bb;
                token_terms(sw[i], r, beta, bi, vi, bb);
                const float Vr = fmaxf(VL - vi, 0.0f);
                float gD;
                if (base + i != id1 || b2 == b1) {
                    const float den = R + sqrtf(fmaf(A, A, 2.0f * Vr * l));
                    gD = bi + (den > 0.0f ? __fdiv_rn(2.0f * vi * l, den) : 0.0f);
                } else {
                    const float A2 = b2 * l * (1.0f / 3.0f);
                    const float R2 = sqrtf(fmaf(A2, A2, 2.0f * Vr * l));
                    const float den = R + R2;
                    gD = bi + (A - A2) +
                         (den > 0.0f ? __fdiv_rn(fmaf(A - A2, A + A2, 2.0f * vi * l), den) : 0.0f);
                }
                key = __float_as_uint(fmaxf(gD, 0.0f));
            }
            skey[i] = key;
        }
        float Bb = 0.f, Bv = 0.f, Bm = 0.f;  // the remaining set below the current prefix
        int above = 0;
        for (int d = 0; d < 7; ++d) {
            HistBin *hb = hist + (d & 1) * 256;
            for (int j = tid; j < 256; j += CT_NT) hb[j] = HistBin{0u, 0.f, 0.f, 0u};
            __syncthreads();
            const int shift = 48 - 8 * d;
            for (int i = tid; i < chunk; i += CT_NT) {
                const float r = sr[i];
                if (r < 1.0f) {
                    const unsigned long long key =
                        ((unsigned long long)skey[i] << 24) | (unsigned long long)(0xFFFFFF - (base + i));
                    if ((key >> (shift + 8)) == P) {
                        const int dig = (int)((key >> shift) & 255ull);
                        float bi, vi, bb;
                        token_terms(sw[i], r, beta, bi, vi, bb);
                        atomicAdd(&hb[dig].cnt, 1u);
                        atomicAdd(&hb[dig].sb, bi);
                        atomicAdd(&hb[dig].sv, vi);
                        atomicMax(&hb[dig].bm, __float_as_uint(bb));
                    }
                }
            }
            cluster.sync();
            for (int j = tid; j < 256; j += CT_NT) {
                HistBin acc{0u, 0.f, 0.f, 0u};
                for (int c2 = 0; c2 < a.cl; ++c2) {
                    const HistBin *p = cluster.map_shared_rank(hb, c2);
                    const HistBin x = p[j];
                    acc.cnt += x.cnt;
                    acc.sb += x.sb;
                    acc.sv += x.sv;
                    acc.bm = max(acc.bm, x.bm);
                }
                mh[j] = acc;
            }
            __syncthreads();
            if (warp == 0) {
                // Lane j owns bins 8j..8j+7; exclusive scan over lanes of the bins below.
                float sb = 0.f, sv = 0.f;
                uint32_t bm = 0u;
                int cnt = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const HistBin x = mh[8 * lane + k];
                    sb += x.sb;
                    sv += x.sv;
                    bm = max(bm, x.bm);
                    cnt += (int)x.cnt;
                }
                float eb = sb, ev = sv;
                uint32_t em = bm;
                int ec = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float yb = __shfl_up_sync(0xFFFFFFFFu, eb, o);
                    const float yv = __shfl_up_sync(0xFFFFFFFFu, ev, o);
                    const uint32_t ym = __shfl_up_sync(0xFFFFFFFFu, em, o);
                    const int yc = __shfl_up_sync(0xFFFFFFFFu, ec, o);
                    if (lane >= o) {
                        eb += yb; ev += yv; em = max(em, ym); ec += yc;
                    }
                }
                const int total_cnt = __shfl_sync(0xFFFFFFFFu, ec, 31);
                // exclusive values for this lane's first bin
                float cb = eb - sb, cv = ev - sv;
                uint32_t cm = __shfl_up_sync(0xFFFFFFFFu, em, 1);
                int cc = ec - cnt;
                if (lane == 0) cm = 0u;
                int best = -1;
                float best_eps = 0.f, best_b = 0.f, best_v = 0.f, best_m = 0.f;
                int best_cc = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = 8 * lane + k;
                    // remaining = below + bins < j
                    const float rb = Bb + cb, rv = Bv + cv;
                    const float rm = fmaxf(Bm, __uint_as_float(cm));
                    const float e = (rb + bern(rm, rv, l)) / D;
                    if (e < eps) {
                        best = j;
                        best_eps = e;
                        best_b = rb;
                        best_v = rv;
                        best_m = rm;
                        best_cc = cc;
                    }
                    const HistBin x = mh[j];
                    cb += x.sb;
                    cv += x.sv;
                    cm = max(cm, x.bm);
                    cc += (int)x.cnt;
                }
                // the largest qualifying bin over the warp
                int jb = best;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) jb = max(jb, __shfl_xor_sync(0xFFFFFFFFu, jb, o));
                if (jb < 0) {
                    // Rounding left no bin qualifying: take every candidate.
                    if (lane == 0) {
                        bc_j = 0;
                        bc_cnt_above = 0;
                        bc_cnt_j = total_cnt;
                        bc_final = 1;
                        bc_b = Bb;
                        bc_v = Bv;
                        bc_m = Bm;
                        bc_eps = (Bb + bern(Bm, Bv, l)) / D;
                    }
                } else if (best == jb) {
                    const int cj = (int)mh[jb].cnt;
                    bc_j = jb;
                    bc_cnt_j = cj;
                    bc_cnt_above = total_cnt - best_cc - cj;
                    bc_final = (cj <= 1) || d == 6;
                    bc_b = best_b;
                    bc_v = best_v;
                    bc_m = best_m;
                    bc_eps = best_eps;
                }
            }
            __syncthreads();
            P = (P << 8) | (unsigned long long)bc_j;
            above += bc_cnt_above;
            Bb = bc_b;
            Bv = bc_v;
            Bm = bc_m;
            eps_final = bc_eps;
            ndig = d + 1;
            if (bc_final) {
                kstar = above + bc_cnt_j;
                break;
            }
        }
    }
    // Phase 5: F bitmap: L tokens whose key prefix (ndig digits) is >= P.
    uint32_t *Fq = a.F + (size_t)qh * a.W;
    for (int w = warp; w < chunk / 32; w += CT_NW) {
        const int i = 32 * w + lane;
        bool inF = false;
        if (!certified && sr[i] < 1.0f) {
            const unsigned long long key =
                ((unsigned long long)skey[i] << 24) | (unsigned long long)(0xFFFFFF - (base + i));
            inF = (key >> (56 - 8 * ndig)) >= P;
        }
        const uint32_t word = __ballot_sync(0xFFFFFFFFu, inF);
        const int gw = base / 32 + w;
        if (lane == 0 && gw < a.W) Fq[gw] = word;
    }
    if (tid == 0 && crank == 0) {
        verkv_head_stats st;
        st.m = m;
        st.D = D;
        st.beta = betaL;
        st.V = VL;
        st.b = b1;
        st.eps_hat = eps_hat;
        st.eps_final = certified ? eps_hat : eps_final;
        st.D_hat = 0.f;
        st.M2 = 0.f;
        st.lse = 0.f;
        st.certified = certified ? 1 : 0;
        st.k_star = kstar;
        st.n_L = (int)nL;
        st.n_fetch = 0;
        st.iters = iters;
        st.flags = flags;
        a.qstats[qh] = st;
        if (flags) raise_error(a.err, ERR_NOCONVERGE);
    }
}

cudaError_t launch_certify(const CertifyArgs &a, int qheads, size_t smem, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(k_certify, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(qheads * a.cl);
    cfg.blockDim = dim3(CT_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_certify, a);
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
