// k_certify.cu -- KVFetch steps 2-4 on the GPU: the beta fixed point of Definition 2, the
// Bernstein certificate of Lemma 1 / Eq. (7), and the selection of Eqs. (9)-(10) ("Verify Before
// You Fetch", summary page, KVFETCH: Verification and Adaptive Fetching).
//
// One thread-block cluster per query head.  Each CTA keeps three words per token in shared
// memory (the logit, then w-hat; r; r/(1-r), later the g key) and every global quantity is one
// cluster-wide exchange over distributed shared memory:
//   1  max logit, D, sum_L w (1 - r) and |L| in one exchange (per-warp online-softmax records);
//   2+ beta = sum_L w (1 - lambda(beta)) by safeguarded piece-wise Newton: each pass classifies
//      every token at the current beta -- at its floor (A += w (1 - r)), in the middle (B += w,
//      S += r / (1 - r)) or at lambda = 1 -- and moves to the root (A + B) / (1 + S) of that
//      linear piece, a ratio of positive sums; about five passes from the top of the bracket;
//   +1 beta(L), V(L), the top two b_i (with the argmax id) of Lemma 1;
//   +k when the certificate fails, a windowed most-significant-digit select over the 56-bit key
//      (g bits << 24 | 2^24-1-token id) -- g descending, ties to the lower id.  Each pass builds a
//      256-bin histogram of (count, max b_i, sum beta_i, sum v_i) with the sums in 64-bit fixed
//      point scaled by beta(L) and V(L), added as two 32-bit halves (native integer atomics;
//      exact, order-independent sums),
//      and eight warps scan it for the bin in which eps-hat of the remaining tokens drops below
//      eps.  The first window spans 32 octaves under the largest possible g at 8 bins per octave
//      and folds everything below into bin 0; the select ends when the cut bin holds one token.
// Per-token terms use lambda w = clip(beta rho, r w, w) with rho = r / (1 - r): no division.
#include <math.h>

#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

constexpr int CT_NT = 1024;
constexpr int CT_NW = CT_NT / 32;
constexpr int CT_MAX_CL = 8;
constexpr int CT_REC = 8;   // floats per warp record in a cluster exchange
constexpr int BETA_MAXIT = 64;
constexpr int SEL_MAXPASS = 16;
constexpr int SCAN_WARPS = 8;

// Per-CTA histogram bin, built with 32-bit atomics.  A sum is kept in 64-bit fixed point split
// into a high part (q >> 18) and the low 18 bits, added separately: with the whole mapped to
// 2^49 the high parts sum below 2^31 and at most 16384 low parts below 2^32, so neither wraps.
struct HistBin {
    uint32_t cnt;
    uint32_t bm;    // max b_i (float bits; b_i >= 0)
    uint32_t sbh, sbl, svh, svl;
};
// The cluster-merged bin, with the split sums recombined.
struct MergedBin {
    uint32_t cnt;
    uint32_t bm;
    unsigned long long sb, sv;
};
constexpr int FIX_SPLIT = 18;

int certify_cluster_size(int n) {
    if (n <= 8192) return 1;
    if (n <= 32768) return 4;
    return CT_MAX_CL;
}
int certify_chunk(int n, int cl) {
    const int chunk = (n + cl - 1) / cl;
    return (chunk + 31) / 32 * 32;
}
size_t certify_smem_bytes(int chunk) {
    return (size_t)2 * CT_MAX_CL * CT_NW * CT_REC * 4   // exchange slots
           + 2 * 256 * sizeof(HistBin)                  // two histogram buffers
           + 256 * sizeof(MergedBin)                    // merged copy
           + (size_t)chunk * 12 + 64;
}

// Every warp contributes one record (identical in its lanes).  Lane c writes the record into
// slot [my rank][warp] of CTA c; after one cluster barrier every CTA holds the cl * NW records in
// the same order.  Two buffers alternate so a slot is rewritten only after the next barrier.
template <int K>
__device__ __forceinline__ const float *cluster_exchange(float *slots, int &parity, int cl,
                                                         const float (&rec)[K]) {
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned me = cluster.block_rank();
    float *buf = slots + parity * (CT_MAX_CL * CT_NW * CT_REC);
    if (lane < cl) {
        float *peer = cluster.map_shared_rank(buf, lane);
#pragma unroll
        for (int k = 0; k < K; ++k) peer[(me * CT_NW + warp) * CT_REC + k] = rec[k];
    }
    cluster.sync();
    parity ^= 1;
    return buf;
}

// Sum of field k over all records of an exchange, in a fixed order (same bits everywhere).
__device__ __forceinline__ float records_sum(const float *buf, int total, int k) {
    const int lane = threadIdx.x & 31;
    float acc = 0.0f;
    for (int e = lane; e < total; e += 32) acc += buf[e * CT_REC + k];
    return warp_sum(acc);
}

__device__ __forceinline__ float bern(float b, float V, float l) {
    const float A = b * l * (1.0f / 3.0f);
    return A + sqrtf(fmaf(A, A, 2.0f * V * l));
}

__device__ __forceinline__ float rho_of(float r) { return r * __frcp_rn(1.0f - r); }

// lambda at beta and the three per-token terms of Lemma 1 for a token of L (0 < r < 1):
// lambda w = clip(beta rho, r w, w);  beta_i = w - lambda w;  v_i = (lambda w)^2 (1 - r) / r =
// (lambda w)^2 / rho;  b_i = lambda w max(r, 1 - r) / r = lambda w max(1, 1 / rho).
__device__ __forceinline__ void token_terms(float w, float r, float rho, float beta, float &bi,
                                            float &vi, float &bb) {
    const float t = fminf(w, fmaxf(r * w, beta * rho));
    const float inv_rho = __frcp_rn(rho);
    bi = w - t;
    vi = t * t * inv_rho;
    bb = t * fmaxf(1.0f, inv_rho);
}

__device__ __forceinline__ unsigned long long key64(uint32_t gbits, int token) {
    return ((unsigned long long)gbits << 24) | (unsigned long long)(0xFFFFFF - token);
}

__device__ __forceinline__ unsigned long long to_fixed(float x, float scale) {
    const float y = x * scale;
    return y < 1.8e19f ? __float2ull_rn(y) : 18000000000000000000ull;
}

__global__ void __launch_bounds__(CT_NT, 1) k_certify(CertifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *slots = reinterpret_cast<float *>(smem_raw);
    MergedBin *mh = reinterpret_cast<MergedBin *>(slots + 2 * CT_MAX_CL * CT_NW * CT_REC);
    HistBin *hist = reinterpret_cast<HistBin *>(mh + 256);
    float *W = reinterpret_cast<float *>(hist + 512);  // logit, then w-hat
    float *R = W + a.chunk;                          // r (1 for H and padding)
    uint32_t *X = reinterpret_cast<uint32_t *>(R + a.chunk);  // r/(1-r), later the g key
    __shared__ unsigned long long s_wsb[SCAN_WARPS], s_wsv[SCAN_WARPS];
    __shared__ uint32_t s_wcnt[SCAN_WARPS], s_wbm[SCAN_WARPS];
    __shared__ int s_wbest[SCAN_WARPS];
    __shared__ int bc_int[3];
    __shared__ unsigned long long bc_u64[2];
    __shared__ uint32_t bc_bm;
    __shared__ float bc_e;

    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.li.G;
    const int qh = blockIdx.x / a.cl;
    const int ul = qh / G;
    const int ug = a.li.unit_global(ul);
    const int n = a.n, chunk = a.chunk, cl = a.cl;
    const int base = crank * chunk;
    const int total_rec = cl * CT_NW;
    const float *sc = a.scores + (size_t)qh * n;
    const float *rf = a.r_full + (size_t)ug * n;
    const float eps = a.eps, l = a.ldelta;
    const float NEG_INF = -__int_as_float(0x7F800000);
    int parity = 0;

    // ---- 1. logits, r; max logit, D, sum_L w (1 - r), |L| in one exchange ----
    float m, D, C, nL;
    {
        float tmax = NEG_INF;
        for (int i = tid; i < chunk; i += CT_NT) {
            const int t = base + i;
            float s = NEG_INF, r = 1.0f;
            if (t < n) {
                s = sc[t];
                r = rf[t];
            }
            W[i] = s;
            R[i] = r;
            tmax = fmaxf(tmax, s);
        }
        float d = 0.f, c = 0.f, cnt = 0.f;
        for (int i = tid; i < chunk; i += CT_NT) {
            const float e = tmax == NEG_INF ? 0.0f : expf(W[i] - tmax);  // 0 for padding
            d += e;
            const float r = R[i];
            if (r < 1.0f) {
                c += e * (1.0f - r);
                cnt += 1.0f;
            }
        }
        const float wmax = warp_max(tmax);
        const float sc_t = tmax == NEG_INF ? 0.0f : expf(tmax - wmax);
        const float rec[4] = {wmax, warp_sum(d * sc_t), warp_sum(c * sc_t), warp_sum(cnt)};
        const float *buf = cluster_exchange<4>(slots, parity, cl, rec);
        float mm = NEG_INF;
        for (int e = lane; e < total_rec; e += 32) mm = fmaxf(mm, buf[e * CT_REC]);
        m = warp_max(mm);
        float dd = 0.f, ccs = 0.f;
        for (int e = lane; e < total_rec; e += 32) {
            const float mj = buf[e * CT_REC];
            const float f = mj == NEG_INF ? 0.0f : expf(mj - m);
            dd += buf[e * CT_REC + 1] * f;
            ccs += buf[e * CT_REC + 2] * f;
        }
        D = warp_sum(dd);
        C = warp_sum(ccs);
        nL = records_sum(buf, total_rec, 3);
    }

    // ---- 2. beta: safeguarded piece-wise Newton from the top of the bracket ----
    float beta = 0.0f;
    int iters = 0, flags = 0;
    bool first = true;
    if (C > 0.0f) {
        float lo = 0.0f, hi = C;  // h(0) <= 0 <= h(C)
        beta = C;
        for (iters = 1; iters <= BETA_MAXIT; ++iters) {
            float ab = 0.f, S = 0.f;
            for (int i = tid; i < chunk; i += CT_NT) {
                const float r = R[i];
                float w;
                if (first) {
                    w = expf(W[i] - m);
                    W[i] = w;
                    if (r < 1.0f) X[i] = __float_as_uint(rho_of(r));
                } else {
                    w = W[i];
                }
                if (r < 1.0f) {
                    const float fl = w * (1.0f - r);
                    if (beta <= fl) {
                        ab += fl;
                    } else if (beta * r < fl) {
                        ab += w;
                        S += __uint_as_float(X[i]);
                    }
                }
            }
            first = false;
            const float rec[2] = {warp_sum(ab), warp_sum(S)};
            const float *buf = cluster_exchange<2>(slots, parity, cl, rec);
            ab = records_sum(buf, total_rec, 0);
            S = records_sum(buf, total_rec, 1);
            // The root of the linear piece through beta.  When it reproduces beta (to 1e-6
            // relative: float32 sums jitter by an ulp or two), beta is the fixed point; this is
            // tested before the bracket, which rounding can leave an ulp off the root.
            float nb = __fdiv_rn(ab, 1.0f + S);
            if (fabsf(nb - beta) <= 1e-6f * beta) {
                beta = nb;
                break;
            }
            const float hval = fmaf(beta, 1.0f + S, -ab);
            if (hval < 0.0f) lo = beta; else hi = beta;
            if (!(nb > lo && nb < hi)) nb = (lo > 0.0f) ? sqrtf(lo) * sqrtf(hi) : hi * 0.0625f;
            beta = nb;
            if ((hi - lo) <= 1e-6f * hi) break;
        }
        if (iters > BETA_MAXIT) {
            iters = BETA_MAXIT;
            flags = 1;
        }
    }
    if (first) {  // no Newton pass ran: convert the logits now
        for (int i = tid; i < chunk; i += CT_NT) {
            W[i] = expf(W[i] - m);
            if (R[i] < 1.0f) X[i] = __float_as_uint(rho_of(R[i]));
        }
        __syncthreads();
    }

    // ---- 3. certificate terms ----
    float betaL, VL;
    Top2 tb{-1.0f, 0x7FFFFFFF, -1.0f};
    {
        float sb = 0.f, sv = 0.f;
        for (int i = tid; i < chunk; i += CT_NT) {
            const float r = R[i];
            if (r < 1.0f) {
                float bi, vi, bb;
                token_terms(W[i], r, __uint_as_float(X[i]), beta, bi, vi, bb);
                sb += bi;
                sv += vi;
                tb = top2_merge(tb, Top2{bb, base + i, -1.0f});
            }
        }
        tb = warp_top2(tb);
        const float rec[5] = {warp_sum(sb), warp_sum(sv), tb.b1, __int_as_float(tb.id1), tb.b2};
        const float *buf = cluster_exchange<5>(slots, parity, cl, rec);
        betaL = records_sum(buf, total_rec, 0);
        VL = records_sum(buf, total_rec, 1);
        Top2 acc{-1.0f, 0x7FFFFFFF, -1.0f};
        for (int e = lane; e < total_rec; e += 32)
            acc = top2_merge(acc, Top2{buf[e * CT_REC + 2], __float_as_int(buf[e * CT_REC + 3]),
                                       buf[e * CT_REC + 4]});
        tb = warp_top2(acc);
    }
    const float b1 = fmaxf(tb.b1, 0.0f), b2 = fmaxf(tb.b2, 0.0f);
    const int id1 = tb.id1;
    const float eps_hat = (betaL + bern(b1, VL, l)) / D;
    const bool certified = eps_hat < eps;

    // ---- 4. selection ----
    int kstar = 0;
    unsigned long long fthr = ~0ull;  // F = { L tokens with key >= fthr }
    float eps_final = eps_hat;
    if (!certified) {
        const float A = b1 * l * (1.0f / 3.0f);
        const float Rr = sqrtf(fmaf(A, A, 2.0f * VL * l));
        const float epsD = eps * D;
        // Fixed-point scales: every partial sum is at most the whole, which maps to 2^49 (a scale
        // is capped below the float range; a zero total gives zero sums).
        const float SB = betaL > 0.0f ? fminf(562949953421312.0f / betaL, 1e38f) : 0.0f;
        const float SV = VL > 0.0f ? fminf(562949953421312.0f / VL, 1e38f) : 0.0f;
        const float iSB = SB > 0.0f ? 1.0f / SB : 0.0f;
        const float iSV = SV > 0.0f ? 1.0f / SV : 0.0f;
        // Every g_i D is at most eps-hat(L) D; the first window ends just above that.
        const uint32_t top = __float_as_uint(betaL + bern(b1, VL, l)) + 256u;
        const unsigned long long wend = ((unsigned long long)top + 1ull) << 24;
        unsigned long long lo = wend > (1ull << 52) ? wend - (1ull << 52) : 0ull;
        int shift = 44;
        bool absorb = true;  // bin 0 also takes every candidate below lo
        unsigned long long cand_lo = 0ull, cand_hi = ~0ull;
        unsigned long long Bb = 0ull, Bv = 0ull;  // tokens known to remain below the candidates
        uint32_t Bm = 0u;
        int above = 0;
        for (int pass = 0; pass < SEL_MAXPASS; ++pass) {
            HistBin *hb = hist + (pass & 1) * 256;
            for (int j = tid; j < 256; j += CT_NT) hb[j] = HistBin{0u, 0u, 0u, 0u, 0u, 0u};
            __syncthreads();
            uint32_t bc = 0u, bbm = 0u, bsbh = 0u, bsbl = 0u, bsvh = 0u, bsvl = 0u;
            for (int i = tid; i < chunk; i += CT_NT) {
                const float r = R[i];
                if (r < 1.0f) {
                    float bi, vi, bb;
                    unsigned long long k;
                    if (pass == 0) {  // the g key (Eq. (9), rationalised) of every token of L
                        token_terms(W[i], r, __uint_as_float(X[i]), beta, bi, vi, bb);
                        const float Vr = fmaxf(VL - vi, 0.0f);
                        float gD;
                        if (base + i != id1 || b2 == b1) {
                            const float den = Rr + sqrtf(fmaf(A, A, 2.0f * Vr * l));
                            gD = bi + (den > 0.0f ? __fdiv_rn(2.0f * vi * l, den) : 0.0f);
                        } else {
                            const float A2 = b2 * l * (1.0f / 3.0f);
                            const float R2 = sqrtf(fmaf(A2, A2, 2.0f * Vr * l));
                            const float den = Rr + R2;
                            gD = bi + (A - A2) +
                                 (den > 0.0f ? __fdiv_rn(fmaf(A - A2, A + A2, 2.0f * vi * l), den) : 0.0f);
                        }
                        const uint32_t g = __float_as_uint(fmaxf(gD, 0.0f));
                        X[i] = g;
                        k = key64(g, base + i);
                    } else {
                        k = key64(X[i], base + i);
                        if (!(k >= cand_lo && k < cand_hi)) continue;
                        token_terms(W[i], r, rho_of(r), beta, bi, vi, bb);
                    }
                    const unsigned long long qb = to_fixed(bi, SB), qv = to_fixed(vi, SV);
                    const uint32_t qbh = (uint32_t)(qb >> FIX_SPLIT), qbl = (uint32_t)qb & ((1u << FIX_SPLIT) - 1u);
                    const uint32_t qvh = (uint32_t)(qv >> FIX_SPLIT), qvl = (uint32_t)qv & ((1u << FIX_SPLIT) - 1u);
                    if (absorb && k < lo) {
                        bc += 1u;
                        bsbh += qbh;
                        bsbl += qbl;
                        bsvh += qvh;
                        bsvl += qvl;
                        bbm = max(bbm, __float_as_uint(bb));
                    } else {
                        const unsigned long long dj = (k - lo) >> shift;
                        const int bin = dj > 255ull ? 255 : (int)dj;
                        HistBin *hx = &hb[bin];
                        atomicAdd(&hx->cnt, 1u);
                        atomicMax(&hx->bm, __float_as_uint(bb));
                        atomicAdd(&hx->sbh, qbh);
                        atomicAdd(&hx->sbl, qbl);
                        atomicAdd(&hx->svh, qvh);
                        atomicAdd(&hx->svl, qvl);
                    }
                }
            }
            if (absorb) {
                bc = warp_sum(bc);
                bsbh = warp_sum(bsbh);
                bsbl = warp_sum(bsbl);
                bsvh = warp_sum(bsvh);
                bsvl = warp_sum(bsvl);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bbm = max(bbm, __shfl_xor_sync(0xFFFFFFFFu, bbm, o));
                if (lane == 0 && bc) {
                    atomicAdd(&hb[0].cnt, bc);
                    atomicMax(&hb[0].bm, bbm);
                    atomicAdd(&hb[0].sbh, bsbh);
                    atomicAdd(&hb[0].sbl, bsbl);
                    atomicAdd(&hb[0].svh, bsvh);
                    atomicAdd(&hb[0].svl, bsvl);
                }
            }
            cluster.sync();
            {
                // thread t merges field t / 256 of bin t % 256 over the cluster, in rank order
                const int j = tid & 255, f = tid >> 8;
                MergedBin *mj = &mh[j];
                if (f <= 1) {
                    uint32_t acc = 0u;
#pragma unroll
                    for (int c2 = 0; c2 < CT_MAX_CL; ++c2) {
                        if (c2 < cl) {
                            const HistBin *p = cluster.map_shared_rank(hb, c2) + j;
                            const uint32_t v = f == 0 ? p->cnt : p->bm;
                            acc = f == 0 ? acc + v : max(acc, v);
                        }
                    }
                    if (f == 0) mj->cnt = acc; else mj->bm = acc;
                } else {
                    unsigned long long acc = 0ull;
#pragma unroll
                    for (int c2 = 0; c2 < CT_MAX_CL; ++c2) {
                        if (c2 < cl) {
                            const HistBin *p = cluster.map_shared_rank(hb, c2) + j;
                            const uint32_t hi = f == 2 ? p->sbh : p->svh;
                            const uint32_t lo32 = f == 2 ? p->sbl : p->svl;
                            acc += ((unsigned long long)hi << FIX_SPLIT) + lo32;
                        }
                    }
                    if (f == 2) mj->sb = acc; else mj->sv = acc;
                }
            }
            __syncthreads();
            // Eight warps scan the 256 bins: remaining(j) = below + bins < j (exact integers).
            unsigned long long xsb = 0ull, xsv = 0ull;
            uint32_t xcnt = 0u, xbm = 0u, bcnt = 0u;
            if (warp < SCAN_WARPS) {
                const MergedBin hbin = mh[warp * 32 + lane];
                bcnt = hbin.cnt;
                unsigned long long isb = hbin.sb, isv = hbin.sv;
                uint32_t icnt = hbin.cnt, ibm = hbin.bm;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y1 = __shfl_up_sync(0xFFFFFFFFu, isb, o);
                    const unsigned long long y2 = __shfl_up_sync(0xFFFFFFFFu, isv, o);
                    const uint32_t y3 = __shfl_up_sync(0xFFFFFFFFu, icnt, o);
                    const uint32_t y4 = __shfl_up_sync(0xFFFFFFFFu, ibm, o);
                    if (lane >= o) {
                        isb += y1;
                        isv += y2;
                        icnt += y3;
                        ibm = max(ibm, y4);
                    }
                }
                xsb = isb - hbin.sb;   // exclusive within the warp (integer: exact)
                xsv = isv - hbin.sv;
                xcnt = icnt - hbin.cnt;
                xbm = __shfl_up_sync(0xFFFFFFFFu, ibm, 1);
                if (lane == 0) xbm = 0u;
                if (lane == 31) {
                    s_wsb[warp] = isb;
                    s_wsv[warp] = isv;
                    s_wcnt[warp] = icnt;
                    s_wbm[warp] = ibm;
                }
            }
            __syncthreads();
            int mybest = -1;
            if (warp < SCAN_WARPS) {
                for (int w2 = 0; w2 < warp; ++w2) {
                    xsb += s_wsb[w2];
                    xsv += s_wsv[w2];
                    xcnt += s_wcnt[w2];
                    xbm = max(xbm, s_wbm[w2]);
                }
                const unsigned long long rsb = Bb + xsb, rsv = Bv + xsv;
                const float rb = (float)rsb * iSB, rv = (float)rsv * iSV;
                const float rm = __uint_as_float(max(Bm, xbm));
                const float e = rb + bern(rm, rv, l);  // eps-hat of the remaining set, times D
                if (bcnt > 0u && e < epsD) mybest = warp * 32 + lane;
                int wb = mybest;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wb = max(wb, __shfl_xor_sync(0xFFFFFFFFu, wb, o));
                if (lane == 0) s_wbest[warp] = wb;
            }
            __syncthreads();
            int jb = -1;
#pragma unroll
            for (int w2 = 0; w2 < SCAN_WARPS; ++w2) jb = max(jb, s_wbest[w2]);
            uint32_t total_cnt = 0u;
#pragma unroll
            for (int w2 = 0; w2 < SCAN_WARPS; ++w2) total_cnt += s_wcnt[w2];
            if (jb >= 0 && warp * 32 + lane == jb) {
                bc_int[0] = (int)(total_cnt - xcnt - bcnt);  // above the cut bin
                bc_int[1] = (int)bcnt;
                bc_u64[0] = Bb + xsb;
                bc_u64[1] = Bv + xsv;
                bc_bm = max(Bm, xbm);
                bc_e = ((float)(Bb + xsb) * iSB +
                        bern(__uint_as_float(max(Bm, xbm)), (float)(Bv + xsv) * iSV, l)) / D;
            }
            __syncthreads();
            if (jb < 0) {  // rounding left no bin qualifying: take every candidate
                kstar = above + (int)total_cnt;
                fthr = absorb ? 0ull : cand_lo;
                eps_final = ((float)Bb * iSB + bern(__uint_as_float(Bm), (float)Bv * iSV, l)) / D;
                break;
            }
            const int cnt_above = bc_int[0], cj = bc_int[1];
            Bb = bc_u64[0];
            Bv = bc_u64[1];
            Bm = bc_bm;
            eps_final = bc_e;
            above += cnt_above;
            const unsigned long long cut_lo = lo + ((unsigned long long)jb << shift);
            if (absorb && jb == 0) {
                // The cut lies in bin 0, which also holds every candidate below the window.
                if (cj == 1) {  // one token left: it is taken, and so is every other token
                    kstar = above + 1;
                    fthr = 0ull;
                    break;
                }
                // Slide the window down at the same resolution; it ends where bin 0 ended.
                cand_lo = 0ull;
                cand_hi = lo + (1ull << shift);
                const unsigned long long span = 255ull << shift;
                if (lo > span) {
                    lo -= span;
                } else {
                    lo = 0ull;
                    absorb = false;
                }
                continue;
            }
            if (cj == 1 || shift == 0) {
                kstar = above + cj;
                fthr = cut_lo;
                break;
            }
            cand_lo = cut_lo;
            cand_hi = cut_lo + (1ull << shift);
            lo = cut_lo;
            shift = shift >= 8 ? shift - 8 : 0;
            absorb = false;
        }
        // Peers may still be reading this CTA's last histogram: no CTA leaves before all have.
        cluster.sync();
    }

    // ---- 5. F bitmap and statistics ----
    uint32_t *Fq = a.F + (size_t)qh * a.W;
    for (int w = warp; w < chunk / 32; w += CT_NW) {
        const int i = 32 * w + lane;
        bool inF = false;
        if (!certified && R[i] < 1.0f) inF = key64(X[i], base + i) >= fthr;
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
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(k_certify, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
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

}  // namespace verkv
