// k_certify.cu -- KVFetch steps 2-4 on the GPU: the beta fixed point of Definition 2, the
// Bernstein certificate of Lemma 1 / Eq. (7), and the selection of Eqs. (9)-(10) ("Verify Before
// You Fetch", summary page, KVFETCH: Verification and Adaptive Fetching).
//
// One thread-block cluster per query head.  Each CTA keeps three words per token in shared
// memory (w-hat, r and r/(1-r), the last later replaced by the g key) and every global quantity is
// one cluster-wide exchange over distributed shared memory, so a decision takes about ten cluster
// barriers:
//   1  max logit m;
//   2  D, sum_L w (1 - r) (the upper end of the beta bracket), |L|;
//   3+ safeguarded piece-wise Newton for beta = sum_L w (1 - lambda(beta)): on the linear piece
//      through beta every token is at its floor (A += w (1 - r)), in the middle (B += w,
//      S += r / (1 - r)) or at lambda = 1, and the piece's root is (A + B) / (1 + S), a ratio of
//      positive sums; about five passes from the upper end of the bracket;
//   +1 beta(L), V(L), the top two b_i (with the argmax id) of Lemma 1;
//   +k when the certificate fails, a windowed most-significant-digit select over the 56-bit key
//      (g bits << 24 | 2^24-1-token id) -- g descending, ties to the lower id -- where each pass
//      builds a 256-bin histogram of (count, sum beta_i, sum v_i, max b_i) and scans it for the
//      bin in which eps-hat of the remaining tokens drops below eps (the first window covers 32
//      octaves under the largest possible g with 8 bins per octave and folds everything below
//      into bin 0); the pass ends as soon as the cut bin holds one token.
// Per-token terms use lambda w = clip(beta rho, r w, w) with rho = r / (1 - r): no division.
#include <math.h>

#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

constexpr int CT_NT = 1024;
constexpr int CT_NW = CT_NT / 32;
constexpr int CT_MAX_CL = 8;
constexpr int CT_REC = 8;              // floats per warp record in a cluster exchange
constexpr int BETA_MAXIT = 64;
constexpr int SEL_MAXPASS = 16;

struct HistBin {
    uint32_t cnt;
    float sb;     // sum of beta_i = w (1 - lambda)
    float sv;     // sum of v_i = lambda^2 w^2 (1 - r) / r
    uint32_t bm;  // max b_i = lambda w max(r, 1 - r) / r (float bits; b_i >= 0)
};

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
           + 3 * 256 * sizeof(HistBin)                  // two histogram buffers + merged copy
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
__device__ __forceinline__ float records_max(const float *buf, int total, int k) {
    const int lane = threadIdx.x & 31;
    float acc = -__int_as_float(0x7F800000);
    for (int e = lane; e < total; e += 32) acc = fmaxf(acc, buf[e * CT_REC + k]);
    return warp_max(acc);
}

__device__ __forceinline__ float bern(float b, float V, float l) {
    const float A = b * l * (1.0f / 3.0f);
    return A + sqrtf(fmaf(A, A, 2.0f * V * l));
}

// lambda at beta and the three per-token terms of Lemma 1 for a token of L (0 < r < 1), with
// rho = r / (1 - r):  lambda w = clip(beta rho, r w, w);  beta_i = w - lambda w;
// v_i = (lambda w)^2 (1 - r) / r = (lambda w)^2 / rho;  b_i = lambda w max(r, 1 - r) / r.
__device__ __forceinline__ void token_terms(float w, float r, float rho, float beta, float &bi,
                                            float &vi, float &bb) {
    const float t = fminf(w, fmaxf(r * w, beta * rho));
    const float inv_rho = __frcp_rn(rho);
    bi = w - t;
    vi = t * t * inv_rho;
    bb = t * fmaxf(1.0f, inv_rho);
}

__device__ __forceinline__ float rho_of(float r) { return r * __frcp_rn(1.0f - r); }

__device__ __forceinline__ unsigned long long key64(uint32_t gbits, int token) {
    return ((unsigned long long)gbits << 24) | (unsigned long long)(0xFFFFFF - token);
}

__global__ void __launch_bounds__(CT_NT, 1) k_certify(CertifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *slots = reinterpret_cast<float *>(smem_raw);
    HistBin *hist = reinterpret_cast<HistBin *>(slots + 2 * CT_MAX_CL * CT_NW * CT_REC);
    HistBin *mh = hist + 512;
    float *W = reinterpret_cast<float *>(mh + 256);  // w-hat (logit before phase 1)
    float *R = W + a.chunk;                          // r (1 for H and padding)
    uint32_t *X = reinterpret_cast<uint32_t *>(R + a.chunk);  // r/(1-r), later the g key
    __shared__ int bc_int[4];
    __shared__ float bc_f[4];

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
    int parity = 0;

    // ---- 1. logits, r; the max logit ----
    float lmax = -__int_as_float(0x7F800000);
    for (int i = tid; i < chunk; i += CT_NT) {
        const int t = base + i;
        float s = -__int_as_float(0x7F800000), r = 1.0f;
        if (t < n) {
            s = sc[t];
            r = rf[t];
        }
        W[i] = s;
        R[i] = r;
        lmax = fmaxf(lmax, s);
    }
    float m;
    {
        const float rec[1] = {warp_max(lmax)};
        const float *buf = cluster_exchange<1>(slots, parity, cl, rec);
        m = records_max(buf, total_rec, 0);
    }

    // ---- 2. w-hat, D, the upper end of the beta bracket ----
    float D, C, nL;
    {
        float d = 0.f, c = 0.f, cnt = 0.f;
        for (int i = tid; i < chunk; i += CT_NT) {
            const float w = expf(W[i] - m);
            W[i] = w;
            d += w;
            const float r = R[i];
            if (r < 1.0f) {
                cnt += 1.0f;
                c += w * (1.0f - r);
                X[i] = __float_as_uint(rho_of(r));
            }
        }
        const float rec[3] = {warp_sum(d), warp_sum(c), warp_sum(cnt)};
        const float *buf = cluster_exchange<3>(slots, parity, cl, rec);
        D = records_sum(buf, total_rec, 0);
        C = records_sum(buf, total_rec, 1);
        nL = records_sum(buf, total_rec, 2);
    }

    // ---- 3. beta ----
    float beta = 0.0f;
    int iters = 0, flags = 0;
    if (C > 0.0f) {
        float lo = 0.0f, hi = C;  // h(0) <= 0 <= h(C)
        beta = C;
        for (iters = 1; iters <= BETA_MAXIT; ++iters) {
            float ab = 0.f, S = 0.f;
            for (int i = tid; i < chunk; i += CT_NT) {
                const float r = R[i], w = W[i];
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

    // ---- 4. certificate terms ----
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

    // ---- 5. selection ----
    int kstar = 0;
    unsigned long long fthr = ~0ull;  // F = { L tokens with key >= fthr }
    float eps_final = eps_hat;
    if (!certified) {
        const float A = b1 * l * (1.0f / 3.0f);
        const float Rr = sqrtf(fmaf(A, A, 2.0f * VL * l));
        for (int i = tid; i < chunk; i += CT_NT) {
            const float r = R[i];
            if (r < 1.0f) {
                float bi, vi, bb;
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
                X[i] = __float_as_uint(fmaxf(gD, 0.0f));
            }
        }
        // Every g_i D is at most eps-hat(L) D; the first window ends just above that.
        const uint32_t top = __float_as_uint(betaL + bern(b1, VL, l)) + 256u;
        const unsigned long long wend = ((unsigned long long)top + 1ull) << 24;
        unsigned long long lo = wend > (1ull << 52) ? wend - (1ull << 52) : 0ull;
        int shift = 44;
        bool absorb = true;  // bin 0 also takes every candidate below lo
        unsigned long long cand_lo = 0ull, cand_hi = ~0ull;
        float Bb = 0.f, Bv = 0.f, Bm = 0.f;  // tokens known to remain (below the candidates)
        int above = 0;
        const float epsD = eps * D;
        for (int pass = 0; pass < SEL_MAXPASS; ++pass) {
            HistBin *hb = hist + (pass & 1) * 256;
            for (int j = tid; j < 256; j += CT_NT) hb[j] = HistBin{0u, 0.f, 0.f, 0u};
            __syncthreads();
            uint32_t bc = 0u, bbm = 0u;
            float bsb = 0.f, bsv = 0.f;
            for (int i = tid; i < chunk; i += CT_NT) {
                const float r = R[i];
                if (r < 1.0f) {
                    const unsigned long long k = key64(X[i], base + i);
                    if (k >= cand_lo && k < cand_hi) {
                        float bi, vi, bb;
                        token_terms(W[i], r, rho_of(r), beta, bi, vi, bb);
                        if (absorb && k < lo) {
                            bc += 1u;
                            bsb += bi;
                            bsv += vi;
                            bbm = max(bbm, __float_as_uint(bb));
                        } else {
                            unsigned long long dj = (k - lo) >> shift;
                            const int bin = dj > 255ull ? 255 : (int)dj;
                            atomicAdd(&hb[bin].cnt, 1u);
                            atomicAdd(&hb[bin].sb, bi);
                            atomicAdd(&hb[bin].sv, vi);
                            atomicMax(&hb[bin].bm, __float_as_uint(bb));
                        }
                    }
                }
            }
            if (absorb) {
                bc = warp_sum(bc);
                bsb = warp_sum(bsb);
                bsv = warp_sum(bsv);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bbm = max(bbm, __shfl_xor_sync(0xFFFFFFFFu, bbm, o));
                if (lane == 0 && bc) {
                    atomicAdd(&hb[0].cnt, bc);
                    atomicAdd(&hb[0].sb, bsb);
                    atomicAdd(&hb[0].sv, bsv);
                    atomicMax(&hb[0].bm, bbm);
                }
            }
            cluster.sync();
            {
                // thread t merges field t / 256 of bin t % 256 over the cluster, in rank order
                const int j = tid & 255, f = tid >> 8;
                const uint32_t *hw = reinterpret_cast<const uint32_t *>(hb);
                uint32_t v[CT_MAX_CL];
#pragma unroll
                for (int c2 = 0; c2 < CT_MAX_CL; ++c2)
                    v[c2] = c2 < cl ? cluster.map_shared_rank(hw, c2)[4 * j + f] : 0u;
                uint32_t acc = v[0];
#pragma unroll
                for (int c2 = 1; c2 < CT_MAX_CL; ++c2) {
                    if (c2 < cl) {
                        if (f == 0) acc += v[c2];
                        else if (f == 3) acc = max(acc, v[c2]);
                        else acc = __float_as_uint(__uint_as_float(acc) + __uint_as_float(v[c2]));
                    }
                }
                reinterpret_cast<uint32_t *>(mh)[4 * j + f] = acc;
            }
            __syncthreads();
            if (warp == 0) {
                // lane j owns bins 8j..8j+7; remaining(j) = below + bins < j
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
                int ec = cnt;
                uint32_t em = bm;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float yb = __shfl_up_sync(0xFFFFFFFFu, eb, o);
                    const float yv = __shfl_up_sync(0xFFFFFFFFu, ev, o);
                    const int yc = __shfl_up_sync(0xFFFFFFFFu, ec, o);
                    const uint32_t ym = __shfl_up_sync(0xFFFFFFFFu, em, o);
                    if (lane >= o) {
                        eb += yb;
                        ev += yv;
                        ec += yc;
                        em = max(em, ym);
                    }
                }
                const int total_cnt = __shfl_sync(0xFFFFFFFFu, ec, 31);
                float cb = __shfl_up_sync(0xFFFFFFFFu, eb, 1);
                float cv = __shfl_up_sync(0xFFFFFFFFu, ev, 1);
                int cc = __shfl_up_sync(0xFFFFFFFFu, ec, 1);
                uint32_t cm = __shfl_up_sync(0xFFFFFFFFu, em, 1);
                if (lane == 0) {
                    cb = 0.f;
                    cv = 0.f;
                    cc = 0;
                    cm = 0u;
                }
                int best = -1, best_cc = 0;
                float best_e = 0.f, best_b = 0.f, best_v = 0.f, best_m = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = 8 * lane + k;
                    const HistBin x = mh[j];
                    const float rb = Bb + cb, rv = Bv + cv;
                    const float rm = fmaxf(Bm, __uint_as_float(cm));
                    const float e = rb + bern(rm, rv, l);  // eps-hat of the remaining set, times D
                    if (x.cnt > 0u && e < epsD) {
                        best = j;
                        best_e = e;
                        best_b = rb;
                        best_v = rv;
                        best_m = rm;
                        best_cc = cc;
                    }
                    cb += x.sb;
                    cv += x.sv;
                    cm = max(cm, x.bm);
                    cc += (int)x.cnt;
                }
                int jb = best;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) jb = max(jb, __shfl_xor_sync(0xFFFFFFFFu, jb, o));
                if (jb < 0) {
                    if (lane == 0) {  // rounding left no bin qualifying: take every candidate
                        bc_int[0] = -1;
                        bc_int[1] = 0;
                        bc_int[2] = total_cnt;
                        bc_f[0] = Bb + bern(Bm, Bv, l);
                        bc_f[1] = Bb;
                        bc_f[2] = Bv;
                        bc_f[3] = Bm;
                    }
                } else if (best == jb) {
                    const int cj = (int)mh[jb].cnt;
                    bc_int[0] = jb;
                    bc_int[1] = total_cnt - best_cc - cj;  // above the cut bin
                    bc_int[2] = cj;
                    bc_f[0] = best_e;
                    bc_f[1] = best_b;
                    bc_f[2] = best_v;
                    bc_f[3] = best_m;
                }
            }
            __syncthreads();
            const int jb = bc_int[0], cnt_above = bc_int[1], cj = bc_int[2];
            eps_final = bc_f[0] / D;
            Bb = bc_f[1];
            Bv = bc_f[2];
            Bm = bc_f[3];
            if (jb < 0) {
                kstar = above + cj;
                fthr = absorb ? 0ull : cand_lo;
                break;
            }
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
    }

    // ---- 6. F bitmap and statistics ----
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
