// k_certify.cu -- KVFetch steps 2-4 on the GPU: the beta fixed point of Definition 2, the
// Bernstein certificate of Lemma 1 / Eq. (7), and the selection of Eqs. (9)-(10) ("Verify Before
// You Fetch", summary page, KVFETCH: Verification and Adaptive Fetching).
//
// One thread-block cluster per query head.  Each CTA keeps three words per token in shared
// memory (the logit, then w-hat; r; r/(1-r), later the g key) and every global quantity is one
// cluster-wide all-reduce: the warps' records are combined into one record per CTA, each CTA
// sends its record to every peer over distributed shared memory, and after one cluster barrier
// every thread combines the CTA records in rank order (the same bits everywhere):
//   1  max logit, D, sum_L w (1 - r) and |L| in one exchange (per-warp online-softmax records);
//   2+ beta = sum_L w (1 - lambda(beta)) by safeguarded piece-wise Newton: each pass classifies
//      every token at the current beta -- at its floor (A += w (1 - r)), in the middle (B += w,
//      S += r / (1 - r)) or at lambda = 1 -- and moves to the root (A + B) / (1 + S) of that
//      linear piece, a ratio of positive sums; the pass also finds the nearest breakpoints on
//      either side, and the solve ends as soon as the new root lies between them.  The first
//      pass evaluates two points, C/2 and C/8, in one exchange, which brackets the root and starts
//      Newton closer to it than the top of the bracket (2.5 passes on average instead of 3.4);
//   +1 beta(L), V(L), the top two b_i (with the argmax id) of Lemma 1;
//   +k when the certificate fails, a windowed most-significant-digit select over the 56-bit key
//      (g bits << 24 | 2^24-1-token id) -- g descending, ties to the lower id.  Each pass builds a
//      256-bin histogram of (count, max b_i, sum beta_i, sum v_i) with the sums in 64-bit fixed
//      point scaled by beta(L) and V(L), added as two 32-bit halves (native integer atomics;
//      exact, order-independent sums); the CTAs' histograms are merged over distributed shared
//      memory and 256 threads, one per bin, scan them for the bin in which eps-hat of the
//      remaining tokens drops below eps.  The first window spans 32 octaves under the largest possible g
//      at 8 bins per octave and folds everything below into bin 0; the select ends when the cut
//      bin holds one token.  With clusters of 1 and 4, once the cut bin holds at most SEL_GATHER
//      tokens they are gathered into rank 0 and ranked there instead (the same result bits);
//   tail  the last of a KV head's G clusters to finish builds that head's fetch list (KVFetch
//      step 5: the rows of the union of the G sets F that are not resident), so the list is
//      ready when the kernel ends.
// Per-token terms use lambda w = clip(beta rho, r w, w) with rho = r / (1 - r).
#include <math.h>
#include <stddef.h>

#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

constexpr int CT_NT = 1024;
constexpr int CT_NW = CT_NT / 32;
constexpr int CT_MAX_CL = 8;
constexpr int CT_REC = 16;  // floats per record in a cluster all-reduce
// Points of the beta solve's first pass: C/2 and C/8.  (Measured against 1, 3 and 4 points on the
// bench; a simulation of the solve over the bench's heads gave 2.53 passes on average with the
// pair C/2, C/8 against 2.54 with C, C/4, and 52 heads of 1536 needing four passes or more
// against 132.)
constexpr int BETA_GRID = 2;
constexpr float BETA_GRID_FIRST = 0.5f;
constexpr float BETA_GRID_STEP = 0.25f;
constexpr int BETA_MAXIT = 64;
constexpr int SEL_MAXPASS = 16;

// Per-CTA 256-bin histogram, built with 32-bit atomics, one array per field (consecutive bins in
// consecutive banks).  A sum is kept in 64-bit fixed point split into a high part (q >> 18) and
// the low 18 bits, added separately: with the whole mapped to 2^49 the high parts sum below 2^31
// and at most 16384 low parts below 2^32, so neither wraps.
struct Hist {
    uint32_t cnt[256];
    uint32_t bm[256];  // max b_i (float bits; b_i >= 0)
    uint32_t sbh[256], sbl[256], svh[256], svl[256];
};
// The cluster-merged histogram, with the split sums recombined.
struct Merged {
    uint32_t cnt[256];
    uint32_t bm[256];
    unsigned long long sb[256], sv[256];
};
constexpr int FIX_SPLIT = 18;
// A candidate token of the select's cut bin, gathered into rank 0 when the bin holds at most
// SEL_GATHER tokens: its g bits, token id, w-hat and r (its Lemma 1 terms are recomputed there).
struct GatherCand {
    uint32_t g;
    int token;
    float w, r;
};
constexpr int SEL_GATHER = 512;
static_assert(SEL_GATHER * 12 <= 6 * 256 * 4, "the rank scratch (order and keys) fits a histogram buffer");

int certify_cluster_size(int n, int qheads, int sms) {
    if (n <= 8192) return 1;
    // Up to 32K tokens: clusters of 4 while the grid fits the GPU in one wave (the kernel then
    // ends with its slowest head), else clusters of 2 with twice the tokens per CTA: half the CTAs,
    // and half the exchanges and barriers per token, for grids that take several waves.
    if (n <= 32768) return (long long)qheads * 4 <= sms ? 4 : 2;
    return CT_MAX_CL;
}
int certify_chunk(int n, int cl) {
    const int chunk = (n + cl - 1) / cl;
    return (chunk + 31) / 32 * 32;
}
size_t certify_smem_bytes(int chunk) {
    return (size_t)CT_NW * CT_REC * 4                   // warp records of this CTA
           + (size_t)2 * CT_MAX_CL * CT_REC * 4         // CTA records from the cluster, two buffers
           + 2 * sizeof(Hist)                           // two histogram buffers
           + sizeof(Merged)                             // merged copy
           + (size_t)chunk * 12 + 64
           + (size_t)SEL_GATHER * sizeof(GatherCand);    // gathered select candidates (clusters of 1, 4)
}

// Cluster-wide all-reduce of a K-float record held identically by the lanes of each warp.
// `comb(x, y)` sets x to x (+) y.  Warp 0 combines the CTA's warp records with a butterfly and
// takes lane 0's result as the CTA record: a butterfly pairs comb(x, y) on one lane with
// comb(y, x) on the other, and a comb that is not bitwise symmetric (a multiply-add the compiler
// contracts) would leave the lanes a rounding apart.  Lanes 0..CL-1 send that one record into
// slot [my rank] of each peer, and after one cluster barrier every thread combines the CL
// records in rank order, so every thread of every CTA holds the same bits.  That is what keeps
// the cluster's control flow uniform: every branch after an exchange (the certificate, the beta
// passes, the select's passes) is decided from these values, and CTAs that took different
// branches would meet different cluster barriers.  The two CTA-record buffers alternate: a
// buffer is rewritten two calls later, after a barrier every peer passes only once it has read
// it.
template <int CL, int K, class Comb>
__device__ __forceinline__ void cluster_allreduce(float (&v)[K], float *wrec, float *xrec,
                                                  int &parity, Comb comb) {
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < K; ++k) wrec[warp * CT_REC + k] = v[k];
    }
    __syncthreads();
    float *buf = xrec + parity * (CT_MAX_CL * CT_REC);
    if (warp == 0) {
        float x[K];
#pragma unroll
        for (int k = 0; k < K; ++k) x[k] = wrec[lane * CT_REC + k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float y[K];
#pragma unroll
            for (int k = 0; k < K; ++k) y[k] = __shfl_xor_sync(0xFFFFFFFFu, x[k], o);
            comb(x, y);
        }
#pragma unroll
        for (int k = 0; k < K; ++k) x[k] = __shfl_sync(0xFFFFFFFFu, x[k], 0);
        if (lane < CL) {
            float *peer = cluster.map_shared_rank(buf, lane);
            const int me = (int)cluster.block_rank();
#pragma unroll
            for (int k = 0; k < K; ++k) peer[me * CT_REC + k] = x[k];
        }
    }
    cluster.sync();
    parity ^= 1;
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = buf[k];
#pragma unroll
    for (int c = 1; c < CL; ++c) {
        float y[K];
#pragma unroll
        for (int k = 0; k < K; ++k) y[k] = buf[c * CT_REC + k];
        comb(v, y);
    }
}

__device__ __forceinline__ float bern(float b, float V, float l) {
    const float A = b * l * (1.0f / 3.0f);
    return A + sqrtf(fmaf(A, A, 2.0f * V * l));
}

// Per-token terms use the hardware's approximate reciprocal, quotient and square root (about one
// ulp): their errors stay far below the 1e-5 relative resolution the decisions are held to.
__device__ __forceinline__ float sqrt_approx(float x) {
    float y;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rho_of(float r) { return __fdividef(r, 1.0f - r); }

// lambda at beta and the three per-token terms of Lemma 1 for a token of L (0 < r < 1):
// lambda w = clip(beta rho, r w, w);  beta_i = w - lambda w;  v_i = (lambda w)^2 (1 - r) / r =
// (lambda w)^2 / rho;  b_i = lambda w max(r, 1 - r) / r = lambda w max(1, 1 / rho).
__device__ __forceinline__ void token_terms(float w, float r, float rho, float beta, float &bi,
                                            float &vi, float &bb) {
    const float t = fminf(w, fmaxf(r * w, beta * rho));
    const float inv_rho = __fdividef(1.0f, rho);
    bi = w - t;
    vi = t * t * inv_rho;
    bb = t * fmaxf(1.0f, inv_rho);
}

// g_i D of Eq. (9) in the rationalised form, as the bits of a non-negative float.
__device__ __forceinline__ uint32_t g_bits(float bi, float vi, bool is_argmax, float A, float Rr,
                                           float b2, float VL, float l) {
    const float Vr = fmaxf(VL - vi, 0.0f);
    float gD;
    if (!is_argmax) {
        const float den = Rr + sqrt_approx(fmaf(A, A, 2.0f * Vr * l));
        gD = bi + (den > 0.0f ? __fdividef(2.0f * vi * l, den) : 0.0f);
    } else {
        const float A2 = b2 * l * (1.0f / 3.0f);
        const float R2 = sqrt_approx(fmaf(A2, A2, 2.0f * Vr * l));
        const float den = Rr + R2;
        gD = bi + (A - A2) +
             (den > 0.0f ? __fdividef(fmaf(A - A2, A + A2, 2.0f * vi * l), den) : 0.0f);
    }
    return __float_as_uint(fmaxf(gD, 0.0f));
}

__device__ __forceinline__ unsigned long long key64(uint32_t gbits, int token) {
    return ((unsigned long long)gbits << 24) | (unsigned long long)(0xFFFFFF - token);
}

// round(x * scale) as its high part (>> FIX_SPLIT) and its low FIX_SPLIT bits, in 32-bit
// arithmetic (64-bit conversions are slow on this part).  x * scale < 2^50 by construction: a
// term is at most the whole, which maps to 2^49.  Both the split y = yh 2^18 + rem and rem are
// exact in float, and yh 2^18 is even, so this is round-half-even of y.
__device__ __forceinline__ void fixed_split(float x, float scale, uint32_t &hi, uint32_t &lo) {
    const float y = fminf(x * scale, 1.0e15f);
    const float yh = truncf(y * (1.0f / (float)(1u << FIX_SPLIT)));
    const float rem = fmaf(-yh, (float)(1u << FIX_SPLIT), y);
    uint32_t h = __float2uint_rz(yh), l = __float2uint_rn(rem);
    if (l >= (1u << FIX_SPLIT)) {
        l -= 1u << FIX_SPLIT;
        h += 1u;
    }
    hi = h;
    lo = l;
}

// Nearest float of a 64-bit integer from two 32-bit conversions (within an ulp).
__device__ __forceinline__ float u64_to_float(unsigned long long x) {
    return fmaf((float)(uint32_t)(x >> 32), 4294967296.0f, (float)(uint32_t)x);
}

// 32-bit shared::cluster address of a local shared-memory address in CTA `rank`.
__device__ __forceinline__ uint32_t map_cluster(uint32_t local, int rank) {
    uint32_t r;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// State of the windowed select, uniform over the CTA.
struct SelState {
    unsigned long long lo;                // key of the window's first bin
    unsigned long long cand_lo, cand_hi;  // candidates: keys in [cand_lo, cand_hi)
    unsigned long long Bb, Bv;            // fixed-point sums of the tokens known to remain
    unsigned long long fthr;              // result: F = { keys >= fthr }
    uint32_t Bm;                          // max b of the tokens known to remain (float bits)
    int shift;                            // bin width 2^shift keys
    int absorb;                           // bin 0 also takes every candidate below lo
    int above;                            // tokens known to be in F
    int ncand;                            // tokens with keys in [cand_lo, cand_hi)
    int done, kstar;
    float eps_final;
};

// eps-hat D of a remaining set from its exact fixed-point sums and its max b (float bits), as
// every select decision evaluates it (Eq. (10)).
__device__ __forceinline__ float remaining_epsD(unsigned long long sb, unsigned long long sv, uint32_t mb,
                                                float iSB, float iSV, float l) {
    return u64_to_float(sb) * iSB + bern(__uint_as_float(mb), u64_to_float(sv) * iSV, l);
}

// One pass's scan of the merged histogram and the select's next state (Eq. (10): eps-hat of the
// remaining set, nonincreasing as tokens are taken in g order).  Threads 0..SEL_NT-1 take one bin
// each: exact integer prefix sums (and a running max) of the bins below it give the remaining
// set if the cut falls there; the cut bin is the last non-empty bin whose remaining set already
// certifies, and its thread moves the select on.  The other threads do not take part.
constexpr int SEL_NT = 256;  // = bins per pass
struct SelScratch {
    uint32_t c[SEL_NT / 32], m[SEL_NT / 32];
    unsigned long long b[SEL_NT / 32], v[SEL_NT / 32];
    int best[SEL_NT / 32];
};
__device__ __forceinline__ void sel_bar() { asm volatile("bar.sync 1, %0;" ::"n"(SEL_NT) : "memory"); }

__device__ __forceinline__ void select_step(const Merged &mh, SelState &ss, SelScratch &sx, int tid,
                                            float SB, float SV, float l, float epsD, float D) {
    const int lane = tid & 31, w = tid >> 5;
    const float iSB = SB > 0.0f ? 1.0f / SB : 0.0f;
    const float iSV = SV > 0.0f ? 1.0f / SV : 0.0f;
    const unsigned long long Bb = ss.Bb, Bv = ss.Bv;
    const uint32_t Bm = ss.Bm;
    const uint32_t c = mh.cnt[tid], m = mh.bm[tid];
    const unsigned long long sb = mh.sb[tid], sv = mh.sv[tid];
    uint32_t ic = c, im = m;
    unsigned long long ib = sb, iv = sv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t yc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        const uint32_t ym = __shfl_up_sync(0xFFFFFFFFu, im, o);
        const unsigned long long yb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
        const unsigned long long yv = __shfl_up_sync(0xFFFFFFFFu, iv, o);
        if (lane >= o) {
            ic += yc;
            im = max(im, ym);
            ib += yb;
            iv += yv;
        }
    }
    uint32_t xm = __shfl_up_sync(0xFFFFFFFFu, im, 1);
    if (lane == 0) xm = 0u;
    if (lane == 31) {
        sx.c[w] = ic;
        sx.m[w] = im;
        sx.b[w] = ib;
        sx.v[w] = iv;
    }
    sel_bar();
    uint32_t pc = 0u, pm = 0u, total = 0u;
    unsigned long long pb = 0ull, pv = 0ull;
#pragma unroll
    for (int k = 0; k < SEL_NT / 32; ++k) {
        if (k < w) {
            pc += sx.c[k];
            pm = max(pm, sx.m[k]);
            pb += sx.b[k];
            pv += sx.v[k];
        }
        total += sx.c[k];
    }
    // The bins below this one: all earlier warps, then the earlier lanes of this warp.
    const uint32_t best_c = pc + ic - c;
    const uint32_t best_m = max(Bm, max(pm, xm));
    const unsigned long long best_b = Bb + pb + ib - sb, best_v = Bv + pv + iv - sv;
    const float best_e = remaining_epsD(best_b, best_v, best_m, iSB, iSV, l);
    const uint32_t best_n = c;
    int jb = (c > 0u && best_e < epsD) ? tid : -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) jb = max(jb, __shfl_xor_sync(0xFFFFFFFFu, jb, o));
    if (lane == 0) sx.best[w] = jb;
    sel_bar();
#pragma unroll
    for (int k = 0; k < SEL_NT / 32; ++k) jb = max(jb, sx.best[k]);
    if (jb < 0) {
        if (tid == 0) {  // rounding left no bin qualifying: take every candidate
            ss.kstar = ss.above + (int)total;
            ss.fthr = ss.absorb ? 0ull : ss.cand_lo;
            ss.eps_final = remaining_epsD(Bb, Bv, Bm, iSB, iSV, l) / D;
            ss.done = 1;
        }
        return;
    }
    if (tid != jb) return;
    const int cj = (int)best_n;
    ss.Bb = best_b;
    ss.Bv = best_v;
    ss.Bm = best_m;
    ss.eps_final = best_e / D;
    const int above = ss.above + (int)(total - best_c - best_n);  // bins above the cut
    ss.above = above;
    const unsigned long long lo = ss.lo;
    const int shift = ss.shift;
    const unsigned long long cut_lo = lo + ((unsigned long long)jb << shift);
    if (ss.absorb && jb == 0) {
        // The cut lies in bin 0, which also holds every candidate below the window.
        if (cj == 1) {  // one token left: it is taken, and so is every other token
            ss.kstar = above + 1;
            ss.fthr = 0ull;
            ss.done = 1;
            return;
        }
        // Slide the window down at the same resolution; it ends where bin 0 ended.
        ss.ncand = cj;
        ss.cand_lo = 0ull;
        ss.cand_hi = lo + (1ull << shift);
        const unsigned long long span = 255ull << shift;
        if (lo > span) {
            ss.lo = lo - span;
        } else {
            ss.lo = 0ull;
            ss.absorb = 0;
        }
        return;
    }
    if (cj == 1 || shift == 0) {
        ss.kstar = above + cj;
        ss.fthr = cut_lo;
        ss.done = 1;
        return;
    }
    ss.ncand = cj;
    ss.cand_lo = cut_lo;
    ss.cand_hi = cut_lo + (1ull << shift);
    ss.lo = cut_lo;
    ss.shift = shift >= 8 ? shift - 8 : 0;
    ss.absorb = 0;
}

// The per-KV-head fetch list, built by the last of the KV head's G clusters to finish.  The
// cluster barrier orders every CTA's F words before rank 0's acquire-release increment of the
// KV head's counter; the cluster that completes the count (its rank-0 CTA) ORs the G bitmaps,
// removes the resident tokens, scans the counts and writes the ascending ids, one coalesced
// store per bitmap word and warp; it then rearms the counter for the next call.
constexpr int FL_MAX_WPT = 4;  // bitmap words per thread: n <= 131072 = 4 * 32 * CT_NT
// Tokens (and bitmap words) a thread holds: clusters of 1 and 4 cover n <= 8192 and n <= 32768
// with a CTA's chunk at most 8 * CT_NT tokens; clusters of 2 (n <= 32768) and of 8 take up to
// 16 * CT_NT; the whole bitmap is at most CT_NT words except with clusters of 8.
template <int CL>
struct PerThread {
    static constexpr int tokens = (CL == CT_MAX_CL || CL == 2) ? 16 : 8;
    static constexpr int words = CL == CT_MAX_CL ? FL_MAX_WPT : 1;
};

__device__ __forceinline__ int atomic_add_acq_rel(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

template <int CL>
__device__ __forceinline__ void fetch_list_tail(const CertifyArgs &a, int ul, int ug) {
    __shared__ int s_last;
    __shared__ int s_wsum[CT_NW];
    __shared__ int s_nf[CT_NW][8];
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.li.G, W = a.W;
    cluster.sync();
    if (cluster.block_rank() != 0) return;
    if (tid == 0) {
        const int old = atomic_add_acq_rel(&a.fl_counter[ul], 1);
        s_last = old == G - 1;
        if (old == G - 1) a.fl_counter[ul] = 0;
    }
    __syncthreads();
    if (!s_last) return;
    const uint32_t *res = a.resident + (size_t)ug * W;
    const uint32_t *F0 = a.F + (size_t)ul * G * W;
    constexpr int WPT = PerThread<CL>::words;
    const int wpt = (W + CT_NT - 1) / CT_NT;  // <= WPT
    const int w0 = tid * wpt;
    uint32_t fw[WPT];
    int cnt[WPT];
    int my = 0;
    int nf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
        const int w = w0 + i;
        uint32_t f = 0u;
        if (i < wpt && w < W) {
            const uint32_t rw = __ldcg(res + w);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g < G) {
                    const uint32_t fg = __ldcg(F0 + (size_t)g * W + w) & ~rw;
                    f |= fg;
                    nf[g] += __popc(fg);
                }
            }
        }
        fw[i] = f;
        cnt[i] = __popc(f);
        my += cnt[i];
    }
    int incl = my;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    for (int g = 0; g < G; ++g) {
        const int t = warp_sum(nf[g]);
        if (lane == 0) s_nf[warp][g] = t;
    }
    __syncthreads();
    if (warp == 0) {
        const int v = lane < CT_NW ? s_wsum[lane] : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane < CT_NW) s_wsum[lane] = x - v;  // exclusive
        if (lane == 31) {
            a.counts[ul] = x;
            if (a.counts_user) a.counts_user[ul] = x;
            if (a.counts_host) a.counts_host[ul] = x;
        }
        if (lane < G) {
            int t = 0;
            for (int w = 0; w < CT_NW; ++w) t += s_nf[w][lane];
            a.qstats[ul * G + lane].n_fetch = t;
        }
    }
    __syncthreads();
    // Lane j's words, in order, are written by the whole warp: lane l stores the id of bit l.
    int pos = s_wsum[warp] + incl - my;
    int32_t *ids = a.ids + (size_t)ul * a.n;
    int32_t *idsu = a.ids_user ? a.ids_user + (size_t)ul * a.n : nullptr;
    int32_t *idsh = a.ids_host ? a.ids_host + (size_t)ul * a.n : nullptr;
    const uint32_t below = (1u << lane) - 1u;
    for (int j = 0; j < 32; ++j) {
        int base = __shfl_sync(0xFFFFFFFFu, pos, j);
        const int wj = __shfl_sync(0xFFFFFFFFu, w0, j);
#pragma unroll
        for (int i = 0; i < WPT; ++i) {
            const uint32_t f = __shfl_sync(0xFFFFFFFFu, fw[i], j);
            if ((f >> lane) & 1u) {
                const int p = base + __popc(f & below);
                const int id = 32 * (wj + i) + lane;
                ids[p] = id;
                if (idsu) idsu[p] = id;
                if (idsh) idsh[p] = id;
            }
            base += __popc(f);
        }
    }
}

// The end of the select when the candidates (keys in [cand_lo, cand_hi), ss.ncand of them, at most
// SEL_GATHER) are few.  Every CTA appends its candidates to rank 0's buffer; rank 0 orders them by
// key (g descending, ties to the lower id: the keys are unique), recomputes each one's Lemma 1
// terms and fixed-point parts exactly as the histogram passes do, and forms for every k the sums
// of the set that remains when the first k are taken: the tokens known to remain plus the
// candidates after rank k (exact 64-bit suffix sums, a suffix max of b).  k* is the smallest k in
// [1, ncand] whose remaining set certifies (all of them if rounding leaves none), evaluated with
// the same expression as the histogram scan, so F, k* and eps-hat are the bits the finer passes
// would give.  Rank 0 writes the result into every CTA's select state; `ord` is rank 0's scratch
// of SEL_GATHER ints followed by SEL_GATHER 64-bit keys.
template <int CL>
__device__ __noinline__ void gather_select(cg::cluster_group &cluster, int crank, int tid, SelState &ss,
                                           int &s_gn, GatherCand *gbuf, int *ord, const float *W,
                                           const float *R, const uint32_t *X, int chunk, int base,
                                           float beta, float SB, float SV, float l, float epsD,
                                           float D) {
    constexpr int TPT = PerThread<CL>::tokens;
    const int lane = tid & 31, warp = tid >> 5;
    {
        // The thread's candidates, their offsets in this CTA (a block scan of the counts) and one
        // remote atomic per CTA for the CTA's place in rank 0's buffer.
        __shared__ int s_wc[CT_NW];
        __shared__ int s_base;
        const unsigned long long clo = ss.cand_lo, chi = ss.cand_hi;
        uint32_t cm = 0u;
#pragma unroll
        for (int q = 0; q < TPT; ++q) {
            const int i = tid + q * CT_NT;
            if (i < chunk && R[i] < 1.0f) {
                const unsigned long long key = key64(X[i], base + i);
                if (key >= clo && key < chi) cm |= 1u << q;
            }
        }
        const int c = __popc(cm);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wc[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int t = s_wc[lane];
            int x = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            s_wc[lane] = x - t;  // exclusive
            if (lane == 31 && x > 0) s_base = atomicAdd(cluster.map_shared_rank(&s_gn, 0), x);
        }
        __syncthreads();
        if (cm) {
            GatherCand *gb0 = cluster.map_shared_rank(gbuf, 0);
            int slot = s_base + s_wc[warp] + incl - c;
            for (uint32_t m = cm; m; m &= m - 1u, ++slot) {
                const int i = tid + (__ffs(m) - 1) * CT_NT;
                if (slot < SEL_GATHER) gb0[slot] = GatherCand{X[i], base + i, W[i], R[i]};
            }
        }
    }
    cluster.sync();  // every candidate is in rank 0's buffer
    if (crank == 0) {
        __shared__ unsigned long long s_sb[CT_NW], s_sv[CT_NW];
        __shared__ uint32_t s_mb[CT_NW];
        __shared__ int s_k;
        const int nc = min(s_gn, SEL_GATHER);
        unsigned long long *keys = reinterpret_cast<unsigned long long *>(ord + SEL_GATHER);
        if (tid < nc) keys[tid] = key64(gbuf[tid].g, gbuf[tid].token);
        if (tid == 0) s_k = nc;  // none certifies: take every candidate
        __syncthreads();
        // Rank of candidate j: how many keys exceed its own, counted by P lanes of one warp
        // (P the largest power of two with P nc <= CT_NT, at most 32) over interleaved keys.
        {
            int P = 32;
            while (P > 1 && P * nc > CT_NT) P >>= 1;
            const int j = tid / P, part = tid - j * P;
            int rk = 0;
            if (j < nc) {
                const unsigned long long kj = keys[j];
                int q = part;
#pragma unroll 1
                for (; q + 3 * P < nc; q += 4 * P)
                    rk += (keys[q] > kj ? 1 : 0) + (keys[q + P] > kj ? 1 : 0) +
                          (keys[q + 2 * P] > kj ? 1 : 0) + (keys[q + 3 * P] > kj ? 1 : 0);
                for (; q < nc; q += P) rk += keys[q] > kj ? 1 : 0;
            }
            for (int o = 1; o < P; o <<= 1) rk += __shfl_xor_sync(0xFFFFFFFFu, rk, o);
            if (j < nc && part == 0) ord[rk] = j;
        }
        __syncthreads();
        // Thread p holds the candidate of rank p.
        const float iSB = SB > 0.0f ? 1.0f / SB : 0.0f;
        const float iSV = SV > 0.0f ? 1.0f / SV : 0.0f;
        unsigned long long qb = 0ull, qv = 0ull;
        uint32_t mb = 0u;
        if (tid < nc) {
            const GatherCand c = gbuf[ord[tid]];
            float bi, vi, bb;
            token_terms(c.w, c.r, rho_of(c.r), beta, bi, vi, bb);
            uint32_t h, lo;
            fixed_split(bi, SB, h, lo);
            qb = ((unsigned long long)h << FIX_SPLIT) + lo;
            fixed_split(vi, SV, h, lo);
            qv = ((unsigned long long)h << FIX_SPLIT) + lo;
            mb = __float_as_uint(bb);
        }
        // Exclusive suffix sums (ranks after p) within the warp, then over the later warps.
        unsigned long long eb = 0ull, ev = 0ull;
        uint32_t em = 0u;
        {
            unsigned long long ib = qb, iv = qv;
            uint32_t im = mb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long yb = __shfl_down_sync(0xFFFFFFFFu, ib, o);
                const unsigned long long yv = __shfl_down_sync(0xFFFFFFFFu, iv, o);
                const uint32_t ym = __shfl_down_sync(0xFFFFFFFFu, im, o);
                if (lane + o < 32) {
                    ib += yb;
                    iv += yv;
                    im = max(im, ym);
                }
            }
            if (lane == 0) {
                s_sb[warp] = ib;
                s_sv[warp] = iv;
                s_mb[warp] = im;
            }
            eb = ib - qb;
            ev = iv - qv;
            const uint32_t xm = __shfl_down_sync(0xFFFFFFFFu, im, 1);
            em = lane == 31 ? 0u : xm;
        }
        __syncthreads();
        if (warp == 0) {  // exclusive suffix over the warps' totals, in place
            unsigned long long tb = s_sb[lane], tv = s_sv[lane];
            uint32_t tm = s_mb[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long yb = __shfl_down_sync(0xFFFFFFFFu, tb, o);
                const unsigned long long yv = __shfl_down_sync(0xFFFFFFFFu, tv, o);
                const uint32_t ym = __shfl_down_sync(0xFFFFFFFFu, tm, o);
                if (lane + o < 32) {
                    tb += yb;
                    tv += yv;
                    tm = max(tm, ym);
                }
            }
            const unsigned long long xb = __shfl_down_sync(0xFFFFFFFFu, tb, 1);
            const unsigned long long xv = __shfl_down_sync(0xFFFFFFFFu, tv, 1);
            const uint32_t xm = __shfl_down_sync(0xFFFFFFFFu, tm, 1);
            __syncwarp();
            s_sb[lane] = lane == 31 ? 0ull : xb;
            s_sv[lane] = lane == 31 ? 0ull : xv;
            s_mb[lane] = lane == 31 ? 0u : xm;
        }
        __syncthreads();
        eb += s_sb[warp];
        ev += s_sv[warp];
        em = max(em, s_mb[warp]);
        // Taking ranks 0..p (k = p + 1) leaves the known remainder and the ranks after p.
        float e = 0.0f;
        bool ok = false;
        if (tid < nc) {
            e = remaining_epsD(ss.Bb + eb, ss.Bv + ev, max(ss.Bm, em), iSB, iSV, l);
            ok = e < epsD;
        }
        if (ok) atomicMin(&s_k, tid + 1);
        __syncthreads();
        const int ks = s_k;
        if (tid == ks - 1) {
            const GatherCand c = gbuf[ord[tid]];
            const unsigned long long ft = key64(c.g, c.token);
            const int kstar = ss.above + ks;
            const float efin = e / D;
            for (int c2 = 0; c2 < CL; ++c2) {
                SelState *r = cluster.map_shared_rank(&ss, c2);
                r->fthr = ft;
                r->kstar = kstar;
                r->eps_final = efin;
                r->done = 1;
            }
        }
    }
    cluster.sync();  // every CTA holds the result
}

template <int CL, bool SL>
__global__ void __launch_bounds__(CT_NT, 1) k_certify(CertifyArgs a) {
    pdl_trigger();  // the refine kernel after this one may be scheduled early
    cluster_arrive_relaxed();  // waited on before the first exchange with the peers
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *wrec = reinterpret_cast<float *>(smem_raw);
    float *xrec = wrec + CT_NW * CT_REC;
    Merged &mh = *reinterpret_cast<Merged *>(xrec + 2 * CT_MAX_CL * CT_REC);
    Hist *hist = reinterpret_cast<Hist *>(&mh + 1);
    float *W = reinterpret_cast<float *>(hist + 2);  // logit, then w-hat
    float *R = W + a.chunk;                          // r (1 for H and padding)
    uint32_t *X = reinterpret_cast<uint32_t *>(R + a.chunk);  // r/(1-r), later the g key
    GatherCand *gbuf = reinterpret_cast<GatherCand *>(X + a.chunk);  // rank 0: the select's candidates

    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.li.G;
    const int qh = blockIdx.x / CL;
    const int ul = qh / G;
    const int ug = a.li.unit_global(ul);
    const int n = a.n, chunk = a.chunk;
    const int base = crank * chunk;
    const float *sc = a.scores + (size_t)qh * n;
    const float *rf = a.r_full + (size_t)ug * n;
    const float eps = a.eps, l = a.ldelta;
    const float NEG_INF = -__int_as_float(0x7F800000);
    int parity = 0;

    // ---- 1. logits, r; max logit, D, sum_L w (1 - r), |L| in one exchange ----
    float m, D, C, nL;
    float tmax = NEG_INF;
    {
        // All of the thread's loads are issued before any is used.
        constexpr int TPT = PerThread<CL>::tokens;
        float sv[TPT], rv[TPT];
#pragma unroll
        for (int k = 0; k < TPT; ++k) {
            const int i = tid + k * CT_NT, t = base + i;
            rv[k] = (i < chunk && t < n) ? rf[t] : 1.0f;
        }
        pdl_wait();  // the logits come from the kernel before this one
#pragma unroll
        for (int k = 0; k < TPT; ++k) {
            const int i = tid + k * CT_NT, t = base + i;
            sv[k] = (i < chunk && t < n) ? sc[t] : NEG_INF;
            tmax = fmaxf(tmax, sv[k]);
        }
        float d = 0.f, c = 0.f, cnt = 0.f;
#pragma unroll
        for (int k = 0; k < TPT; ++k) {
            const int i = tid + k * CT_NT;
            if (i >= chunk) break;
            const float e = tmax == NEG_INF ? 0.0f : expf(sv[k] - tmax);  // 0 for padding
            W[i] = e;  // exp(logit - this thread's max); rescaled to w-hat once m is known
            R[i] = rv[k];
            d += e;
            const float r = rv[k];
            if (r < 1.0f) {
                c += e * (1.0f - r);
                cnt += 1.0f;
            }
        }
        const float wmax = warp_max(tmax);
        const float sc_t = tmax == NEG_INF ? 0.0f : expf(tmax - wmax);
        // (max logit, D, C) combine as online-softmax partials; |L| adds.
        float rec[4] = {wmax, warp_sum(d * sc_t), warp_sum(c * sc_t), warp_sum(cnt)};
        cluster_wait_all();  // every CTA of the cluster is running: its shared memory may be written
        cluster_allreduce<CL>(rec, wrec, xrec, parity, [&](float (&x)[4], const float (&y)[4]) {
            const float M = fmaxf(x[0], y[0]);
            const float fx = x[0] == NEG_INF ? 0.0f : expf(x[0] - M);
            const float fy = y[0] == NEG_INF ? 0.0f : expf(y[0] - M);
            x[0] = M;  // products rounded separately: the same bits for (x, y) and (y, x)
            x[1] = __fadd_rn(__fmul_rn(x[1], fx), __fmul_rn(y[1], fy));
            x[2] = __fadd_rn(__fmul_rn(x[2], fx), __fmul_rn(y[2], fy));
            x[3] = x[3] + y[3];
        });
        m = rec[0];
        D = rec[1];
        C = rec[2];
        nL = rec[3];
    }

    // ---- 2. beta: safeguarded piece-wise Newton ----
    // h(beta) = beta - sum_L w-hat (1 - lambda(beta)) rises from h(0) <= 0 to h(C) >= 0.  Every
    // pass evaluates, at a point beta, the sums of the linear piece of h through it and the
    // nearest breakpoints on either side: the largest one below (pl) and the smallest one at or
    // above (ph).  A token's breakpoints are w (1 - r), where lambda leaves its floor, and
    // w (1 - r) / r, where it reaches 1.  The root of the piece through beta is the fixed point
    // when it lies strictly between pl and ph, or when it reproduces beta (to 1e-6 relative:
    // float32 sums jitter by an ulp or two).  The first pass evaluates BETA_GRID points C/2, C/8
    // together (one cluster exchange), which brackets the root and gives the Newton start; later
    // passes take one point each.
    float beta = 0.0f;
    int iters = 0, flags = 0;
    const float wscale = tmax == NEG_INF ? 0.0f : expf(tmax - m);  // w-hat = W * wscale
    // Classify one token of L at beta into the piece sums and nearest breakpoints (fl = w (1 - r)):
    // at its floor, in the middle, or at lambda = 1; a breakpoint fl / r is computed only where it
    // can move pl or ph (most tokens sit at their floor: the branches are nearly uniform).
    auto piece = [](float beta, float w, float r, float fl, float rho, float &ab, float &S,
                    float &pl, float &ph) {
        if (beta <= fl) {
            ab += fl;
            ph = fminf(ph, fl);
        } else if (beta * r < fl) {
            ab += w;
            S += rho;
            pl = fmaxf(pl, fl);
            if (fl < r * ph) ph = fminf(ph, __fdividef(fl, r));
        } else if (fl > r * pl) {
            pl = fmaxf(pl, __fdividef(fl, r));
        }
    };
    if (C > 0.0f) {
        constexpr int NG = BETA_GRID;
        float gb[NG], gab[NG], gS[NG], gpl[NG], gph[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) {
            gb[k] = k == 0 ? BETA_GRID_FIRST * C : gb[k - 1] * BETA_GRID_STEP;
            gab[k] = 0.f;
            gS[k] = 0.f;
            gpl[k] = 0.f;
            gph[k] = INFINITY;
        }
        // Pass 1 also turns the logits into w-hat and r into rho = r / (1 - r).
        for (int i = tid; i < chunk; i += CT_NT) {
            const float r = R[i];
            const float w = W[i] * wscale;
            W[i] = w;
            if (r < 1.0f) {
                const float rho = rho_of(r);
                X[i] = __float_as_uint(rho);
                const float fl = w * (1.0f - r);
#pragma unroll
                for (int k = 0; k < NG; ++k) piece(gb[k], w, r, fl, rho, gab[k], gS[k], gpl[k], gph[k]);
            }
        }
        float rec[4 * NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) {
            rec[4 * k] = warp_sum(gab[k]);
            rec[4 * k + 1] = warp_sum(gS[k]);
            rec[4 * k + 2] = warp_max(gpl[k]);
            rec[4 * k + 3] = warp_min(gph[k]);
        }
        cluster_allreduce<CL>(rec, wrec, xrec, parity, [](float (&x)[4 * NG], const float (&y)[4 * NG]) {
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                x[4 * k] += y[4 * k];
                x[4 * k + 1] += y[4 * k + 1];
                x[4 * k + 2] = fmaxf(x[4 * k + 2], y[4 * k + 2]);
                x[4 * k + 3] = fminf(x[4 * k + 3], y[4 * k + 3]);
            }
        });
        // The bracket from the signs of h at the grid points; Newton roots of their pieces are
        // below the root where h is concave, so the largest inside the bracket starts the rest.
        float lo = 0.0f, hi = C, start = 0.0f;
        bool found = false;
#pragma unroll
        for (int k = 0; k < NG; ++k) {
            const float bk = gb[k];
            const float ab = rec[4 * k], S = rec[4 * k + 1];
            const float nb = __fdiv_rn(ab, 1.0f + S);
            if (!found && ((nb > rec[4 * k + 2] && nb < rec[4 * k + 3]) || fabsf(nb - bk) <= 1e-6f * bk)) {
                beta = nb;
                found = true;
            }
            if (fmaf(bk, 1.0f + S, -ab) < 0.0f) lo = fmaxf(lo, bk);
            else hi = fminf(hi, bk);
            start = fmaxf(start, nb);
        }
        iters = 1;
        if (!found) {
            beta = (start > lo && start < hi) ? start : ((lo > 0.0f) ? sqrtf(lo) * sqrtf(hi) : hi * 0.0625f);
            const int maxit = a.beta_maxit > 0 ? a.beta_maxit : BETA_MAXIT;
            for (iters = 2; iters <= maxit; ++iters) {
                float ab = 0.f, S = 0.f, pl = 0.f, ph = INFINITY;
                for (int i = tid; i < chunk; i += CT_NT) {
                    const float r = R[i];
                    if (r < 1.0f) {
                        const float w = W[i];
                        piece(beta, w, r, w * (1.0f - r), __uint_as_float(X[i]), ab, S, pl, ph);
                    }
                }
                float rec1[4] = {warp_sum(ab), warp_sum(S), warp_max(pl), warp_min(ph)};
                cluster_allreduce<CL>(rec1, wrec, xrec, parity,
                                      [](float (&x)[4], const float (&y)[4]) {
                                          x[0] += y[0];
                                          x[1] += y[1];
                                          x[2] = fmaxf(x[2], y[2]);
                                          x[3] = fminf(x[3], y[3]);
                                      });
                ab = rec1[0];
                S = rec1[1];
                pl = rec1[2];
                ph = rec1[3];
                float nb = __fdiv_rn(ab, 1.0f + S);
                if ((nb > pl && nb < ph) || fabsf(nb - beta) <= 1e-6f * beta) {
                    beta = nb;
                    break;
                }
                const float hval = fmaf(beta, 1.0f + S, -ab);
                if (hval < 0.0f) lo = beta; else hi = beta;
                if (!(nb > lo && nb < hi)) nb = (lo > 0.0f) ? sqrtf(lo) * sqrtf(hi) : hi * 0.0625f;
                beta = nb;
                if ((hi - lo) <= 1e-6f * hi) break;
            }
            if (iters > maxit) {
                iters = maxit;
                flags = 1;
            }
        }
    } else {  // no token of L carries weight: only convert the logits
        for (int i = tid; i < chunk; i += CT_NT) {
            W[i] *= wscale;
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
        float rec[5] = {warp_sum(sb), warp_sum(sv), tb.b1, __int_as_float(tb.id1), tb.b2};
        cluster_allreduce<CL>(rec, wrec, xrec, parity, [](float (&x)[5], const float (&y)[5]) {
            x[0] += y[0];
            x[1] += y[1];
            const Top2 t = top2_merge(Top2{x[2], __float_as_int(x[3]), x[4]},
                                      Top2{y[2], __float_as_int(y[3]), y[4]});
            x[2] = t.b1;
            x[3] = __int_as_float(t.id1);
            x[4] = t.b2;
        });
        betaL = rec[0];
        VL = rec[1];
        tb = Top2{rec[2], __float_as_int(rec[3]), rec[4]};
    }
    const float b1 = fmaxf(tb.b1, 0.0f), b2 = fmaxf(tb.b2, 0.0f);
    const int id1 = tb.id1;
    const float eps_hat = (betaL + bern(b1, VL, l)) / D;
    const bool certified = eps_hat < eps;

    // ---- 4. selection ----
    // The select's state is uniform over the CTA and lives in shared memory: one lane of warp 0
    // decides each pass and every thread reads the outcome after a barrier.
    __shared__ SelState ss;
    __shared__ SelScratch sx;
    int kstar = 0;
    unsigned long long fthr = ~0ull;  // F = { L tokens with key >= fthr }
    float eps_final = eps_hat;
    bool exhausted = false;
    if constexpr (SL) if (!certified) {
        // Only the KV head's shortlist may be fetched.  Candidates (at most SHORTLIST_MAX) carry
        // their key and Lemma 1 terms into a list in rank 0 (the histogram region is free here);
        // every other token of L stays in the remaining set (its sums all-reduced).  Rank 0 ranks
        // the list by key and scans it from the end for the first k with eps-hat < eps; the cut
        // key is sent back to every CTA.
        struct Cand {
            unsigned long long key;
            float bi, vi, bb, pad;
        };
        __shared__ int s_nc, s_kstar, s_exh;
        __shared__ unsigned long long s_fthr;
        __shared__ float s_efin;
        Cand *list = reinterpret_cast<Cand *>(hist);                 // [SHORTLIST_MAX]
        int *rank_of = reinterpret_cast<int *>(list + SHORTLIST_MAX);  // sorted position -> entry
        const float A = b1 * l * (1.0f / 3.0f);
        const float Rr = sqrtf(fmaf(A, A, 2.0f * VL * l));
        const uint32_t *sl = a.shortlist + (size_t)ul * a.W;
        if (tid == 0) s_nc = 0;
        cluster.sync();  // rank 0's counter is zero before anyone appends
        int *cnt0 = cluster.map_shared_rank(&s_nc, 0);
        Cand *list0 = cluster.map_shared_rank(list, 0);
        float osb = 0.0f, osv = 0.0f, obm = 0.0f;
        for (int i = tid; i < chunk; i += CT_NT) {
            const float r = R[i];
            if (r < 1.0f) {
                const int t = base + i;
                float bi, vi, bb;
                token_terms(W[i], r, __uint_as_float(X[i]), beta, bi, vi, bb);
                if ((sl[t >> 5] >> (t & 31)) & 1u) {
                    const uint32_t g = g_bits(bi, vi, t == id1 && b2 != b1, A, Rr, b2, VL, l);
                    X[i] = g;
                    const int slot = atomicAdd(cnt0, 1);
                    if (slot < SHORTLIST_MAX) list0[slot] = Cand{key64(g, t), bi, vi, bb, 0.0f};
                } else {
                    X[i] = 0u;
                    osb += bi;
                    osv += vi;
                    obm = fmaxf(obm, bb);
                }
            }
        }
        float rec[3] = {warp_sum(osb), warp_sum(osv), warp_max(obm)};
        cluster_allreduce<CL>(rec, wrec, xrec, parity, [](float (&x)[3], const float (&y)[3]) {
            x[0] += y[0];
            x[1] += y[1];
            x[2] = fmaxf(x[2], y[2]);
        });
        if (crank == 0) {
            const int nc = min(s_nc, SHORTLIST_MAX);
            for (int j = tid; j < nc; j += CT_NT) {  // keys are unique: ranks are a permutation
                const unsigned long long kj = list[j].key;
                int rk = 0;
                for (int q = 0; q < nc; ++q) rk += list[q].key > kj ? 1 : 0;
                rank_of[rk] = j;
            }
            __syncthreads();
            if (tid == 0) {
                float sbv = rec[0], svv = rec[1], smx = rec[2];
                float ek_next = (sbv + bern(smx, svv, l)) / D;  // eps-hat with every candidate taken
                int kk = -1;
                float efin = ek_next;
                // eps-hat(k) for k = nc .. 1; k* is the smallest k >= 1 with eps-hat(k) < eps
                for (int k = nc; k >= 1; --k) {
                    if (ek_next < eps) {
                        kk = k;
                        efin = ek_next;
                    }
                    const Cand &cd = list[rank_of[k - 1]];
                    sbv += cd.bi;
                    svv += cd.vi;
                    smx = fmaxf(smx, cd.bb);
                    ek_next = (sbv + bern(smx, svv, l)) / D;
                }
                const bool exh = kk < 0;
                if (exh) {
                    kk = nc;
                    efin = (rec[0] + bern(rec[2], rec[1], l)) / D;
                }
                const unsigned long long ft = kk >= 1 ? list[rank_of[kk - 1]].key : ~0ull;
                for (int c2 = 0; c2 < CL; ++c2) {
                    *cluster.map_shared_rank(&s_fthr, c2) = ft;
                    *cluster.map_shared_rank(&s_kstar, c2) = kk;
                    *cluster.map_shared_rank(&s_exh, c2) = exh ? 1 : 0;
                    *cluster.map_shared_rank(&s_efin, c2) = efin;
                }
            }
        }
        cluster.sync();
        fthr = s_fthr;
        kstar = s_kstar;
        exhausted = s_exh != 0;
        eps_final = s_efin;
        if (s_nc > SHORTLIST_MAX) flags |= 2;  // more candidates than the list holds
    }
    if constexpr (!SL) if (!certified) {
        const float A = b1 * l * (1.0f / 3.0f);
        const float Rr = sqrtf(fmaf(A, A, 2.0f * VL * l));
        // Fixed-point scales: every partial sum is at most the whole, which maps to 2^49 (a scale
        // is capped below the float range; a zero total gives zero sums).
        const float SB = betaL > 0.0f ? fminf(562949953421312.0f / betaL, 1e38f) : 0.0f;
        const float SV = VL > 0.0f ? fminf(562949953421312.0f / VL, 1e38f) : 0.0f;
        __shared__ int s_gn;  // rank 0: candidates gathered
        if (tid == 0) s_gn = 0;  // before the first pass's cluster barrier; appends come after it
        if (tid == 0) {
            // Every g_i D is at most eps-hat(L) D; the first window ends just above that.
            const uint32_t top = __float_as_uint(betaL + bern(b1, VL, l)) + 256u;
            const unsigned long long wend = ((unsigned long long)top + 1ull) << 24;
            ss.lo = wend > (1ull << 52) ? wend - (1ull << 52) : 0ull;
            ss.cand_lo = 0ull;
            ss.cand_hi = ~0ull;
            ss.Bb = 0ull;  // tokens known to remain below the candidates
            ss.Bv = 0ull;
            ss.fthr = ~0ull;
            ss.Bm = 0u;
            ss.shift = 44;
            ss.absorb = 1;  // bin 0 also takes every candidate below lo
            ss.above = 0;
            ss.ncand = 0;
            ss.done = 0;
            ss.kstar = 0;
            ss.eps_final = eps_hat;
        }
        for (int pass = 0; pass < SEL_MAXPASS; ++pass) {
            Hist &hb = hist[pass & 1];
            for (int j = tid; j < 6 * 256; j += CT_NT) (&hb.cnt[0])[j] = 0u;
            __syncthreads();
            const unsigned long long lo = ss.lo, cand_lo = ss.cand_lo, cand_hi = ss.cand_hi;
            const int shift = ss.shift;
            const bool absorb = ss.absorb != 0;
            uint32_t bc = 0u, bbm = 0u, bsbh = 0u, bsbl = 0u, bsvh = 0u, bsvl = 0u;
            // Bin one token of L (its key k and Lemma 1 terms given).
            auto bin_token = [&](unsigned long long k, float bi, float vi, float bb) {
                uint32_t qbh, qbl, qvh, qvl;
                fixed_split(bi, SB, qbh, qbl);
                fixed_split(vi, SV, qvh, qvl);
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
                    atomicAdd(&hb.cnt[bin], 1u);
                    atomicMax(&hb.bm[bin], __float_as_uint(bb));
                    atomicAdd(&hb.sbh[bin], qbh);
                    atomicAdd(&hb.sbl[bin], qbl);
                    atomicAdd(&hb.svh[bin], qvh);
                    atomicAdd(&hb.svl[bin], qvl);
                }
            };
            if (pass == 0) {
                // The g key (Eq. (9), rationalised) of every token of L.
                for (int i = tid; i < chunk; i += CT_NT) {
                    const float r = R[i];
                    if (r < 1.0f) {
                        float bi, vi, bb;
                        token_terms(W[i], r, __uint_as_float(X[i]), beta, bi, vi, bb);
                        const uint32_t g = g_bits(bi, vi, base + i == id1 && b2 != b1, A, Rr, b2,
                                                  VL, l);
                        X[i] = g;
                        bin_token(key64(g, base + i), bi, vi, bb);
                    }
                }
            } else {
                // Only the candidates (keys in [cand_lo, cand_hi)): the thread's keys are read
                // with all loads in flight, then its few candidates visited in token order.
                constexpr int TPT = PerThread<CL>::tokens;
                uint32_t todo = 0u;
#pragma unroll
                for (int q = 0; q < TPT; ++q) {
                    const int i = tid + q * CT_NT;
                    if (i < chunk && R[i] < 1.0f) {
                        const unsigned long long key = key64(X[i], base + i);
                        if (key >= cand_lo && key < cand_hi) todo |= 1u << q;
                    }
                }
                for (; todo; todo &= todo - 1u) {
                    const int i = tid + (__ffs(todo) - 1) * CT_NT;
                    const float r = R[i];
                    float bi, vi, bb;
                    token_terms(W[i], r, rho_of(r), beta, bi, vi, bb);
                    bin_token(key64(X[i], base + i), bi, vi, bb);
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
                    atomicAdd(&hb.cnt[0], bc);
                    atomicMax(&hb.bm[0], bbm);
                    atomicAdd(&hb.sbh[0], bsbh);
                    atomicAdd(&hb.sbl[0], bsbl);
                    atomicAdd(&hb.svh[0], bsvh);
                    atomicAdd(&hb.svl[0], bsvl);
                }
            }
            cluster.sync();
            {
                // Thread t merges field t / 256 of bin t % 256 over the cluster, in rank order;
                // the CL remote loads are independent and issue together.
                const int j = tid & 255, f = tid >> 8;
                if (f <= 1) {
                    const uint32_t local = (uint32_t)__cvta_generic_to_shared(f == 0 ? &hb.cnt[j] : &hb.bm[j]);
                    uint32_t v[CL];
#pragma unroll
                    for (int c2 = 0; c2 < CL; ++c2) v[c2] = ld_cluster_u32(map_cluster(local, c2));
                    uint32_t acc = v[0];
#pragma unroll
                    for (int c2 = 1; c2 < CL; ++c2) acc = f == 0 ? acc + v[c2] : max(acc, v[c2]);
                    if (f == 0) mh.cnt[j] = acc; else mh.bm[j] = acc;
                } else {
                    const uint32_t lh = (uint32_t)__cvta_generic_to_shared(f == 2 ? &hb.sbh[j] : &hb.svh[j]);
                    const uint32_t ll = (uint32_t)__cvta_generic_to_shared(f == 2 ? &hb.sbl[j] : &hb.svl[j]);
                    uint32_t hi[CL], lw[CL];
#pragma unroll
                    for (int c2 = 0; c2 < CL; ++c2) {
                        hi[c2] = ld_cluster_u32(map_cluster(lh, c2));
                        lw[c2] = ld_cluster_u32(map_cluster(ll, c2));
                    }
                    unsigned long long acc = 0ull;
#pragma unroll
                    for (int c2 = 0; c2 < CL; ++c2)
                        acc += ((unsigned long long)hi[c2] << FIX_SPLIT) + lw[c2];
                    if (f == 2) mh.sb[j] = acc; else mh.sv[j] = acc;
                }
            }
            __syncthreads();
            // Threads 0..255 scan the 256 bins: remaining(j) = below + bins < j (exact
            // integers); the cut bin is the last non-empty bin whose remaining set already
            // certifies.  Its thread then moves the select on.
            if (tid < SEL_NT) select_step(mh, ss, sx, tid, SB, SV, l, eps * D, D);
            __syncthreads();
            if (ss.done) break;
            // Few candidates left (one-wave grids, where the slowest head sets the launch time):
            // gather them into rank 0, rank them by key and take k* from exact suffix sums, with
            // the bits the histogram passes would reach.  Measured faster for clusters of 4 at
            // batch 1 (38.6 against 39.2 us) and slower for clusters of 2 at batch 8, where most
            // heads need one more pass at most; clusters of 2 and 8 keep the passes.
            if constexpr (CL == 1 || CL == 4) {
                if (a.sel_gather && ss.ncand <= SEL_GATHER) {
                    gather_select<CL>(cluster, crank, tid, ss, s_gn, gbuf,
                                      reinterpret_cast<int *>(&hist[(pass + 1) & 1]), W, R, X, chunk,
                                      base, beta, SB, SV, l, eps * D, D);
                    flags |= 8;
                    break;
                }
            }
        }
        // Peers may still be reading this CTA's last histogram: no CTA leaves before all have.
        cluster.sync();
        if (!ss.done) flags |= 2;  // the select ran out of passes
        kstar = ss.kstar;
        fthr = ss.fthr;
        eps_final = ss.eps_final;
    }

    // ---- 5. F bitmap and statistics ----
    uint32_t *Fq = a.F + (size_t)qh * a.W;
    for (int w = warp; w < chunk / 32; w += CT_NW) {
        const int i = 32 * w + lane;
        bool inF = false;
        if (!certified && R[i] < 1.0f) {
            inF = key64(X[i], base + i) >= fthr;
            if constexpr (SL) {
                const int t = base + i;
                inF = inF && t < a.n && ((a.shortlist[(size_t)ul * a.W + (t >> 5)] >> (t & 31)) & 1u);
            }
        }
        const uint32_t word = __ballot_sync(0xFFFFFFFFu, inF);
        const int gw = base / 32 + w;
        if (lane == 0 && gw < a.W) Fq[gw] = word;
    }
    // The refine's non-empty-range mask of this KV head starts empty.
    if (a.rmask && crank == 0 && qh == ul * G && tid < RMASK_W) a.rmask[ul * RMASK_W + tid] = 0u;
    // So does the refine's item counter (the refine of the previous call ended before this call's
    // scoring kernel, a plain launch, began).
    if (a.refine_next && blockIdx.x == 0 && tid == 0) *a.refine_next = 0;
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
        st.flags = flags | (exhausted ? 4 : 0);
        a.qstats[qh] = st;
        if (flags & 3) raise_error(a.err, ERR_NOCONVERGE);  // 8 only records the gathered finish
    }
    if (a.fl_counter) fetch_list_tail<CL>(a, ul, ug);
}

template <int CL, bool SL>
static cudaError_t launch_certify_cl(const CertifyArgs &a, int qheads, size_t smem, cudaStream_t s) {
    const cudaError_t e = ensure_smem((const void *)k_certify<CL, SL>, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(qheads * a.cl);
    cfg.blockDim = dim3(CT_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // When the grid fits the GPU in one wave it may be scheduled while the scoring kernel
    // finishes: it first loads r (written by a call that completed before the scoring kernel, a
    // plain launch, began) and waits for the scoring kernel before it reads the logits.  A grid
    // of several waves is launched in plain stream order (an early start showed no gain there).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.attrs = attr;
    cfg.numAttrs = (int)cfg.gridDim.x <= sms ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k_certify<CL, SL>, a);
}

cudaError_t launch_certify(const CertifyArgs &a, int qheads, size_t smem, cudaStream_t s) {
    const bool sl = a.shortlist != nullptr;
    switch (a.cl) {
        case 1: return sl ? launch_certify_cl<1, true>(a, qheads, smem, s)
                          : launch_certify_cl<1, false>(a, qheads, smem, s);
        case 2: return sl ? launch_certify_cl<2, true>(a, qheads, smem, s)
                          : launch_certify_cl<2, false>(a, qheads, smem, s);
        case 4: return sl ? launch_certify_cl<4, true>(a, qheads, smem, s)
                          : launch_certify_cl<4, false>(a, qheads, smem, s);
        case CT_MAX_CL: return sl ? launch_certify_cl<CT_MAX_CL, true>(a, qheads, smem, s)
                                  : launch_certify_cl<CT_MAX_CL, false>(a, qheads, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------------------------
// k_shortlist: one CTA per KV head.  A token of L gets the order-preserving 32-bit image of its
// largest sketch logit over the G query heads (0 for tokens outside L; kept in shared memory
// between passes when the unit's keys fit, recomputed otherwise); a most-significant-digit
// radix select (12, 12 and 8 bits, each pass a 4096-bin shared histogram over the tokens that
// still match the prefix) finds the size-th largest value T and how many tokens equal to T are
// still needed; a last pass in token order keeps every token above T and the lowest ids equal to
// T, writing the bitmap one warp word at a time.
constexpr int SL_NT = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <bool CACHED>
__global__ void __launch_bounds__(SL_NT, 1) k_shortlist(ShortlistArgs a) {
    extern __shared__ uint32_t s_ord[];  // CACHED: the order key of every token of the unit
    __shared__ uint32_t hist[4096];
    __shared__ uint32_t s_prefix, s_need, s_eq, s_nl;
    pdl_wait();  // the logits come from the kernel before this one
    pdl_trigger();
    __shared__ int s_wcnt[SL_NT / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ul = blockIdx.x;
    const int ug = a.li.unit_global(ul);
    const int G = a.li.G, n = a.n;
    const float *rf = a.r_full + (size_t)ug * n;
    const float *sc = a.scores + (size_t)ul * G * n;
    auto ord_load = [&](int t) -> uint32_t {
        if (!(rf[t] < 1.0f)) return 0u;
        float m = sc[t];
        for (int g = 1; g < G; ++g) m = fmaxf(m, sc[(size_t)g * n + t]);
        return order_key(m);
    };
    if constexpr (CACHED) {
#pragma unroll 8
        for (int t = tid; t < n; t += SL_NT) s_ord[t] = ord_load(t);
    }
    auto ord = [&](int t) -> uint32_t {
        if constexpr (CACHED) return s_ord[t];
        else return ord_load(t);
    };
    if (tid == 0) {
        s_prefix = 0u;
        s_need = (uint32_t)a.size;
        s_nl = 0u;
    }
    // |L|: when it does not exceed the size, the whole of L is the shortlist
    uint32_t cl = 0u;
    for (int t = tid; t < n; t += SL_NT) cl += ord(t) != 0u ? 1u : 0u;
    cl = warp_sum(cl);
    __syncthreads();
    if (lane == 0) atomicAdd(&s_nl, cl);
    __syncthreads();
    const bool all_of_L = s_nl <= (uint32_t)a.size;
    uint32_t T = 0u, need = 0u, eq = 0u;
    if (!all_of_L) {
        const int shifts[3] = {20, 8, 0}, widths[3] = {12, 12, 8};
        uint32_t mask = 0u;
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = shifts[pass], nb = 1 << widths[pass];
            for (int j = tid; j < 4096; j += SL_NT) hist[j] = 0u;
            __syncthreads();
            const uint32_t prefix = s_prefix;
#pragma unroll 4
            for (int t = tid; t < n; t += SL_NT) {
                const uint32_t o = ord(t);
                if (o != 0u && (o & mask) == prefix) atomicAdd(&hist[(o >> sh) & (uint32_t)(nb - 1)], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // bins from the top: lane j takes bins [nb - (j+1) * per, nb - j * per)
                const int per = nb / 32;
                uint32_t tot = 0u;
                for (int q = 0; q < per; ++q) tot += hist[nb - 1 - (lane * per + q)];
                uint32_t incl = tot;  // inclusive prefix over lanes (lane 0 = the highest bins)
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t excl = incl - tot, nd = s_need;
                if (excl < nd && nd <= incl) {  // the cut is in this lane's bins
                    uint32_t acc = excl;
                    for (int q = 0; q < per; ++q) {
                        const int bin = nb - 1 - (lane * per + q);
                        const uint32_t hb = hist[bin];
                        if (acc + hb >= nd) {
                            s_need = nd - acc;
                            s_prefix = prefix | ((uint32_t)bin << sh);
                            s_eq = hb;
                            break;
                        }
                        acc += hb;
                    }
                }
            }
            __syncthreads();
            mask |= (uint32_t)(nb - 1) << sh;
        }
        T = s_prefix;
        need = s_need;
        eq = s_eq;  // tokens equal to T
    }
    // Keep: every token above T, and the `need` lowest ids among those equal to T.
    uint32_t *out = a.out + (size_t)ul * a.W;
    uint32_t taken_eq = 0u;
    for (int c0 = 0; c0 < n; c0 += SL_NT) {
        const int t = c0 + tid;
        bool keep = false, tie = false;
        if (t < n) {
            if (all_of_L) {
                keep = ord(t) != 0u;
            } else {
                const uint32_t o = ord(t);
                keep = o > T;
                tie = o == T;
            }
        }
        if (!all_of_L && eq > need) {  // rank the ties in token order
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, tie);
            if (lane == 0) s_wcnt[warp] = __popc(bal);
            __syncthreads();
            uint32_t before = taken_eq;
            for (int w2 = 0; w2 < warp; ++w2) before += (uint32_t)s_wcnt[w2];
            before += __popc(bal & ((1u << lane) - 1u));
            keep = keep || (tie && before < need);
            uint32_t chunk_ties = 0u;
            for (int w2 = 0; w2 < SL_NT / 32; ++w2) chunk_ties += (uint32_t)s_wcnt[w2];
            taken_eq += chunk_ties;
            __syncthreads();
        } else {
            keep = keep || tie;
        }
        const uint32_t word = __ballot_sync(0xFFFFFFFFu, keep);
        const int wi = (c0 >> 5) + warp;
        if (lane == 0 && wi < a.W) out[wi] = word;
    }
}

cudaError_t launch_shortlist(const ShortlistArgs &a, int units_layer, cudaStream_t s) {
    if (a.size < 1 || a.size > SHORTLIST_MAX) return cudaErrorInvalidValue;
    // The keys of up to 40960 tokens stay in shared memory between the passes.
    const size_t smem = (size_t)a.n * 4;
    if (smem <= 160 * 1024) {
        const cudaError_t e = ensure_smem((const void *)k_shortlist<true>, 160 * 1024);
        if (e != cudaSuccess) return e;
        return launch_pdl(k_shortlist<true>, dim3(units_layer), dim3(SL_NT), smem, s, a);
    }
    return launch_pdl(k_shortlist<false>, dim3(units_layer), dim3(SL_NT), 0, s, a);
}

}  // namespace verkv
