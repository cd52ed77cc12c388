/*
 * verkv_oracle.c -- plain, slow fp64 CPU oracle for VerKV's decode-time hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load this file.  The CUDA library never links, loads or calls it, and the two share no
 * source, header, table, constant generator or helper.  Inputs reach both sides from the seeded
 * generators in verified_kv_cache_poissoncomp_gb300/inputs.py, which hold none of the method.
 *
 * What it restates: "Verify Before You Fetch: Reliable KV Cache Compression for LLM Inference"
 * (arXiv abstract page, and the Markdown summary page of the same title).  Section, equation,
 * definition, lemma and theorem names below are those of the summary page.
 *
 * Precision: fp64 everywhere, except where a float32 value is itself part of the definition of a
 * decision: r_i is published as float32 and the Bernoulli draw compares a 24-bit uniform against
 * it (vo_poissoncomp), and the 2-bit sketch's float32 / binary16 quantiser (vo_q2_build) whose
 * codes are part of the sketch's definition.  Every loop is serial; the only library primitives
 * are qsort, exp, log, sqrt, floor, ceil, frexp, ldexp and rintf.
 *
 * Parity status: every exported function is pinned by tests/test_oracle_*.py against closed
 * forms, brute force, an independent Philox (Triton's, run by its CPU interpreter), high-precision
 * recomputation (mpmath) or Monte-Carlo statistics.  None is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { VO_OK = 0, VO_EINVAL = 1, VO_EBUDGET = 2, VO_ENOMEM = 3 };

/* ------------------------------------------------------------------------------------------- */
/* Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3" (SC'11).  The pages only ask for independent Bernoulli draws
 * (summary page, Methodology, PoissonComp, the sample S); which generator produces them is our
 * reading, chosen so a draw depends only on (seed, token) and so is reproducible bit for bit.
 * One round multiplies counter words 0 and 2 by the two Philox multipliers, swaps the 32-bit
 * halves into a new counter and xors in the round key; the key advances by the two Weyl
 * constants between rounds. */
static void philox_round(uint32_t c[4], const uint32_t k[2])
{
    const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k[0];
    const uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

void vo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int round = 0; round < 10; ++round) {
        philox_round(c, k);
        k[0] += 0x9E3779B9u;
        k[1] += 0xBB67AE85u;
    }
    memcpy(out, c, sizeof c);
}

/* The uniform u_i in [0, 1) behind token i's draw in head (seq, layer, head): counter
 * (floor(i/4), head, layer, seq), key (seed low word, seed high word), output word i mod 4,
 * top 24 bits scaled by 2^-24 (exact in float32 and fp64). */
double vo_uniform24(uint64_t seed, uint32_t seq, uint32_t layer, uint32_t head, uint64_t i)
{
    const uint32_t ctr[4] = {(uint32_t)(i >> 2), head, layer, seq};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    vo_philox4x32_10(ctr, key, out);
    return (double)(out[i & 3u] >> 8) * 0x1p-24;
}

/* ------------------------------------------------------------------------------------------- */
/* PoissonComp (summary page, Methodology, "POISSONCOMP: Stochastic KV Cache Compression",
 * Eq. (3) and the H / L partition and Poisson sample that follow it).
 *
 *   r_i = min{1, c tau_i}, c chosen so that sum_i min(1, c tau_i) = eta n.
 *   H = tokens kept with probability 1, including the sink and local tokens;  L = 0 < r_i < 1.
 *   S = { i in L : Z_i = 1 },  Z_i ~ Bernoulli(r_i) independent.
 *
 * Readings (the pages are silent): the first n_sink and the last n_local tokens are forced into
 * H with r_i = 1 and count 1 each in the budget sum; tau of those tokens is ignored; every other
 * tau must be finite and in (0, 1] (tau = 0 would give r_i = 0, a token in neither H nor L);
 * eta n must exceed the forced count whenever other tokens exist.
 *
 * c is the exact root of the piecewise-linear budget equation, found by sorting tau descending
 * and trying s = 0, 1, ... saturated tokens: c_s = (B_rest - s) / (sum of the unsaturated tau),
 * accepted when c_s saturates exactly the top s.  r_i is then published as the float32 product
 * fminf(1, float(c) * tau_i) -- the precision in which both this oracle and the CUDA library take
 * the sampling decision -- and Z_i = [u_i < r_i] with u_i from vo_uniform24.  A token with
 * published r_i = 1 is in H.
 *
 * Outputs: c_exact (fp64 root, +inf when every token is kept), c32 = float(c_exact), r32[n],
 * resident[n] (1 for H and S), count = |H| + |S|.  Returns VO_OK, VO_EINVAL or VO_EBUDGET. */
static int cmp_double_desc(const void *a, const void *b)
{
    const double x = *(const double *)a, y = *(const double *)b;
    return (x < y) - (x > y);
}

int vo_poissoncomp(const float *tau, int64_t n, double eta, int64_t n_sink, int64_t n_local,
                   uint64_t seed, uint32_t seq, uint32_t layer, uint32_t head,
                   double *c_exact, float *c32_out, float *r32, uint8_t *resident,
                   int64_t *count)
{
    if (n <= 0 || n_sink < 0 || n_local < 0 || !(eta > 0.0) || eta > 1.0)
        return VO_EINVAL;

    int64_t n_forced = 0;
    for (int64_t i = 0; i < n; ++i)
        n_forced += (i < n_sink || i >= n - n_local);
    const int64_t n_rest = n - n_forced;
    const double b_rest = eta * (double)n - (double)n_forced;

    for (int64_t i = 0; i < n; ++i) {
        if (i < n_sink || i >= n - n_local)
            continue;
        const float t = tau[i];
        if (!isfinite(t) || !(t > 0.0f) || t > 1.0f)
            return VO_EINVAL;
    }
    if (n_rest > 0 && !(b_rest > 0.0))
        return VO_EBUDGET;

    double c = INFINITY;
    if (n_rest > 0 && b_rest < (double)n_rest) {
        double *t = (double *)malloc(sizeof(double) * (size_t)n_rest);
        double *suffix = (double *)malloc(sizeof(double) * (size_t)(n_rest + 1));
        if (!t || !suffix) {
            free(t);
            free(suffix);
            return VO_ENOMEM;
        }
        int64_t m = 0;
        for (int64_t i = 0; i < n; ++i)
            if (!(i < n_sink || i >= n - n_local))
                t[m++] = (double)tau[i];
        qsort(t, (size_t)n_rest, sizeof(double), cmp_double_desc);
        suffix[n_rest] = 0.0;
        for (int64_t j = n_rest - 1; j >= 0; --j)
            suffix[j] = suffix[j + 1] + t[j];

        int found = 0;
        double best_c = 0.0, best_violation = INFINITY;
        for (int64_t s = 0; s < n_rest && (double)s < b_rest; ++s) {
            const double cs = (b_rest - (double)s) / suffix[s];
            const double top_unsat = cs * t[s];              /* must stay below 1 */
            const double last_sat = s > 0 ? cs * t[s - 1] : INFINITY; /* must reach 1 */
            if (last_sat >= 1.0 && top_unsat < 1.0) {
                c = cs;
                found = 1;
                break;
            }
            /* Rounding guard: if fp64 rounding rejects both neighbours of an exact piece
             * boundary, keep the candidate whose conditions are violated least. */
            double viol = 0.0;
            if (last_sat < 1.0)
                viol += 1.0 - last_sat;
            if (top_unsat >= 1.0)
                viol += top_unsat - 1.0;
            if (viol < best_violation) {
                best_violation = viol;
                best_c = cs;
            }
        }
        if (!found)
            c = best_c;
        free(t);
        free(suffix);
    }

    const float c32 = (float)c;
    int64_t cnt = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (i < n_sink || i >= n - n_local) {
            r32[i] = 1.0f;
        } else {
            const float prod = c32 * tau[i];
            r32[i] = prod < 1.0f ? prod : 1.0f;
        }
        const double u = vo_uniform24(seed, seq, layer, head, (uint64_t)i);
        resident[i] = (uint8_t)(u < (double)r32[i]);
        cnt += resident[i];
    }
    *c_exact = c;
    *c32_out = c32;
    *count = cnt;
    return VO_OK;
}

/* ------------------------------------------------------------------------------------------- */
/* Scaled dot-product logits s_i = q . k_i / sqrt(d) for n keys stored row-major [n][d].
 * The pages cite SDPA without printing it (summary page, Theoretical Foundation: the numerator
 * N and denominator D of the attention computation); we read the weights as the standard
 * w_i = exp(q . k_i / sqrt(d)) and N = sum_i w_i v_i, D = sum_i w_i. */
void vo_logits(const double *q, const double *keys, int64_t n, int d, double *s)
{
    const double scale = 1.0 / sqrt((double)d);
    for (int64_t i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += q[c] * keys[i * d + c];
        s[i] = acc * scale;
    }
}

/* Dense attention over all n tokens.  out = [m, D, N[0..d), o[0..d)] with
 * m = max_i s_i, w_i = exp(s_i - m), D = sum w_i, N = sum w_i v_i, o = N / D. */
void vo_dense(const double *s, const double *values, int64_t n, int d, double *out)
{
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (s[i] > m)
            m = s[i];
    double D = 0.0;
    double *N = out + 2;
    for (int c = 0; c < d; ++c)
        N[c] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double w = exp(s[i] - m);
        D += w;
        for (int c = 0; c < d; ++c)
            N[c] += w * values[i * d + c];
    }
    out[0] = m;
    out[1] = D;
    for (int c = 0; c < d; ++c)
        out[2 + d + c] = N[c] / D;
}

/* ------------------------------------------------------------------------------------------- */
/* The 2-bit token sketch (summary page, Error Bound Guarantee: the "2-bit sketch" compared with
 * the perfect one; abstract page: a token-level sketch of the full KV cache).  The pages give no
 * layout; ours, per token of a head with d channels, in groups of 32 channels:
 *   lo    = the largest IEEE binary16 value <= min of the group (clamped to +-65504),
 *   step  = the smallest binary16 value >= fl((max - lo) / 3) (float32 subtract and divide),
 *   code  = min(3, max(0, rint(fl(fl(x - lo) / step)))) (0 if step == 0; rint rounds half to even),
 *   k-hat = lo + code * step, exactly (the key the certificate scores).
 * Bytes of a row: d/4 bytes of codes (channel c in bits 2(c mod 4) of byte c/4), then per group
 * lo and step as little-endian binary16, zero-padded to a multiple of 16 bytes. */

/* The binary16 value next to a finite x in direction dir (< 0: largest <= x, > 0: smallest >= x),
 * with x first clamped to the finite binary16 range. */
double vo_f16_round(double x, int dir)
{
    const double maxf16 = 65504.0;
    if (x > maxf16) x = maxf16;
    if (x < -maxf16) x = -maxf16;
    const double a = fabs(x);
    double q; /* spacing of binary16 values at |x| */
    if (a < ldexp(1.0, -14)) {
        q = ldexp(1.0, -24);
    } else {
        int e;
        frexp(a, &e); /* a in [2^(e-1), 2^e) */
        q = ldexp(1.0, e - 1 - 10);
    }
    const double k = x / q; /* exact: q is a power of two */
    return (dir < 0 ? floor(k) : ceil(k)) * q;
}

/* Bits of a binary16 value v (exactly representable). */
uint16_t vo_f16_bits(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u; /* -0 keeps its sign */
    const double a = fabs(v);
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)(a / ldexp(1.0, -24)));
    int e;
    const double m = frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
    const uint16_t exp16 = (uint16_t)(e - 1 + 15);
    const uint16_t mant = (uint16_t)((2.0 * m - 1.0) * 1024.0);
    return (uint16_t)(sign | (uint16_t)(exp16 << 10) | mant);
}

/* Value of binary16 bits (finite). */
double vo_f16_value(uint16_t h)
{
    const double sign = (h & 0x8000u) ? -1.0 : 1.0;
    const int e = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    if (e == 0) return sign * ldexp((double)m, -24);
    return sign * ldexp(1024.0 + (double)m, e - 25);
}

int vo_q2_row_bytes(int d)
{
    const int raw = d / 4 + 4 * (d / 32);
    return (raw + 15) / 16 * 16;
}

/* Quantise n keys (float32 values of bf16 keys, row-major [n][d], d a multiple of 32) into rows
 * of vo_q2_row_bytes(d) bytes, and write the exact dequantised keys k-hat [n][d]. */
void vo_q2_build(const float *keys, int64_t n, int d, uint8_t *rows, double *khat)
{
    const int rb = vo_q2_row_bytes(d);
    for (int64_t i = 0; i < n; ++i) {
        uint8_t *row = rows + i * rb;
        memset(row, 0, (size_t)rb);
        for (int gr = 0; gr < d / 32; ++gr) {
            const float *x = keys + i * d + 32 * gr;
            float mn = x[0], mx = x[0];
            for (int c = 1; c < 32; ++c) {
                if (x[c] < mn) mn = x[c];
                if (x[c] > mx) mx = x[c];
            }
            const float lo = (float)vo_f16_round((double)mn, -1);
            const float span = mx - lo;         /* float32 */
            const float third = span / 3.0f;    /* float32 */
            const float step = (float)vo_f16_round((double)third, +1);
            for (int c = 0; c < 32; ++c) {
                int code = 0;
                if (step > 0.0f) {
                    const float t = (x[c] - lo) / step; /* float32 subtract, float32 divide */
                    const float rq = rintf(t);
                    code = rq < 0.0f ? 0 : (rq > 3.0f ? 3 : (int)rq);
                }
                const int ch = 32 * gr + c;
                row[ch / 4] |= (uint8_t)(code << (2 * (ch % 4)));
                khat[i * d + ch] = (double)lo + (double)code * (double)step;
            }
            const uint16_t lb = vo_f16_bits((double)lo), sb = vo_f16_bits((double)step);
            uint8_t *par = row + d / 4 + 4 * gr;
            par[0] = (uint8_t)(lb & 0xFF);
            par[1] = (uint8_t)(lb >> 8);
            par[2] = (uint8_t)(sb & 0xFF);
            par[3] = (uint8_t)(sb >> 8);
        }
    }
}

/* ------------------------------------------------------------------------------------------- */
/* Bounded shrinkage estimator (summary page, Definition 2, Eq. (5)):
 *   lambda_i = clip_[r_i, 1]( beta r_i / (w_i (1 - r_i)) ),  beta = sum_{i in L} w_i (1 - lambda_i).
 * beta is the fixed point of that pair.  Reading: a token with w_i = 0 has lambda_i = 1 (its
 * ratio is +inf before clipping). */
static double shrink_lambda(double beta, double w, double r)
{
    if (!(w > 0.0))
        return 1.0;
    const double x = beta * r / (w * (1.0 - r));
    return x < r ? r : (x > 1.0 ? 1.0 : x);
}

/* h(beta) = beta - sum_{i in L} w_i (1 - lambda_i(beta)); its root is the fixed point. */
static double fixed_point_gap(double beta, const double *w, const float *r32, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (!((double)r32[i] < 1.0))
            continue;
        const double r = (double)r32[i];
        acc += w[i] * (1.0 - shrink_lambda(beta, w[i], r));
    }
    return beta - acc;
}

static int cmp_double_asc(const void *a, const void *b)
{
    const double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

/* Exact root of h.  h(0) = -sum_L w(1-r) <= 0 <= h(sum_L w(1-r)); h is continuous, strictly
 * increasing and linear between the breakpoints w_i (1 - r_i) (lambda_i leaves r_i) and
 * w_i (1 - r_i) / r_i (lambda_i reaches 1).  Binary search over the sorted breakpoints finds the
 * piece holding the root.  On that piece every token is in a fixed state: at its floor
 * (lambda = r, contributes A += w (1 - r)), in the middle (contributes w - beta r / (1 - r), so
 * B += w and S += r / (1 - r)) or at 1 (contributes 0).  h = beta (1 + S) - A - B there, so the
 * root is (A + B) / (1 + S), a ratio of sums of positive terms (no cancellation). */
static int solve_beta(const double *w, const float *r32, int64_t n, double *beta_out)
{
    double upper = 0.0;
    int64_t nl = 0;
    for (int64_t i = 0; i < n; ++i)
        if ((double)r32[i] < 1.0) {
            upper += w[i] * (1.0 - (double)r32[i]);
            ++nl;
        }
    if (!(upper > 0.0)) {
        *beta_out = 0.0;
        return VO_OK;
    }
    double *bp = (double *)malloc(sizeof(double) * (size_t)(2 * nl + 2));
    if (!bp)
        return VO_ENOMEM;
    int64_t nb = 0;
    bp[nb++] = 0.0;
    bp[nb++] = upper;
    for (int64_t i = 0; i < n; ++i) {
        const double r = (double)r32[i];
        if (!(r < 1.0) || !(w[i] > 0.0))
            continue;
        const double lo = w[i] * (1.0 - r), hi = w[i] * (1.0 - r) / r;
        if (lo < upper)
            bp[nb++] = lo;
        if (hi < upper)
            bp[nb++] = hi;
    }
    qsort(bp, (size_t)nb, sizeof(double), cmp_double_asc);
    int64_t lo = 0, hi = nb - 1; /* h(bp[lo]) <= 0 <= h(bp[hi]) */
    while (hi - lo > 1) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (fixed_point_gap(bp[mid], w, r32, n) <= 0.0)
            lo = mid;
        else
            hi = mid;
    }
    const double probe = 0.5 * (bp[lo] + bp[hi]);
    double A = 0.0, B = 0.0, S = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double r = (double)r32[i];
        if (!(r < 1.0) || !(w[i] > 0.0))
            continue;
        const double floor_end = w[i] * (1.0 - r), cap_start = w[i] * (1.0 - r) / r;
        if (probe <= floor_end) {
            A += floor_end;
        } else if (probe < cap_start) {
            B += w[i];
            S += r / (1.0 - r);
        }
    }
    double beta = (A + B) / (1.0 + S);
    /* Keep the root inside the bracket found by the search (rounding guard). */
    if (beta < bp[lo])
        beta = bp[lo];
    if (beta > bp[hi])
        beta = bp[hi];
    free(bp);
    *beta_out = beta;
    return VO_OK;
}

/* Bernstein radius of Lemma 1 (summary page, Bernstein Certificate, Eq. (7)):
 *   b l/3 + sqrt((b l/3)^2 + 2 V l),  l = log(2/delta) (natural log; the page writes log). */
static double bernstein(double b, double V, double l)
{
    const double a = b * l / 3.0;
    return a + sqrt(a * a + 2.0 * V * l);
}

typedef struct {
    double g;
    int64_t id;
} vo_gkey;

/* Order of Eq. (10): g descending; equal g by token id ascending (our tie-break). */
static int cmp_gkey(const void *a, const void *b)
{
    const vo_gkey *x = (const vo_gkey *)a, *y = (const vo_gkey *)b;
    if (x->g > y->g)
        return -1;
    if (x->g < y->g)
        return 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* KVFetch for one query head (summary page, "KVFETCH: Verification and Adaptive Fetching",
 * steps 1-5, with Definition 2, Lemma 1 and Eqs. (5), (7), (9), (10)).
 *
 * Inputs: s_hat[n] = logits from the sketch (step 1: w-hat_i = exp(s_hat_i - m)), r32[n] and
 * resident[n] from PoissonComp, eps, delta.
 *
 * Readings: D in Eq. (7) is unknown at run time and is taken as sum_i w-hat_i over all tokens
 * (exact for an exact sketch); the certificate is on D alone and uses all of delta; lambda is
 * solved once on L and held fixed for every subset in Eqs. (9)-(10) (any lambda in [r, 1] fixed
 * before the draw keeps Lemma 1's bound); g is evaluated in the algebraically equal form
 *   g_i D = beta_i + Bern(b, V) - Bern(b_{-i}, V - v_i)
 * with the difference of square roots rationalised; ties in g go to the lower token id.
 *
 * Outputs:
 *   scal[8]  = m, D, beta(L), V(L), b(L), l_delta, eps_hat(L), eps_hat(L_g[k*:])
 *   ints[4]  = certified, k*, |L|, |F \ S|
 *   lambda[n] (1 outside L), g[n] (0 outside L), F[n] (1 for the k* fetched tokens of L),
 *   order[|L|] (token ids in Eq. (10) order; may be NULL),
 *   eps_k[|L|+1] (eps_hat(L_g[k:]) for every k; may be NULL).
 *
 * With a candidate mask cand (vo_certify_cand), only tokens of L with cand[i] may be fetched:
 * the order of Eq. (10) runs over L n cand and every other token of L stays in the remaining set;
 * order and eps_k then cover the candidates only, and if even all of them leave eps-hat >= eps,
 * k* is their number and *exhausted is set (the certificate is not met). */
static int certify_core(const double *s_hat, const float *r32, const uint8_t *resident, int64_t n,
                        double eps, double delta, double *scal, int64_t *ints, double *lambda,
                        double *g, uint8_t *F, int64_t *order, double *eps_k, const uint8_t *cand,
                        int64_t *exhausted)
{
    if (n <= 0 || !(delta > 0.0) || !(delta < 1.0) || !(eps > 0.0))
        return VO_EINVAL;

    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (s_hat[i] > m)
            m = s_hat[i];
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    double *bi = (double *)malloc(sizeof(double) * (size_t)n);
    double *vi = (double *)malloc(sizeof(double) * (size_t)n);
    double *ci = (double *)malloc(sizeof(double) * (size_t)n);
    vo_gkey *keys = (vo_gkey *)malloc(sizeof(vo_gkey) * (size_t)n);
    if (!w || !bi || !vi || !ci || !keys) {
        free(w); free(bi); free(vi); free(ci); free(keys);
        return VO_ENOMEM;
    }
    double D = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        w[i] = exp(s_hat[i] - m);
        D += w[i];
    }

    double beta = 0.0;
    int st = solve_beta(w, r32, n, &beta);
    if (st != VO_OK) {
        free(w); free(bi); free(vi); free(ci); free(keys);
        return st;
    }

    /* Per-token terms of Eq. (7) with lambda frozen at the solution on L. */
    double beta_L = 0.0, V_L = 0.0, b_L = 0.0, b_second = 0.0;
    int64_t argmax = -1, nl = 0;
    for (int64_t i = 0; i < n; ++i) {
        const double r = (double)r32[i];
        lambda[i] = 1.0;
        g[i] = 0.0;
        F[i] = 0;
        bi[i] = vi[i] = ci[i] = 0.0;
        if (!(r < 1.0))
            continue;
        ++nl;
        const double lam = shrink_lambda(beta, w[i], r);
        lambda[i] = lam;
        ci[i] = w[i] * (1.0 - lam);                                  /* bias term   */
        vi[i] = lam * lam * w[i] * w[i] * (1.0 - r) / r;            /* variance    */
        bi[i] = lam * w[i] / r * (r > 1.0 - r ? r : 1.0 - r);       /* range bound */
        beta_L += ci[i];
        V_L += vi[i];
        if (bi[i] > b_L || argmax < 0) {
            b_second = b_L;
            b_L = bi[i];
            argmax = i;
        } else if (bi[i] > b_second) {
            b_second = bi[i];
        }
    }
    const double l = log(2.0 / delta);
    const double eps_L = (beta_L + bernstein(b_L, V_L, l)) / D;
    const int certified = eps_L < eps;

    /* Eq. (9): g_i = eps_hat(L) - eps_hat(L \ {i}), in the rationalised form. */
    const double A = b_L * l / 3.0;
    const double R = sqrt(A * A + 2.0 * V_L * l);
    int b_tied = 0; /* another token shares the maximal b: removing one leaves b unchanged */
    for (int64_t i = 0; i < n; ++i)
        if ((double)r32[i] < 1.0 && i != argmax && bi[i] == b_L)
            b_tied = 1;
    int64_t k = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (!((double)r32[i] < 1.0))
            continue;
        double V_rest = V_L - vi[i];
        if (V_rest < 0.0)
            V_rest = 0.0;
        double gD;
        if (i != argmax || b_tied) {
            const double R_rest = sqrt(A * A + 2.0 * V_rest * l);
            const double den = R + R_rest;
            gD = ci[i] + (den > 0.0 ? 2.0 * vi[i] * l / den : 0.0);
        } else {
            const double A2 = b_second * l / 3.0;
            const double R2 = sqrt(A2 * A2 + 2.0 * V_rest * l);
            const double den = R + R2;
            gD = ci[i] + (A - A2) +
                 (den > 0.0 ? ((A - A2) * (A + A2) + 2.0 * vi[i] * l) / den : 0.0);
        }
        g[i] = gD / D;
        if (cand && !cand[i])
            continue;
        keys[k].g = g[i];
        keys[k].id = i;
        ++k;
    }
    const int64_t nc = k; /* tokens the order runs over: L, or L n cand */
    qsort(keys, (size_t)nc, sizeof(vo_gkey), cmp_gkey);
    /* Tokens of L outside the candidates always remain. */
    double base_beta = 0.0, base_var = 0.0, base_bmax = 0.0;
    if (cand)
        for (int64_t i = 0; i < n; ++i)
            if ((double)r32[i] < 1.0 && !cand[i]) {
                base_beta += ci[i];
                base_var += vi[i];
                if (bi[i] > base_bmax)
                    base_bmax = bi[i];
            }

    /* Eq. (10): eps_hat(L_g[k:]) from suffix sums along the order; nonincreasing in k and 0 at
     * k = |L|.  k* = 0 when certified, else the first k >= 1 below eps. */
    double s_beta = base_beta, s_var = base_var, s_bmax = base_bmax;
    double *ek = (double *)malloc(sizeof(double) * (size_t)(nc + 1));
    if (!ek) {
        free(w); free(bi); free(vi); free(ci); free(keys);
        return VO_ENOMEM;
    }
    ek[nc] = cand ? (s_beta + bernstein(s_bmax, s_var, l)) / D : 0.0;
    for (int64_t j = nc - 1; j >= 0; --j) {
        const int64_t i = keys[j].id;
        s_beta += ci[i];
        s_var += vi[i];
        if (bi[i] > s_bmax)
            s_bmax = bi[i];
        ek[j] = (s_beta + bernstein(s_bmax, s_var, l)) / D;
    }
    int64_t kstar = 0;
    int64_t exh = 0;
    if (!certified) {
        kstar = nc;
        for (int64_t j = 1; j <= nc; ++j)
            if (ek[j] < eps) {
                kstar = j;
                break;
            }
        exh = !(ek[kstar] < eps);
    }
    if (exhausted)
        *exhausted = exh;
    int64_t nfetch = 0;
    for (int64_t j = 0; j < kstar; ++j) {
        const int64_t i = keys[j].id;
        F[i] = 1;
        nfetch += !resident[i];
    }
    if (order)
        for (int64_t j = 0; j < nc; ++j)
            order[j] = keys[j].id;
    if (eps_k)
        for (int64_t j = 0; j <= nc; ++j)
            eps_k[j] = ek[j];

    scal[0] = m;
    scal[1] = D;
    scal[2] = beta_L;
    scal[3] = V_L;
    scal[4] = b_L;
    scal[5] = l;
    scal[6] = eps_L;
    scal[7] = certified ? eps_L : ek[kstar];
    ints[0] = certified;
    ints[1] = kstar;
    ints[2] = nl;
    ints[3] = nfetch;

    free(ek);
    free(w); free(bi); free(vi); free(ci); free(keys);
    return VO_OK;
}

int vo_certify(const double *s_hat, const float *r32, const uint8_t *resident, int64_t n,
               double eps, double delta, double *scal, int64_t *ints, double *lambda, double *g,
               uint8_t *F, int64_t *order, double *eps_k)
{
    return certify_core(s_hat, r32, resident, n, eps, delta, scal, ints, lambda, g, F, order,
                        eps_k, NULL, NULL);
}

int vo_certify_cand(const double *s_hat, const float *r32, const uint8_t *resident, int64_t n,
                    double eps, double delta, const uint8_t *cand, double *scal, int64_t *ints,
                    double *lambda, double *g, uint8_t *F, int64_t *order, double *eps_k,
                    int64_t *exhausted)
{
    return certify_core(s_hat, r32, resident, n, eps, delta, scal, ints, lambda, g, F, order,
                        eps_k, cand, exhausted);
}

/* ------------------------------------------------------------------------------------------- */
/* The returned estimator after fetching (summary page, KVFETCH step 5 and Theorem 2; abstract
 * page: fetched tokens refine the attention computation).  Eq. (5) restricted to L' = L_g[k*:]:
 *   D-hat = sum_{H} w_i + sum_{F} w_i + sum_{S \ F} (lambda_i / r_i) w_i,
 * N-hat likewise with w_i v_i (the numerator the pages verify alongside D), o = N-hat / D-hat,
 * lse = m + log D-hat, and M2 = sum_{S \ F} (lambda_i w_i / r_i)^2 (1 - r_i), whose expectation is
 * V(L') of Eq. (7).  s[n] are the logits from the resident or fetched keys (exact), m the shift
 * used by vo_certify, lambda[n] its frozen lambda.
 * out = [D-hat, M2, lse, N-hat[0..d), o[0..d)]. */
void vo_refine(const double *s, const double *values, const float *r32, const uint8_t *resident,
               const uint8_t *F, const double *lambda, double m, int64_t n, int d, double *out)
{
    double Dh = 0.0, M2 = 0.0;
    double *N = out + 3;
    for (int c = 0; c < d; ++c)
        N[c] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double r = (double)r32[i];
        double coef;
        if (!(r < 1.0) || F[i]) {
            coef = 1.0;                          /* H, or fetched: exact */
        } else if (resident[i]) {
            coef = lambda[i] / r;                /* sampled, not fetched */
        } else {
            continue;                            /* L \ (S u F): Z_i = 0 */
        }
        const double w = exp(s[i] - m);
        if (r < 1.0 && !F[i]) {
            const double t = coef * w;
            M2 += t * t * (1.0 - r);
        }
        Dh += coef * w;
        for (int c = 0; c < d; ++c)
            N[c] += coef * w * values[i * d + c];
    }
    out[0] = Dh;
    out[1] = M2;
    out[2] = m + log(Dh);
    for (int c = 0; c < d; ++c)
        out[3 + d + c] = N[c] / Dh;
}
