// k_poissoncomp.cu -- PoissonComp on the GPU ("Verify Before You Fetch", summary page,
// Methodology, POISSONCOMP: Eq. (3), the H / L partition and the Poisson sample S).
//
// One thread-block cluster per unit (sequence, layer, KV head); each CTA holds up to 32768
// importance scores in shared memory.  F(c) = sum_i min(1, c tau_i) is concave and piecewise
// linear, so the budget constant is found by Newton on it, climbing from c = B / sum tau (where
// F <= B): on the current piece F(c) = s + c T (s saturated tokens, T the unsaturated sum), the
// next c is (B - s) / T, until the saturated set stops changing (one to three passes on lognormal
// scores).  The sums are exact: T in 64-bit fixed point (2^-46 per unit of tau) from 32-bit
// arithmetic, s an integer count, and a token saturates when tau >= the float32 rounded up from
// 1 / c, so the float32 c every decision uses is the correctly rounded root.  A float32 bisection
// followed by the same finish is kept as the fallback if Newton has not settled in 8 passes.  Each token's Bernoulli draw is word i%4 of one Philox4x32-10 block per four
// tokens; warp shuffles assemble the keep bits into the resident bitmap and a cluster-wide scan
// compacts H u S in ascending token order into the pivotal buffer.
#include <cuda_fp16.h>
#include <math.h>

#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

constexpr int PC_NT = 1024;
constexpr int PC_NW = PC_NT / 32;
constexpr int PC_MAX_CL = 8;
constexpr int PC_LD = 4;  // four-token tau loads in flight per thread

struct PcSmem {
    float *tau;        // [chunk]: tau of non-forced tokens, 0 for forced tokens and padding
    uint32_t *bits;    // [chunk / 32]
    float *fslots;     // [2][PC_MAX_CL][PC_NW][2]
    double *dslots;    // [2][PC_MAX_CL][PC_NW][2]
    int *wcount;       // [PC_NW]
    int *cta_total;    // [PC_MAX_CL]
    double *bc_c;      // [1]: the current c, written by thread 0
    float *bc_thr;     // [1]: its float32 saturation threshold
};

static size_t pc_smem_bytes(int chunk) {
    return 16 + (size_t)chunk * 4 + (size_t)(chunk / 32) * 4 + 2 * PC_MAX_CL * PC_NW * 2 * 4 +
           2 * PC_MAX_CL * PC_NW * 2 * 8 + PC_NW * 4 + PC_MAX_CL * 4 + 64;
}

// tau (in [0, 1]) as 64-bit fixed point with 46 fractional bits, truncated: floor(tau 2^46).
// With tau = m 2^(e - 150) (m the significand with its implicit bit, e the biased exponent, at
// most 127 here), floor(tau 2^46) = (m 2^23) >> (127 - e): integer operations only.
__device__ __forceinline__ unsigned long long tau_fixed(float x) {
    const uint32_t bits = __float_as_uint(x);
    const uint32_t e = bits >> 23;
    const unsigned long long m =
        (unsigned long long)((bits & 0x7FFFFFu) | (e ? 0x800000u : 0u)) << 23;
    const uint32_t rs = 127u - e;
    return rs < 64u ? m >> rs : 0ull;
}
// r (in [0, 1]) in units of 2^-24, truncated: floor(r 2^24) = m >> (126 - e) below 1 (m the
// significand with its implicit bit, e the biased exponent), 2^24 at 1.  The budget check sums
// these: n 2^-24 of truncation is far inside its tolerance.
__device__ __forceinline__ uint32_t r_fixed24(float r) {
    const uint32_t bits = __float_as_uint(r);
    const uint32_t e = bits >> 23;
    const uint32_t m = (bits & 0x7FFFFFu) | (e ? 0x800000u : 0u);
    if (e >= 127u) return 1u << 24;
    const uint32_t rs = 126u - e;
    return rs < 32u ? m >> rs : 0u;
}
constexpr double R_FIXED_UNIT = 1.0 / 16777216.0;  // 2^-24
constexpr double TAU_FIXED_UNIT = 1.0 / 70368744177664.0;  // 2^-46

__global__ void __launch_bounds__(PC_NT, 1) k_pc_solve(PcArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    PcSmem sm;
    sm.bc_c = reinterpret_cast<double *>(smem_raw);
    sm.bc_thr = reinterpret_cast<float *>(smem_raw + 8);
    sm.dslots = reinterpret_cast<double *>(smem_raw + 16);
    sm.fslots = reinterpret_cast<float *>(sm.dslots + 2 * PC_MAX_CL * PC_NW * 2);
    sm.tau = sm.fslots + 2 * PC_MAX_CL * PC_NW * 2;
    sm.bits = reinterpret_cast<uint32_t *>(sm.tau + a.chunk);
    sm.wcount = reinterpret_cast<int *>(sm.bits + a.chunk / 32);
    sm.cta_total = sm.wcount + PC_NW;

    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = blockIdx.x / a.cl;
    const int h = u % a.kv_heads;
    const int l = (u / a.kv_heads) % a.layers;
    const int b = u / (a.kv_heads * a.layers);
    const int base = crank * a.chunk;
    const int n = a.n;
    const float *tau = a.tau + (size_t)u * n;

    ClusterReducer<PC_NW, 2> red{sm.fslots, a.cl, 0};
    ClusterReducer64<PC_NW> red64{sm.dslots, a.cl, 0};
    cluster_arrive_relaxed();  // waited on before the first exchange with the peers

    // 1. Load tau of the non-forced tokens; validate it.  Each thread keeps PC_LD four-token
    //    loads in flight (16-byte vectors when the tau rows are 16-byte aligned).
    unsigned long long tfix = 0ull;  // exact sum of tau
    bool bad = false;
    const bool vec = (reinterpret_cast<uintptr_t>(a.tau) & 15u) == 0 && (n & 3) == 0;
    const int nvec = a.chunk / 4;
    for (int v0 = 0; v0 < nvec; v0 += PC_NT * PC_LD) {
        float4 xs[PC_LD];
#pragma unroll
        for (int k = 0; k < PC_LD; ++k) {
            const int v = v0 + k * PC_NT + tid;
            const int t = base + 4 * v;
            float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (v < nvec && t < n) {
                if (vec) {
                    x = __ldg(reinterpret_cast<const float4 *>(tau + t));
                } else {
                    x.x = tau[t];
                    if (t + 1 < n) x.y = tau[t + 1];
                    if (t + 2 < n) x.z = tau[t + 2];
                    if (t + 3 < n) x.w = tau[t + 3];
                }
            }
            xs[k] = x;
        }
#pragma unroll
        for (int k = 0; k < PC_LD; ++k) {
            const int v = v0 + k * PC_NT + tid;
            if (v >= nvec) break;
            float e[4] = {xs[k].x, xs[k].y, xs[k].z, xs[k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = base + 4 * v + j;
                float x = 0.0f;
                if (t < n && !(t < a.n_sink || t >= n - a.n_local)) {
                    x = e[j];
                    if (!(x > 0.0f && x <= 1.0f)) {  // also catches NaN
                        bad = true;
                        x = 1.0f;
                    }
                    tfix += tau_fixed(x);
                }
                e[j] = x;
            }
            *reinterpret_cast<float4 *>(sm.tau + 4 * v) = make_float4(e[0], e[1], e[2], e[3]);
        }
    }
    if (bad) raise_error(a.err, ERR_TAU);
    cluster_wait_all();  // every CTA of the cluster is running: its shared memory may be written
    {
        unsigned long long z = 0ull;
        red64.run_u64(tfix, z);
    }

    double c = __longlong_as_double(0x7FF0000000000000LL);  // +inf: every token kept
    bool solved = false;
    if (a.n_rest > 0 && a.b_rest < (double)a.n_rest) {
        // 2. Newton on the concave piecewise-linear F from below.  A token saturates at c when
        //    tau >= 1 / c, i.e. tau >= the float32 rounded up from 1 / c.
        // The unsaturated sum is the total less the saturated tokens' sum (exact integers), so
        // a pass converts only the few saturated tau.
        // The unsaturated sum is the total less the saturated tokens' sum (exact integers), so
        // a pass converts only the few saturated tau, on a branch the other tokens skip.  thr is
        // positive, so padding and forced tokens (tau 0 here) never count.
        auto eval_exact = [&](float thr, unsigned long long &sat, unsigned long long &tun) {
            unsigned long long s = 0ull, Ts = 0ull;
            const float4 *t4 = reinterpret_cast<const float4 *>(sm.tau);
            for (int v = tid; v < a.chunk / 4; v += PC_NT) {
                const float4 q = t4[v];
                const uint32_t m = (q.x >= thr ? 1u : 0u) | (q.y >= thr ? 2u : 0u) |
                                   (q.z >= thr ? 4u : 0u) | (q.w >= thr ? 8u : 0u);
                if (m) {
                    s += (unsigned long long)__popc(m);
                    if (m & 1u) Ts += tau_fixed(q.x);
                    if (m & 2u) Ts += tau_fixed(q.y);
                    if (m & 4u) Ts += tau_fixed(q.z);
                    if (m & 8u) Ts += tau_fixed(q.w);
                }
            }
            red64.run_u64(Ts, s);
            sat = s;
            tun = tfix - Ts;
        };
        // The scalar fp64 steps (a divide per pass) run on thread 0 and reach the other threads
        // through shared memory: fp64 throughput is a few operations per clock per SM here, so a
        // divide on every thread would cost microseconds a pass.  The next write comes after the
        // next reduction's barrier, so one slot suffices.
        auto share = [&](double &cc) -> float {
            if (tid == 0) {
                *sm.bc_c = cc;
                *sm.bc_thr = fmaxf(__double2float_ru(1.0 / cc), __int_as_float(1));
            }
            __syncthreads();
            cc = *sm.bc_c;
            return *sm.bc_thr;
        };
        double cc = 0.0;
        if (tid == 0) cc = a.b_rest / ((double)tfix * TAU_FIXED_UNIT) * (1.0 - 0x1p-40);  // F(c) <= c sum tau <= B
        float thr = share(cc);
        c = cc;
        unsigned long long s, T;
        eval_exact(thr, s, T);
        for (int it = 0; it < 8 && T > 0ull; ++it) {
            double cn = 0.0;
            if (tid == 0) cn = (a.b_rest - (double)s) / ((double)T * TAU_FIXED_UNIT);
            thr = share(cn);
            unsigned long long s2, T2;
            eval_exact(thr, s2, T2);
            c = cn;
            if (s2 == s) {
                solved = true;
                break;
            }
            s = s2;
            T = T2;
        }
    }
    if (!solved && a.n_rest > 0 && a.b_rest < (double)a.n_rest) {
        const float B = (float)a.b_rest;
        // Fallback.  Bisection on float32 c: F(lo) <= B <= F(hi): at lo every tau is scaled below its
        //    unclipped sum; at hi = 2 / min tau every token saturates.
        float tsum = 0.0f, tmin = __int_as_float(0x7F800000);
        for (int i = tid; i < a.chunk; i += PC_NT) {
            const float x = sm.tau[i];
            if (x > 0.0f) {
                tmin = fminf(tmin, x);
                tsum += x;
            }
        }
        {
            float v[2] = {tsum, 0.0f};
            red.run(v, OpSum());
            tsum = v[0];
            float m[2] = {-tmin, 0.0f};
            red.run(m, OpMax());
            tmin = -m[0];
        }
        float lo = (float)(a.b_rest / (double)tsum) * 0.999f;
        float hi = 2.0f / tmin;
        for (int it = 0; it < 64; ++it) {
            if (hi - lo <= lo * 1e-4f) break;
            const float mid = (hi > 4.0f * lo) ? sqrtf(lo) * sqrtf(hi) : 0.5f * (lo + hi);
            float acc = 0.0f;
            for (int i = tid; i < a.chunk; i += PC_NT) acc += fminf(1.0f, mid * sm.tau[i]);
            float v[2] = {acc, 0.0f};
            red.run(v, OpSum());
            if (v[0] < B) lo = mid; else hi = mid;
        }
        // 3. Exact finish in fp64.  From any c, the line s(c) + c' T(c) lies above the budget
        //    function, so c' = (B - s) / T is at most the root and at least c when c is below it:
        //    the iteration climbs to the root and stops when the saturated set is stable.
        c = (double)lo * (1.0 - 1.0 / 1024.0);
        auto eval = [&](double cc, double &sat, double &unsat_sum) {
            double s = 0.0, T = 0.0;
            for (int i = tid; i < a.chunk; i += PC_NT) {
                const float x = sm.tau[i];
                if (x > 0.0f) {
                    if (cc * (double)x >= 1.0) s += 1.0; else T += (double)x;
                }
            }
            red64.run(T, s);
            sat = s;
            unsat_sum = T;
        };
        double s, T;
        eval(c, s, T);
        bool done = false;
        for (int it = 0; it < 64; ++it) {
            const double cn = (a.b_rest - s) / T;
            double s2, T2;
            eval(cn, s2, T2);
            c = cn;
            if (s2 == s) {
                done = true;
                break;
            }
            s = s2;
            T = T2;
        }
        if (!done && tid == 0 && crank == 0) raise_error(a.err, ERR_NOCONVERGE);
    }
    const float c32 = (float)c;

    // 4-5. r_i = min(1, c tau_i) as a float32 product (1 for forced H), written out and summed
    //    (in units of 2^-24) for the budget check, and the draws: lane j of a warp takes tokens 4j..4j+3 of a
    //    128-token group (one Philox block), and shuffles turn the four keep bits of eight lanes
    //    into one bitmap word.
    float *r_full = a.r_full + (size_t)u * n;
    const bool rvec = (reinterpret_cast<uintptr_t>(a.r_full) & 15u) == 0 && (n & 3) == 0;
    uint32_t rfix = 0u;  // sum of floor(r 2^24): chunk / 1024 <= 32 tokens a thread, below 2^30
    const int wchunk = a.chunk / PC_NW;  // tokens per warp, a multiple of 32
    const int wbase = warp * wchunk;
    int wcnt = 0;
    for (int g0 = 0; g0 < wchunk; g0 += 128) {
        const int i0 = wbase + g0 + 4 * lane;  // CTA-local index of my first token
        const int t0 = base + i0;
        const uint4 blk = philox4x32_10(make_uint4((uint32_t)t0 >> 2, (uint32_t)h, (uint32_t)l,
                                                   (uint32_t)(a.seq0 + b)), a.seed_lo, a.seed_hi);
        const uint32_t words[4] = {blk.x, blk.y, blk.z, blk.w};
        uint32_t nib = 0;
        if (g0 + 4 * lane < wchunk && t0 < n) {
            const float4 q = *reinterpret_cast<const float4 *>(sm.tau + i0);
            const float xs[4] = {q.x, q.y, q.z, q.w};
            float rr[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = t0 + k;
                const float x = xs[k];
                const float r = (x > 0.0f) ? fminf(1.0f, __fmul_rn(c32, x)) : 1.0f;
                rr[k] = r;
                if (t < n) {
                    rfix += r_fixed24(r);
                    const float uu = (float)(words[k] >> 8) * 0x1p-24f;
                    nib |= (uu < r ? 1u : 0u) << k;
                }
            }
            if (rvec) {
                *reinterpret_cast<float4 *>(r_full + t0) = make_float4(rr[0], rr[1], rr[2], rr[3]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (t0 + k < n) r_full[t0 + k] = rr[k];
            }
        }
        uint32_t val = nib << (4 * (lane & 7));
        val |= __shfl_xor_sync(0xFFFFFFFFu, val, 1);
        val |= __shfl_xor_sync(0xFFFFFFFFu, val, 2);
        val |= __shfl_xor_sync(0xFFFFFFFFu, val, 4);
        if ((lane & 7) == 0 && g0 + 32 * (lane >> 3) < wchunk) {
            sm.bits[(wbase + g0) / 32 + (lane >> 3)] = val;
            wcnt += __popc(val);
        }
    }
    wcnt = warp_sum(wcnt);
    if (lane == 0) sm.wcount[warp] = wcnt;
    __syncthreads();
    unsigned long long rtot = rfix, zero = 0ull;
    red64.run_u64(rtot, zero);
    if (tid == 0 && crank == 0) {
        const double rsum = (double)rtot * R_FIXED_UNIT;
        if (!(fabs(rsum - a.eta_n) < 1e-6 * (double)n)) raise_error(a.err, ERR_BUDGET_SUM);
    }

    // Cluster-wide exclusive scan of the per-CTA counts (distributed shared memory).
    if (tid == 0) {
        int tot = 0;
        for (int w = 0; w < PC_NW; ++w) tot += sm.wcount[w];
        for (int c2 = 0; c2 < a.cl; ++c2) {
            int *peer = cluster.map_shared_rank(sm.cta_total, c2);
            peer[crank] = tot;
        }
    }
    cluster.sync();
    int cta_off = 0, total = 0;
    for (int c2 = 0; c2 < a.cl; ++c2) {
        if (c2 < crank) cta_off += sm.cta_total[c2];
        total += sm.cta_total[c2];
    }
    int woff = cta_off;
    for (int w = 0; w < warp; ++w) woff += sm.wcount[w];

    // 6. Compaction in ascending id order; the resident bitmap.
    int32_t *ids = a.ids + (size_t)u * a.cap;
    float *pr = a.pr + (size_t)u * a.cap;
    for (int w0 = 0; w0 < wchunk / 32; w0 += 32) {
        const int wi = w0 + lane;
        uint32_t word = 0;
        if (wi < wchunk / 32) word = sm.bits[wbase / 32 + wi];
        const int cnt = __popc(word);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        int pos = woff + incl - cnt;
        const int gword = (base + wbase) / 32 + wi;
        if (wi < wchunk / 32 && gword * 32 < n) a.resident[(size_t)u * a.W + gword] = word;
        while (word) {
            const int bit = __ffs(word) - 1;
            word &= word - 1;
            const int i = wbase + 32 * wi + bit;
            if (pos < a.cap) {
                const float x = sm.tau[i];
                ids[pos] = base + i;
                pr[pos] = (x > 0.0f) ? fminf(1.0f, __fmul_rn(c32, x)) : 1.0f;
            }
            ++pos;
        }
        woff += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (tid == 0 && crank == 0) {
        a.count[u] = total < a.cap ? total : a.cap;
        a.c_out[u] = c32;
        if (total > a.cap) raise_error(a.err, ERR_CAPACITY);
    }
}

cudaError_t launch_pc_solve(const PcArgs &a, int units, cudaStream_t s) {
    const size_t smem = pc_smem_bytes(a.chunk);
    cudaError_t e = ensure_smem((const void *)k_pc_solve, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units * a.cl);
    cfg.blockDim = dim3(PC_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_pc_solve, a);
}

// ---------------------------------------------------------------------------------------------
// Row copies: a warp takes 32 consecutive pivotal slots of one unit, reads their ids at once (a
// lane each) and keeps PG_ROWS rows of 4d bytes in flight, in 16-byte vectors.
constexpr int PG_ROWS = 8;
__global__ void __launch_bounds__(256) k_pc_gather(const uint4 *kv_full, const int32_t *ids,
                                                   const int32_t *count, uint4 *pkv, int units,
                                                   int cap, int n, int row16) {
    const int lane = threadIdx.x & 31;
    const int groups = (cap + 31) / 32;  // 32-slot groups per unit
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t total = (int64_t)units * groups;
    for (int64_t item = gw; item < total; item += nw) {
        const int u = (int)(item / groups);
        const int s0 = (int)(item - (int64_t)u * groups) * 32;
        const int cnt = count[u];
        if (s0 >= cnt) continue;
        const int rows = cnt - s0 < 32 ? cnt - s0 : 32;
        const int my_id = lane < rows ? ids[(size_t)u * cap + s0 + lane] : 0;
        const uint4 *src = kv_full + (size_t)u * n * row16;
        uint4 *dst = pkv + ((size_t)u * cap + s0) * row16;
        for (int r0 = 0; r0 < rows; r0 += PG_ROWS) {
            int id[PG_ROWS];
#pragma unroll
            for (int k = 0; k < PG_ROWS; ++k) id[k] = __shfl_sync(0xFFFFFFFFu, my_id, (r0 + k) & 31);
            for (int v = lane; v < row16; v += 32) {
                uint4 buf[PG_ROWS];
#pragma unroll
                for (int k = 0; k < PG_ROWS; ++k)
                    if (r0 + k < rows) buf[k] = ldg_stream(src + (size_t)id[k] * row16 + v);
#pragma unroll
                for (int k = 0; k < PG_ROWS; ++k)
                    if (r0 + k < rows) dst[(size_t)(r0 + k) * row16 + v] = buf[k];
            }
        }
    }
}

cudaError_t launch_pc_gather(const uint16_t *kv_full, const int32_t *ids, const int32_t *count,
                             uint16_t *pkv, int units, int cap, int n, int d, cudaStream_t s) {
    const int row16 = d / 4;  // 2 * d bf16 = 4d bytes = d/4 16-byte vectors
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_pc_gather, 256, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t warps = (int64_t)units * ((cap + 31) / 32);
    int blocks = (int)((warps + 7) / 8);
    if (blocks > sms * per_sm) blocks = sms * per_sm;
    if (blocks < 1) blocks = 1;
    k_pc_gather<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4 *>(kv_full), ids, count,
                                       reinterpret_cast<uint4 *>(pkv), units, cap, n, row16);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_sketch_exact(const uint4 *kv_full, uint4 *sketch,
                                                      int64_t rows, int half16) {
    const int64_t total = rows * half16;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = v / half16;
        const int c = (int)(v - row * half16);
        sketch[v] = ldg_stream(kv_full + row * 2 * half16 + c);
    }
}

cudaError_t launch_sketch_exact(const uint16_t *kv_full, uint16_t *sketch, int64_t rows, int d,
                                cudaStream_t s) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int half16 = d / 8;
    int64_t blocks = (rows * half16 + 255) / 256;
    if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
    if (blocks < 1) blocks = 1;
    k_sketch_exact<<<(int)blocks, 256, 0, s>>>(reinterpret_cast<const uint4 *>(kv_full),
                                               reinterpret_cast<uint4 *>(sketch), rows, half16);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// The 2-bit sketch: one thread per (token, 32-channel group).  floor = the largest binary16 at or
// below the group minimum, step = the smallest binary16 at or above fl((max - floor) / 3) (both
// clamped to the finite binary16 range first), code = rint(fl(fl(x - floor) / step)) in 0..3.
// Row layout (q2_row_bytes(d) bytes): d/4 bytes of codes, channel c in bits 2(c mod 4) of byte
// c/4, then per group floor and step as binary16, then zero padding to 16 bytes.
__global__ void __launch_bounds__(256) k_sketch_q2(const uint16_t *kv_full, uint8_t *sketch,
                                                   int64_t rows, int d, int row_bytes) {
    const int ng = d / 32;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * ng) return;
    const int64_t i = t / ng;
    const int gr = (int)(t - i * ng);
    const uint4 *x4 = reinterpret_cast<const uint4 *>(kv_full + i * 2 * d + 32 * gr);  // K row
    float x[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        float f[8];
        unpack8(ldg_stream(x4 + v), f);
#pragma unroll
        for (int c = 0; c < 8; ++c) x[8 * v + c] = f[c];
    }
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int c = 1; c < 32; ++c) {
        mn = fminf(mn, x[c]);
        mx = fmaxf(mx, x[c]);
    }
    const __half lo_h = __float2half_rd(fminf(fmaxf(mn, -65504.0f), 65504.0f));
    const float lo = __half2float(lo_h);
    const float third = __fdiv_rn(__fsub_rn(mx, lo), 3.0f);
    const __half st_h = __float2half_ru(fminf(third, 65504.0f));
    const float st = __half2float(st_h);
    uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        int code = 0;
        if (st > 0.0f) {
            const float rq = rintf(__fdiv_rn(__fsub_rn(x[c], lo), st));
            code = rq < 0.0f ? 0 : (rq > 3.0f ? 3 : (int)rq);
        }
        if (c < 16) w0 |= (uint32_t)code << (2 * c);
        else w1 |= (uint32_t)code << (2 * (c - 16));
    }
    uint8_t *row = sketch + i * row_bytes;
    *reinterpret_cast<uint2 *>(row + 8 * gr) = make_uint2(w0, w1);
    *reinterpret_cast<uint32_t *>(row + d / 4 + 4 * gr) =
        (uint32_t)__half_as_ushort(lo_h) | ((uint32_t)__half_as_ushort(st_h) << 16);
    if (gr == 0)
        for (int b = d / 4 + 4 * ng; b < row_bytes; b += 4) *reinterpret_cast<uint32_t *>(row + b) = 0u;
}

int q2_row_bytes(int d) { return (d / 4 + 4 * (d / 32) + 15) / 16 * 16; }

cudaError_t launch_sketch_q2(const uint16_t *kv_full, uint8_t *sketch, int64_t rows, int d,
                             cudaStream_t s) {
    const int64_t threads = rows * (d / 32);
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    k_sketch_q2<<<(int)(blocks < 1 ? 1 : blocks), 256, 0, s>>>(kv_full, sketch, rows, d,
                                                              q2_row_bytes(d));
    return cudaGetLastError();
}

}  // namespace verkv
