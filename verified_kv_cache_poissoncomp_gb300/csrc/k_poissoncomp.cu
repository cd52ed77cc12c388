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

struct PcSmem {
    float *tau;        // [chunk]: tau of non-forced tokens, 0 for forced tokens and padding
    uint32_t *bits;    // [chunk / 32]
    float *fslots;     // [2][PC_MAX_CL][PC_NW][2]
    double *dslots;    // [2][PC_MAX_CL][PC_NW][2]
    int *wcount;       // [PC_NW]
    int *cta_total;    // [PC_MAX_CL]
};

static size_t pc_smem_bytes(int chunk) {
    return (size_t)chunk * 4 + (size_t)(chunk / 32) * 4 + 2 * PC_MAX_CL * PC_NW * 2 * 4 +
           2 * PC_MAX_CL * PC_NW * 2 * 8 + PC_NW * 4 + PC_MAX_CL * 4 + 64;
}

// tau (in (0, 1]) as 64-bit fixed point with 46 fractional bits, from 32-bit arithmetic:
// the integer part of tau 2^14 and 32 bits of what remains (truncated below 2^-46).
__device__ __forceinline__ unsigned long long tau_fixed(float x) {
    const float y = x * 16384.0f;
    const float hi = truncf(y);
    return ((unsigned long long)__float2uint_rz(hi) << 32) |
           (unsigned long long)__float2uint_rz((y - hi) * 4294967296.0f);
}
constexpr double TAU_FIXED_UNIT = 1.0 / 70368744177664.0;  // 2^-46

__global__ void __launch_bounds__(PC_NT, 1) k_pc_solve(PcArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    PcSmem sm;
    sm.dslots = reinterpret_cast<double *>(smem_raw);
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

    // 1. Load tau of the non-forced tokens; validate it.
    float tsum = 0.0f, tmin = __int_as_float(0x7F800000);
    unsigned long long tfix = 0ull;  // exact sum of tau
    bool bad = false;
    for (int i = tid; i < a.chunk; i += PC_NT) {
        const int t = base + i;
        float x = 0.0f;
        if (t < n && !(t < a.n_sink || t >= n - a.n_local)) {
            x = tau[t];
            if (!(x > 0.0f && x <= 1.0f)) {  // also catches NaN
                bad = true;
                x = 1.0f;
            }
            tmin = fminf(tmin, x);
            tsum += x;
            tfix += tau_fixed(x);
        }
        sm.tau[i] = x;
    }
    if (bad) raise_error(a.err, ERR_TAU);
    {
        float v[2] = {tsum, 0.0f};
        red.run(v, OpSum());
        tsum = v[0];
        float m[2] = {-tmin, 0.0f};
        red.run(m, OpMax());
        tmin = -m[0];
        unsigned long long z = 0ull;
        red64.run_u64(tfix, z);
    }

    double c = __longlong_as_double(0x7FF0000000000000LL);  // +inf: every token kept
    bool solved = false;
    if (a.n_rest > 0 && a.b_rest < (double)a.n_rest) {
        // 2. Newton on the concave piecewise-linear F from below.  A token saturates at c when
        //    tau >= 1 / c, i.e. tau >= the float32 rounded up from 1 / c.
        auto eval_exact = [&](double cc, unsigned long long &sat, unsigned long long &tun) {
            const float thr = __double2float_ru(1.0 / cc);
            unsigned long long s = 0ull, T = 0ull;
            for (int i = tid; i < a.chunk; i += PC_NT) {
                const float x = sm.tau[i];
                if (x > 0.0f) {
                    if (x >= thr) s += 1ull; else T += tau_fixed(x);
                }
            }
            red64.run_u64(T, s);
            sat = s;
            tun = T;
        };
        const double tsum_exact = (double)tfix * TAU_FIXED_UNIT;
        c = a.b_rest / tsum_exact * (1.0 - 0x1p-40);  // F(c) <= c sum tau <= B
        unsigned long long s, T;
        eval_exact(c, s, T);
        for (int it = 0; it < 8 && T > 0ull; ++it) {
            const double cn = (a.b_rest - (double)s) / ((double)T * TAU_FIXED_UNIT);
            unsigned long long s2, T2;
            eval_exact(cn, s2, T2);
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

    // 4. r_i = min(1, c tau_i) as a float32 product (1 for forced H); the budget check in fp64.
    float *r_full = a.r_full + (size_t)u * n;
    unsigned long long rfix = 0ull, zero = 0ull;  // exact sum of the float32 r
    for (int i = tid; i < a.chunk; i += PC_NT) {
        const int t = base + i;
        if (t >= n) break;
        const float x = sm.tau[i];
        const float r = (x > 0.0f) ? fminf(1.0f, __fmul_rn(c32, x)) : 1.0f;
        r_full[t] = r;
        rfix += tau_fixed(r);
    }
    red64.run_u64(rfix, zero);
    const double rsum = (double)rfix * TAU_FIXED_UNIT;
    if (!(fabs(rsum - a.eta_n) < 1e-6 * (double)n) && tid == 0 && crank == 0)
        raise_error(a.err, ERR_BUDGET_SUM);

    // 5. Draws: lane j of a warp takes tokens 4j..4j+3 of a 128-token group (one Philox block),
    //    and shuffles turn the four keep bits of eight lanes into one bitmap word.
    const int wchunk = a.chunk / PC_NW;  // tokens per warp, a multiple of 32
    const int wbase = warp * wchunk;
    int wcnt = 0;
    for (int g0 = 0; g0 < wchunk; g0 += 128) {
        const int i0 = wbase + g0 + 4 * lane;  // CTA-local index of my first token
        const int t0 = base + i0;
        const uint4 blk = philox4x32_10(make_uint4((uint32_t)t0 >> 2, (uint32_t)h, (uint32_t)l,
                                                   (uint32_t)b), a.seed_lo, a.seed_hi);
        const uint32_t words[4] = {blk.x, blk.y, blk.z, blk.w};
        uint32_t nib = 0;
        if (g0 + 4 * lane < wchunk) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = t0 + k;
                if (t < n) {
                    const float x = sm.tau[i0 + k];
                    const float r = (x > 0.0f) ? fminf(1.0f, __fmul_rn(c32, x)) : 1.0f;
                    const float uu = (float)(words[k] >> 8) * 0x1p-24f;
                    nib |= (uu < r ? 1u : 0u) << k;
                }
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
    cudaError_t e = cudaFuncSetAttribute(k_pc_solve, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
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
// Row copies: one warp per 4d-byte row, 16-byte vectors.
__global__ void __launch_bounds__(256) k_pc_gather(const uint4 *kv_full, const int32_t *ids,
                                                   const int32_t *count, uint4 *pkv, int units,
                                                   int cap, int n, int row16) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t total = (int64_t)units * cap;
    for (int64_t item = gw; item < total; item += nw) {
        const int u = (int)(item / cap);
        const int slot = (int)(item - (int64_t)u * cap);
        if (slot >= count[u]) continue;
        const int id = ids[(size_t)u * cap + slot];
        const uint4 *src = kv_full + ((size_t)u * n + id) * row16;
        uint4 *dst = pkv + ((size_t)u * cap + slot) * row16;
        for (int v = lane; v < row16; v += 32) dst[v] = ldg_stream(src + v);
    }
}

cudaError_t launch_pc_gather(const uint16_t *kv_full, const int32_t *ids, const int32_t *count,
                             uint16_t *pkv, int units, int cap, int n, int d, cudaStream_t s) {
    const int row16 = d / 4;  // 2 * d bf16 = 4d bytes = d/4 16-byte vectors
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t warps = (int64_t)units * cap;
    int blocks = (int)((warps + 7) / 8);
    if (blocks > sms * 8) blocks = sms * 8;
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
