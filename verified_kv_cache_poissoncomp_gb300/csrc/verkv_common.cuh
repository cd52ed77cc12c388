// verkv_common.cuh -- device helpers shared by libverkv's kernels (sm_103a).
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "verkv_internal.h"

namespace verkv {

namespace cg = cooperative_groups;

__device__ __forceinline__ void raise_error(uint32_t *err, uint32_t bit) { atomicOr(err, bit); }

// Programmatic dependent launch.  A kernel started through launch_pdl may begin while the kernel
// before it on the stream is still running: pdl_wait() returns once that kernel has completed
// and its memory is visible, so every such kernel calls it before touching anything the stream
// produced.  pdl_trigger() lets the next kernel be scheduled early; it only waits in turn.
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Cluster start-up.  A CTA may touch a peer's shared memory only once the peer is known to be
// running: the CTAs of a cluster are co-scheduled, but nothing orders their start, and a
// distributed-shared-memory access to a CTA that has not begun (or has already exited) is a
// launch failure.  Every thread calls cluster_arrive_relaxed() first thing and
// cluster_wait_all() before its first access to another CTA's shared memory; the barrier's
// latency hides behind whatever the kernel loads in between.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_all() {
    __syncwarp();  // the .aligned form wants the whole warp converged
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// bf16 pairs packed in a 32-bit word: element 0 in the low half.
__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// Streaming 16-byte load that does not allocate in L1 (data read once per launch).
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------------------------
// Warp reductions (fixed butterfly order: deterministic).
template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Largest b with its token id (lower id wins a tie) and the second-largest b.
struct Top2 {
    float b1;
    int id1;
    float b2;
};
__device__ __forceinline__ Top2 top2_merge(Top2 x, Top2 y) {
    const bool x_wins = x.b1 > y.b1 || (x.b1 == y.b1 && x.id1 < y.id1);
    Top2 r;
    if (x_wins) {
        r.b1 = x.b1; r.id1 = x.id1; r.b2 = fmaxf(x.b2, y.b1);
    } else {
        r.b1 = y.b1; r.id1 = y.id1; r.b2 = fmaxf(y.b2, x.b1);
    }
    return r;
}
__device__ __forceinline__ Top2 warp_top2(Top2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Top2 p;
        p.b1 = __shfl_xor_sync(0xFFFFFFFFu, v.b1, o);
        p.id1 = __shfl_xor_sync(0xFFFFFFFFu, v.id1, o);
        p.b2 = __shfl_xor_sync(0xFFFFFFFFu, v.b2, o);
        // Order the operands by lane so every lane computes the same merge.
        v = (threadIdx.x & o) ? top2_merge(p, v) : top2_merge(v, p);
    }
    return v;
}

// ---------------------------------------------------------------------------------------------
// All-reduce over every thread of a thread-block cluster.  Each warp reduces with shuffles and
// stores its partial into slot [my rank][warp] of every CTA's shared buffer (distributed shared
// memory); one cluster barrier; then every warp reduces the CL*NW partials itself, in the same
// fixed order, so every thread of every CTA gets bitwise the same result.  Two buffers alternate
// between calls: a CTA can only overwrite a buffer after the next barrier, i.e. after every peer
// has finished reading it.
template <int NW, int K>
struct ClusterReducer {
    float *slots;  // [2][cl][NW][K] floats in shared memory
    int cl;
    int parity;

    __device__ __forceinline__ float *buf(int p) const { return slots + p * cl * NW * K; }

    template <typename Op>
    __device__ __forceinline__ void run(float (&v)[K], Op op) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int k = 0; k < K; ++k) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v[k] = op(v[k], __shfl_xor_sync(0xFFFFFFFFu, v[k], o));
            v[k] = __shfl_sync(0xFFFFFFFFu, v[k], 0);  // one value per warp, whatever op's symmetry
        }
        cg::cluster_group cluster = cg::this_cluster();
        const unsigned me = cluster.block_rank();
        float *b = buf(parity);
        if (lane < cl) {
            float *peer = cluster.map_shared_rank(b, lane);
#pragma unroll
            for (int k = 0; k < K; ++k) peer[(me * NW + warp) * K + k] = v[k];
        }
        cluster.sync();
        const int total = cl * NW;  // <= 8 * 32
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float acc = (lane < total) ? b[lane * K + k] : op.identity();
            for (int e = lane + 32; e < total; e += 32) acc = op(acc, b[e * K + k]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc = op(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
            v[k] = __shfl_sync(0xFFFFFFFFu, acc, 0);
        }
        parity ^= 1;
    }
};

struct OpSum {
    __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
    __device__ __forceinline__ float identity() const { return 0.0f; }
};
struct OpMax {
    __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
    __device__ __forceinline__ float identity() const { return -__int_as_float(0x7F800000); }
};

// Same pattern for fp64 sums and int counts (PoissonComp's exact finish and compaction).
template <int NW>
struct ClusterReducer64 {
    double *slots;  // [2][cl][NW][2]
    int cl;
    int parity;

    // Exact integer sums (a, b) over the cluster, on the same buffers and parity.
    __device__ __forceinline__ void run_u64(unsigned long long &a, unsigned long long &b) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
        }
        cg::cluster_group cluster = cg::this_cluster();
        const unsigned me = cluster.block_rank();
        unsigned long long *buf = reinterpret_cast<unsigned long long *>(slots + parity * cl * NW * 2);
        if (lane < cl) {
            unsigned long long *peer = cluster.map_shared_rank(buf, lane);
            peer[(me * NW + warp) * 2 + 0] = a;
            peer[(me * NW + warp) * 2 + 1] = b;
        }
        cluster.sync();
        const int total = cl * NW;
        unsigned long long sa = 0ull, sb = 0ull;
        for (int e = lane; e < total; e += 32) {
            sa += buf[e * 2 + 0];
            sb += buf[e * 2 + 1];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sa += __shfl_xor_sync(0xFFFFFFFFu, sa, o);
            sb += __shfl_xor_sync(0xFFFFFFFFu, sb, o);
        }
        a = sa;
        b = sb;
        parity ^= 1;
    }

    // Sums (a, b) over the cluster: a fp64 and b an integer count carried exactly in fp64.
    __device__ __forceinline__ void run(double &a, double &b) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
        }
        cg::cluster_group cluster = cg::this_cluster();
        const unsigned me = cluster.block_rank();
        double *buf = slots + parity * cl * NW * 2;
        if (lane < cl) {
            double *peer = cluster.map_shared_rank(buf, lane);
            peer[(me * NW + warp) * 2 + 0] = a;
            peer[(me * NW + warp) * 2 + 1] = b;
        }
        cluster.sync();
        const int total = cl * NW;
        double sa = 0.0, sb = 0.0;
        for (int e = lane; e < total; e += 32) {
            sa += buf[e * 2 + 0];
            sb += buf[e * 2 + 1];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sa += __shfl_xor_sync(0xFFFFFFFFu, sa, o);
            sb += __shfl_xor_sync(0xFFFFFFFFu, sb, o);
        }
        a = sa;
        b = sb;
        parity ^= 1;
    }
};

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32->64 multiplies
// with the round key xored in, the key advancing by two Weyl constants per round.
// TMA bulk copies into shared memory that complete on an mbarrier, and bounded waits on it: a
// wait gives up after TMA_WAIT_NS of %globaltimer and returns false (the caller latches
// ERR_TIMEOUT, waits again, bounded, for its own copies in flight and returns).
constexpr unsigned long long TMA_WAIT_NS = 1000000000ull;  // 1 s
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Wait for phase `parity` of the barrier; false if limit_ns (TMA_WAIT_NS) elapsed first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned long long limit_ns = TMA_WAIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

// The same wait, which also gives up as soon as *abort is set (by another thread that timed out).
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (*abort || globaltimer_ns() - t0 > TMA_WAIT_NS) return false;
    return true;
}

// Orders this thread's earlier generic-proxy accesses to shared memory before its later async-proxy
// ones (a bulk copy refilling a stage that was just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

}  // namespace verkv
