// pivotal_mma.cuh -- the bounded shrinkage estimator over the pivotal set on the tensor cores
// ("Verify Before You Fetch", summary page, Definition 2 / Eq. (5): D-hat and N-hat over H u S
// with weight 1 on H and on tokens of F, lambda_i / r_i on sampled, unfetched tokens).
//
// A pivotal row is 4d bytes (K then V, bf16).  Rows are staged in shared memory PIV_STAGE_ROWS at a
// time, in boxes of 64 rows x 64 channels (128 bytes a row) -- K channels 0-63, (64-127,) then V
// the same -- with the 128-byte swizzle of the tensor-memory-access unit: the 16-byte chunk c of
// box row r sits at chunk c xor (r mod 8), so the eight rows of an 8x8 ldmatrix tile fall in eight
// different bank groups.  Per stage, consumer warp w takes rows 16w .. 16w + 15:
// After the chunk's stages, the four warps' O^T tiles and sums are added in warp order through
// shared memory into one partial [G][d + 2] (N-hat, D-hat, second moment).  Every path that sums
// pivotal rows (the pipelined MEMCPY-mode kernel, the zero-copy refine, the unaligned fallback)
// runs these functions in the same order, so all of them produce the same bits.
#pragma once

#include <cuda.h>

#include "verkv_common.cuh"
#include "verkv_internal.h"

namespace verkv {

// ---------------------------------------------------------------------------------------------
// Tensor copies.  One box into shared memory, completing on `bar` (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point (no link against the
// driver library); null where the driver does not provide it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                               cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
            encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return encode;
}

// ---------------------------------------------------------------------------------------------
// PTX wrappers.  Fragment layouts follow the PTX ISA for mma.m16n8k16 with .bf16 operands: with
// g = lane / 4 and t = lane % 4, A holds (row g | g + 8, columns 2t, 2t + 1 | + 8), B holds
// (rows 2t, 2t + 1 | + 8, column g) and the f32 accumulator (row g | g + 8, columns 2t, 2t + 1).
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// Transpose of an 8x8 b16 tile held in the ldmatrix fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// Two floats rounded to bf16 (nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t y;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(y) : "f"(hi), "f"(lo));
    return y;
}
__device__ __forceinline__ float bf16_lo_f(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// ---------------------------------------------------------------------------------------------
// Shared-memory stage: NB boxes of 64 rows x 128 bytes (swizzled), then the rows' token ids and r;
// stages are a multiple of 1024 bytes so that every box keeps the swizzle's 1024-byte alignment.
template <int D>
struct PivLayout {
    static constexpr int ROWB = 4 * D;        // a K|V row in global memory
    static constexpr int ROWS = PIV_STAGE_ROWS;
    static constexpr int HALVES = D / 64;     // 64-channel boxes per K (or V) row
    static constexpr int NB = 2 * HALVES;     // boxes per stage
    static constexpr int BOX = ROWS * 128;    // bytes per box
    static constexpr int IDS = NB * BOX;      // int32 [ROWS]
    static constexpr int RS = IDS + ROWS * 4; // float [ROWS]
    static constexpr int BYTES = (RS + ROWS * 4 + 1023) / 1024 * 1024;
    static_assert(ROWS == 64 && D % 64 == 0, "boxes of 64 rows x 64 channels");
    // Byte offset of channels c .. c + 7 (c a multiple of 8) of row r of part p (0 K, 1 V).
    __host__ __device__ static constexpr int off(int p, int r, int c) {
        return (p * HALVES + c / 64) * BOX + r * 128 + ((((c % 64) >> 3) ^ (r & 7)) << 4);
    }
};
// Zero row r of a stage (every box's 128-byte line of it), with the 32 lanes of a warp.
template <int D>
__device__ __forceinline__ void piv_zero_row(unsigned char *st, int r) {
    using LY = PivLayout<D>;
    const int lane = threadIdx.x & 31;
    if (lane < LY::NB * 8) {
        uint4 *line = reinterpret_cast<uint4 *>(st + (lane >> 3) * LY::BOX + r * 128);
        line[lane & 7] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Bytes of the chunk-end reduction: [4 warps][G][D] floats, then [4 warps][G][2].
template <int D, int G>
__host__ __device__ constexpr int piv_red_bytes() { return 4 * G * D * 4 + 4 * G * 2 * 4; }

// Per consumer warp, the state of one chunk (one partial) of one layer unit.
template <int D, int G, bool SKL>
struct PivChunk {
    static constexpr int KS = D / 16;  // k-steps of S = K Q^T, and m-tiles of O^T
    uint32_t qb[KS][2];                // B fragments of Q^T (query head g, channels 2t, 2t+1 | +8)
    float acc[KS][4];                  // O^T: tile mt holds channels 16 mt + g | + 8, heads 2t, 2t+1
    float dsum[2], m2[2];              // D-hat and second moment of heads 2t, 2t+1 (this lane's rows)
    float mh[2], bh[2];                // shift m and beta of heads 2t, 2t+1
    const uint32_t *Fh[2];             // selection bitmaps of heads 2t, 2t+1
    const float *sh[2];                // their sketch logits (2-bit sketch only)

    // The unit's query fragments and per-head values (a chunk of another unit needs them anew).
    __device__ __forceinline__ void load_unit(const PartialArgs &a, int ul) {
        const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
        const int b = ul / a.li.kv_heads, h = ul - b * a.li.kv_heads;
        const int hq = a.li.kv_heads * G;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.q + ((size_t)b * hq + h * G + (g < G ? g : 0)) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qb[ks][0] = g < G ? qrow[ks * 8 + t] : 0u;
            qb[ks][1] = g < G ? qrow[ks * 8 + 4 + t] : 0u;
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int hd = 2 * t + k;
            mh[k] = 0.0f;
            bh[k] = 0.0f;
            Fh[k] = a.F;
            sh[k] = a.scores;
            if (hd < G) {
                const int qh = ul * G + hd;
                mh[k] = a.qstats[qh].m;
                bh[k] = a.qstats[qh].beta;
                Fh[k] = a.F + (size_t)qh * a.W;
                if (SKL) sh[k] = a.scores + (size_t)qh * a.n;
            }
        }
    }
    // Zero sums for a new chunk.
    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            dsum[k] = 0.0f;
            m2[k] = 0.0f;
        }
    }
    __device__ __forceinline__ void init(const PartialArgs &a, int ul) {
        load_unit(a, ul);
        reset();
    }

    // One stage of `rows` (<= PIV_STAGE_ROWS) rows at `st` (shared memory), this warp's 16 rows.
    // Rows at or beyond `rows` must hold finite values (the callers keep zeros there).
    __device__ __forceinline__ void stage(const PartialArgs &a, const unsigned char *st, int rows) {
        using LY = PivLayout<D>;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
        const int row0 = warp * 16;
        const int32_t *s_id = reinterpret_cast<const int32_t *>(st + LY::IDS);
        const float *s_r = reinterpret_cast<const float *>(st + LY::RS);
        // The lane's rows and what they need from global memory, loaded first.
        int id[2];
        float rr[2];
        bool ok[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = row0 + g + 8 * k;
            ok[k] = r < rows;
            id[k] = ok[k] ? s_id[r] : 0;
            rr[k] = ok[k] ? s_r[r] : 1.0f;
            if ((unsigned)id[k] >= (unsigned)a.n) {  // not a token of the unit: skip the row
                if (ok[k]) raise_error(a.err, ERR_BADID);
                ok[k] = false;
                id[k] = 0;
                rr[k] = 1.0f;
            }
        }
        uint32_t fw[4];
        float shat[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = e >> 1, hk = e & 1;
            fw[e] = 0u;
            shat[e] = 0.0f;
            if (ok[k] && rr[k] < 1.0f && 2 * t + hk < G) {
                fw[e] = __ldcg(Fh[hk] + (id[k] >> 5));
                if (SKL) shat[e] = __ldcg(sh[hk] + id[k]);
            }
        }
        // 1. S = K Q^T for the warp's 16 rows (even and odd k-steps in two accumulators).
        const uint32_t base = smem_addr(st);
        float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        {
            float c1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: tile mi, row ri of it
            const int ar = row0 + (mi & 1) * 8 + ri;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t af[4];
                ldsm_x4(af, base + (uint32_t)LY::off(0, ar, ks * 16 + (mi >> 1) * 8));
                mma_bf16((ks & 1) ? c1 : c, af, qb[ks][0], qb[ks][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) c[e] += c1[e];
        }
        // 2. The weight of each (row, head) element: c[e] is row g + 8 (e >> 1), head 2t + (e & 1).
        //    For a sampled, unfetched token the weight is (lambda / r) w with
        //    lambda / r = clip(beta / (w-hat (1 - r)), 1, 1 / r); with the exact sketch (w-hat = w)
        //    that is min(w / r, max(w, beta / (1 - r))), so 1 / r and 1 / (1 - r) are taken once
        //    per row and no element divides.  1 / r when w-hat underflows (lambda = 1).
        const float scale = a.scale;
        float ir[2], i1r[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            ir[k] = __fdividef(1.0f, rr[k]);
            i1r[k] = __fdividef(1.0f, 1.0f - rr[k]);
        }
        float cw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = e >> 1, hk = e & 1;
            cw[e] = 0.0f;
            if (ok[k] && 2 * t + hk < G) {
                const float w = __expf(fmaf(c[e], scale, -mh[hk]));
                const float r = rr[k];
                const bool inF = (fw[e] >> (id[k] & 31)) & 1u;
                float v = w;
                if (r < 1.0f && !inF) {
                    const float lo = bh[hk] * i1r[k];  // beta / (1 - r)
                    if (SKL) {
                        const float wh = __expf(shat[e] - mh[hk]);
                        v = wh > 0.0f ? w * fminf(ir[k], fmaxf(1.0f, __fdividef(lo, wh))) : w * ir[k];
                    } else {
                        v = w > 0.0f ? fminf(w * ir[k], fmaxf(w, lo)) : 0.0f;
                    }
                    m2[hk] = fmaf(v * v, 1.0f - r, m2[hk]);
                }
                cw[e] = v;
                dsum[hk] += v;
            }
        }
        // 3. P^T as the B operand, hi and lo parts; O^T += V^T P^T.
        const uint32_t h01 = pack_bf16x2(cw[0], cw[1]), h23 = pack_bf16x2(cw[2], cw[3]);
        const uint32_t l01 = pack_bf16x2(cw[0] - bf16_lo_f(h01), cw[1] - bf16_hi_f(h01));
        const uint32_t l23 = pack_bf16x2(cw[2] - bf16_lo_f(h23), cw[3] - bf16_hi_f(h23));
        const uint32_t bh0 = movmatrix_t(h01), bh1 = movmatrix_t(h23);
        const uint32_t bl0 = movmatrix_t(l01), bl1 = movmatrix_t(l23);
        {
            // ldmatrix.trans: tile mi covers rows 8 (mi >> 1) .. + 7 and channels 8 (mi & 1) .. + 7
            const int mi = lane >> 3, ri = lane & 7;
            const int vr = row0 + (mi >> 1) * 8 + ri;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t vf[4];
                ldsm_x4_t(vf, base + (uint32_t)LY::off(1, vr, mt * 16 + (mi & 1) * 8));
                mma_bf16(acc[mt], vf, bh0, bh1);
                mma_bf16(acc[mt], vf, bl0, bl1);
            }
        }
    }

    // Adds the four consumer warps' sums in warp order into the partial at `out` ([G][D + 2]).
    // `red` is shared memory of piv_red_bytes<D, G>() bytes; bar() synchronises the four warps.
    template <class Bar>
    __device__ __forceinline__ void finish(float *red, float *out, bool write, Bar bar) {
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                dsum[k] += __shfl_xor_sync(0xFFFFFFFFu, dsum[k], o);
                m2[k] += __shfl_xor_sync(0xFFFFFFFFu, m2[k], o);
            }
        }
        float *rn = red + (size_t)warp * G * D;
        float *rs = red + 4 * G * D + warp * G * 2;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int hd = 2 * t + k;
                if (hd < G) {
                    rn[hd * D + 16 * mt + g] = acc[mt][k];
                    rn[hd * D + 16 * mt + g + 8] = acc[mt][2 + k];
                }
            }
        }
        if (g == 0) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int hd = 2 * t + k;
                if (hd < G) {
                    rs[hd * 2] = dsum[k];
                    rs[hd * 2 + 1] = m2[k];
                }
            }
        }
        bar();
        if (write) {
            for (int e = tid; e < G * (D + 2); e += 128) {
                const int hd = e / (D + 2), cc = e - hd * (D + 2);
                float s;
                if (cc < D) {
                    s = red[hd * D + cc];
#pragma unroll
                    for (int w = 1; w < 4; ++w) s += red[(w * G + hd) * D + cc];
                } else {
                    const int f = cc - D;
                    const float *r2 = red + 4 * G * D;
                    s = r2[hd * 2 + f];
#pragma unroll
                    for (int w = 1; w < 4; ++w) s += r2[(w * G + hd) * 2 + f];
                }
                out[e] = s;
            }
        }
        bar();
    }
};

}  // namespace verkv
