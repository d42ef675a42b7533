// xattn.cuh -- pieces shared by the output-copy cross-attention kernel (Eq. 5)
// and the fused decode step: a warp-level "16 query rows x 16 keys" online-softmax
// step over K/V staged in shared memory with the TMA 128-byte swizzle.
#pragma once

#include "common.cuh"

namespace orthros {

// Per-warp flash state for 16 query rows (fragment rows gr and gr + 8 of this lane).
template <int D>
struct WarpRows16 {
    uint32_t qa[D / 16][4];  // bf16 query fragments (already scale-offset and scaled): high part
    uint32_t ql[D / 16][4];  // bf16 residual q - high part: QK runs twice, hi and lo, into one sum
    float o[D / 8][4];       // unnormalised output accumulator
    float mA, mB;            // running max (log2 domain) of rows gr, gr + 8
    float lA, lB;            // running sum (this lane's partial; quad-reduced at the end)

    __device__ __forceinline__ void reset()
    {
        const float NEG_INF = -__int_as_float(0x7f800000);
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        mA = mB = NEG_INF;
        lA = lB = 0.f;
    }

    // One 16-key chunk: keys j0 .. j0+15 whose K rows start at shared-memory row
    // `krow0` of a block staged as D/64 slabs of `slab_bytes` each (K at kbase,
    // V at vbase).  Key j is valid for row A iff j <= limA (likewise B); pass
    // full = true when every key of the chunk is valid for every row.
    __device__ __forceinline__ void step(uint32_t kbase, uint32_t vbase, int slab_bytes, int krow0,
                                         int j0, int limA, int limB, bool full)
    {
        const int lane = threadIdx.x & 31;
        const int qd = (lane & 3) * 2;
        const int kld_row = (lane & 7) + ((lane >> 4) << 3);
        const int kld_hi = (lane >> 3) & 1;
        const int vld_row = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int vld_hi = lane >> 4;
        const float NEG_INF = -__int_as_float(0x7f800000);
        float s[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + (kt * 16 / 64) * slab_bytes +
                        sw128_offset(krow0 + kld_row, ((kt * 16) % 64) / 8 + kld_hi),
                    b0, b1, b2, b3);
            mma_16816(s[0], qa[kt], b0, b1);
            mma_16816(s[1], qa[kt], b2, b3);
            mma_16816(s[0], ql[kt], b0, b1);
            mma_16816(s[1], ql[kt], b2, b3);
        }
        if (!full) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = j0 + i * 8 + qd + (e & 1);
                    if (j > ((e & 2) ? limB : limA))
                        s[i][e] = NEG_INF;
                }
        }
        float cmA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float cmB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        cmA = fmaxf(cmA, __shfl_xor_sync(0xffffffffu, cmA, 1));
        cmA = fmaxf(cmA, __shfl_xor_sync(0xffffffffu, cmA, 2));
        cmB = fmaxf(cmB, __shfl_xor_sync(0xffffffffu, cmB, 1));
        cmB = fmaxf(cmB, __shfl_xor_sync(0xffffffffu, cmB, 2));
        const float nmA = fmaxf(mA, cmA), nmB = fmaxf(mB, cmB);
        const float uA = (nmA == NEG_INF) ? 0.f : nmA;
        const float uB = (nmB == NEG_INF) ? 0.f : nmB;
        const float corrA = fast_exp2(mA - uA), corrB = fast_exp2(mB - uB);
        mA = nmA;
        mB = nmB;
        float pr[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            pr[i][0] = fast_exp2(s[i][0] - uA);
            pr[i][1] = fast_exp2(s[i][1] - uA);
            pr[i][2] = fast_exp2(s[i][2] - uB);
            pr[i][3] = fast_exp2(s[i][3] - uB);
        }
        lA = lA * corrA + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
        lB = lB * corrB + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
        if (corrA != 1.f || corrB != 1.f) {
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= corrA;
                o[i][1] *= corrA;
                o[i][2] *= corrB;
                o[i][3] *= corrB;
            }
        }
        uint32_t pa[4];
        pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(vbase + (dp * 16 / 64) * slab_bytes +
                              sw128_offset(krow0 + vld_row, ((dp * 16) % 64) / 8 + vld_hi),
                          v0, v1, v2, v3);
            mma_16816(o[2 * dp], pa, v0, v1);
            mma_16816(o[2 * dp + 1], pa, v2, v3);
        }
    }

    __device__ __forceinline__ void finish_sums()
    {
        lA += __shfl_xor_sync(0xffffffffu, lA, 1);
        lA += __shfl_xor_sync(0xffffffffu, lA, 2);
        lB += __shfl_xor_sync(0xffffffffu, lB, 1);
        lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    }
};

// Split a pair of fp32 query values into bf16 high parts and bf16 residuals, so
// that q . k = hi . k + lo . k keeps ~16 significant bits of the scaled query
// (one bf16 rounding of q alone is amplified by large keys).
__device__ __forceinline__ void split_q_pair(float a, float b, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16x2(a, b);
    const float2 h = unpack_bf16x2(hi);
    lo = pack_bf16x2(a - h.x, b - h.y);
}

// Load a query element pair from global bf16 memory, apply the stream's
// scale-offset q = (x * alpha + beta) * qscale, and split it into hi / lo bf16.
__device__ __forceinline__ void load_q_pair(const orthros_bf16 *row, const float *alpha, const float *beta,
                                            int dcol, float qscale, uint32_t &hi, uint32_t &lo)
{
    const uint32_t raw = __ldg(reinterpret_cast<const unsigned int *>(row + dcol));
    const float2 x = unpack_bf16x2(raw);
    const float2 al = __ldg(reinterpret_cast<const float2 *>(alpha + dcol));
    const float2 be = __ldg(reinterpret_cast<const float2 *>(beta + dcol));
    split_q_pair(fmaf(x.x, al.x, be.x) * qscale, fmaf(x.y, al.y, be.y) * qscale, hi, lo);
}

}  // namespace orthros
