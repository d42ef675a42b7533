// xattn.cuh -- pieces shared by the output-copy cross-attention kernel (Eq. 5)
// and the fused decode step: a warp-level "16 query rows x 16 keys" online-softmax
// step over K/V staged in shared memory with the TMA 128-byte swizzle.
#pragma once

#include "common.cuh"

namespace orthros {

// Per-warp flash state for 16 query rows (fragment rows gr and gr + 8 of this lane).
// F16: q and K are fp16 (one QK pass); otherwise bf16 with q split into high part
// and residual (two QK passes into one sum).  P V is bf16 either way.
template <int D, bool F16 = false>
struct WarpRows16 {
    uint32_t qa[D / 16][4];              // query fragments (already scale-offset and scaled): high part
    uint32_t ql[F16 ? 1 : D / 16][4];    // bf16 residual q - high part (bf16 mode only)
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
    // `krow0` of a block staged as D/64 slabs (K at kbase, slabs kslab bytes apart;
    // V at vbase, vslab apart).  Key j is valid for row A iff j <= limA (likewise
    // B); pass full = true when every key of the chunk is valid for every row.
    __device__ __forceinline__ void step(uint32_t kbase, int kslab, uint32_t vbase, int vslab, int krow0,
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
            ldsm_x4(kbase + (kt * 16 / 64) * kslab + sw128_offset(krow0 + kld_row, ((kt * 16) % 64) / 8 + kld_hi),
                    b0, b1, b2, b3);
            if constexpr (F16) {
                mma_16816_f16(s[0], qa[kt], b0, b1);
                mma_16816_f16(s[1], qa[kt], b2, b3);
            } else {
                mma_16816(s[0], qa[kt], b0, b1);
                mma_16816(s[1], qa[kt], b2, b3);
                mma_16816(s[0], ql[kt], b0, b1);
                mma_16816(s[1], ql[kt], b2, b3);
            }
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
            ldsm_x4_trans(vbase + (dp * 16 / 64) * vslab + sw128_offset(krow0 + vld_row, ((dp * 16) % 64) / 8 + vld_hi),
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

// Per-warp online-softmax state for up to 8 * NT query rows that share one KV head,
// with the 16-key chunk on the MMA's M side: S^T = K q^T (keys x rows) and
// O^T += V^T P^T, P^T reaching the second MMA through an in-register transpose.
// For a handful of rows (a few output copies of one KV head) this takes half the
// MMAs and half the accumulator registers of WarpRows16.  Lane l owns rows
// 8 nt + 2 (l % 4) + {0, 1} of n-tile nt, and output columns d = 16 mt + l / 4 (+ 8).
// F16: q and K are fp16 (one QK pass); otherwise bf16, q split into high part and
// residual.  P V is bf16.
template <int D, int NT, bool F16>
struct WarpKeys16 {
    uint32_t qb[NT][D / 16][2];                      // q^T B fragments (row l / 4 of the n-tile)
    uint32_t ql[F16 ? 1 : NT][F16 ? 1 : D / 16][2];  // bf16 residual (bf16 mode only)
    float o[NT][D / 16][4];                          // O^T: d = 16 mt + l / 4 (+8), rows 2 (l % 4) + {0, 1}
    float m[NT][2], l[NT][2];                        // running max (log2 units) and partial sum per row

    __device__ __forceinline__ void reset()
    {
        const float NEG_INF = -__int_as_float(0x7f800000);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
                o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
            m[nt][0] = m[nt][1] = NEG_INF;
            l[nt][0] = l[nt][1] = 0.f;
        }
    }

    // Keys j0 .. j0+15 at shared-memory rows krow0.. of a block staged as D/64 slabs
    // with the TMA 128-byte swizzle (K at kbase, slabs kslab bytes apart; V at vbase,
    // vslab apart).  Key j counts for row (nt, i) iff j <= lim[nt][i]; pass whole =
    // true when every key counts for every row this warp keeps.
    __device__ __forceinline__ void step(uint32_t kbase, int kslab, uint32_t vbase, int vslab, int krow0, int j0,
                                         const int (&lim)[NT][2], bool whole)
    {
        const int lane = threadIdx.x & 31;
        const float NEG_INF = -__int_as_float(0x7f800000);
        // ldmatrix addresses: A of K (16 keys x 16 d, row-major) and A of V^T (16 d x 16 keys)
        const int ka_row = krow0 + (lane & 7) + (((lane >> 3) & 1) << 3), ka_hi = lane >> 4;
        const int va_row = krow0 + (lane & 7) + ((lane >> 4) << 3), va_hi = (lane >> 3) & 1;
        // two accumulator chains (even / odd 16-wide d steps) for more MMAs in flight
        float s[NT][4], s2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt) {
            uint32_t a[4];
            ldsm_x4(kbase + (kt * 16 / 64) * kslab + sw128_offset(ka_row, ((kt * 16) % 64) / 8 + ka_hi), a[0], a[1],
                    a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float *acc = (kt & 1) ? s2[nt] : s[nt];
                if constexpr (F16) {
                    mma_16816_f16(acc, a, qb[nt][kt][0], qb[nt][kt][1]);
                } else {
                    mma_16816(acc, a, qb[nt][kt][0], qb[nt][kt][1]);
                    mma_16816(acc, a, ql[nt][kt][0], ql[nt][kt][1]);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s[nt][e] += s2[nt][e];
        // s[nt][e]: key j0 + l / 4 + 8 (e >> 1), row 8 nt + 2 (l % 4) + (e & 1)
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (!whole) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (j0 + (lane >> 2) + ((e >> 1) << 3) > lim[nt][e & 1])
                        s[nt][e] = NEG_INF;
            }
            float cm0 = fmaxf(s[nt][0], s[nt][2]), cm1 = fmaxf(s[nt][1], s[nt][3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, off));
                cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, off));
            }
            const float n0 = fmaxf(m[nt][0], cm0), n1 = fmaxf(m[nt][1], cm1);
            const float u0 = (n0 == NEG_INF) ? 0.f : n0, u1 = (n1 == NEG_INF) ? 0.f : n1;
            const float c0 = fast_exp2(m[nt][0] - u0), c1 = fast_exp2(m[nt][1] - u1);
            m[nt][0] = n0;
            m[nt][1] = n1;
            const float p0 = fast_exp2(s[nt][0] - u0), p1 = fast_exp2(s[nt][1] - u1);
            const float p2 = fast_exp2(s[nt][2] - u0), p3 = fast_exp2(s[nt][3] - u1);
            l[nt][0] = l[nt][0] * c0 + (p0 + p2);
            l[nt][1] = l[nt][1] * c1 + (p1 + p3);
            if (c0 != 1.f || c1 != 1.f) {
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    o[nt][mt][0] *= c0;
                    o[nt][mt][1] *= c1;
                    o[nt][mt][2] *= c0;
                    o[nt][mt][3] *= c1;
                }
            }
            // P^T as the B operand (keys x rows): transpose the (key, row) pairs per 8 keys
            pb[nt][0] = movmatrix_trans(pack_bf16x2(p0, p1));
            pb[nt][1] = movmatrix_trans(pack_bf16x2(p2, p3));
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(vbase + (mt * 16 / 64) * vslab + sw128_offset(va_row, ((mt * 16) % 64) / 8 + va_hi), a[0],
                          a[1], a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_16816(o[nt][mt], a, pb[nt][0], pb[nt][1]);
        }
    }

    // full row sums (the keys of a row are spread over the 8 lanes with equal l % 4)
    __device__ __forceinline__ void finish_sums()
    {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1)
                    l[nt][i] += __shfl_xor_sync(0xffffffffu, l[nt][i], off);
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
