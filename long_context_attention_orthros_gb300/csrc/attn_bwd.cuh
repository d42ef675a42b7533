// attn_bwd.cuh -- gradients of "Orthros: Phase-Aware Heterogeneous Attention" for
// the training modes (Sec. 3.2: SFT / PT compute every base position and T_out
// copies): the base stream, Eq. (4), and the output copies, Eq. (5), each with its
// scale-offset q = Q_raw * alpha + beta (Sec. 3.1).  For an output gradient dO and,
// per query row with the keys j it attends,
//   p_j = softmax_j(s_j), s_j = scale * (q . k_j);  dp_j = dO . v_j
//   D = dO . o = sum_j p_j dp_j;  ds_j = p_j (dp_j - D)
//   dq = scale * sum_j ds_j k_j;  dk_j += scale * ds_j q;  dv_j += p_j dO
//   dq_raw = dq * alpha;  dalpha += q_raw * dq;  dbeta += dq
// A query row is a "unit" (a base token, or a copy) times a head; the unit sits at
// position P (the token itself, or the copy's original position) and sees keys
// P - window + 1 .. P (window = T_kv for the copies: keys 0 .. P).
// Launches (bf16 / fp16 operands, fp32 accumulation, fp32 outputs):
//   attn_bwd_k16_kernel     an exact fp16 copy of K (for q . k on tensor memory);
//   attn_bwd_rows_kernel    the scale-offset q of the stream's rows as fp16, D = dO . o per row
//                           (and a given forward log-sum-exp in log2 units), one pass;
//   attn_bwd_dq_kernel      (base stream without the forward's log-sum-exp) warp MMAs, rows
//                           on the MMA's M side: K/V stream through a two-stage shared-memory
//                           ring of 64-key blocks (cp.async); pass 1 takes each row's
//                           log2-sum-exp (kept for the dK/dV kernel), pass 2 dP = dO V^T,
//                           dS = P (dP - D), dQ += dS K (q as bf16 high part + residual);
//                           then dq_raw, and dalpha / dbeta through shared, then global,
//                           atomics;
//   attn_bwd_dq_tc_base_kernel + attn_bwd_dab_kernel  (base stream with it) the same on
//                           tcgen05, persistent, then the dalpha / dbeta column sums;
//   attn_bwd_dq_band_kernel (base stream with it, G >= 4, narrow windows) tcgen05, each row
//                           tile's whole key band per MMA, dalpha / dbeta folded in (below);
//   attn_bwd_dq_tc_kernel   (copies) the same on tcgen05, one or two passes, optionally
//                           split over the keys (below);
//   attn_bwd_dq_copies_keys_kernel  (copies with it, at most 8 rows per KV head) warp MMAs
//                           with the rows on N, keys split over CTAs (below);
//   attn_bwd_dkv_tc_kernel  keys on tcgen05's M side, dK and dV in tensor memory (below),
//                           for one stream or for both of a layer.
// P enters dV as bf16; dS enters dQ as bf16 and dK as fp16 (beside the fp16 q).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"
#include "xattn.cuh"

namespace orthros {

namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr int BWD_ROWS = 64;  // query rows of a warp-MMA dq CTA
constexpr int BWD_KEYS = 64;  // keys per streamed block of the warp-MMA dq kernel

// [rows][D] bf16 tile in shared memory as D/64 slabs of rows x 128 bytes, 128-byte swizzle
__device__ __forceinline__ uint32_t tile_off(int row, int col, int slab_bytes)
{
    return static_cast<uint32_t>((col / 64) * slab_bytes) + sw128_offset(row, (col % 64) / 8);
}

// 16-byte asynchronous copy global -> shared; valid = false writes zeros (nothing is read)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// position of unit u of sequence b, or -1 when it has none in [0, T_kv)
template <bool COPY>
__device__ __forceinline__ int unit_pos(const AttnBwdParams &p, int b, int u)
{
    if (u >= p.n_units)
        return -1;
    if (!COPY)
        return u;
    const int P = __ldg(p.pos + static_cast<long long>(b) * p.n_units + u);
    return (P >= 0 && P < p.T_kv) ? P : -1;
}


// ------------------------------------------------------------------ fp16 copy of K

// The tensor-memory kernels take q . k in fp16 (as the forward's tensor-memory path): K is
// converted once per call.  A key row whose largest |k| reaches 65520 (beyond fp16) is stored
// as k * 2^-e with its largest element in [2^14, 2^15); the row's e goes to kexp and its
// 64-key block's flag to kflag, so that the kernels reading S multiply its logits back by 2^e.
// One CTA per 64-key block of one (batch, KV head); D / 8 lanes per key row.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_k16_kernel(const orthros_bf16 *k, uint16_t *k16, int8_t *kexp,
                                                           uint8_t *kflag, int T, int Hkv, int nkb, int32_t *dev_err)
{
    constexpr int CPR = D / 8;      // 16-byte chunks per key row
    constexpr int RPI = 256 / CPR;  // rows per pass of the CTA
    const int kb = static_cast<int>(blockIdx.x % nkb);
    const int bh = static_cast<int>(blockIdx.x / nkb);
    const int b = bh / Hkv, g = bh % Hkv;
    const int c = threadIdx.x % CPR, rr = threadIdx.x / CPR;
    bool shifted = false, bad = false;
#pragma unroll
    for (int r0 = 0; r0 < 64; r0 += RPI) {
        const int key = kb * 64 + r0 + rr;
        const bool valid = key < T;
        const long long off = ((static_cast<long long>(b) * T + key) * Hkv + g) * D + c * 8;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (valid)
            u = __ldg(reinterpret_cast<const uint4 *>(k + off));
        float am = bf16x8_absmax(u);
#pragma unroll
        for (int o = 1; o < CPR; o <<= 1)
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        const int ex = fp16_key_shift(am, bad);
        shifted |= ex != 0;
        if (valid)
            *reinterpret_cast<uint4 *>(k16 + off) = ex != 0 ? k_to_fp16_scaled(u, exp2i(-ex)) : k_to_fp16(u);
        if (c == 0)
            kexp[static_cast<long long>(bh) * nkb * 64 + kb * 64 + r0 + rr] = static_cast<int8_t>(ex);
    }
    shifted = __syncthreads_or(shifted ? 1 : 0) != 0;
    if (threadIdx.x == 0)
        kflag[static_cast<long long>(bh) * nkb + kb] = shifted ? 1 : 0;
    if (bad)
        record_error(dev_err, ORTHROS_DEVERR_RANGE);
}

// ------------------------------------------------------------------ fp16 q and the dalpha / dbeta sums

// q = x alpha + beta of every row of the stream as fp16 (workspace), for the dK/dV kernel
// and the persistent dq kernel; |q| >= 65504 sets ORTHROS_DEVERR_RANGE.  A thread takes two
// 16-byte chunks per step (both loads in flight) and keeps its chunks' column in the row
// [0, hd8) by adding the grid stride modulo hd8.
__device__ __forceinline__ uint4 scale_offset_fp16(uint4 u, const float *alpha, const float *beta, int col,
                                                   bool &bad)
{
    const float4 a0 = __ldg(reinterpret_cast<const float4 *>(alpha + col));
    const float4 a1 = __ldg(reinterpret_cast<const float4 *>(alpha + col + 4));
    const float4 b0 = __ldg(reinterpret_cast<const float4 *>(beta + col));
    const float4 b1 = __ldg(reinterpret_cast<const float4 *>(beta + col + 4));
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        const float qa = fmaf(f.x, av[2 * e], bv[2 * e]), qc = fmaf(f.y, av[2 * e + 1], bv[2 * e + 1]);
        bad |= !(fmaxf(fabsf(qa), fabsf(qc)) < 65504.f);
        __half2 hv = __floats2half2_rn(qa, qc);
        o[e] = *reinterpret_cast<uint32_t *>(&hv);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// dalpha[c] += sum_rows x * dq, dbeta[c] += sum_rows dq over the columns c = h * D + d, with
// dq = dq_raw / alpha (both sums are linear in the rows: one pass after the dq kernel).
// Each thread owns 4 columns over a run of rows; one atomic per column and CTA.
__global__ void __launch_bounds__(256) attn_bwd_dab_kernel(const float *dq_raw, const orthros_bf16 *x,
                                                           const float *alpha, float *dalpha, float *dbeta,
                                                           long long rows, int cols, int rows_per_cta)
{
    const int c4 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;  // first of this thread's columns
    if (c4 >= cols)
        return;
    const long long r0 = static_cast<long long>(blockIdx.y) * rows_per_cta;
    const long long r1 = min(rows, r0 + rows_per_cta);
    const float4 al = __ldg(reinterpret_cast<const float4 *>(alpha + c4));
    const float4 ia = make_float4(1.f / al.x, 1.f / al.y, 1.f / al.z, 1.f / al.w);
    float4 sa = make_float4(0.f, 0.f, 0.f, 0.f), sb = sa;
    for (long long r = r0; r < r1; ++r) {
        const float4 g = __ldcs(reinterpret_cast<const float4 *>(dq_raw + r * cols + c4));
        const uint2 xr = __ldcs(reinterpret_cast<const uint2 *>(x + r * cols + c4));
        const float2 x0 = unpack_bf16x2(xr.x), x1 = unpack_bf16x2(xr.y);
        const float4 dq = make_float4(g.x * ia.x, g.y * ia.y, g.z * ia.z, g.w * ia.w);
        sb.x += dq.x;
        sb.y += dq.y;
        sb.z += dq.z;
        sb.w += dq.w;
        sa.x = fmaf(x0.x, dq.x, sa.x);
        sa.y = fmaf(x0.y, dq.y, sa.y);
        sa.z = fmaf(x1.x, dq.z, sa.z);
        sa.w = fmaf(x1.y, dq.w, sa.w);
    }
    atomicAdd(dalpha + c4, sa.x);
    atomicAdd(dalpha + c4 + 1, sa.y);
    atomicAdd(dalpha + c4 + 2, sa.z);
    atomicAdd(dalpha + c4 + 3, sa.w);
    atomicAdd(dbeta + c4, sb.x);
    atomicAdd(dbeta + c4 + 1, sb.y);
    atomicAdd(dbeta + c4 + 2, sb.z);
    atomicAdd(dbeta + c4 + 3, sb.w);
}

// ------------------------------------------------------------------ fp16 q and D = dO . o

// One pass over the stream's query rows: q = x alpha + beta as fp16 into the workspace (read by
// the dK/dV kernel and the persistent dQ; |q| >= 65504 sets ORTHROS_DEVERR_RANGE), D = dO . o
// per row, and a given forward log-sum-exp in log2 units.  D / 8 lanes per row, 16 bytes of
// each of x, o and dO per lane, all three loads in flight.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_rows_kernel(const orthros_bf16 *x, const float *alpha,
                                                            const float *beta, uint16_t *q16, const orthros_bf16 *o,
                                                            const orthros_bf16 *dO, float *Dout, const float *lse_in,
                                                            float *lse_out, long long rows, int Hq, int32_t *dev_err)
{
    constexpr int LPR = D / 8;  // lanes per row
    const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / LPR;
    const int sub = threadIdx.x % LPR;
    bool bad = false;
    float acc = 0.f;
    if (row < rows) {
        const long long off = row * D + sub * 8;
        const uint4 xa = __ldg(reinterpret_cast<const uint4 *>(x + off));
        const uint4 oa = __ldg(reinterpret_cast<const uint4 *>(o + off));
        const uint4 ga = __ldg(reinterpret_cast<const uint4 *>(dO + off));
        const int h = static_cast<int>(row % Hq);
        *reinterpret_cast<uint4 *>(q16 + off) = scale_offset_fp16(xa, alpha + h * D, beta + h * D, sub * 8, bad);
        const uint32_t aw[4] = {oa.x, oa.y, oa.z, oa.w}, bw[4] = {ga.x, ga.y, ga.z, ga.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 u = unpack_bf16x2(aw[e]), v = unpack_bf16x2(bw[e]);
            acc = fmaf(u.x, v.x, fmaf(u.y, v.y, acc));
        }
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && sub == 0) {
        Dout[row] = acc;
        if (lse_in != nullptr)  // the forward's log-sum-exp, to log2 units
            lse_out[row] = lse_in[row] * kLog2eF;
    }
    if (bad)
        record_error(dev_err, ORTHROS_DEVERR_RANGE);
}

// ------------------------------------------------------------------ dQ (rows on M)

template <int D, int G, bool COPY>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const AttnBwdParams p)
{
    constexpr int UNITS = BWD_ROWS / G;
    constexpr int SLAB = BWD_KEYS * 128;  // one 64-column slab of a 64-key block
    constexpr int BLK = (D / 64) * SLAB;  // one K (or V) block
    const int u0 = blockIdx.x * UNITS, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    float *red = reinterpret_cast<float *>(smem + 4 * BLK);  // [2][G][D]: dalpha, dbeta
    int *krange = reinterpret_cast<int *>(red + 2 * G * D);  // the CTA's lowest and highest key
    const uint32_t sbase = smem_u32(smem);

    // this warp's 16 rows: r = 16 warp + 0..15 -> unit u0 + r / G, head g G + r % G
    const int gr = lane >> 2, qd = (lane & 3) * 2;
    const int rowA = 16 * warp + gr, rowB = rowA + 8;
    const int uA = u0 + rowA / G, uB = u0 + rowB / G;
    const int hA = g * G + rowA % G, hB = g * G + rowB % G;
    const int PA = unit_pos<COPY>(p, b, uA), PB = unit_pos<COPY>(p, b, uB);
    const bool vA = PA >= 0, vB = PB >= 0;
    if (COPY && (lane & 3) == 0 && ((uA < p.n_units && !vA) || (uB < p.n_units && !vB)))
        record_error(p.dev_err, ORTHROS_DEVERR_POSITION);
    const int loA = PA - p.window + 1, loB = PB - p.window + 1;
    int wlo = 0x7fffffff, whi = -1;  // the warp's key range
    if (vA) {
        wlo = max(0, loA);
        whi = PA;
    }
    if (vB) {
        wlo = min(wlo, max(0, loB));
        whi = max(whi, PB);
    }
    wlo = __reduce_min_sync(0xffffffffu, wlo);
    whi = __reduce_max_sync(0xffffffffu, whi);
    if (threadIdx.x == 0) {
        krange[0] = 0x7fffffff;
        krange[1] = -1;
    }
    for (int i = threadIdx.x; i < 2 * G * D; i += 128)
        red[i] = 0.f;
    __syncthreads();
    if (lane == 0 && whi >= 0) {
        atomicMin(&krange[0], wlo);
        atomicMax(&krange[1], whi);
    }
    __syncthreads();
    const int cb0 = krange[1] >= 0 ? krange[0] / BWD_KEYS : 0;
    const int cb1 = krange[1] >= 0 ? krange[1] / BWD_KEYS + 1 : 0;  // key blocks [cb0, cb1)

    const long long q_bs = static_cast<long long>(p.n_units) * p.Hq * D;
    const float c2 = p.scale * kLog2eF;  // logits in log2 units
    WarpRows16<D> st;                    // q fragments (unscaled q = x alpha + beta) + dQ accumulators
    uint32_t ga[D / 16][4];              // dO fragments (A operand)
#pragma unroll
    for (int kt2 = 0; kt2 < D / 16; ++kt2)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const bool isB = r & 1;
            const int u = isB ? uB : uA, h = isB ? hB : hA;
            const int dcol = kt2 * 16 + qd + ((r & 2) ? 8 : 0);
            uint32_t hi = 0, lo = 0, gw = 0;
            if (isB ? vB : vA) {
                const long long off = b * q_bs + (static_cast<long long>(u) * p.Hq + h) * D;
                load_q_pair(p.q + off, p.alpha + h * D, p.beta + h * D, dcol, 1.f, hi, lo);
                gw = *reinterpret_cast<const uint32_t *>(p.dO + off + dcol);
            }
            st.qa[kt2][r] = hi;
            st.ql[kt2][r] = lo;
            ga[kt2][r] = gw;
        }
    st.reset();
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int kld_row = (lane & 7) + ((lane >> 4) << 3), kld_hi = (lane >> 3) & 1;
    const int vld_row = (lane & 7) + (((lane >> 3) & 1) << 3), vld_hi = lane >> 4;

    // stream key block blk into ring slot buf: K, and V when withV
    const long long kv_rs = static_cast<long long>(p.Hkv) * D;
    const orthros_bf16 *kb = p.k + static_cast<long long>(b) * p.T_kv * kv_rs + static_cast<long long>(g) * D;
    const orthros_bf16 *vb = p.v + static_cast<long long>(b) * p.T_kv * kv_rs + static_cast<long long>(g) * D;
    auto stage = [&](int blk, int buf, bool withV) {
        const int key0 = blk * BWD_KEYS;
        for (int i = threadIdx.x; i < BWD_KEYS * (D / 8); i += 128) {
            const int r = i / (D / 8), c = (i % (D / 8)) * 8;
            const int key = key0 + r;
            const bool ok = key < p.T_kv;
            const long long off = static_cast<long long>(ok ? key : 0) * kv_rs + c;
            const uint32_t o = sbase + buf * 2 * BLK + tile_off(r, c, SLAB);
            cp_async16(o, kb + off, ok);
            if (withV)
                cp_async16(o + BLK, vb + off, ok);
        }
        cp_async_commit();
    };

    // S chunk (16 rows x keys kc .. kc+15 at block row jc) in log2 units, masked
    auto s_chunk = [&](uint32_t kbase, int jc, int kc, float (&s)[2][4]) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kt2 = 0; kt2 < D / 16; ++kt2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + tile_off(jc + kld_row, kt2 * 16 + kld_hi * 8, SLAB), b0, b1, b2, b3);
            mma_16816(s[0], st.qa[kt2], b0, b1);
            mma_16816(s[1], st.qa[kt2], b2, b3);
            mma_16816(s[0], st.ql[kt2], b0, b1);
            mma_16816(s[1], st.ql[kt2], b2, b3);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = kc + i * 8 + qd + (e & 1);
                const bool isB = e & 2;
                const int P = isB ? PB : PA, lo = isB ? loB : loA;
                s[i][e] = (key <= P && key >= lo) ? s[i][e] * c2 : NEG_INF;  // P = -1: no key
            }
    };

    float mA = NEG_INF, mB = NEG_INF, lA = 0.f, lB = 0.f, lseA = 0.f, lseB = 0.f, DA = 0.f, DB = 0.f;
    const long long rA = (static_cast<long long>(b) * p.n_units + uA) * p.Hq + hA;
    const long long rB = (static_cast<long long>(b) * p.n_units + uB) * p.Hq + hB;
    // pass 1 (each row's log-sum-exp) is skipped when the forward's is given
#pragma unroll 1
    for (int pass = p.lse_in != nullptr ? 2 : 1; pass <= 2; ++pass) {
        if (pass == 2) {
            if (p.lse_in != nullptr) {  // converted to log2 units by the rows kernel
                lseA = vA ? p.lse[rA] : 0.f;
                lseB = vB ? p.lse[rB] : 0.f;
            } else {
                // log2-sum-exp of each row over its keys (every valid row holds at least its own key)
                lA += __shfl_xor_sync(0xffffffffu, lA, 1);
                lA += __shfl_xor_sync(0xffffffffu, lA, 2);
                lB += __shfl_xor_sync(0xffffffffu, lB, 1);
                lB += __shfl_xor_sync(0xffffffffu, lB, 2);
                lseA = vA ? mA + __log2f(lA) : 0.f;
                lseB = vB ? mB + __log2f(lB) : 0.f;
                if ((lane & 3) == 0) {
                    if (vA)
                        p.lse[rA] = lseA;
                    if (vB)
                        p.lse[rB] = lseB;
                }
            }
            DA = vA ? p.Drow[rA] : 0.f;
            DB = vB ? p.Drow[rB] : 0.f;
        }
        if (cb0 < cb1)
            stage(cb0, 0, pass == 2);
#pragma unroll 1
        for (int blk = cb0; blk < cb1; ++blk) {
            const int buf = (blk - cb0) & 1;
            if (blk + 1 < cb1) {
                stage(blk + 1, buf ^ 1, pass == 2);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const uint32_t kbase = sbase + buf * 2 * BLK, vbase = kbase + BLK;
#pragma unroll 1
            for (int jc = 0; jc < BWD_KEYS; jc += 16) {
                const int kc = blk * BWD_KEYS + jc;
                if (kc + 15 < wlo || kc > whi)
                    continue;  // warp-uniform: no key of this chunk is seen by the warp's rows
                float s[2][4];
                s_chunk(kbase, jc, kc, s);
                if (pass == 1) {
                    float cA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
                    float cB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
                    cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 1));
                    cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 2));
                    cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 1));
                    cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 2));
                    const float nA = fmaxf(mA, cA), nB = fmaxf(mB, cB);
                    const float zA = nA == NEG_INF ? 0.f : nA, zB = nB == NEG_INF ? 0.f : nB;
                    lA = lA * fast_exp2(mA - zA) + fast_exp2(s[0][0] - zA) + fast_exp2(s[0][1] - zA) +
                         fast_exp2(s[1][0] - zA) + fast_exp2(s[1][1] - zA);
                    lB = lB * fast_exp2(mB - zB) + fast_exp2(s[0][2] - zB) + fast_exp2(s[0][3] - zB) +
                         fast_exp2(s[1][2] - zB) + fast_exp2(s[1][3] - zB);
                    mA = nA;
                    mB = nB;
                } else {
                    float dp[2][4];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
#pragma unroll
                    for (int kt2 = 0; kt2 < D / 16; ++kt2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(vbase + tile_off(jc + kld_row, kt2 * 16 + kld_hi * 8, SLAB), b0, b1, b2, b3);
                        mma_16816(dp[0], ga[kt2], b0, b1);
                        mma_16816(dp[1], ga[kt2], b2, b3);
                    }
                    uint32_t da[4];
                    float ds[2][4];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const bool isB = e & 2;
                            ds[i][e] = fast_exp2(s[i][e] - (isB ? lseB : lseA)) * (dp[i][e] - (isB ? DB : DA));
                        }
                    da[0] = pack_bf16x2(ds[0][0], ds[0][1]);
                    da[1] = pack_bf16x2(ds[0][2], ds[0][3]);
                    da[2] = pack_bf16x2(ds[1][0], ds[1][1]);
                    da[3] = pack_bf16x2(ds[1][2], ds[1][3]);
#pragma unroll
                    for (int dp2 = 0; dp2 < D / 16; ++dp2) {
                        uint32_t v0, v1, v2, v3;
                        ldsm_x4_trans(kbase + tile_off(jc + vld_row, dp2 * 16 + vld_hi * 8, SLAB), v0, v1, v2, v3);
                        mma_16816(st.o[2 * dp2], da, v0, v1);
                        mma_16816(st.o[2 * dp2 + 1], da, v2, v3);
                    }
                }
            }
            __syncthreads();  // slot buf is refilled by the next iteration's prefetch
        }
    }
    // epilogue: dq = scale * dQ; dq_raw = dq * alpha; dalpha += x * dq, dbeta += dq
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const bool live = half ? vB : vA;
        const int u = half ? uB : uA, h = half ? hB : hA, hh = h - g * G;
        const long long off = b * q_bs + (static_cast<long long>(u) * p.Hq + h) * D;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const int dcol = i * 8 + qd;
            if (!live)
                continue;
            const float dq0 = st.o[i][2 * half] * p.scale, dq1 = st.o[i][2 * half + 1] * p.scale;
            const float2 al = __ldg(reinterpret_cast<const float2 *>(p.alpha + h * D + dcol));
            *reinterpret_cast<float2 *>(p.dq + off + dcol) = make_float2(dq0 * al.x, dq1 * al.y);
            const float2 x = unpack_bf16x2(*reinterpret_cast<const uint32_t *>(p.q + off + dcol));
            atomicAdd(&red[hh * D + dcol], x.x * dq0);
            atomicAdd(&red[hh * D + dcol + 1], x.y * dq1);
            atomicAdd(&red[G * D + hh * D + dcol], dq0);
            atomicAdd(&red[G * D + hh * D + dcol + 1], dq1);
        }
        if (!live && u < p.n_units) {  // a copy without a valid position: zero gradient row
#pragma unroll
            for (int i = 0; i < D / 8; ++i)
                *reinterpret_cast<float2 *>(p.dq + off + i * 8 + qd) = make_float2(0.f, 0.f);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += 128) {
        atomicAdd(p.dalpha + g * G * D + i, red[i]);
        atomicAdd(p.dbeta + g * G * D + i, red[G * D + i]);
    }
}

// ------------------------------------------------------------------ dK, dV on tcgen05

// A CTA owns 128 keys of one (batch, KV head): the MMA's M side, K and V resident in
// shared memory (one TMA load each).  The query rows that can see them stream through
// a four-stage ring in rounds of 64 (64/G units x G heads, in the order the 4-D TMA box
// lands them): q as fp16 (the scale-offset applied and rounded once by
// attn_bwd_rows_kernel, which also flags a query outside the fp16 range) and dO.  Per round
//   S^T  = K q^T          (fp16: K from the call's exact fp16 copy)
//   dP^T = V dO^T         (bf16) fp32 in tensor memory (two buffers each)
//   P^T  = exp2(S^T c - lse_row) on the row's keys, dS^T = P^T (dP^T - D_row), written
//          back over S^T (P^T, bf16) and dP^T (dS^T, fp16; |dS| >= 65504 sets
//          ORTHROS_DEVERR_RANGE) by the softmax warps (lane = key)
//   dV  += P^T dO,  dK += dS^T q           (A from tensor memory, B = the row tiles)
// and dK, dV (fp32, tensor memory) leave once at the end.  The MMA issuer computes S^T,
// dP^T of round i + 1 while the softmax works on round i.
// Roles (256 threads, one CTA per SM):
//   warp 0      TMA producer (K, V once; q and dO per round)
//   warp 1      allocates tensor memory; lane 0 issues every tcgen05.mma
//   warps 2-3   stage each round's per-row lse, D and position (one row per thread)
//   warps 4-7   P^T, dS^T (tensor-memory lane = key), then the dK / dV epilogue
// Tensor memory: S^T at 64 u, dP^T at 128 + 64 u (buffer u), dK at 256, dV at 256 + D.
// Every wait is bounded; a timeout records ORTHROS_DEVERR_TIMEOUT and every role drains
// to the common exit, where tensor memory is released.
template <int D>
struct BtCfg {
    static constexpr int KEYS = 128;          // keys of a CTA (the MMA's M)
    static constexpr int RB = 64;             // query rows per round (N of S^T, dP^T)
    static constexpr int SLABS = D / 64;
    static constexpr int STG = 4;
    static constexpr int KSLAB = KEYS * 128;  // one 64-wide slab of the K (or V) tile
    static constexpr int RSLAB = RB * 128;    // one 64-wide slab of a row tile
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + SLABS * KSLAB;
    static constexpr int ST_OFF = V_OFF + SLABS * KSLAB;
    static constexpr int ST_Q16 = 0;                  // scale-offset q as fp16 (from the workspace)
    static constexpr int ST_DO = SLABS * RSLAB;       // dO
    static constexpr int ST_BYTES = 2 * SLABS * RSLAB;
    static constexpr int META_OFF = ST_OFF + STG * ST_BYTES;  // [STG][3][RB]: lse, D, position
    static constexpr int BAR_OFF = META_OFF + STG * 3 * RB * 4;
    static constexpr int NBARS = 1 + 3 * STG + 3 * 2 + 1;
    static constexpr int HOLD_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = HOLD_OFF + 16 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DK = 256, TM_DV = 256 + D;
};

// q = x alpha + beta for 8 elements of head h at column d0: fp16 and bf16 copies
__device__ __forceinline__ void scale_offset8(uint4 x4, const float *alpha, const float *beta, int d0, uint4 &q16,
                                              uint4 &qb, bool &bad)
{
    const float4 a0 = __ldg(reinterpret_cast<const float4 *>(alpha + d0));
    const float4 a1 = __ldg(reinterpret_cast<const float4 *>(alpha + d0 + 4));
    const float4 b0 = __ldg(reinterpret_cast<const float4 *>(beta + d0));
    const float4 b1 = __ldg(reinterpret_cast<const float4 *>(beta + d0 + 4));
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
    uint32_t hw[4], bw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 xv = unpack_bf16x2(xw[e]);
        const float qa = fmaf(xv.x, av[2 * e], bv[2 * e]), qc = fmaf(xv.y, av[2 * e + 1], bv[2 * e + 1]);
        bad |= !(fmaxf(fabsf(qa), fabsf(qc)) < 65504.f);
        __half2 hv = __floats2half2_rn(qa, qc);
        hw[e] = *reinterpret_cast<uint32_t *>(&hv);
        bw[e] = pack_bf16x2(qa, qc);
    }
    q16 = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    qb = make_uint4(bw[0], bw[1], bw[2], bw[3]);
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// wait on an mbarrier as a whole warp (lane 0 polls); false after the time limit
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = mbar_wait(bar, parity);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// the next round (of `units` units) at or after r that holds a unit seeing keys >= kt0
// (copies; base rounds are a contiguous range).  Called by whole warps.
template <bool COPY>
__device__ __forceinline__ int next_round(const AttnBwdParams &p, int b, int kt0, int r, int r_end, int units)
{
    if (!COPY)
        return r;
    const int lane = threadIdx.x & 31;
    for (; r < r_end; ++r) {
        bool hit = false;
        for (int u = lane; u < units; u += 32)
            hit |= unit_pos<COPY>(p, b, r * units + u) >= kt0;
        if (__any_sync(0xffffffffu, hit))
            return r;
    }
    return r_end;
}

constexpr int DKV_TC_THREADS = 384;
constexpr int DKV_TC_CONV = 192;  // preparation threads of the dQ kernel (warps 2-3 and 8-11)
constexpr int DKV_THREADS = 256;  // the dK/dV kernel: producer, MMA, 2 metadata warps, 4 softmax warps

// The rounds of query rows a dK/dV CTA takes, in order: phase 0 is the stream of p (base
// rows: rounds kt0/UNITS .. while a row can see the block; copies: the rounds holding a copy at
// a position >= kt0), phase 1 (STREAMS == 2) the copies of pc.  seek moves (ph, r) to the first
// round at or after it and returns false once none is left.  Called by whole warps.
template <int STREAMS>
struct DkvRounds {
    const AttnBwdParams &p, &pc;
    int b, kt0, units, base_end;
    __device__ __forceinline__ bool seek(int &ph, int &r) const
    {
        if (ph == 0) {
            if (STREAMS == 1) {
                const int e = (p.n_units + units - 1) / units;
                r = next_round<true>(p, b, kt0, r, e, units);
                return r < e;
            }
            if (r < base_end)
                return true;
            if (STREAMS == 0)
                return false;
            ph = 1;
            r = 0;
        }
        const int e = (pc.n_units + units - 1) / units;
        r = next_round<true>(pc, b, kt0, r, e, units);
        return r < e;
    }
};

// position of unit u of the round's stream (copies: pos, -1 when out of range or past the end)
__device__ __forceinline__ int round_unit_pos(const AttnBwdParams &p, const AttnBwdParams &pc, bool from_pc,
                                              bool copy, int b, int u)
{
    const int n = from_pc ? pc.n_units : p.n_units;
    if (u >= n)
        return -1;
    if (!copy)
        return u;
    const int32_t *pos = from_pc ? pc.pos : p.pos;
    const int P = __ldg(pos + static_cast<long long>(b) * n + u);
    return (P >= 0 && P < p.T_kv) ? P : -1;
}

// STREAMS: 0 the base stream (p), 1 copies (p), 2 the base stream (p) and then the copies (pc,
// with its own row maps qcmap / ocmap) into the same dK / dV, written once.
template <int D, int G, int STREAMS>
__global__ void __launch_bounds__(DKV_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                           const __grid_constant__ CUtensorMap qcmap, const __grid_constant__ CUtensorMap ocmap,
                           const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const AttnBwdParams p, const AttnBwdParams pc)
{
    using C = BtCfg<D>;
    constexpr int UNITS = C::RB / G;  // units per round
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *kv_full = bars;                     // K, V landed
    uint64_t *st_full = bars + 1;                 // [STG] row tiles landed
    uint64_t *qconv = bars + 1 + C::STG;          // [STG] row metadata staged
    uint64_t *st_empty = bars + 1 + 2 * C::STG;   // [STG] round's MMAs done with the stage
    uint64_t *s_full = bars + 1 + 3 * C::STG;     // [2] S^T, dP^T of a round complete
    uint64_t *p_full = s_full + 2;                // [2] P^T, dS^T written
    uint64_t *pv_done = s_full + 4;               // [2] dV, dK of a round issued and complete
    uint64_t *acc_final = s_full + 6;             // dV, dK of the last round complete
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::HOLD_OFF);
    float *meta = reinterpret_cast<float *>(smem + C::META_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt0 = blockIdx.x * C::KEYS, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    // rounds r cover units r*UNITS .. r*UNITS+UNITS-1 of their stream
    const int r_begin = STREAMS == 1 ? 0 : kt0 / UNITS;
    const int base_end = static_cast<int>((min(static_cast<long long>(p.n_units),
                                                static_cast<long long>(kt0) + C::KEYS - 1 + p.window) +
                                            UNITS - 1) /
                                           UNITS);
    const DkvRounds<STREAMS> rounds{p, pc, b, kt0, UNITS, base_end};

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < C::STG; ++s) {
            mbar_init(&st_full[s], 1);
            mbar_init(&qconv[s], 2);
            mbar_init(&st_empty[s], 1);
        }
        for (int u = 0; u < 2; ++u) {
            mbar_init(&s_full[u], 1);
            mbar_init(&p_full[u], 4);
            mbar_init(&pv_done[u], 1);
        }
        mbar_init(acc_final, 1);
        fence_barrier_init();
    }
    if (warp == 1)
        tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&omap);
            if (STREAMS == 2) {
                tma_prefetch_desc(&qcmap);
                tma_prefetch_desc(&ocmap);
            }
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            mbar_arrive_expect_tx(kv_full, 2 * C::SLABS * C::KSLAB);
#pragma unroll
            for (int sl = 0; sl < C::SLABS; ++sl) {
                tma_load_4d(smem + C::K_OFF + sl * C::KSLAB, &kmap, kv_full, sl * 64, g, kt0, b);
                tma_load_4d(smem + C::V_OFF + sl * C::KSLAB, &vmap, kv_full, sl * 64, g, kt0, b);
            }
        }
        int i = 0, ph = 0, r = r_begin;
        for (bool more = rounds.seek(ph, r); more; ++r, more = rounds.seek(ph, r), ++i) {
            const int s = i % C::STG;
            if (i >= C::STG && !(ok = warp_wait(&st_empty[s], static_cast<uint32_t>(((i / C::STG) - 1) & 1))))
                break;
            if (lane == 0) {
                uint8_t *st = smem + C::ST_OFF + s * C::ST_BYTES;
                const CUtensorMap *qm = (STREAMS == 2 && ph == 1) ? &qcmap : &qmap;
                const CUtensorMap *om = (STREAMS == 2 && ph == 1) ? &ocmap : &omap;
                mbar_arrive_expect_tx(&st_full[s], 2 * C::SLABS * C::RSLAB);
#pragma unroll
                for (int sl = 0; sl < C::SLABS; ++sl) {
                    tma_load_4d(st + C::ST_Q16 + sl * C::RSLAB, qm, &st_full[s], sl * 64, g * G, r * UNITS, b);
                    tma_load_4d(st + C::ST_DO + sl * C::RSLAB, om, &st_full[s], sl * 64, g * G, r * UNITS, b);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        constexpr uint32_t IDESC_S = umma_idesc(128, C::RB, false, false);   // fp16
        constexpr uint32_t IDESC_DP = umma_idesc(128, C::RB, true, false);   // bf16
        constexpr uint32_t IDESC_DV = umma_idesc(128, D, true, true);    // bf16 P^T, dO
        constexpr uint32_t IDESC_DK = umma_idesc(128, D, false, true);   // fp16 dS^T, q
        const uint64_t kdesc = umma_desc_sw128(sbase + C::K_OFF, 16, 1024);
        const uint64_t vdesc = umma_desc_sw128(sbase + C::V_OFF, 16, 1024);
        // dV += P^T dO and dK += dS^T q of round j
        auto accumulate = [&](int j) -> bool {
            const int u = j & 1, s = j % C::STG;
            if (!warp_wait(&p_full[u], static_cast<uint32_t>((j >> 1) & 1)))
                return false;
            if (lane == 0) {
                tc_fence_after();
                const uint32_t st = sbase + C::ST_OFF + s * C::ST_BYTES;
                const uint64_t odesc = umma_desc_sw128(st + C::ST_DO, C::RSLAB, 1024);
                const uint64_t qdesc = umma_desc_sw128(st + C::ST_Q16, C::RSLAB, 1024);
#pragma unroll
                for (int kk = 0; kk < C::RB / 16; ++kk) {
                    const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                    umma_ts(tbase + C::TM_DV, tbase + C::TM_S + 64 * u + 8 * kk,
                            odesc + static_cast<uint64_t>(kk * (2048 >> 4)), IDESC_DV, acc);
                    umma_ts(tbase + C::TM_DK, tbase + C::TM_DP + 64 * u + 8 * kk,
                            qdesc + static_cast<uint64_t>(kk * (2048 >> 4)), IDESC_DK, acc);
                }
                umma_commit(&pv_done[u]);
                umma_commit(&st_empty[s]);
            }
            __syncwarp();
            return true;
        };
        ok = warp_wait(kv_full, 0);
        int i = 0, ph = 0, r = r_begin;
        for (bool more = rounds.seek(ph, r); ok && more; ++r, more = rounds.seek(ph, r), ++i) {
            const int s = i % C::STG, u = i & 1;
            if (!(ok = warp_wait(&st_full[s], static_cast<uint32_t>((i / C::STG) & 1))))
                break;
            // S^T / dP^T buffer u is free once dV, dK of round i - 2 have read P^T, dS^T from it
            if (i >= 2 && !(ok = warp_wait(&pv_done[u], static_cast<uint32_t>(((i - 2) >> 1) & 1))))
                break;
            if (lane == 0) {
                tc_fence_after();
                const uint32_t st = sbase + C::ST_OFF + s * C::ST_BYTES;
                const uint64_t qdesc = umma_desc_sw128(st + C::ST_Q16, 16, 1024);
                const uint64_t odesc = umma_desc_sw128(st + C::ST_DO, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = static_cast<uint32_t>((kk >> 2) * C::KSLAB + (kk & 3) * 32) >> 4;
                    const uint32_t ro = static_cast<uint32_t>((kk >> 2) * C::RSLAB + (kk & 3) * 32) >> 4;
                    umma_ss(tbase + C::TM_S + 64 * u, kdesc + ko, qdesc + ro, IDESC_S, kk != 0);
                    umma_ss(tbase + C::TM_DP + 64 * u, vdesc + ko, odesc + ro, IDESC_DP, kk != 0);
                }
                umma_commit(&s_full[u]);
            }
            __syncwarp();
            if (i >= 1 && !(ok = accumulate(i - 1)))
                break;
        }
        if (ok && i >= 1) {
            ok = accumulate(i - 1);
            if (ok && lane == 0)
                umma_commit(acc_final);
            __syncwarp();
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------------ row metadata
        const int ct = threadIdx.x - 64;  // 0..63: one row of the round each
        int i = 0, ph = 0, r = r_begin;
        for (bool more = rounds.seek(ph, r); ok && more; ++r, more = rounds.seek(ph, r), ++i) {
            const int s = i % C::STG;
            const bool from_pc = STREAMS == 2 && ph == 1;
            // loaded before the wait so that the latency overlaps it
            float m_lse = 0.f, m_d = 0.f;
            int m_pos = -1;
            {
                const int u = r * UNITS + ct / G, h = g * G + ct % G;
                m_pos = round_unit_pos(p, pc, from_pc, STREAMS != 0 && (STREAMS == 1 || ph == 1), b, u);
                if (m_pos >= 0) {
                    const long long ri =
                        (static_cast<long long>(b) * (from_pc ? pc.n_units : p.n_units) + u) * p.Hq + h;
                    m_lse = (from_pc ? pc.lse : p.lse)[ri];
                    m_d = (from_pc ? pc.Drow : p.Drow)[ri];
                }
            }
            // the slot is free once the stage of this round has landed: its producer waited
            // for the MMAs of round i - STG, which waited for that round's softmax
            if (!(ok = warp_wait(&st_full[s], static_cast<uint32_t>((i / C::STG) & 1))))
                break;
            float *m = meta + s * 3 * C::RB;
            m[ct] = m_lse;
            m[C::RB + ct] = m_d;
            m[2 * C::RB + ct] = __int_as_float(m_pos);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&qconv[s]);
        }
    } else {
        // ------------------------------------------------------------------ P^T, dS^T + epilogue
        const int rw = warp - 4;
        const int key = kt0 + rw * 32 + lane;
        const uint32_t tl = tbase + (static_cast<uint32_t>(rw * 32) << 16);
        // logit scale of this key's row of S^T (its fp16 copy is k * 2^-e: the logits are times 2^e)
        const float c2 = p.scale * kLog2eF *
                         exp2i(key < p.T_kv ? p.kexp[static_cast<long long>(bh) * p.nkb * 64 + key] : 0);
        float ds_max = 0.f;  // dS^T goes to fp16: |dS| < 65504 or the range error
        int i = 0, ph = 0, r = r_begin;
        for (bool more = rounds.seek(ph, r); more; ++r, more = rounds.seek(ph, r), ++i) {
            const int s = i % C::STG, u = i & 1;
            const int window = (STREAMS == 2 && ph == 1) ? pc.window : p.window;
            if (!(ok = warp_wait(&s_full[u], static_cast<uint32_t>((i >> 1) & 1)) &&
                       warp_wait(&qconv[s], static_cast<uint32_t>((i / C::STG) & 1))))
                break;
            tc_fence_after();
            const float *m = meta + s * 3 * C::RB;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t sv[32], dv[32];
                tmem_ld32(tl + C::TM_S + 64 * u + 32 * half, sv);
                tmem_ld32(tl + C::TM_DP + 64 * u + 32 * half, dv);
                tmem_wait_ld();
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float pr[2], ds[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int c = 32 * half + 2 * e + q;
                        const int P = __float_as_int(m[2 * C::RB + c]);
                        const bool valid = key <= P && key >= P - window + 1;  // P = -1: none
                        pr[q] = valid ? fast_exp2(__uint_as_float(sv[2 * e + q]) * c2 - m[c]) : 0.f;
                        ds[q] = pr[q] * (__uint_as_float(dv[2 * e + q]) - m[C::RB + c]);
                    }
                    ds_max = fmaxf(ds_max, fmaxf(fabsf(ds[0]), fabsf(ds[1])));
                    pw[e] = pack_bf16x2(pr[0], pr[1]);
                    __half2 hv = __floats2half2_rn(ds[0], ds[1]);
                    dw[e] = *reinterpret_cast<uint32_t *>(&hv);
                }
                tmem_st16(tl + C::TM_S + 64 * u + 16 * half, pw);
                tmem_st16(tl + C::TM_DP + 64 * u + 16 * half, dw);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[u]);
        }
        if (!(ds_max < 65504.f))
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
        // ---- epilogue: dK (scaled), dV of this key -> global (written, or added)
        const bool have = ok && i > 0;
        if (have && !(ok = warp_wait(acc_final, 0))) {
        } else {
            if (have)
                tc_fence_after();
            const long long off =
                (static_cast<long long>(b) * p.T_kv + key) * p.Hkv * D + static_cast<long long>(g) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t wk[32], wv[32];
                if (have) {
                    tmem_ld32(tl + C::TM_DK + c, wk);
                    tmem_ld32(tl + C::TM_DV + c, wv);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        wk[e] = wv[e] = 0u;
                }
                if (key < p.T_kv) {  // whole 32-byte sectors per store (rows are 32-byte aligned)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        wk[e] = __float_as_uint(__uint_as_float(wk[e]) * p.scale);
                    float *pk = p.dk + off + c, *pv = p.dv + off + c;
                    if (p.accumulate) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float4 ok4 = *reinterpret_cast<const float4 *>(pk + e);
                            const float4 ov4 = *reinterpret_cast<const float4 *>(pv + e);
                            wk[e] = __float_as_uint(__uint_as_float(wk[e]) + ok4.x);
                            wk[e + 1] = __float_as_uint(__uint_as_float(wk[e + 1]) + ok4.y);
                            wk[e + 2] = __float_as_uint(__uint_as_float(wk[e + 2]) + ok4.z);
                            wk[e + 3] = __float_as_uint(__uint_as_float(wk[e + 3]) + ok4.w);
                            wv[e] = __float_as_uint(__uint_as_float(wv[e]) + ov4.x);
                            wv[e + 1] = __float_as_uint(__uint_as_float(wv[e + 1]) + ov4.y);
                            wv[e + 2] = __float_as_uint(__uint_as_float(wv[e + 2]) + ov4.z);
                            wv[e + 3] = __float_as_uint(__uint_as_float(wv[e + 3]) + ov4.w);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        st_global_v8(pk + e, make_uint4(wk[e], wk[e + 1], wk[e + 2], wk[e + 3]),
                                     make_uint4(wk[e + 4], wk[e + 5], wk[e + 6], wk[e + 7]));
                        st_global_v8(pv + e, make_uint4(wv[e], wv[e + 1], wv[e + 2], wv[e + 3]),
                                     make_uint4(wv[e + 4], wv[e + 5], wv[e + 6], wv[e + 7]));
                    }
                }
            }
        }
    }
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ------------------------------------------------------------------ dQ on tcgen05

// A CTA owns 128 query rows (128/G units x G heads of one KV head): the MMA's M side,
// q (fp16, rounded once) and dO resident in shared memory.  The keys its rows see stream
// through a three-stage TMA ring in blocks of 64 (K from the call's fp16 copy for S; in
// pass 2 also K itself, bf16, for dQ, and V), twice:
//   pass 1  S = q K^T -> per-row running max / sum (lane = row) -> log2-sum-exp, stored
//           for the dK/dV kernel;
//   pass 2  S = q K^T, dP = dO V^T (fp32 in tensor memory, two buffers each);
//           dS = P (dP - D) with P = exp2(S c - lse), written over dP as bf16;
//           dQ += dS K  (A from tensor memory, B = the key block, MN-major)
// then dq_raw = scale dQ * alpha, and dalpha / dbeta reduced across the CTA's rows of
// each head (shuffles, then shared memory) and added with global atomics.
// Roles (384 threads, one CTA per SM): warp 0 TMA producer; warp 1 tensor-memory
// allocation and MMA issue; warps 2-3 and 8-11 query preparation; warps 4-7 softmax and
// epilogue.
// Tensor memory: S at 64 u, dP at 128 + 64 u (buffer u), dQ at 256.
template <int D>
struct BqCfg {
    static constexpr int ROWS = 128;          // query rows of a CTA (the MMA's M)
    static constexpr int KB = 64;             // keys per block (N of S, dP)
    static constexpr int SLABS = D / 64;
    static constexpr int STG = 3;
    static constexpr int QSLAB = ROWS * 128;
    static constexpr int KSLAB = KB * 128;
    static constexpr int Q16_OFF = 0;                         // raw x, then q as fp16
    static constexpr int DO_OFF = Q16_OFF + SLABS * QSLAB;    // dO
    static constexpr int K_OFF = DO_OFF + SLABS * QSLAB;      // [STG] K blocks (bf16)
    static constexpr int V_OFF = K_OFF + STG * SLABS * KSLAB; // [STG] V blocks
    static constexpr int K16_OFF = V_OFF + STG * SLABS * KSLAB;   // [STG] K blocks as fp16
    static constexpr int RED_OFF = K16_OFF + STG * SLABS * KSLAB; // [2][16][D+1] dalpha, dbeta partials
    static constexpr int RS = D + 1;                              // padded row: no bank conflicts
    static constexpr int RANGE_OFF = RED_OFF + 2 * 16 * RS * 4;
    static constexpr int BAR_OFF = RANGE_OFF + 16;
    static constexpr int NBARS = 2 + 2 * STG + 3 * 2 + 1;
    static constexpr int HOLD_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = HOLD_OFF + 16 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256;
};

template <int D, int G, bool COPY>
__global__ void __launch_bounds__(DKV_TC_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                          const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ CUtensorMap k16map, const AttnBwdParams p)
{
    using C = BqCfg<D>;
    constexpr int UNITS = C::ROWS / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *q_full = bars;                    // raw query and dO tiles landed
    uint64_t *q_conv = bars + 1;                // q prepared
    uint64_t *kv_full = bars + 2;               // [STG] key block landed
    uint64_t *kv_empty = bars + 2 + C::STG;     // [STG] key block released
    uint64_t *s_full = bars + 2 + 2 * C::STG;   // [2] S (and dP) of a block complete
    uint64_t *buf_free = s_full + 2;            // [2] S / dP buffer may be overwritten
    uint64_t *p_full = s_full + 4;              // [2] dS written (pass 2)
    uint64_t *dq_final = s_full + 6;            // dQ complete
    float *red = reinterpret_cast<float *>(smem + C::RED_OFF);
    int *krange = reinterpret_cast<int *>(smem + C::RANGE_OFF);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::HOLD_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u0 = blockIdx.x * UNITS, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;

    // ---- each row's position and the CTA's key range
    if (threadIdx.x == 0) {
        krange[0] = 0x7fffffff;
        krange[1] = -1;
    }
    int Prow = -1;
    if (threadIdx.x < C::ROWS)
        Prow = unit_pos<COPY>(p, b, u0 + static_cast<int>(threadIdx.x) / G);
    if (COPY && threadIdx.x < C::ROWS && Prow < 0 && u0 + static_cast<int>(threadIdx.x) / G < p.n_units &&
        threadIdx.x % G == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_POSITION);
    const int wlo = __reduce_min_sync(0xffffffffu, Prow >= 0 ? max(0, Prow - p.window + 1) : 0x7fffffff);
    const int whi = __reduce_max_sync(0xffffffffu, Prow);
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_conv, DKV_TC_CONV / 32);
        for (int s = 0; s < C::STG; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int u = 0; u < 2; ++u) {
            mbar_init(&s_full[u], 1);
            mbar_init(&buf_free[u], 4);
            mbar_init(&p_full[u], 4);
        }
        mbar_init(dq_final, 1);
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < 2 * G * C::RS; i += DKV_TC_THREADS)
        red[i] = 0.f;
    if (warp == 1)
        tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    if (lane == 0 && whi >= 0) {
        atomicMin(&krange[0], wlo);
        atomicMax(&krange[1], whi);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;
    int kb0 = krange[1] >= 0 ? krange[0] / C::KB : 0;
    int nb = krange[1] >= 0 ? krange[1] / C::KB - kb0 + 1 : 0;  // key blocks
    const int mode = p.split_mode;
    if (mode != 0) {  // this CTA's share of the key blocks
        const int chunk = (nb + p.splits - 1) / p.splits, z = static_cast<int>(blockIdx.z);
        kb0 += z * chunk;
        nb = max(0, min(chunk, nb - z * chunk));
    }
    // steps n = 0 .. nsteps - 1: pass 1 (log-sum-exp; skipped when it is known) over the
    // blocks, then pass 2 over them again (none in mode 1)
    const int n1 = (p.lse_in != nullptr || mode == 2) ? 0 : nb;
    const int nsteps = mode == 1 ? nb : n1 + nb;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0 && nb > 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&omap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            tma_prefetch_desc(&k16map);
            mbar_arrive_expect_tx(q_full, 2 * C::SLABS * C::QSLAB);
#pragma unroll
            for (int sl = 0; sl < C::SLABS; ++sl) {
                tma_load_4d(smem + C::Q16_OFF + sl * C::QSLAB, &qmap, q_full, sl * 64, g * G, u0, b);
                tma_load_4d(smem + C::DO_OFF + sl * C::QSLAB, &omap, q_full, sl * 64, g * G, u0, b);
            }
        }
        for (int n = 0; n < nsteps; ++n) {
            const bool pass2 = n >= n1;
            const int slot = n % C::STG, kb = kb0 + (pass2 ? n - n1 : n);
            if (n >= C::STG && !(ok = warp_wait(&kv_empty[slot], static_cast<uint32_t>(((n / C::STG) - 1) & 1))))
                break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&kv_full[slot], (pass2 ? 3 : 1) * C::SLABS * C::KSLAB);
#pragma unroll
                for (int sl = 0; sl < C::SLABS; ++sl) {
                    tma_load_4d(smem + C::K16_OFF + (slot * C::SLABS + sl) * C::KSLAB, &k16map, &kv_full[slot], sl * 64,
                                g, kb * C::KB, b);
                    if (pass2) {
                        tma_load_4d(smem + C::K_OFF + (slot * C::SLABS + sl) * C::KSLAB, &kmap, &kv_full[slot], sl * 64,
                                    g, kb * C::KB, b);
                        tma_load_4d(smem + C::V_OFF + (slot * C::SLABS + sl) * C::KSLAB, &vmap, &kv_full[slot],
                                    sl * 64, g, kb * C::KB, b);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        constexpr uint32_t IDESC_S = umma_idesc(128, C::KB, false, false);   // fp16
        constexpr uint32_t IDESC_DP = umma_idesc(128, C::KB, true, false);   // bf16
        constexpr uint32_t IDESC_DQ = umma_idesc(128, D, true, true);
        const uint64_t qdesc = umma_desc_sw128(sbase + C::Q16_OFF, 16, 1024);
        const uint64_t odesc = umma_desc_sw128(sbase + C::DO_OFF, 16, 1024);
        // dQ += dS K of pass-2 block n
        auto issue_dq = [&](int n) -> bool {
            const int u = n & 1, slot = n % C::STG;
            if (!warp_wait(&p_full[u], static_cast<uint32_t>(((n - n1) >> 1) & 1)))
                return false;
            if (lane == 0) {
                tc_fence_after();
                const uint64_t kdesc = umma_desc_sw128(sbase + C::K_OFF + slot * C::SLABS * C::KSLAB, C::KSLAB, 1024);
#pragma unroll
                for (int kk = 0; kk < C::KB / 16; ++kk)
                    umma_ts(tbase + C::TM_DQ, tbase + C::TM_DP + 64 * u + 8 * kk,
                            kdesc + static_cast<uint64_t>(kk * (2048 >> 4)), IDESC_DQ, (n > n1 || kk > 0) ? 1u : 0u);
                // buf_free counts 4 arrivals (the four softmax warps in pass 1): here the
                // commit completes the phase once the dQ MMAs are done, after 3 plain arrivals
                umma_commit(&buf_free[u]);
                mbar_arrive_cnt(&buf_free[u], 3);
                umma_commit(&kv_empty[slot]);
            }
            __syncwarp();
            return true;
        };
        if (nb > 0)
            ok = warp_wait(q_full, 0) && warp_wait(q_conv, 0);
        for (int n = 0; ok && n < nsteps; ++n) {
            const int slot = n % C::STG, u = n & 1;
            const bool pass2 = n >= n1;
            if (!(ok = warp_wait(&kv_full[slot], static_cast<uint32_t>((n / C::STG) & 1))))
                break;
            if (n >= 2 && !(ok = warp_wait(&buf_free[u], static_cast<uint32_t>(((n - 2) >> 1) & 1))))
                break;
            if (lane == 0) {
                tc_fence_after();
                const uint64_t kdesc = umma_desc_sw128(sbase + C::K16_OFF + slot * C::SLABS * C::KSLAB, 16, 1024);
                const uint64_t vdesc = umma_desc_sw128(sbase + C::V_OFF + slot * C::SLABS * C::KSLAB, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = static_cast<uint32_t>((kk >> 2) * C::QSLAB + (kk & 3) * 32) >> 4;
                    const uint32_t ko = static_cast<uint32_t>((kk >> 2) * C::KSLAB + (kk & 3) * 32) >> 4;
                    umma_ss(tbase + C::TM_S + 64 * u, qdesc + qo, kdesc + ko, IDESC_S, kk != 0);
                    if (pass2)
                        umma_ss(tbase + C::TM_DP + 64 * u, odesc + qo, vdesc + ko, IDESC_DP, kk != 0);
                }
                umma_commit(&s_full[u]);
                if (!pass2)
                    umma_commit(&kv_empty[slot]);  // pass 1 reads K only through S
            }
            __syncwarp();
            if (n > n1 && !(ok = issue_dq(n - 1)))
                break;
        }
        if (ok && nsteps > n1) {  // there is a pass 2: the last block's dQ
            ok = issue_dq(nsteps - 1);
            if (ok && lane == 0)
                umma_commit(dq_final);
            __syncwarp();
        }
    } else if (warp < 4 || warp >= 8) {
        // ------------------------------------------------------------------ query preparation
        const int ct = warp < 4 ? threadIdx.x - 64 : threadIdx.x - 256 + 64;  // 0..191
        bool bad = false;
        if (nb > 0 && (ok = warp_wait(q_full, 0))) {
#pragma unroll 2
            for (int idx = ct; idx < C::ROWS * C::SLABS * 8; idx += DKV_TC_CONV) {
                const int row = idx / (C::SLABS * 8), rem = idx % (C::SLABS * 8);
                const int sl = rem / 8, c8 = rem % 8;
                const int h = g * G + row % G, d0 = sl * 64 + c8 * 8;
                uint4 *qp = reinterpret_cast<uint4 *>(smem + C::Q16_OFF + sl * C::QSLAB + sw128_offset(row, c8));
                uint4 q16, qb;
                scale_offset8(*qp, p.alpha + h * D, p.beta + h * D, d0, q16, qb, bad);
                *qp = q16;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(q_conv);
        }
        if (bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
    } else {
        // ------------------------------------------------------------------ softmax + epilogue
        const int rw = warp - 4;
        const int r = rw * 32 + lane;  // row of the tile = tensor-memory lane
        const int P = unit_pos<COPY>(p, b, u0 + r / G);
        const int lo = P - p.window + 1;
        const int uu = u0 + r / G, h = g * G + r % G;
        const long long ri = (static_cast<long long>(b) * p.n_units + uu) * p.Hq + h;
        const float Drow = P >= 0 ? p.Drow[ri] : 0.f;
        const uint32_t tl = tbase + (static_cast<uint32_t>(rw * 32) << 16);
        const float c2 = p.scale * kLog2eF;
        const float NEG_INF = -__int_as_float(0x7f800000);
        float m = NEG_INF, l = 0.f;
        // known beforehand (log2 units): from the forward via the rows kernel, or the split combine
        float lse = ((p.lse_in != nullptr || mode == 2) && P >= 0) ? p.lse[ri] : 0.f;
        bool kshift_bad = false;
        for (int n = 0; ok && n < nsteps; ++n) {
            const int u = n & 1;
            const bool pass2 = n >= n1;
            const int k0 = (kb0 + (pass2 ? n - n1 : n)) * C::KB;
            const bool kshift = p.kflag[static_cast<long long>(bh) * p.nkb + k0 / 64] != 0;  // rare
            if (!(ok = warp_wait(&s_full[u], static_cast<uint32_t>((n >> 1) & 1))))
                break;
            tc_fence_after();
            if (kshift)  // logits of shifted key rows times 2^e_j, in tensor memory
                for (int half = 0; half < 2; ++half)
                    unshift_chunk32(tl + C::TM_S + 64 * u + 32 * half, p.kexp + static_cast<long long>(bh) * p.nkb * 64 + k0,
                                    32 * half, 1u, 1, 1, kshift_bad);
            if (!pass2) {
                uint32_t sa[32], sb[32];
                tmem_ld32(tl + C::TM_S + 64 * u, sa);
                tmem_ld32(tl + C::TM_S + 64 * u + 32, sb);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&buf_free[u]);  // this warp has read its lanes of S (4 arrivals)
                float mb = NEG_INF;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int ka = k0 + c, kb = k0 + 32 + c;
                    const float va = (ka <= P && ka >= lo) ? __uint_as_float(sa[c]) * c2 : NEG_INF;
                    const float vb = (kb <= P && kb >= lo) ? __uint_as_float(sb[c]) * c2 : NEG_INF;
                    sa[c] = __float_as_uint(va);
                    sb[c] = __float_as_uint(vb);
                    mb = fmax3(mb, va, vb);
                }
                const float mn = fmaxf(m, mb);
                const float z = mn == NEG_INF ? 0.f : mn;
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    acc += fast_exp2(__uint_as_float(sa[c]) - z) + fast_exp2(__uint_as_float(sb[c]) - z);
                l = l * fast_exp2(m - z) + acc;
                m = mn;
                if (n == n1 - 1 && mode == 0) {
                    lse = P >= 0 ? m + __log2f(l) : 0.f;  // every valid row holds its own key
                    if (P >= 0)
                        p.lse[ri] = lse;
                }
            } else {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t sv[32], dv[32];
                    tmem_ld32(tl + C::TM_S + 64 * u + 32 * half, sv);
                    tmem_ld32(tl + C::TM_DP + 64 * u + 32 * half, dv);
                    tmem_wait_ld();
                    uint32_t dw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float ds[2];
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int key = k0 + 32 * half + 2 * e + q;
                            const float pr = (key <= P && key >= lo)
                                                 ? fast_exp2(__uint_as_float(sv[2 * e + q]) * c2 - lse)
                                                 : 0.f;
                            ds[q] = pr * (__uint_as_float(dv[2 * e + q]) - Drow);
                        }
                        dw[e] = pack_bf16x2(ds[0], ds[1]);
                    }
                    tmem_st16(tl + C::TM_DP + 64 * u + 16 * half, dw);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[u]);
            }
        }
        if (kshift_bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
        // ---- epilogue: dq_raw = scale dQ alpha; dalpha, dbeta summed over the warp's rows per head
        if (mode == 1 && ok)  // this split's (max, sum) of every row of the tile (log2 units)
            p.part_ml[(static_cast<long long>(bh) * p.splits + blockIdx.z) * C::ROWS + r] = make_float2(m, l);
        const bool have = ok && nsteps > n1;  // a pass 2 ran: dQ is in tensor memory
        const bool any_live = __any_sync(0xffffffffu, uu < p.n_units);
        // mode 0 writes every live row (zeros without keys); mode 2 adds its split's share
        const bool write = mode == 0 ? any_live : (mode == 2 && have && any_live);
        if (have && !(ok = warp_wait(dq_final, 0))) {
        } else if (write) {
            if (have)
                tc_fence_after();
            const long long off = ri * D;
            const bool live = uu < p.n_units;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t w[32];
                if (have) {
                    tmem_ld32(tl + C::TM_DQ + c, w);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        w[e] = 0u;
                }
                float dqv[32], xv[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    dqv[e] = __uint_as_float(w[e]) * p.scale;
                if (live && P >= 0) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        const uint4 x4 = *reinterpret_cast<const uint4 *>(p.q + off + c + e);
                        const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = unpack_bf16x2(xw[q]);
                            xv[e + 2 * q] = f.x;
                            xv[e + 2 * q + 1] = f.y;
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        xv[e] = 0.f;
                }
                if (live) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 al = __ldg(reinterpret_cast<const float4 *>(p.alpha + h * D + c + e));
                        const float4 y =
                            make_float4(dqv[e] * al.x, dqv[e + 1] * al.y, dqv[e + 2] * al.z, dqv[e + 3] * al.w);
                        float *dst = p.dq + off + c + e;
                        if (mode == 2) {  // dq_raw is linear in dQ: the splits add up (dq zeroed first)
                            atomicAdd(dst, y.x);
                            atomicAdd(dst + 1, y.y);
                            atomicAdd(dst + 2, y.z);
                            atomicAdd(dst + 3, y.w);
                        } else {
                            *reinterpret_cast<float4 *>(dst) = y;
                        }
                    }
                }
                // rows of one head are the lanes congruent mod G: butterfly over the other bits
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float sa = xv[e] * dqv[e], sb = dqv[e];
#pragma unroll
                    for (int o = G; o < 32; o <<= 1) {
                        sa += __shfl_xor_sync(0xffffffffu, sa, o);
                        sb += __shfl_xor_sync(0xffffffffu, sb, o);
                    }
                    if (lane < G) {
                        atomicAdd(&red[lane * C::RS + c + e], sa);
                        atomicAdd(&red[(G + lane) * C::RS + c + e], sb);
                    }
                }
            }
        }
        named_barrier(1, 128);  // every softmax warp reaches this point (all waits are bounded)
        for (int i = r; i < G * D; i += 128) {
            const int hh = i / D, dd = i % D;
            atomicAdd(p.dalpha + g * G * D + i, red[hh * C::RS + dd]);
            atomicAdd(p.dbeta + g * G * D + i, red[(G + hh) * C::RS + dd]);
        }
    }
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ------------------------------------------------------------------ base-stream dQ, persistent

// The base stream's rows see at most w + 128/G keys (two to four 64-key blocks per tile of
// 128 rows), so a CTA per tile would spend most of its time on set-up, loads and the
// epilogue.  Here one CTA per SM walks a contiguous run of row tiles with the forward's
// log-sum-exp given (pass 2 only), and overlaps them: two dQ accumulators in tensor memory
// let the epilogue of tile i run while tile i + 1's MMAs do, and tile i + 1's q / dO load
// lands in the other of two query buffers while tile i computes.  Per key block (64 keys,
// through a two-stage ring, so that the two query buffers fit in shared memory beside it)
// as in the dq kernel above: S = q K16^T (fp16), dP = dO V^T, dS = P (dP - D) over dP as
// bf16, dQ += dS K.
// The query tile arrives as fp16 q = x alpha + beta, made for the whole tensor beforehand
// (attn_bwd_rows_kernel), and dalpha / dbeta are summed afterwards from dq_raw
// (attn_bwd_dab_kernel): both were measured to pace this kernel when done per tile here
// (q preparation 7.8 us and the per-head butterfly 14.6 us of a 21 us tile).
// Roles (384 threads): warp 0 TMA producer; warp 1 tensor-memory allocation and MMA issue;
// warps 4-7 dS (lane = row); warps 8-11 the epilogue (lane = row: the same tensor-memory
// lanes), so that one tile's epilogue runs beside the next tile's dS; warps 2-3 idle.
// Tensor memory: S at 64 u, dP at 128 + 64 u (block buffer u of 2), dQ at 256 + D t (tile
// buffer t).
template <int D>
struct BpCfg {
    static constexpr int ROWS = 128;
    static constexpr int KB = 64;
    static constexpr int SLABS = D / 64;
    static constexpr int STG = 2;
    static constexpr int QSLAB = ROWS * 128;
    static constexpr int KSLAB = KB * 128;
    static constexpr int QBUF = 2 * SLABS * QSLAB;                 // one query buffer: q, dO
    static constexpr int Q16_OFF = 0;                              // [2] q as fp16
    static constexpr int DO_OFF = Q16_OFF + SLABS * QSLAB;         // [2] dO (QBUF apart)
    static constexpr int K_OFF = 2 * QBUF;                         // [STG] K blocks (bf16)
    static constexpr int V_OFF = K_OFF + STG * SLABS * KSLAB;      // [STG] V blocks
    static constexpr int K16_OFF = V_OFF + STG * SLABS * KSLAB;    // [STG] K blocks as fp16
    static constexpr int BAR_OFF = K16_OFF + STG * SLABS * KSLAB;
    static constexpr int NBUF = 2;                                 // S / dP buffers
    static constexpr int NBARS = 2 * 2 + 2 * STG + 3 * NBUF + 2 * 2;
    static constexpr int HOLD_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = HOLD_OFF + 16 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static constexpr uint32_t TM_S = 0, TM_DP = NBUF * KB, TM_DQ = 2 * NBUF * KB;
};

template <int D, int G>
__global__ void __launch_bounds__(DKV_TC_THREADS, 1)
    attn_bwd_dq_tc_base_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                               const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                               const __grid_constant__ CUtensorMap k16map, const AttnBwdParams p)
{
    using C = BpCfg<D>;
    constexpr int UNITS = C::ROWS / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *q_full = bars;                     // [2] a tile's fp16 q and dO landed
    uint64_t *q_free = bars + 2;                 // [2] a tile's last S, dP done: the buffer may be reloaded
    uint64_t *kv_full = bars + 4;                // [STG] key block landed
    uint64_t *kv_empty = kv_full + C::STG;       // [STG] key block released
    uint64_t *s_full = kv_empty + C::STG;        // [NBUF] S, dP of a block complete
    uint64_t *buf_free = s_full + C::NBUF;       // [NBUF] S / dP buffer may be overwritten
    uint64_t *p_full = buf_free + C::NBUF;       // [NBUF] dS written
    uint64_t *dq_final = p_full + C::NBUF;       // [2] a tile's dQ complete
    uint64_t *dq_free = dq_final + 2;            // [2] a tile's dQ read by the epilogue
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::HOLD_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's tiles: a contiguous run of (batch, KV head, 128-row tile) in that order
    const int n_xt = (p.n_units + UNITS - 1) / UNITS;
    const long long n_tiles = static_cast<long long>(p.B) * p.Hkv * n_xt;
    const long long per = (n_tiles + gridDim.x - 1) / gridDim.x;
    const long long t_begin = blockIdx.x * per, t_end = min(n_tiles, t_begin + per);
    // tile tau: sequence b, KV head g, first unit u0, key blocks kb0 .. kb0 + nb - 1
    auto tile = [&](long long tau, int &b, int &g, int &u0, int &kb0, int &nb) {
        const int bh = static_cast<int>(tau / n_xt);
        b = bh / p.Hkv;
        g = bh % p.Hkv;
        u0 = static_cast<int>(tau % n_xt) * UNITS;
        const int klo = max(0, u0 - p.window + 1), khi = min(p.n_units, u0 + UNITS) - 1;
        kb0 = klo / C::KB;
        nb = khi / C::KB - kb0 + 1;
    };

    if (threadIdx.x == 0) {
        for (int qb = 0; qb < 2; ++qb) {
            mbar_init(&q_full[qb], 1);
            mbar_init(&q_free[qb], 1);
        }
        for (int s = 0; s < C::STG; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int u = 0; u < C::NBUF; ++u) {
            mbar_init(&s_full[u], 1);
            mbar_init(&buf_free[u], 1);
            mbar_init(&p_full[u], 4);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&dq_final[t], 1);
            mbar_init(&dq_free[t], 4);
        }
        fence_barrier_init();
    }
    if (warp == 1)
        tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&omap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            tma_prefetch_desc(&k16map);
        }
        long long n = 0;  // key blocks issued so far, over all tiles
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            int b, g, u0, kb0, nb;
            tile(tau, b, g, u0, kb0, nb);
            const int qb = static_cast<int>(i & 1);
            // query buffer qb is free once tile i - 2's last S, dP products are done
            if (i >= 2 && !(ok = warp_wait(&q_free[qb], static_cast<uint32_t>(((i - 2) >> 1) & 1))))
                break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&q_full[qb], 2 * C::SLABS * C::QSLAB);
#pragma unroll
                for (int sl = 0; sl < C::SLABS; ++sl) {
                    tma_load_4d(smem + qb * C::QBUF + C::Q16_OFF + sl * C::QSLAB, &qmap, &q_full[qb], sl * 64, g * G,
                                u0, b);
                    tma_load_4d(smem + qb * C::QBUF + C::DO_OFF + sl * C::QSLAB, &omap, &q_full[qb], sl * 64, g * G,
                                u0, b);
                }
            }
            for (int j = 0; j < nb; ++j, ++n) {
                const int slot = static_cast<int>(n % C::STG);
                if (n >= C::STG && !(ok = warp_wait(&kv_empty[slot], static_cast<uint32_t>(((n / C::STG) - 1) & 1))))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&kv_full[slot], 3 * C::SLABS * C::KSLAB);
                    const int key0 = (kb0 + j) * C::KB;
#pragma unroll
                    for (int sl = 0; sl < C::SLABS; ++sl) {
                        const int o = (slot * C::SLABS + sl) * C::KSLAB;
                        tma_load_4d(smem + C::K16_OFF + o, &k16map, &kv_full[slot], sl * 64, g, key0, b);
                        tma_load_4d(smem + C::K_OFF + o, &kmap, &kv_full[slot], sl * 64, g, key0, b);
                        tma_load_4d(smem + C::V_OFF + o, &vmap, &kv_full[slot], sl * 64, g, key0, b);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        constexpr uint32_t IDESC_S = umma_idesc(128, C::KB, false, false);  // fp16
        constexpr uint32_t IDESC_DP = umma_idesc(128, C::KB, true, false);  // bf16
        constexpr uint32_t IDESC_DQ = umma_idesc(128, D, true, true);
        // dQ[t] (+)= dS K of block m
        auto issue_dq = [&](long long m, bool first, int t) -> bool {
            const int u = static_cast<int>(m % C::NBUF), slot = static_cast<int>(m % C::STG);
            if (!warp_wait(&p_full[u], static_cast<uint32_t>((m / C::NBUF) & 1)))
                return false;
            if (lane == 0) {
                tc_fence_after();
                const uint64_t kdesc = umma_desc_sw128(sbase + C::K_OFF + slot * C::SLABS * C::KSLAB, C::KSLAB, 1024);
#pragma unroll
                for (int kk = 0; kk < C::KB / 16; ++kk)
                    umma_ts(tbase + C::TM_DQ + D * t, tbase + C::TM_DP + C::KB * u + 8 * kk,
                            kdesc + static_cast<uint64_t>(kk * (2048 >> 4)), IDESC_DQ, (!first || kk > 0) ? 1u : 0u);
                umma_commit(&buf_free[u]);
                umma_commit(&kv_empty[slot]);
            }
            __syncwarp();
            return true;
        };
        long long n = 0;
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            int b, g, u0, kb0, nb;
            tile(tau, b, g, u0, kb0, nb);
            const int t = static_cast<int>(i & 1), qb = t;
            const uint32_t qph = static_cast<uint32_t>((i >> 1) & 1);
            if (!(ok = warp_wait(&q_full[qb], qph)))
                break;
            const uint64_t qdesc = umma_desc_sw128(sbase + qb * C::QBUF + C::Q16_OFF, 16, 1024);
            const uint64_t odesc = umma_desc_sw128(sbase + qb * C::QBUF + C::DO_OFF, 16, 1024);
            // dQ[t] is free once the epilogue of tile i - 2 has read it
            if (i >= 2 && !(ok = warp_wait(&dq_free[t], static_cast<uint32_t>(((i - 2) >> 1) & 1))))
                break;
            for (int j = 0; j < nb; ++j, ++n) {
                const int slot = static_cast<int>(n % C::STG), u = static_cast<int>(n % C::NBUF);
                if (!(ok = warp_wait(&kv_full[slot], static_cast<uint32_t>((n / C::STG) & 1))))
                    break;
                // S / dP buffer u is free once the dQ product of block n - NBUF has read dS
                if (n >= C::NBUF &&
                    !(ok = warp_wait(&buf_free[u], static_cast<uint32_t>(((n - C::NBUF) / C::NBUF) & 1))))
                    break;
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t kdesc = umma_desc_sw128(sbase + C::K16_OFF + slot * C::SLABS * C::KSLAB, 16, 1024);
                    const uint64_t vdesc = umma_desc_sw128(sbase + C::V_OFF + slot * C::SLABS * C::KSLAB, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qo = static_cast<uint32_t>((kk >> 2) * C::QSLAB + (kk & 3) * 32) >> 4;
                        const uint32_t ko = static_cast<uint32_t>((kk >> 2) * C::KSLAB + (kk & 3) * 32) >> 4;
                        umma_ss(tbase + C::TM_S + C::KB * u, qdesc + qo, kdesc + ko, IDESC_S, kk != 0);
                        umma_ss(tbase + C::TM_DP + C::KB * u, odesc + qo, vdesc + ko, IDESC_DP, kk != 0);
                    }
                    umma_commit(&s_full[u]);
                    if (j == nb - 1)
                        umma_commit(&q_free[qb]);  // the tile's q and dO are no longer read
                }
                __syncwarp();
                if (j >= 1 && !(ok = issue_dq(n - 1, j == 1, t)))
                    break;
            }
            if (!ok)
                break;
            if (!(ok = issue_dq(n - 1, nb == 1, t)))
                break;
            if (lane == 0)
                umma_commit(&dq_final[t]);
            __syncwarp();
        }
    } else if (warp < 4) {
        // warps 2-3: no role (the query tile arrives prepared)
    } else if (warp < 8) {
        // ------------------------------------------------------------------ dS (lane = row)
        const int rw = warp - 4;
        const int r = rw * 32 + lane;  // row of the tile = tensor-memory lane
        const uint32_t tl = tbase + (static_cast<uint32_t>(rw * 32) << 16);
        const float c2 = p.scale * kLog2eF;
        bool kshift_bad = false;
        long long n = 0;
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            int b, g, u0, kb0, nb;
            tile(tau, b, g, u0, kb0, nb);
            const int uu = u0 + r / G, h = g * G + r % G;
            const bool live = uu < p.n_units;
            const int P = live ? uu : -1, lo = P - p.window + 1;
            const long long ri = (static_cast<long long>(b) * p.n_units + uu) * p.Hq + h;
            const float lse = live ? p.lse[ri] : 0.f;  // log2 units (the rows kernel converted it)
            const float Drow = live ? p.Drow[ri] : 0.f;
            for (int j = 0; j < nb; ++j, ++n) {
                const int u = static_cast<int>(n % C::NBUF);
                const int k0 = (kb0 + j) * C::KB;
                const long long bh = static_cast<long long>(b) * p.Hkv + g;
                const bool kshift = p.kflag[bh * p.nkb + k0 / 64] != 0;  // rare
                if (!(ok = warp_wait(&s_full[u], static_cast<uint32_t>((n / C::NBUF) & 1))))
                    break;
                tc_fence_after();
                if (kshift)  // logits of shifted key rows times 2^e_j, in tensor memory
                    for (int half = 0; half < C::KB / 32; ++half)
                        unshift_chunk32(tl + C::TM_S + C::KB * u + 32 * half, p.kexp + bh * p.nkb * 64 + k0, 32 * half,
                                        1u, 1, 1, kshift_bad);
#pragma unroll
                for (int half = 0; half < C::KB / 32; ++half) {
                    uint32_t sv[32], dv[32];
                    tmem_ld32(tl + C::TM_S + C::KB * u + 32 * half, sv);
                    tmem_ld32(tl + C::TM_DP + C::KB * u + 32 * half, dv);
                    tmem_wait_ld();
                    uint32_t dw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float ds[2];
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int key = k0 + 32 * half + 2 * e + q;
                            const float pr = (key <= P && key >= lo)
                                                 ? fast_exp2(__uint_as_float(sv[2 * e + q]) * c2 - lse)
                                                 : 0.f;
                            ds[q] = pr * (__uint_as_float(dv[2 * e + q]) - Drow);
                        }
                        dw[e] = pack_bf16x2(ds[0], ds[1]);
                    }
                    tmem_st16(tl + C::TM_DP + C::KB * u + 16 * half, dw);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[u]);
            }
        }
        if (kshift_bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
    } else {
        // ------------------------------------------------------------------ epilogue (warps 8-11)
        // dq_raw = scale dQ alpha (dalpha, dbeta follow from it in attn_bwd_dab_kernel)
        const int rw = warp - 8;
        const int r = rw * 32 + lane;  // row of the tile = tensor-memory lane
        const uint32_t tl = tbase + (static_cast<uint32_t>(rw * 32) << 16);
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            int b, g, u0, kb0, nb;
            tile(tau, b, g, u0, kb0, nb);
            const int t = static_cast<int>(i & 1);
            const int uu = u0 + r / G, h = g * G + r % G;
            const bool live = uu < p.n_units;
            const long long off = ((static_cast<long long>(b) * p.n_units + uu) * p.Hq + h) * D;
            if (!(ok = warp_wait(&dq_final[t], static_cast<uint32_t>((i >> 1) & 1))))
                break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t w[32];
                tmem_ld32(tl + C::TM_DQ + D * t + c, w);
                tmem_wait_ld();
                if (live) {  // dq_raw = scale dQ alpha, whole 32-byte sectors per store
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        const float4 a0 = __ldg(reinterpret_cast<const float4 *>(p.alpha + h * D + c + e));
                        const float4 a1 = __ldg(reinterpret_cast<const float4 *>(p.alpha + h * D + c + e + 4));
                        const float sc = p.scale;
                        st_global_v8(p.dq + off + c + e,
                                     make_uint4(__float_as_uint(__uint_as_float(w[e]) * sc * a0.x),
                                                __float_as_uint(__uint_as_float(w[e + 1]) * sc * a0.y),
                                                __float_as_uint(__uint_as_float(w[e + 2]) * sc * a0.z),
                                                __float_as_uint(__uint_as_float(w[e + 3]) * sc * a0.w)),
                                     make_uint4(__float_as_uint(__uint_as_float(w[e + 4]) * sc * a1.x),
                                                __float_as_uint(__uint_as_float(w[e + 5]) * sc * a1.y),
                                                __float_as_uint(__uint_as_float(w[e + 6]) * sc * a1.z),
                                                __float_as_uint(__uint_as_float(w[e + 7]) * sc * a1.w)));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&dq_free[t]);  // this warp's lanes of dQ[t] are read
        }
    }
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ------------------------------------------------------------------ copies' dQ, few rows

// At most 8 copy rows of one (batch, KV head) (one copy of G = 4 heads, say) with the forward's
// log-sum-exp known: a tensor-memory tile would carry 120 empty rows of its 128.  Here the rows
// sit on the warp MMA's N side and 16 keys on M, as in the forward's split-KV kernel:
//   S^T = K q^T (q = (x alpha + beta) scale log2(e) as bf16 high part + residual, so S is in
//   log2 units), dP^T = V dO^T, P^T = exp2(S^T - lse2), dS^T = P^T (dP^T - D) (rounded to bf16),
//   dQ^T += K^T dS^T,
// with K and V read as bf16 straight from the inputs.  Grid (split, 1, batch * KV head); the keys
// 0 .. max(pos) of the CTA's rows are split into chunks of 64-key blocks, which stream through a
// 3-stage TMA ring; warp w takes keys 16 w .. 16 w + 15 of every block, and the four warps' dQ
// are summed through shared memory.  The CTA then adds its share: dq_raw += scale dQ alpha,
// dalpha += x scale dQ, dbeta += scale dQ (all linear in dQ; dq_raw zeroed first unless there is
// one split, which stores it, zeros included for rows without a valid position).
template <int D>
struct BkCfg {
    static constexpr int KB = 64;
    static constexpr int SLAB = KB * 128;
    static constexpr int KV_BYTES = KB * D * 2;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int STAGES = 3;
    static constexpr int CWARPS = 4;
    static constexpr int THREADS = (CWARPS + 1) * 32;
    static constexpr int RMAX = 8;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int MISC_OFF = BAR_OFF + 2 * STAGES * 8;  // int [RMAX] positions
    static constexpr int SMEM = MISC_OFF + RMAX * 4 + 1024;
    static_assert(CWARPS * RMAX * D * 4 <= BAR_OFF, "the dQ merge fits in the ring");
};

template <int D>
__global__ void __launch_bounds__(BkCfg<D>::THREADS)
    attn_bwd_dq_copies_keys_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                                   const AttnBwdParams p)
{
    using C = BkCfg<D>;
    constexpr int RMAX = C::RMAX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    int *s_pos = reinterpret_cast<int *>(smem + C::MISC_OFF);

    const int G = p.Hq / p.Hkv, R = p.n_units * G;
    const int split = blockIdx.x, bh = blockIdx.z;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x < RMAX) {
        const int r = threadIdx.x;
        const int P = r < R ? unit_pos<true>(p, b, r / G) : -1;
        if (r < R && P < 0 && r % G == 0 && split == 0)
            record_error(p.dev_err, ORTHROS_DEVERR_POSITION);
        s_pos[r] = P;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::CWARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();
    int kmax = -1;
    for (int i = 0; i < RMAX; ++i)
        kmax = max(kmax, s_pos[i]);
    const int nbk = (kmax + C::KB) / C::KB;  // blocks of keys 0 .. kmax
    const int per = (nbk + p.splits - 1) / p.splits;
    const int blk0 = split * per, nblk = max(0, min(per, nbk - blk0));

    if (warp == C::CWARPS) {
        // ------------------------------------------------------------------ producer
        if (lane != 0)
            return;
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        for (int i = 0; i < nblk; ++i) {
            const int s = i % C::STAGES;
            if (i >= C::STAGES && !mbar_wait(&empty[s], static_cast<uint32_t>(((i / C::STAGES) - 1) & 1))) {
                record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
                return;
            }
            uint8_t *dst = smem + s * C::STAGE_BYTES;
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
            for (int sl = 0; sl < D / 64; ++sl) {
                tma_load_4d(dst + sl * C::SLAB, &kmap, &full[s], sl * 64, g, (blk0 + i) * C::KB, b);
                tma_load_4d(dst + C::KV_BYTES + sl * C::SLAB, &vmap, &full[s], sl * 64, g, (blk0 + i) * C::KB, b);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // B fragments hold row lane / 4 (q^T high / residual, dO^T); the lane's accumulators hold rows
    // 2 (lane % 4) + {0, 1} and, for dQ^T, d = 16 mt + lane / 4 (+ 8)
    const float c2 = p.scale * kLog2eF;
    uint32_t qb[D / 16][2], ql[D / 16][2], ob[D / 16][2];
    {
        const int row = lane >> 2;
        const bool valid = row < R && s_pos[row] >= 0;
        const int h = g * G + row % G;
        const long long ri = (static_cast<long long>(b) * p.n_units + row / G) * p.Hq + h;
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int dcol = kt * 16 + 2 * (lane & 3) + 8 * hf;
                uint32_t hi = 0, lo = 0, ow = 0;
                if (valid) {
                    load_q_pair(p.q + ri * D, p.alpha + h * D, p.beta + h * D, dcol, c2, hi, lo);
                    ow = __ldg(reinterpret_cast<const unsigned int *>(p.dO + ri * D + dcol));
                }
                qb[kt][hf] = hi;
                ql[kt][hf] = lo;
                ob[kt][hf] = ow;
            }
    }
    int lim[2];
    float lse2[2], Dr[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int row = 2 * (lane & 3) + i;
        const int P = row < R ? s_pos[row] : -1;
        lim[i] = P;
        const long long ri = (static_cast<long long>(b) * p.n_units + row / G) * p.Hq + g * G + row % G;
        lse2[i] = P >= 0 ? p.lse[ri] : 0.f;
        Dr[i] = P >= 0 ? p.Drow[ri] : 0.f;
    }
    float dq[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
        dq[mt][0] = dq[mt][1] = dq[mt][2] = dq[mt][3] = 0.f;
    // ldmatrix rows: A of K and of V (16 keys x 16 d, row-major), A of K^T (16 d x 16 keys)
    const int ka_row = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), ka_hi = lane >> 4;
    const int ta_row = warp * 16 + (lane & 7) + ((lane >> 4) << 3), ta_hi = (lane >> 3) & 1;

    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
        const int s = i % C::STAGES;
        if (!mbar_wait(&full[s], static_cast<uint32_t>((i / C::STAGES) & 1))) {
            ok = false;
            break;
        }
        const uint32_t kbase = sbase + s * C::STAGE_BYTES, vbase = kbase + C::KV_BYTES;
        const int j0 = (blk0 + i) * C::KB + warp * 16;
        if (j0 <= kmax) {
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kt = 0; kt < D / 16; ++kt) {
                uint32_t a[4], v[4];
                const uint32_t off = (kt * 16 / 64) * C::SLAB + sw128_offset(ka_row, ((kt * 16) % 64) / 8 + ka_hi);
                ldsm_x4(kbase + off, a[0], a[1], a[2], a[3]);
                ldsm_x4(vbase + off, v[0], v[1], v[2], v[3]);
                float *s1 = (kt & 1) ? sb : sa, *d1 = (kt & 1) ? db : da;
                mma_16816(s1, a, qb[kt][0], qb[kt][1]);
                mma_16816(s1, a, ql[kt][0], ql[kt][1]);
                mma_16816(d1, v, ob[kt][0], ob[kt][1]);
            }
            // element e: key j0 + lane / 4 + 8 (e >> 1), row 2 (lane % 4) + (e & 1)
            float ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = j0 + (lane >> 2) + ((e >> 1) << 3), ri = e & 1;
                const float pr = key <= lim[ri] ? fast_exp2(sa[e] + sb[e] - lse2[ri]) : 0.f;
                ds[e] = pr * (da[e] + db[e] - Dr[ri]);
            }
            const uint32_t b0 = movmatrix_trans(pack_bf16x2(ds[0], ds[1]));
            const uint32_t b1 = movmatrix_trans(pack_bf16x2(ds[2], ds[3]));
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                uint32_t a[4];
                ldsm_x4_trans(kbase + (mt * 16 / 64) * C::SLAB + sw128_offset(ta_row, ((mt * 16) % 64) / 8 + ta_hi),
                              a[0], a[1], a[2], a[3]);
                mma_16816(dq[mt], a, b0, b1);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[s]);
    }
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);

    // the four warps' dQ^T summed through shared memory (the ring is free once every warp is past
    // its last block), then this CTA's share added to the outputs
    constexpr int CT = C::CWARPS * 32;
    float *os = reinterpret_cast<float *>(smem);  // [CWARPS][RMAX][D]
    named_barrier(2, CT);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float *po = os + (warp * RMAX + 2 * (lane & 3) + i) * D + (lane >> 2);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            po[16 * mt] = dq[mt][i];
            po[16 * mt + 8] = dq[mt][2 + i];
        }
    }
    named_barrier(2, CT);
    for (int i = threadIdx.x; i < R * D; i += CT) {
        const int row = i / D, c = i % D;
        const int h = g * G + row % G;
        const long long ri = (static_cast<long long>(b) * p.n_units + row / G) * p.Hq + h;
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < C::CWARPS; ++w)
            a += os[(w * RMAX + row) * D + c];
        const float dqv = s_pos[row] >= 0 ? a * p.scale : 0.f;
        if (p.splits == 1) {
            p.dq[ri * D + c] = dqv * p.alpha[h * D + c];
        } else if (s_pos[row] >= 0) {
            atomicAdd(p.dq + ri * D + c, dqv * p.alpha[h * D + c]);
        }
        if (s_pos[row] >= 0) {
            const float x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(p.q)[ri * D + c]) << 16);
            atomicAdd(p.dalpha + h * D + c, x * dqv);
            atomicAdd(p.dbeta + h * D + c, dqv);
        }
    }
}

// ------------------------------------------------------------------ base-stream dQ over the key band

// Persistent like the kernel above, but a row tile's whole key band is one MMA wide.  Keys stream
// through a ring of NSLOT 32-key slots (block kb in load order n sits in slot n % NSLOT); a tile's
// band (at most NSLOT - 1 blocks, so that the next tile's first new block loads meanwhile) is a
// run of consecutive loads.  S = q K16^T and dP = dO V^T each take one N = 32 * NSLOT product per
// K step over the whole ring: columns of slots outside the band are never read.  dS (fp16) is
// written over dP and dQ = dS K16 runs from tensor memory, 16 keys per K step, over the band's
// slots only.  The fp16 copy of K holds k * 2^-e for the rare key rows beyond fp16: their logits
// are scaled back by 2^e in tensor memory and their dS columns by 2^e before the fp16 rounding
// (|dS 2^e| >= 65504 sets ORTHROS_DEVERR_RANGE).  With FOLD the epilogue also sums
// dalpha = sum x * dq and dbeta = sum dq over the CTA's rows (lanes of one head reduce-scatter
// each 32-column chunk, so each lane owns G columns of its head; global atomics when the KV
// head changes and at the end).
// Roles (512 threads): warp 0 TMA producer, warp 1 tensor-memory allocation and MMA issue,
// warps 4-7 and 8-11 dS (lane = row; the first group slots 0-2 of the ring, the second slots
// 3-5, each writing its dS over its own slots' dP columns) and, once a tile's dQ is done, the
// dalpha / dbeta sums over their half of the columns (FOLD); warps 12-15 store dq_raw (the same
// lanes); warps 2-3 idle.
// Tensor memory: S at 0, dP (then dS) at N, dQ at 2 N.
template <int D>
struct BbCfg {
    static constexpr int ROWS = 128;
    static constexpr int KB = 32;                      // keys per slot
    static constexpr int NSLOT = 6;
    static constexpr int N = KB * NSLOT;               // S / dP columns
    static constexpr int SLABS = D / 64;
    static constexpr int QSLAB = ROWS * 128;
    static constexpr int SLOT = KB * 128;              // one slot of one 64-column slab
    static constexpr int RSLAB = NSLOT * SLOT;         // one 64-column slab of a ring
    static constexpr int QBUF = 2 * SLABS * QSLAB;     // the query buffer: fp16 q, dO
    static constexpr int Q16_OFF = 0;
    static constexpr int DO_OFF = SLABS * QSLAB;
    static constexpr int DQS_OFF = QBUF;               // dq_raw staging: D / 32 tiles of ROWS x 128 B
    static constexpr int DQS_TILE = ROWS * 128;
    static_assert((D / 32) * DQS_TILE == QBUF, "the staging tiles fill the second buffer");
    static constexpr int K16_OFF = 2 * QBUF;           // ring of the fp16 K
    static constexpr int V_OFF = K16_OFF + SLABS * RSLAB;
    static constexpr int BAR_OFF = V_OFF + SLABS * RSLAB;
    static constexpr int NBARS = 2 + 2 + 2 * NSLOT + 4;
    static constexpr int HOLD_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = HOLD_OFF + 16 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static constexpr uint32_t TM_S = 0, TM_DP = N, TM_DQ = 2 * N;
    static_assert(TM_DQ + D <= 512, "tensor memory budget");
    static constexpr int THREADS = 512;
    // dS of slot j (16 packed fp16 pairs) over dP columns of its own dS group's slots:
    // slots 0-2 at 16 j (dP slots 0-1), slots 3-5 at 48 + 16 j (dP slots 3-4)
    static __device__ __forceinline__ uint32_t ds_col(int j) { return static_cast<uint32_t>(j < 3 ? 16 * j : 48 + 16 * j); }
};

// The band of a CTA's tiles in load order: tiles run in (batch, KV head, row tile) order, so
// within one (batch, KV head) each tile loads the blocks past the previous tile's band; a new
// (batch, KV head) loads its whole band.  Every role steps one of these through the same tiles.
struct BandRun {
    int bh = -1, hi = -1;
    long long nh = -1;  // load index of the current band's last block
    // step to a tile with band blocks lo..hi of sequence bh; returns the first block to load
    __device__ __forceinline__ int step(int bh_t, int lo, int hi_t)
    {
        const int first = (bh_t == bh && hi >= lo) ? hi + 1 : lo;
        nh += hi_t - first + 1;
        bh = bh_t;
        hi = hi_t;
        return first;
    }
};

template <int D, int G, bool FOLD>
__global__ void __launch_bounds__(BbCfg<D>::THREADS, 1)
    attn_bwd_dq_band_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                            const __grid_constant__ CUtensorMap k16map, const __grid_constant__ CUtensorMap vmap,
                            const __grid_constant__ CUtensorMap dqmap, const AttnBwdParams p)
{
    using C = BbCfg<D>;
    constexpr int UNITS = C::ROWS / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *q_full = bars;                     // a tile's fp16 q and dO landed (one phase per tile)
    uint64_t *q_free = bars + 2;                 // a tile's S, dP done: the buffer may be reloaded
    uint64_t *kv_full = bars + 4;                // [NSLOT] block landed
    uint64_t *kv_empty = kv_full + C::NSLOT;     // [NSLOT] block no longer read
    uint64_t *s_full = kv_empty + C::NSLOT;      // S, dP of a tile complete
    uint64_t *p_full = s_full + 1;               // dS written (and S read)
    uint64_t *dq_final = s_full + 2;             // dQ of a tile complete (dS read)
    uint64_t *dq_free = s_full + 3;              // dQ read by the epilogue
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::HOLD_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_xt = (p.n_units + UNITS - 1) / UNITS;
    const long long n_tiles = static_cast<long long>(p.B) * p.Hkv * n_xt;
    const long long per = (n_tiles + gridDim.x - 1) / gridDim.x;
    const long long t_begin = blockIdx.x * per, t_end = min(n_tiles, t_begin + per);
    // tile tau: sequence bh = b * Hkv + g, first unit u0, band blocks lo .. hi
    auto tile = [&](long long tau, int &bh, int &u0, int &lo, int &hi) {
        bh = static_cast<int>(tau / n_xt);
        u0 = static_cast<int>(tau % n_xt) * UNITS;
        lo = max(0, u0 - p.window + 1) / C::KB;
        hi = (min(p.n_units, u0 + UNITS) - 1) / C::KB;
    };

    if (threadIdx.x == 0) {
        for (int qb = 0; qb < 2; ++qb) {
            mbar_init(&q_full[qb], 1);
            mbar_init(&q_free[qb], 1);
        }
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, 8);
        mbar_init(dq_final, 1);
        mbar_init(dq_free, FOLD ? 12 : 4);  // the store warps, and the dS warps once they have summed
        fence_barrier_init();
    }
    if (warp == 1)
        tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&omap);
            tma_prefetch_desc(&k16map);
            tma_prefetch_desc(&vmap);
        }
        BandRun run;
        long long n = 0;  // blocks loaded so far
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            int bh, u0, lo, hi;
            tile(tau, bh, u0, lo, hi);
            const int first = run.step(bh, lo, hi);
            const int b = bh / p.Hkv, g = bh % p.Hkv;
            // the single query buffer is free once tile i - 1's S, dP are done, well before the
            // slot of this tile's new key block (freed by tile i - 1's dQ): q goes first
            if (i >= 1 && !(ok = warp_wait(q_free, static_cast<uint32_t>((i - 1) & 1))))
                break;
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full, 2 * C::SLABS * C::QSLAB);
#pragma unroll
                for (int sl = 0; sl < C::SLABS; ++sl) {
                    tma_load_4d(smem + C::Q16_OFF + sl * C::QSLAB, &qmap, q_full, sl * 64, g * G, u0, b);
                    tma_load_4d(smem + C::DO_OFF + sl * C::QSLAB, &omap, q_full, sl * 64, g * G, u0, b);
                }
            }
            for (int kb = first; kb <= hi; ++kb, ++n) {
                const int slot = static_cast<int>(n % C::NSLOT);
                // the slot's previous block (load n - NSLOT) is released after the dQ of its last tile
                if (n >= C::NSLOT &&
                    !(ok = warp_wait(&kv_empty[slot], static_cast<uint32_t>(((n / C::NSLOT) - 1) & 1))))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&kv_full[slot], 2 * C::SLABS * C::SLOT);
#pragma unroll
                    for (int sl = 0; sl < C::SLABS; ++sl) {
                        const int o = sl * C::RSLAB + slot * C::SLOT;
                        tma_load_4d(smem + C::K16_OFF + o, &k16map, &kv_full[slot], sl * 64, g, kb * C::KB, b);
                        tma_load_4d(smem + C::V_OFF + o, &vmap, &kv_full[slot], sl * 64, g, kb * C::KB, b);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        constexpr uint32_t IDESC_S = umma_idesc(128, C::N, false, false);  // fp16
        constexpr uint32_t IDESC_DP = umma_idesc(128, C::N, true, false);  // bf16
        constexpr uint32_t IDESC_DQ = umma_idesc(128, D, false, true);     // fp16 dS, K16 MN-major
        const uint64_t kdesc = umma_desc_sw128(sbase + C::K16_OFF, 16, 1024);
        const uint64_t vdesc = umma_desc_sw128(sbase + C::V_OFF, 16, 1024);
        BandRun run, ahead;
        long long n = 0, released = 0;  // blocks whose arrival was awaited; blocks released
        bool have_next = false;
        int nbh = 0, nu0 = 0, nlo = 0, nhi = 0;
        if (t_begin < t_end) {
            tile(t_begin, nbh, nu0, nlo, nhi);
            have_next = true;
        }
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            const int bh = nbh, lo = nlo, hi = nhi;
            const int first = run.step(bh, lo, hi);
            const long long nf = run.nh - (hi - lo);  // load index of block lo
            have_next = tau + 1 < t_end;
            if (have_next)
                tile(tau + 1, nbh, nu0, nlo, nhi);
            if (!(ok = warp_wait(q_full, static_cast<uint32_t>(i & 1))))
                break;
            for (int kb = first; ok && kb <= hi; ++kb, ++n)
                ok = warp_wait(&kv_full[n % C::NSLOT], static_cast<uint32_t>((n / C::NSLOT) & 1));
            if (!ok)
                break;
            const uint64_t qdesc = umma_desc_sw128(sbase + C::Q16_OFF, 16, 1024);
            const uint64_t odesc = umma_desc_sw128(sbase + C::DO_OFF, 16, 1024);
            if (lane == 0) {  // S over the whole ring (S was read by the dS of tile i - 1)
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = static_cast<uint32_t>((kk >> 2) * C::QSLAB + (kk & 3) * 32) >> 4;
                    const uint32_t ko = static_cast<uint32_t>((kk >> 2) * C::RSLAB + (kk & 3) * 32) >> 4;
                    umma_ss(tbase + C::TM_S, qdesc + qo, kdesc + ko, IDESC_S, kk != 0);
                }
            }
            __syncwarp();
            // dP overwrites the columns where tile i - 1's dS was read by its dQ
            if (i >= 1 && !(ok = warp_wait(dq_final, static_cast<uint32_t>((i - 1) & 1))))
                break;
            if (lane == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = static_cast<uint32_t>((kk >> 2) * C::QSLAB + (kk & 3) * 32) >> 4;
                    const uint32_t ko = static_cast<uint32_t>((kk >> 2) * C::RSLAB + (kk & 3) * 32) >> 4;
                    umma_ss(tbase + C::TM_DP, odesc + qo, vdesc + ko, IDESC_DP, kk != 0);
                }
                umma_commit(s_full);
                umma_commit(q_free);
            }
            __syncwarp();
            // dQ is free once the epilogue has read tile i - 1's; dS of this tile written
            if ((i >= 1 && !(ok = warp_wait(dq_free, static_cast<uint32_t>((i - 1) & 1)))) ||
                !(ok = warp_wait(p_full, static_cast<uint32_t>(i & 1))))
                break;
            if (lane == 0) {
                tc_fence_after();
                for (int kb = lo; kb <= hi; ++kb) {
                    const int j = static_cast<int>((nf + (kb - lo)) % C::NSLOT);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t bdesc =
                            umma_desc_sw128(sbase + C::K16_OFF + j * C::SLOT + h * 2048, C::RSLAB, 1024);
                        umma_ts(tbase + C::TM_DQ, tbase + C::TM_DP + C::ds_col(j) + 8 * h, bdesc, IDESC_DQ,
                                (kb > lo || h > 0) ? 1u : 0u);
                    }
                }
                umma_commit(dq_final);
            }
            __syncwarp();
            // blocks the next tile's band does not hold are free once this dQ is done
            if (have_next) {
                ahead = run;
                ahead.step(nbh, nlo, nhi);
                const long long next_first = ahead.nh - (nhi - nlo);
                if (lane == 0)
                    for (long long m = released; m < next_first; ++m)
                        umma_commit(&kv_empty[m % C::NSLOT]);
                __syncwarp();
                if (next_first > released)
                    released = next_first;
            }
        }
    } else if (warp < 4) {
        // warps 2-3: no role
    } else if (warp < 12) {
        // ------------------------------------------------------------------ dS (lane = row), sums
        const int rw = warp & 3;
        const int grp = warp < 8 ? 0 : 1;
        const uint32_t gmask = grp == 0 ? 0x07u : 0x38u;  // this group's ring slots
        const int r = rw * 32 + lane;  // row of the tile = tensor-memory lane
        const uint32_t tl = tbase + (static_cast<uint32_t>(rw * 32) << 16);
        const float c2 = p.scale * kLog2eF;
        float ds_max = 0.f;  // dS goes to fp16
        bool kshift_bad = false;
        // FOLD: this group's half of the columns of dalpha += x dq, dbeta += dq (dq = scale dQ).
        // The lanes of one head reduce-scatter each 16-column piece, after which a lane owns G / 2
        // columns of its head (lane / G picks which); sums stay in registers across the CTA's
        // tiles and go to global memory with atomics when the KV head changes and at the end.
        constexpr int OWN = FOLD ? G / 2 : 1;
        constexpr int NP = D / 32;  // 16-column pieces in half the columns
        float acc_a[NP][OWN], acc_b[NP][OWN];
        int cur_g = -1;
        auto flush = [&](int gg) {
            if (FOLD && gg >= 0) {
                const int col0 = (gg * G + lane % G) * D + grp * (D / 2) + (lane / G) * OWN;
#pragma unroll
                for (int pc = 0; pc < NP; ++pc)
#pragma unroll
                    for (int e = 0; e < OWN; ++e) {
                        atomicAdd(p.dalpha + col0 + 16 * pc + e, acc_a[pc][e]);
                        atomicAdd(p.dbeta + col0 + 16 * pc + e, acc_b[pc][e]);
                    }
            }
        };
        BandRun run;
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            int bh, u0, lo, hi;
            tile(tau, bh, u0, lo, hi);
            run.step(bh, lo, hi);
            const int s0 = static_cast<int>((run.nh - (hi - lo)) % C::NSLOT);  // slot of block lo
            const int b = bh / p.Hkv, g = bh % p.Hkv;
            const int uu = u0 + r / G, h = g * G + r % G;
            const bool live = uu < p.n_units;
            const int P = live ? uu : -1, klo = P - p.window + 1;
            const long long ri = (static_cast<long long>(b) * p.n_units + uu) * p.Hq + h;
            const float lse = live ? p.lse[ri] : 0.f;  // log2 units (the rows kernel converted it)
            const float Drow = live ? p.Drow[ri] : 0.f;
            const int8_t *ke = p.kexp + static_cast<long long>(bh) * p.nkb * 64;
            const uint8_t *kf = p.kflag + static_cast<long long>(bh) * p.nkb;
            // this group's band slots (slot s0 + d holds block lo + d); the others are stale or
            // loading, and those of shifted key rows (rare)
            uint32_t band = 0, shifted = 0;
            for (int kb = lo; kb <= hi; ++kb) {
                const uint32_t bit = 1u << ((s0 + kb - lo) % C::NSLOT);
                band |= bit;
                if (kf[kb >> 1] != 0)
                    shifted |= bit;
            }
            band &= gmask;
            shifted &= gmask;
            if (!(ok = warp_wait(s_full, static_cast<uint32_t>(i & 1))))
                break;
            tc_fence_after();
            for (uint32_t m = shifted; m != 0; m &= m - 1) {  // logits of shifted key rows times 2^e
                const int j = __ffs(m) - 1;
                unshift_chunk32(tl + C::TM_S + 32 * j, ke, (lo + (j - s0 + C::NSLOT) % C::NSLOT) * C::KB, 1u, 1, 1,
                                kshift_bad);
            }
            // the group's slots in slot order; dS of slot j goes over dP columns of the group's
            // own slots, below every column it has still to read
#pragma unroll 1
            for (uint32_t m = band; m != 0; m &= m - 1) {
                const int j = __ffs(m) - 1;
                uint32_t sv[32], dv[32];
                tmem_ld32(tl + C::TM_S + 32 * j, sv);
                tmem_ld32(tl + C::TM_DP + 32 * j, dv);
                tmem_wait_ld();
                const int key0 = (lo + (j - s0 + C::NSLOT) % C::NSLOT) * C::KB;
                const bool fl = (shifted >> j) & 1u;
                uint32_t dw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float ds[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int key = key0 + 2 * e + q;
                        const bool valid = key <= P && key >= klo;
                        const float pr = fast_exp2(__uint_as_float(sv[2 * e + q]) * c2 - lse);
                        ds[q] = valid ? pr * (__uint_as_float(dv[2 * e + q]) - Drow) : 0.f;
                    }
                    if (fl) {  // dQ takes K16 = k 2^-e: dS times 2^e
                        ds[0] *= exp2i(ke[key0 + 2 * e]);
                        ds[1] *= exp2i(ke[key0 + 2 * e + 1]);
                    }
                    ds_max = fmax3(ds_max, fabsf(ds[0]), fabsf(ds[1]));
                    __half2 hv = __floats2half2_rn(ds[0], ds[1]);
                    dw[e] = *reinterpret_cast<uint32_t *>(&hv);
                }
                tmem_st16(tl + C::TM_DP + C::ds_col(j), dw);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(p_full);
            if constexpr (FOLD) {
                // the sums of this tile, once its dQ is done (while the next tile's S, dP run)
                if (g != cur_g) {
                    flush(cur_g);
#pragma unroll
                    for (int pc = 0; pc < NP; ++pc)
#pragma unroll
                        for (int e = 0; e < OWN; ++e)
                            acc_a[pc][e] = acc_b[pc][e] = 0.f;
                    cur_g = g;
                }
                // x of the row's half: all loads in flight before the wait (G = 4); piece by piece
                // for G = 8, whose wider per-lane sums leave no registers for them
                constexpr bool XALL = G == 4;
                const long long off = ri * D + grp * (D / 2);
                uint4 xr[XALL ? 2 * NP : 2];
                if (XALL) {
#pragma unroll
                    for (int e = 0; e < (XALL ? 2 * NP : 2); ++e)
                        xr[e] = live ? __ldg(reinterpret_cast<const uint4 *>(p.q + off) + e) : make_uint4(0u, 0u, 0u, 0u);
                }
                if (!(ok = warp_wait(dq_final, static_cast<uint32_t>(i & 1))))
                    break;
                tc_fence_after();
                const float sc = p.scale;
#pragma unroll
                for (int pc = 0; pc < NP; ++pc) {
                    const int xi = XALL ? 2 * pc : 0;
                    if (!XALL) {
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            xr[e] = live ? __ldg(reinterpret_cast<const uint4 *>(p.q + off + 16 * pc) + e)
                                         : make_uint4(0u, 0u, 0u, 0u);
                    }
                    uint32_t w[16];
                    tmem_ld16(tl + C::TM_DQ + grp * (D / 2) + 16 * pc, w);
                    tmem_wait_ld();
                    float va[16], vb[16];
                    const uint32_t xw[8] = {xr[xi].x,     xr[xi].y,     xr[xi].z,     xr[xi].w,
                                            xr[xi + 1].x, xr[xi + 1].y, xr[xi + 1].z, xr[xi + 1].w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 xv = unpack_bf16x2(xw[e]);
                        const float d0 = live ? __uint_as_float(w[2 * e]) * sc : 0.f;
                        const float d1 = live ? __uint_as_float(w[2 * e + 1]) * sc : 0.f;
                        vb[2 * e] = d0;
                        vb[2 * e + 1] = d1;
                        va[2 * e] = xv.x * d0;
                        va[2 * e + 1] = xv.y * d1;
                    }
                    // reduce-scatter over the 32 / G lanes of this head: halve the vector per step
#pragma unroll
                    for (int st = 0; (16 >> st) >= G; ++st) {
                        const int mk = 16 >> st, half = 8 >> st;
                        const bool up = (lane & mk) != 0;
#pragma unroll
                        for (int e = 0; e < half; ++e) {
                            const float sa = up ? va[e] : va[e + half], ka = up ? va[e + half] : va[e];
                            const float sb = up ? vb[e] : vb[e + half], kb2 = up ? vb[e + half] : vb[e];
                            va[e] = ka + __shfl_xor_sync(0xffffffffu, sa, mk);
                            vb[e] = kb2 + __shfl_xor_sync(0xffffffffu, sb, mk);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < OWN; ++e) {
                        acc_a[pc][e] += va[e];
                        acc_b[pc][e] += vb[e];
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(dq_free);  // this warp's share of dQ is read
            }
        }
        if (FOLD && ok)
            flush(cur_g);
        if (!(ds_max < 65504.f) || kshift_bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
    } else {
        // ------------------------------------------------------------------ dq_raw stores (warps 12-15)
        // dq_raw = scale dQ alpha: 32 columns at a time from tensor memory (the next load in flight)
        // into D / 32 staging tiles laid out as the dq map's 128-byte swizzled boxes, which one
        // thread stores by TMA (rows past the stream are clipped).  The four warps meet at a
        // barrier that also ANDs their wait results, so a timeout in one stops all four.
        const int rw = warp - 12;
        const int r = rw * 32 + lane;
        const uint32_t tl = tbase + (static_cast<uint32_t>(rw * 32) << 16);
        const bool issuer = warp == 12 && lane == 0;
        const float sc = p.scale;
        for (long long tau = t_begin, i = 0; ok && tau < t_end; ++tau, ++i) {
            int bh, u0, lo, hi;
            tile(tau, bh, u0, lo, hi);
            const int b = bh / p.Hkv, g = bh % p.Hkv;
            const int h = g * G + r % G;
            if (issuer)
                bulk_wait_read_all();  // the previous tile's stores have read the staging tiles
            const bool got = warp_wait(dq_final, static_cast<uint32_t>(i & 1));
            if (!(ok = bar_red_and(1, 128, got)))
                break;
            tc_fence_after();
            uint32_t wa[32];
            tmem_ld32(tl + C::TM_DQ, wa);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                tmem_wait_ld();
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    w[e] = wa[e];
                if (c + 1 < D / 32) {
                    tmem_ld32(tl + C::TM_DQ + 32 * (c + 1), wa);
                } else {  // every column of dQ is read: the accumulator is free
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(dq_free);
                }
                uint8_t *tile_c = smem + C::DQS_OFF + c * C::DQS_TILE;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 a = __ldg(reinterpret_cast<const float4 *>(p.alpha + h * D + 32 * c + 4 * j));
                    *reinterpret_cast<float4 *>(tile_c + sw128_offset(r, j)) =
                        make_float4(__uint_as_float(w[4 * j]) * sc * a.x, __uint_as_float(w[4 * j + 1]) * sc * a.y,
                                    __uint_as_float(w[4 * j + 2]) * sc * a.z, __uint_as_float(w[4 * j + 3]) * sc * a.w);
                }
            }
            fence_proxy_async_smem();
            named_barrier(1, 128);  // every store warp's rows are in the staging tiles
            if (issuer) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
                    tma_store_4d(&dqmap, smem + C::DQS_OFF + c * C::DQS_TILE, 32 * c, g * G, u0, b);
                bulk_commit();
            }
        }
        if (issuer)
            bulk_wait_all();  // the last stores are complete before the kernel ends
    }
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// the band kernel's limits: G >= 4 (a 128-row tile spans at most 32 units) and every tile's band
// within NSLOT - 1 slots
__host__ inline bool dq_band_fits(int G, int window)
{
    if (G < 4)
        return false;
    const int units = 128 / G, kb = BbCfg<128>::KB;
    int most = 0;
    for (int a = 0; a < kb; a += units) {  // tile starts u0 = a (mod 32), far from the sequence start
        const int u0 = 1 << 20 | a;
        most = max(most, (u0 + units - 1) / kb - (u0 - window + 1) / kb + 1);
    }
    return most <= BbCfg<128>::NSLOT - 1;
}

// ------------------------------------------------------------------ split log-sum-exp

// rows of the single row tile of each (batch, KV head): merge the splits' (max, sum) into
// the row's log2-sum-exp
template <int G>
__global__ void __launch_bounds__(128) attn_bwd_lse_combine_kernel(const AttnBwdParams p)
{
    const int bh = blockIdx.x, r = threadIdx.x;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int u = r / G, h = g * G + r % G;
    if (unit_pos<true>(p, b, u) < 0)
        return;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float2 *part = p.part_ml + static_cast<long long>(bh) * p.splits * 128 + r;
    float M = NEG_INF;
    for (int z = 0; z < p.splits; ++z)
        M = fmaxf(M, part[z * 128].x);
    float L = 0.f;
    for (int z = 0; z < p.splits; ++z) {
        const float2 ml = part[z * 128];
        if (ml.x != NEG_INF)
            L += ml.y * exp2f(ml.x - M);
    }
    p.lse[(static_cast<long long>(b) * p.n_units + u) * p.Hq + h] = M + __log2f(L);  // the row holds its own key
}

// ------------------------------------------------------------------ launches

static size_t dq_smem(int D, int G)
{
    return static_cast<size_t>(4) * (D / 64) * BWD_KEYS * 128 + 2 * G * D * 4 + 16 + 1024;
}

// dalpha, dbeta from dq_raw and x, [B * n_units token rows] x [Hq * D columns]: 4 columns per
// thread, runs of token rows per CTA
static cudaError_t launch_dab(const AttnBwdParams &p, int D, int sms, cudaStream_t stream)
{
    const long long trows = static_cast<long long>(p.B) * p.n_units;
    const int cols = p.Hq * D;
    const unsigned gx = static_cast<unsigned>((cols / 4 + 255) / 256);
    const long long gy_t = (2LL * sms * 4 + gx - 1) / gx, gy = trows < gy_t ? trows : gy_t;
    const int per = static_cast<int>((trows + gy - 1) / gy);
    attn_bwd_dab_kernel<<<dim3(gx, static_cast<unsigned>((trows + per - 1) / per)), 256, 0, stream>>>(
        p.dq, p.q, p.alpha, p.dalpha, p.dbeta, trows, cols, per);
    return cudaGetLastError();
}

// One stream's launches before dK/dV: zeroed dalpha / dbeta, the fp16 copy of K (unless another
// stream's call already made it), the fp16 scale-offset q, D (and the forward's log-sum-exp in
// log2 units), then dq (and, after the persistent base kernel, the dalpha / dbeta sums).
template <int D, int G, bool COPY>
static cudaError_t launch_rows_t(const AttnBwdParams &p, const CUtensorMap *maps, bool make_k16, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(p.B) * p.n_units * p.Hq;
    cudaError_t e = cudaMemsetAsync(p.dalpha, 0, sizeof(float) * p.Hq * D, stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(p.dbeta, 0, sizeof(float) * p.Hq * D, stream);
    if (e != cudaSuccess)
        return e;
    if (make_k16) {
        attn_bwd_k16_kernel<D><<<static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * p.nkb), 256, 0, stream>>>(
            p.k, p.k16, p.kexp, p.kflag, p.T_kv, p.Hkv, p.nkb, p.dev_err);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    // the fp16 scale-offset q (read by the dK/dV kernel and the base stream's persistent dQ),
    // each row's D and the given log-sum-exp in log2 units: one pass
    const bool persistent = !COPY && p.lse_in != nullptr;  // base dq on tensor memory
    if (rows > 0) {
        attn_bwd_rows_kernel<D><<<static_cast<unsigned>((rows * (D / 8) + 255) / 256), 256, 0, stream>>>(
            p.q, p.alpha, p.beta, p.q16, p.o, p.dO, p.Drow, p.lse_in, p.lse, rows, p.Hq, p.dev_err);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        // base rows see at most window + 128/G keys: a tensor-memory CTA (one per SM) spends
        // most of its time filling and draining its pipeline, and the warp-MMA kernel is
        // faster there (whole base gradient of a 2 x 128K-token, 32/8-head, w = 128 layer:
        // 21.6 vs 23.5 ms with the forward's log-sum-exp, 23.4 vs 24.5 ms without); copies
        // see long key ranges (2.54 vs 4.87 ms for 2048 copies of a 16K layer)
        if (COPY && p.lse_in != nullptr && p.n_units * G <= BkCfg<D>::RMAX) {
            // a few copy rows with the forward's log-sum-exp: rows on the warp MMA's N side, the
            // keys split so that the grid fills the GPU (two CTAs' worth per SM)
            int dev = 0, sms = 0;
            if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return e;
            const int nbk = (p.T_kv + BkCfg<D>::KB - 1) / BkCfg<D>::KB;
            AttnBwdParams ps = p;
            ps.splits = max(1, min(min(ATTN_BWD_MAX_SPLITS, 2 * sms / (p.B * p.Hkv)), nbk / 4));
            if (ps.splits >= 2 && (e = cudaMemsetAsync(p.dq, 0, sizeof(float) * rows * D, stream)) != cudaSuccess)
                return e;
            auto k1 = attn_bwd_dq_copies_keys_kernel<D>;
            if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, BkCfg<D>::SMEM)) !=
                cudaSuccess)
                return e;
            k1<<<dim3(ps.splits, 1, p.B * p.Hkv), BkCfg<D>::THREADS, BkCfg<D>::SMEM, stream>>>(maps[6], maps[7], ps);
        } else if (COPY) {
            const size_t s1 = BqCfg<D>::SMEM;
            auto k1 = attn_bwd_dq_tc_kernel<D, G, COPY>;
            if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s1))) !=
                cudaSuccess)
                return e;
            constexpr int UNITS = BqCfg<D>::ROWS / G;
            dim3 g1((p.n_units + UNITS - 1) / UNITS, p.B * p.Hkv);
            // few copies (one row tile per batch and KV head) over many keys: split the keys
            // so that the grid fills the GPU (two CTAs' worth per SM); with the forward's
            // log-sum-exp only the second pass runs
            int splits = 1;
            if (p.n_units <= UNITS && (p.lse_in != nullptr || p.part_ml != nullptr)) {
                int dev = 0, sms = 0;
                if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
                    (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                    return e;
                const int nbk = (p.T_kv + BqCfg<D>::KB - 1) / BqCfg<D>::KB;
                splits = min(min(ATTN_BWD_MAX_SPLITS, 2 * sms / (p.B * p.Hkv)), nbk / 8);
            }
            if (splits >= 2) {
                if ((e = cudaMemsetAsync(p.dq, 0, sizeof(float) * rows * D, stream)) != cudaSuccess)
                    return e;
                AttnBwdParams ps = p;
                ps.splits = splits;
                dim3 gs(1, p.B * p.Hkv, splits);
                if (p.lse_in == nullptr) {  // per-split (max, sum), merged into the log-sum-exp
                    ps.split_mode = 1;
                    k1<<<gs, DKV_TC_THREADS, s1, stream>>>(maps[4], maps[5], maps[6], maps[7], maps[8], ps);
                    if ((e = cudaGetLastError()) != cudaSuccess)
                        return e;
                    attn_bwd_lse_combine_kernel<G><<<p.B * p.Hkv, 128, 0, stream>>>(ps);
                    if ((e = cudaGetLastError()) != cudaSuccess)
                        return e;
                }
                ps.split_mode = 2;
                k1<<<gs, DKV_TC_THREADS, s1, stream>>>(maps[4], maps[5], maps[6], maps[7], maps[8], ps);
            } else {
                k1<<<g1, DKV_TC_THREADS, s1, stream>>>(maps[4], maps[5], maps[6], maps[7], maps[8], p);
            }
        } else if (persistent && G >= 4 && dq_band_fits(G, p.window)) {
            // base stream with the forward's log-sum-exp, each tile's key band one MMA wide; for
            // G <= 8 the dalpha / dbeta sums come out of its dS warps
            if constexpr (G >= 4) {
                constexpr bool FOLD = G <= 8;
                const size_t s1 = BbCfg<D>::SMEM;
                auto k1 = attn_bwd_dq_band_kernel<D, G, FOLD>;
                if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(s1))) != cudaSuccess)
                    return e;
                int dev = 0, sms = 0;
                if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
                    (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                    return e;
                constexpr int UNITS = BbCfg<D>::ROWS / G;
                const long long tiles = static_cast<long long>(p.B) * p.Hkv * ((p.n_units + UNITS - 1) / UNITS);
                k1<<<static_cast<unsigned>(tiles < sms ? tiles : sms), BbCfg<D>::THREADS, s1, stream>>>(
                    maps[9], maps[5], maps[10], maps[11], maps[12], p);
                if (!FOLD) {
                    if ((e = cudaGetLastError()) != cudaSuccess)
                        return e;
                    e = launch_dab(p, D, sms, stream);
                }
            }
        } else if (persistent) {
            // base stream with the forward's log-sum-exp: the persistent tensor-memory kernel
            const size_t s1 = BpCfg<D>::SMEM;
            auto k1 = attn_bwd_dq_tc_base_kernel<D, G>;
            if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s1))) !=
                cudaSuccess)
                return e;
            int dev = 0, sms = 0;
            if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return e;
            constexpr int UNITS = BpCfg<D>::ROWS / G;
            const long long tiles = static_cast<long long>(p.B) * p.Hkv * ((p.n_units + UNITS - 1) / UNITS);
            k1<<<static_cast<unsigned>(tiles < sms ? tiles : sms), DKV_TC_THREADS, s1, stream>>>(
                maps[9], maps[5], maps[6], maps[7], maps[8], p);
            if ((e = cudaGetLastError()) != cudaSuccess)
                return e;
            e = launch_dab(p, D, sms, stream);
        } else {
            const size_t s1 = dq_smem(D, G);
            auto k1 = attn_bwd_dq_kernel<D, G, COPY>;
            if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s1))) !=
                cudaSuccess)
                return e;
            constexpr int UNITS = BWD_ROWS / G;
            dim3 g1((p.n_units + UNITS - 1) / UNITS, p.B * p.Hkv);
            k1<<<g1, 128, s1, stream>>>(p);
        }
        if (e == cudaSuccess)
            e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// dK / dV of the rows of p (STREAMS 0: base, 1: copies) or of both streams (STREAMS 2: p base,
// pc copies).  Also runs without query rows: it writes (or keeps) zeros.
template <int D, int G, int STREAMS>
static cudaError_t launch_dkv_t(const AttnBwdParams &p, const AttnBwdParams &pc, const CUtensorMap *maps,
                                const CUtensorMap *mapsc, cudaStream_t stream)
{
    const size_t s3 = BtCfg<D>::SMEM;
    auto k3 = attn_bwd_dkv_tc_kernel<D, G, STREAMS>;
    cudaError_t e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s3));
    if (e != cudaSuccess)
        return e;
    dim3 g3((p.T_kv + BtCfg<D>::KEYS - 1) / BtCfg<D>::KEYS, p.B * p.Hkv);
    k3<<<g3, DKV_THREADS, s3, stream>>>(maps[0], maps[1], mapsc[0], mapsc[1], maps[3], maps[2], p, pc);
    return cudaGetLastError();
}

template <int D, int G, bool COPY>
static cudaError_t launch_attn_bwd_t(const AttnBwdParams &p, const CUtensorMap *maps, cudaStream_t stream)
{
    const cudaError_t e = launch_rows_t<D, G, COPY>(p, maps, true, stream);
    if (e != cudaSuccess)
        return e;
    return launch_dkv_t<D, G, COPY ? 1 : 0>(p, p, maps, maps, stream);
}

// both streams of a layer: the copies reuse the base stream's fp16 K, and one dK/dV launch
// takes the base rows and then the copies' rows of each key block
template <int D, int G>
static cudaError_t launch_layer_bwd_t(const AttnBwdParams &p, const AttnBwdParams &pc, const CUtensorMap *maps,
                                      const CUtensorMap *mapsc, cudaStream_t stream)
{
    cudaError_t e = launch_rows_t<D, G, false>(p, maps, true, stream);
    if (e == cudaSuccess)
        e = launch_rows_t<D, G, true>(pc, mapsc, false, stream);
    if (e != cudaSuccess)
        return e;
    return pc.n_units > 0 ? launch_dkv_t<D, G, 2>(p, pc, maps, mapsc, stream)
                          : launch_dkv_t<D, G, 0>(p, p, maps, maps, stream);
}

// The launches of one head dimension D for every supported group size G; each D is
// instantiated in its own translation unit (attn_bwd_d128.cu, attn_bwd_d64.cu) so that the
// build compiles them in parallel.
template <int D>
cudaError_t attn_bwd_dispatch(int G, const AttnBwdParams &p, const CUtensorMap *maps, cudaStream_t stream)
{
#define ORTHROS_BWD_CASE(GG) \
    if (G == GG)             \
        return p.pos ? launch_attn_bwd_t<D, GG, true>(p, maps, stream) : launch_attn_bwd_t<D, GG, false>(p, maps, stream);
    ORTHROS_BWD_CASE(1)
    ORTHROS_BWD_CASE(2)
    ORTHROS_BWD_CASE(4)
    ORTHROS_BWD_CASE(8)
    ORTHROS_BWD_CASE(16)
#undef ORTHROS_BWD_CASE
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t attn_bwd_layer_dispatch(int G, const AttnBwdParams &p, const AttnBwdParams &pc, const CUtensorMap *maps,
                                    const CUtensorMap *mapsc, cudaStream_t stream)
{
#define ORTHROS_BWD_CASE(GG) \
    if (G == GG)             \
        return launch_layer_bwd_t<D, GG>(p, pc, maps, mapsc, stream);
    ORTHROS_BWD_CASE(1)
    ORTHROS_BWD_CASE(2)
    ORTHROS_BWD_CASE(4)
    ORTHROS_BWD_CASE(8)
    ORTHROS_BWD_CASE(16)
#undef ORTHROS_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace orthros
