// swa_bwd.cu -- gradient of the base stream, Eq. (4) of "Orthros: Phase-Aware
// Heterogeneous Attention" with its scale-offset q = Q_raw * alpha + beta
// (Sec. 3.1), for SFT / PT training (Sec. 3.2: every base position is computed
// in those modes).  For an output gradient dO and, per row (b, t, h) over its
// window keys j:
//   p_j = softmax_j(s_j), s_j = scale * (q . k_j);  dp_j = dO . v_j
//   D = dO . o = sum_j p_j dp_j;  ds_j = p_j (dp_j - D)
//   dq = scale * sum_j ds_j k_j;  dk_j += scale * ds_j q;  dv_j += p_j dO
//   dq_raw = dq * alpha;  dalpha += q_raw * dq;  dbeta += dq
// Three launches (warp MMAs, bf16 operands, fp32 accumulation):
//   swa_bwd_d_kernel    D = dO . o per row (o: the forward output);
//   swa_bwd_dq_kernel   rows on the MMA's M side: a CTA stages the K/V band of its
//                       64 rows, each warp recomputes S for its 16 rows (q as bf16
//                       high part + residual) and keeps log2-sum-exp (stored for the
//                       next kernel), then dP = dO V^T, dS = P (dP - D), dQ += dS K;
//                       dq_raw, and dalpha / dbeta through shared then global atomics;
//   swa_bwd_dkv_kernel  keys on the M side: a CTA owns 64 keys and streams the rows
//                       of their windows through shared memory; each warp keeps dK, dV
//                       of its 16 keys in registers (S^T = K q^T, dP^T = V dO^T,
//                       dV += P^T dO, dK += dS^T q) and writes them once.
// Outputs are fp32; P and dS enter the second products as bf16.
#include "common.cuh"
#include "kernels.cuh"
#include "xattn.cuh"

namespace orthros {

namespace {

constexpr float kLog2eF = 1.4426950408889634f;

// [rows][D] bf16 tile in shared memory as D/64 slabs of rows x 128 bytes, 128-byte swizzle
__device__ __forceinline__ uint32_t tile_off(int row, int col, int slab_bytes)
{
    return static_cast<uint32_t>((col / 64) * slab_bytes) + sw128_offset(row, (col % 64) / 8);
}

// copy rows [r0, r0 + n) of one KV head (row stride Hkv * D elements) into a swizzled tile;
// rows outside [0, T) are zero-filled
template <int D>
__device__ void stage_kv_rows(uint8_t *tile, int slab_bytes, const orthros_bf16 *base, long long row_stride, int r0,
                              int n, int T, int tid, int nthreads)
{
    constexpr int CPR = D / 8;
    for (int i = tid; i < n * CPR; i += nthreads) {
        const int r = i / CPR, c = (i % CPR) * 8;
        const int key = r0 + r;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (key >= 0 && key < T)
            val = *reinterpret_cast<const uint4 *>(base + key * row_stride + c);
        *reinterpret_cast<uint4 *>(tile + tile_off(r, c, slab_bytes)) = val;
    }
}

}  // namespace

// ------------------------------------------------------------------ D = dO . o

template <int D>
__global__ void __launch_bounds__(256) swa_bwd_d_kernel(const orthros_bf16 *o, const orthros_bf16 *dO, float *Dout,
                                                        long long rows)
{
    const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows)
        return;
    float acc = 0.f;
#pragma unroll
    for (int e = lane * 2; e < D; e += 64) {
        const float2 a = unpack_bf16x2(*reinterpret_cast<const uint32_t *>(o + row * D + e));
        const float2 b = unpack_bf16x2(*reinterpret_cast<const uint32_t *>(dO + row * D + e));
        acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0)
        Dout[row] = acc;
}

// ------------------------------------------------------------------ dQ (rows on M)

template <int D, int G>
__global__ void __launch_bounds__(128) swa_bwd_dq_kernel(const SwaBwdParams p)
{
    constexpr int ROWS = 64;          // rows of a CTA = ROWS / G tokens x G heads
    constexpr int TOKC = ROWS / G;
    const int tile = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = tile * TOKC;                             // first token of the CTA
    const int band0 = max(0, t0 - p.window + 1);            // first key of the band
    const int band1 = min(p.T - 1, t0 + TOKC - 1);          // last key
    const int nband = band1 - band0 + 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int slab = p.band_max * 128;                      // one slab of the K (or V) band
    uint8_t *kt = smem;
    uint8_t *vt = smem + (D / 64) * slab;
    float *red = reinterpret_cast<float *>(smem + 2 * (D / 64) * slab);  // [2][G][D] dalpha, dbeta
    const long long row_stride = static_cast<long long>(p.Hkv) * D;
    const orthros_bf16 *kb = p.k + b * p.kv_bstride + static_cast<long long>(g) * D;
    const orthros_bf16 *vb = p.v + b * p.kv_bstride + static_cast<long long>(g) * D;
    // whole 16-key chunks are read: stage the band rounded up (keys past the band are masked)
    const int nstage = (nband + 15) & ~15;
    stage_kv_rows<D>(kt, slab, kb, row_stride, band0, nstage, p.T, threadIdx.x, 128);
    stage_kv_rows<D>(vt, slab, vb, row_stride, band0, nstage, p.T, threadIdx.x, 128);
    for (int i = threadIdx.x; i < 2 * G * D; i += 128)
        red[i] = 0.f;
    __syncthreads();
    const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);

    // this warp's 16 rows: r = 16 warp + 0..15 -> token t0 + r / G, head g G + r % G
    const int gr = lane >> 2, qd = (lane & 3) * 2;
    const int rowA = 16 * warp + gr, rowB = rowA + 8;
    const int tA = t0 + rowA / G, tB = t0 + rowB / G;
    const int hA = g * G + rowA % G, hB = g * G + rowB % G;
    const bool vA = tA < p.T, vB = tB < p.T;
    const float c2 = p.scale * kLog2eF;  // logits in log2 units
    WarpRows16<D> st;                    // q fragments (unscaled q = x alpha + beta) + dQ accumulators
    uint32_t ga[D / 16][4];              // dO fragments (A operand)
#pragma unroll
    for (int kt2 = 0; kt2 < D / 16; ++kt2)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const bool isB = r & 1;
            const int t = isB ? tB : tA, h = isB ? hB : hA;
            const int dcol = kt2 * 16 + qd + ((r & 2) ? 8 : 0);
            uint32_t hi = 0, lo = 0, gw = 0;
            if (isB ? vB : vA) {
                const long long off = b * p.q_bstride + (static_cast<long long>(t) * p.Hq + h) * D;
                load_q_pair(p.q + off, p.alpha + h * D, p.beta + h * D, dcol, 1.f, hi, lo);
                gw = *reinterpret_cast<const uint32_t *>(p.dO + b * p.o_bstride +
                                                         (static_cast<long long>(t) * p.Hq + h) * D + dcol);
            }
            st.qa[kt2][r] = hi;
            st.ql[kt2][r] = lo;
            ga[kt2][r] = gw;
        }
    st.reset();
    // key range of this warp's rows (band-relative), and each row's window
    const int tw0 = t0 + (16 * warp) / G, tw1 = min(p.T - 1, t0 + (16 * warp + 15) / G);
    const int j_lo = max(0, tw0 - p.window + 1) - band0, j_hi = tw1 - band0;
    const int loA = tA - p.window + 1, loB = tB - p.window + 1;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int kld_row = (lane & 7) + ((lane >> 4) << 3), kld_hi = (lane >> 3) & 1;
    const int vld_row = (lane & 7) + (((lane >> 3) & 1) << 3), vld_hi = lane >> 4;
    const bool warp_live = tw0 < p.T;

    // S chunk (16 rows x 16 keys from band row jc) in log2 units, masked to the windows
    auto s_chunk = [&](int jc, float (&s)[2][4]) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kt2 = 0; kt2 < D / 16; ++kt2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + tile_off(jc + kld_row, kt2 * 16 + kld_hi * 8, slab), b0, b1, b2, b3);
            mma_16816(s[0], st.qa[kt2], b0, b1);
            mma_16816(s[1], st.qa[kt2], b2, b3);
            mma_16816(s[0], st.ql[kt2], b0, b1);
            mma_16816(s[1], st.ql[kt2], b2, b3);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = band0 + jc + i * 8 + qd + (e & 1);
                const bool isB = e & 2;
                const int t = isB ? tB : tA, lo = isB ? loB : loA;
                s[i][e] = (key <= t && key >= lo && key < p.T && (isB ? vB : vA)) ? s[i][e] * c2 : NEG_INF;
            }
    };

    // pass 1: log2-sum-exp of each row over its window
    float mA = NEG_INF, mB = NEG_INF, lA = 0.f, lB = 0.f;
    if (warp_live) {
        for (int jc = j_lo & ~15; jc <= j_hi; jc += 16) {
            float s[2][4];
            s_chunk(jc, s);
            float cA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
            float cB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
            cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 1));
            cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 2));
            cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 1));
            cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 2));
            const float nA = fmaxf(mA, cA), nB = fmaxf(mB, cB);
            const float uA = nA == NEG_INF ? 0.f : nA, uB = nB == NEG_INF ? 0.f : nB;
            lA = lA * fast_exp2(mA - uA) + fast_exp2(s[0][0] - uA) + fast_exp2(s[0][1] - uA) +
                 fast_exp2(s[1][0] - uA) + fast_exp2(s[1][1] - uA);
            lB = lB * fast_exp2(mB - uB) + fast_exp2(s[0][2] - uB) + fast_exp2(s[0][3] - uB) +
                 fast_exp2(s[1][2] - uB) + fast_exp2(s[1][3] - uB);
            mA = nA;
            mB = nB;
        }
    }
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    // every live row holds its own key; rows past T get 0 so that their P is exactly 0
    const float lseA = vA ? mA + __log2f(lA) : 0.f, lseB = vB ? mB + __log2f(lB) : 0.f;
    const long long rA = (static_cast<long long>(b) * p.T + tA) * p.Hq + hA;
    const long long rB = (static_cast<long long>(b) * p.T + tB) * p.Hq + hB;
    if ((lane & 3) == 0) {
        if (vA)
            p.lse[rA] = lseA;
        if (vB)
            p.lse[rB] = lseB;
    }
    const float DA = vA ? p.Drow[rA] : 0.f, DB = vB ? p.Drow[rB] : 0.f;

    // pass 2: dS = P (dP - D), dQ += dS K
    if (warp_live) {
        for (int jc = j_lo & ~15; jc <= j_hi; jc += 16) {
            float s[2][4], dp[2][4];
            s_chunk(jc, s);
#pragma unroll
            for (int i = 0; i < 2; ++i)
                dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
#pragma unroll
            for (int kt2 = 0; kt2 < D / 16; ++kt2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(vbase + tile_off(jc + kld_row, kt2 * 16 + kld_hi * 8, slab), b0, b1, b2, b3);
                mma_16816(dp[0], ga[kt2], b0, b1);
                mma_16816(dp[1], ga[kt2], b2, b3);
            }
            float ds[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool isB = e & 2;
                    const float pr = fast_exp2(s[i][e] - (isB ? lseB : lseA));
                    ds[i][e] = pr * (dp[i][e] - (isB ? DB : DA));
                }
            uint32_t da[4];
            da[0] = pack_bf16x2(ds[0][0], ds[0][1]);
            da[1] = pack_bf16x2(ds[0][2], ds[0][3]);
            da[2] = pack_bf16x2(ds[1][0], ds[1][1]);
            da[3] = pack_bf16x2(ds[1][2], ds[1][3]);
#pragma unroll
            for (int dp2 = 0; dp2 < D / 16; ++dp2) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_trans(kbase + tile_off(jc + vld_row, dp2 * 16 + vld_hi * 8, slab), v0, v1, v2, v3);
                mma_16816(st.o[2 * dp2], da, v0, v1);
                mma_16816(st.o[2 * dp2 + 1], da, v2, v3);
            }
        }
    }
    // epilogue: dq = scale * dQ; dq_raw = dq * alpha; dalpha += x * dq, dbeta += dq
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const bool live = half ? vB : vA;
        const int t = half ? tB : tA, h = half ? hB : hA, hh = h - g * G;
        const long long off = (static_cast<long long>(b) * p.T + t) * p.Hq * D + static_cast<long long>(h) * D;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const int dcol = i * 8 + qd;
            if (!live)
                continue;
            const float dq0 = st.o[i][2 * half] * p.scale, dq1 = st.o[i][2 * half + 1] * p.scale;
            const float2 al = __ldg(reinterpret_cast<const float2 *>(p.alpha + h * D + dcol));
            *reinterpret_cast<float2 *>(p.dq + off + dcol) = make_float2(dq0 * al.x, dq1 * al.y);
            const float2 x = unpack_bf16x2(*reinterpret_cast<const uint32_t *>(
                p.q + b * p.q_bstride + (static_cast<long long>(t) * p.Hq + h) * D + dcol));
            atomicAdd(&red[hh * D + dcol], x.x * dq0);
            atomicAdd(&red[hh * D + dcol + 1], x.y * dq1);
            atomicAdd(&red[G * D + hh * D + dcol], dq0);
            atomicAdd(&red[G * D + hh * D + dcol + 1], dq1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += 128) {
        atomicAdd(p.dalpha + g * G * D + i, red[i]);
        atomicAdd(p.dbeta + g * G * D + i, red[G * D + i]);
    }
}

// ------------------------------------------------------------------ dK, dV (keys on M)

template <int D, int G>
__global__ void __launch_bounds__(128) swa_bwd_dkv_kernel(const SwaBwdParams p)
{
    constexpr int KEYS = 64;     // keys of a CTA (4 warps x 16)
    constexpr int RB = 64;       // rows staged per round = RB / G tokens x G heads
    constexpr int TOKR = RB / G;
    const int kt0 = blockIdx.x * KEYS, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int KSLAB = KEYS * 128, RSLAB = RB * 128;
    uint8_t *kt = smem;                               // K of the CTA's keys
    uint8_t *vt = kt + (D / 64) * KSLAB;              // V
    uint8_t *qh = vt + (D / 64) * KSLAB;              // staged rows: q high part
    uint8_t *ql = qh + (D / 64) * RSLAB;              // q residual
    uint8_t *gt = ql + (D / 64) * RSLAB;              // dO
    float *lse_s = reinterpret_cast<float *>(gt + (D / 64) * RSLAB);  // [RB]
    float *D_s = lse_s + RB;                                          // [RB]
    const long long row_stride = static_cast<long long>(p.Hkv) * D;
    stage_kv_rows<D>(kt, KSLAB, p.k + b * p.kv_bstride + static_cast<long long>(g) * D, row_stride, kt0, KEYS, p.T,
                     threadIdx.x, 128);
    stage_kv_rows<D>(vt, KSLAB, p.v + b * p.kv_bstride + static_cast<long long>(g) * D, row_stride, kt0, KEYS, p.T,
                     threadIdx.x, 128);
    const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
    const uint32_t qhb = smem_u32(qh), qlb = smem_u32(ql), gb = smem_u32(gt);

    const int k_w0 = kt0 + 16 * warp;  // this warp's first key
    const float c2 = p.scale * kLog2eF;
    const float NEG_INF = -__int_as_float(0x7f800000);
    float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
        dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
    // A-operand (keys x d) and row-operand ldmatrix lanes
    const int a_row = (lane & 7) + (((lane >> 3) & 1) << 3), a_hi = lane >> 4;   // A: K / V rows
    const int b_row = (lane & 7) + ((lane >> 4) << 3), b_hi = (lane >> 3) & 1;   // B from row tiles (non-trans)
    const int t_row = (lane & 7) + (((lane >> 3) & 1) << 3), t_hi = lane >> 4;   // B from row tiles (trans)
    const int gk = lane >> 2, gq = (lane & 3) * 2;  // C fragment: key rows gk, gk+8; row columns gq, gq+1

    // rows attending keys kt0 .. kt0+63: tokens kt0 .. kt0 + 63 + w - 1
    const int tok_end = min(p.T, kt0 + KEYS - 1 + p.window);
    for (int tr0 = kt0; tr0 < tok_end; tr0 += TOKR) {
        __syncthreads();  // the previous round's rows are consumed
        // stage RB rows: token tr0 + r / G, head g G + r % G
        for (int i = threadIdx.x; i < RB * (D / 8); i += 128) {
            const int r = i / (D / 8), c = (i % (D / 8)) * 8;
            const int t = tr0 + r / G, h = g * G + r % G;
            uint4 hi4 = make_uint4(0u, 0u, 0u, 0u), lo4 = hi4, g4 = hi4;
            if (t < p.T) {
                const long long off = (static_cast<long long>(t) * p.Hq + h) * D + c;
                const uint4 x4 = *reinterpret_cast<const uint4 *>(p.q + b * p.q_bstride + off);
                g4 = *reinterpret_cast<const uint4 *>(p.dO + b * p.o_bstride + off);
                const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 xv = unpack_bf16x2(xw[e]);
                    const float2 al = __ldg(reinterpret_cast<const float2 *>(p.alpha + h * D + c + 2 * e));
                    const float2 be = __ldg(reinterpret_cast<const float2 *>(p.beta + h * D + c + 2 * e));
                    split_q_pair(fmaf(xv.x, al.x, be.x), fmaf(xv.y, al.y, be.y), hw[e], lw[e]);
                }
                hi4 = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                lo4 = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            const uint32_t o = tile_off(r, c, RSLAB);
            *reinterpret_cast<uint4 *>(qh + o) = hi4;
            *reinterpret_cast<uint4 *>(ql + o) = lo4;
            *reinterpret_cast<uint4 *>(gt + o) = g4;
        }
        for (int r = threadIdx.x; r < RB; r += 128) {
            const int t = tr0 + r / G, h = g * G + r % G;
            const long long ri = (static_cast<long long>(b) * p.T + t) * p.Hq + h;
            lse_s[r] = t < p.T ? p.lse[ri] : 0.f;
            D_s[r] = t < p.T ? p.Drow[ri] : 0.f;
        }
        __syncthreads();
        // this warp's keys k_w0 .. k_w0+15 against 16-row chunks whose tokens can reach them
        for (int rc = 0; rc < RB; rc += 16) {
            const int tc0 = tr0 + rc / G, tc1 = tr0 + (rc + 15) / G;
            if (tc1 < k_w0 || tc0 - p.window + 1 > k_w0 + 15 || tc0 >= p.T)
                continue;  // warp-uniform: no key of this warp is in these rows' windows
            // S^T (16 keys x 16 rows) = K q^T, two 8-row n-tiles, q as high part + residual
            float s[2][4], dpt[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
                s[i][0] = s[i][1] = s[i][2] = s[i][3] = dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t a[4], av[4], bh0, bh1, bh2, bh3, bl0, bl1, bl2, bl3, g0, g1, g2, g3;
                ldsm_x4(kbase + tile_off(16 * warp + a_row, kk * 16 + a_hi * 8, KSLAB), a[0], a[1], a[2], a[3]);
                ldsm_x4(vbase + tile_off(16 * warp + a_row, kk * 16 + a_hi * 8, KSLAB), av[0], av[1], av[2], av[3]);
                ldsm_x4(qhb + tile_off(rc + b_row, kk * 16 + b_hi * 8, RSLAB), bh0, bh1, bh2, bh3);
                ldsm_x4(qlb + tile_off(rc + b_row, kk * 16 + b_hi * 8, RSLAB), bl0, bl1, bl2, bl3);
                ldsm_x4(gb + tile_off(rc + b_row, kk * 16 + b_hi * 8, RSLAB), g0, g1, g2, g3);
                mma_16816(s[0], a, bh0, bh1);
                mma_16816(s[1], a, bh2, bh3);
                mma_16816(s[0], a, bl0, bl1);
                mma_16816(s[1], a, bl2, bl3);
                mma_16816(dpt[0], av, g0, g1);
                mma_16816(dpt[1], av, g2, g3);
            }
            // P^T, dS^T: element (key gk (+8), row column 8 i + gq (+1))
            float pt[2][4], dst[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = k_w0 + gk + ((e & 2) ? 8 : 0);
                    const int rr = rc + 8 * i + gq + (e & 1);
                    const int t = tr0 + rr / G;
                    const bool valid = t < p.T && key <= t && key >= t - p.window + 1 && key < p.T;
                    const float pr = valid ? fast_exp2(s[i][e] * c2 - lse_s[rr]) : 0.f;
                    pt[i][e] = pr;
                    dst[i][e] = pr * (dpt[i][e] - D_s[rr]);
                }
            // as A operands over the 16 rows (k): the two n-tiles' C fragments side by side
            uint32_t pa[4], da[4];
            pa[0] = pack_bf16x2(pt[0][0], pt[0][1]);
            pa[1] = pack_bf16x2(pt[0][2], pt[0][3]);
            pa[2] = pack_bf16x2(pt[1][0], pt[1][1]);
            pa[3] = pack_bf16x2(pt[1][2], pt[1][3]);
            da[0] = pack_bf16x2(dst[0][0], dst[0][1]);
            da[1] = pack_bf16x2(dst[0][2], dst[0][3]);
            da[2] = pack_bf16x2(dst[1][0], dst[1][1]);
            da[3] = pack_bf16x2(dst[1][2], dst[1][3]);
            // dV += P^T dO, dK += dS^T q (rows on k: row tiles through ldmatrix.trans)
#pragma unroll
            for (int dd = 0; dd < D / 16; ++dd) {
                uint32_t g0, g1, g2, g3, q0, q1, q2, q3;
                ldsm_x4_trans(gb + tile_off(rc + t_row, dd * 16 + t_hi * 8, RSLAB), g0, g1, g2, g3);
                ldsm_x4_trans(qhb + tile_off(rc + t_row, dd * 16 + t_hi * 8, RSLAB), q0, q1, q2, q3);
                mma_16816(dv[2 * dd], pa, g0, g1);
                mma_16816(dv[2 * dd + 1], pa, g2, g3);
                mma_16816(dk[2 * dd], da, q0, q1);
                mma_16816(dk[2 * dd + 1], da, q2, q3);
            }
        }
    }
    // write dK (scaled) and dV of the warp's 16 keys
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int key = k_w0 + gk + half * 8;
        if (key >= p.T)
            continue;
        const long long off = (static_cast<long long>(b) * p.T + key) * p.Hkv * D + static_cast<long long>(g) * D;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const int dcol = i * 8 + gq;
            *reinterpret_cast<float2 *>(p.dk + off + dcol) =
                make_float2(dk[i][2 * half] * p.scale, dk[i][2 * half + 1] * p.scale);
            *reinterpret_cast<float2 *>(p.dv + off + dcol) = make_float2(dv[i][2 * half], dv[i][2 * half + 1]);
        }
    }
}

// ------------------------------------------------------------------ host side

int swa_bwd_band_max(int G, int window)
{
    return window - 1 + 64 / G + 16;
}

size_t swa_bwd_workspace_floats(int B, int T, int Hq)
{
    return 2 * static_cast<size_t>(B) * T * Hq;
}

size_t swa_bwd_dq_smem(int D, int G, int window)
{
    return static_cast<size_t>(2 * (D / 64)) * swa_bwd_band_max(G, window) * 128 + 2 * G * D * 4 + 1024;
}

size_t swa_bwd_dkv_smem(int D)
{
    return static_cast<size_t>((D / 64)) * (2 * 64 * 128 + 3 * 64 * 128) + 2 * 64 * 4 + 1024;
}

template <int D, int G>
static cudaError_t launch_swa_bwd_t(const SwaBwdParams &p, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(p.B) * p.T * p.Hq;
    cudaError_t e0 = cudaMemsetAsync(p.dalpha, 0, sizeof(float) * p.Hq * D, stream);
    if (e0 == cudaSuccess)
        e0 = cudaMemsetAsync(p.dbeta, 0, sizeof(float) * p.Hq * D, stream);
    if (e0 != cudaSuccess)
        return e0;
    swa_bwd_d_kernel<D><<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, stream>>>(p.o, p.dO, p.Drow, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const size_t s1 = swa_bwd_dq_smem(D, G, p.window);
    auto k1 = swa_bwd_dq_kernel<D, G>;
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s1))) != cudaSuccess)
        return e;
    dim3 g1((p.T + 64 / G - 1) / (64 / G), p.B * p.Hkv);
    k1<<<g1, 128, s1, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    const size_t s2 = swa_bwd_dkv_smem(D);
    auto k2 = swa_bwd_dkv_kernel<D, G>;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s2))) != cudaSuccess)
        return e;
    dim3 g2((p.T + 63) / 64, p.B * p.Hkv);
    k2<<<g2, 128, s2, stream>>>(p);
    return cudaGetLastError();
}

bool swa_bwd_supported(int D, int G, int window)
{
    return (D == 64 || D == 128) && (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) && window >= 1 &&
           swa_bwd_dq_smem(D, G, window) <= 227 * 1024;
}

cudaError_t launch_swa_bwd(int D, int G, const SwaBwdParams &p, cudaStream_t stream)
{
#define ORTHROS_BWD_CASE(DD, GG) \
    if (D == DD && G == GG)      \
        return launch_swa_bwd_t<DD, GG>(p, stream);
    ORTHROS_BWD_CASE(128, 1)
    ORTHROS_BWD_CASE(128, 2)
    ORTHROS_BWD_CASE(128, 4)
    ORTHROS_BWD_CASE(128, 8)
    ORTHROS_BWD_CASE(128, 16)
    ORTHROS_BWD_CASE(64, 1)
    ORTHROS_BWD_CASE(64, 2)
    ORTHROS_BWD_CASE(64, 4)
    ORTHROS_BWD_CASE(64, 8)
    ORTHROS_BWD_CASE(64, 16)
#undef ORTHROS_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace orthros
