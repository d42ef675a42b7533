// attn_bwd.cu -- gradients of "Orthros: Phase-Aware Heterogeneous Attention" for
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
// Three launches (warp MMAs, bf16 operands, fp32 accumulation):
//   attn_bwd_d_kernel    D = dO . o per row;
//   attn_bwd_dq_kernel   rows on the MMA's M side: K/V stream through a two-stage
//                        shared-memory ring of 64-key blocks (cp.async); pass 1 takes
//                        each row's log2-sum-exp (kept for the next kernel), pass 2
//                        dP = dO V^T, dS = P (dP - D), dQ += dS K; then dq_raw, and
//                        dalpha / dbeta through shared, then global, atomics;
//   attn_bwd_dkv_kernel  keys on the M side: a CTA owns 64 keys and stages, round by
//                        round, the query rows that can see them; each warp keeps dK,
//                        dV of its 16 keys in registers (S^T = K q^T, dP^T = V dO^T,
//                        dV += P^T dO, dK += dS^T q) and writes them once.
// q . k takes q as a bf16 high part plus residual; P and dS enter the second
// products as bf16, and q enters dK as its bf16 high part.  Outputs are fp32.
#include "common.cuh"
#include "kernels.cuh"
#include "xattn.cuh"

namespace orthros {

namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr int BWD_ROWS = 64;  // query rows of a dq CTA, and rows staged per dk/dv round
constexpr int BWD_KEYS = 64;  // keys of a dk/dv CTA, and keys per streamed dq block

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

}  // namespace

// ------------------------------------------------------------------ D = dO . o

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_d_kernel(const orthros_bf16 *o, const orthros_bf16 *dO, float *Dout,
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
#pragma unroll 1
    for (int pass = 1; pass <= 2; ++pass) {
        if (pass == 2) {
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

// ------------------------------------------------------------------ dK, dV (keys on M)

template <int D, int G, bool COPY>
__global__ void __launch_bounds__(128) attn_bwd_dkv_kernel(const AttnBwdParams p)
{
    constexpr int RB = BWD_ROWS;  // rows staged per round = RB / G units x G heads
    constexpr int TOKR = RB / G;
    constexpr int KSLAB = BWD_KEYS * 128, RSLAB = RB * 128;
    const int kt0 = blockIdx.x * BWD_KEYS, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *kt = smem;                   // K of the CTA's keys
    uint8_t *vt = kt + (D / 64) * KSLAB;  // V
    uint8_t *qh = vt + (D / 64) * KSLAB;  // staged rows: q high part
    uint8_t *ql = qh + (D / 64) * RSLAB;  // q residual
    uint8_t *gt = ql + (D / 64) * RSLAB;  // dO
    float *lse_s = reinterpret_cast<float *>(gt + (D / 64) * RSLAB);  // [RB]
    float *D_s = lse_s + RB;                                          // [RB]
    int *P_s = reinterpret_cast<int *>(D_s + RB);                     // [RB] position, -1: none
    const long long kv_rs = static_cast<long long>(p.Hkv) * D;
    const long long kv_b = static_cast<long long>(b) * p.T_kv * kv_rs + static_cast<long long>(g) * D;
    for (int i = threadIdx.x; i < BWD_KEYS * (D / 8); i += 128) {
        const int r = i / (D / 8), c = (i % (D / 8)) * 8;
        const int key = kt0 + r;
        uint4 kv4 = make_uint4(0u, 0u, 0u, 0u), vv4 = kv4;
        if (key < p.T_kv) {
            kv4 = *reinterpret_cast<const uint4 *>(p.k + kv_b + key * kv_rs + c);
            vv4 = *reinterpret_cast<const uint4 *>(p.v + kv_b + key * kv_rs + c);
        }
        *reinterpret_cast<uint4 *>(kt + tile_off(r, c, KSLAB)) = kv4;
        *reinterpret_cast<uint4 *>(vt + tile_off(r, c, KSLAB)) = vv4;
    }
    const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
    const uint32_t qhb = smem_u32(qh), qlb = smem_u32(ql), gb = smem_u32(gt);

    const int k_w0 = kt0 + 16 * warp;  // this warp's first key
    const float c2 = p.scale * kLog2eF;
    const long long q_bs = static_cast<long long>(p.n_units) * p.Hq * D;
    float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
        dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
    const int a_row = (lane & 7) + (((lane >> 3) & 1) << 3), a_hi = lane >> 4;  // A: K / V rows
    const int b_row = (lane & 7) + ((lane >> 4) << 3), b_hi = (lane >> 3) & 1;  // B from row tiles
    const int t_row = a_row, t_hi = a_hi;                                       // B from row tiles, transposed
    const int gk = lane >> 2, gq = (lane & 3) * 2;  // C fragment: key rows gk, gk+8; row columns gq, gq+1

    // units whose keys can include the CTA's: base tokens kt0 .. kt0+63+w-1; every copy
    const int u_begin = COPY ? 0 : kt0;
    const int u_end = COPY ? p.n_units
                           : static_cast<int>(min(static_cast<long long>(p.n_units),
                                                  static_cast<long long>(kt0) + BWD_KEYS - 1 + p.window));
#pragma unroll 1
    for (int tr0 = u_begin; tr0 < u_end; tr0 += TOKR) {
        __syncthreads();  // the previous round's rows are consumed
        if (COPY) {
            int need = 0;
            for (int r = threadIdx.x; r < TOKR; r += 128)
                need |= unit_pos<COPY>(p, b, tr0 + r) >= kt0;
            if (!__syncthreads_or(need))
                continue;  // no copy of this round reaches the CTA's keys
        }
        for (int i = threadIdx.x; i < RB * (D / 8); i += 128) {
            const int r = i / (D / 8), c = (i % (D / 8)) * 8;
            const int u = tr0 + r / G, h = g * G + r % G;
            uint4 hi4 = make_uint4(0u, 0u, 0u, 0u), lo4 = hi4, g4 = hi4;
            if (unit_pos<COPY>(p, b, u) >= 0) {
                const long long off = b * q_bs + (static_cast<long long>(u) * p.Hq + h) * D + c;
                const uint4 x4 = *reinterpret_cast<const uint4 *>(p.q + off);
                g4 = *reinterpret_cast<const uint4 *>(p.dO + off);
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
            const int u = tr0 + r / G, h = g * G + r % G;
            const int P = unit_pos<COPY>(p, b, u);
            const long long ri = (static_cast<long long>(b) * p.n_units + u) * p.Hq + h;
            P_s[r] = P;
            lse_s[r] = P >= 0 ? p.lse[ri] : 0.f;
            D_s[r] = P >= 0 ? p.Drow[ri] : 0.f;
        }
        __syncthreads();
#pragma unroll 1
        for (int rc = 0; rc < RB; rc += 16) {
            // skip chunks none of whose rows sees a key of this warp (warp-uniform)
            const int Pl = P_s[rc + (lane & 15)];
            const int lol = Pl >= 0 ? Pl - p.window + 1 : 0x7fffffff;
            if (__reduce_max_sync(0xffffffffu, Pl) < k_w0 || __reduce_min_sync(0xffffffffu, lol) > k_w0 + 15)
                continue;
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
                    const int P = P_s[rr];
                    const bool valid = key <= P && key >= P - p.window + 1;  // P = -1: none
                    const float pr = valid ? fast_exp2(s[i][e] * c2 - lse_s[rr]) : 0.f;
                    pt[i][e] = pr;
                    dst[i][e] = pr * (dpt[i][e] - D_s[rr]);
                }
            uint32_t pa[4], da[4];
            pa[0] = pack_bf16x2(pt[0][0], pt[0][1]);
            pa[1] = pack_bf16x2(pt[0][2], pt[0][3]);
            pa[2] = pack_bf16x2(pt[1][0], pt[1][1]);
            pa[3] = pack_bf16x2(pt[1][2], pt[1][3]);
            da[0] = pack_bf16x2(dst[0][0], dst[0][1]);
            da[1] = pack_bf16x2(dst[0][2], dst[0][3]);
            da[2] = pack_bf16x2(dst[1][0], dst[1][1]);
            da[3] = pack_bf16x2(dst[1][2], dst[1][3]);
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
    // write (or add) dK (scaled) and dV of the warp's 16 keys
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int key = k_w0 + gk + half * 8;
        if (key >= p.T_kv)
            continue;
        const long long off = (static_cast<long long>(b) * p.T_kv + key) * kv_rs + static_cast<long long>(g) * D;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const int dcol = i * 8 + gq;
            float2 nk = make_float2(dk[i][2 * half] * p.scale, dk[i][2 * half + 1] * p.scale);
            float2 nv = make_float2(dv[i][2 * half], dv[i][2 * half + 1]);
            float2 *pk = reinterpret_cast<float2 *>(p.dk + off + dcol);
            float2 *pv = reinterpret_cast<float2 *>(p.dv + off + dcol);
            if (p.accumulate) {
                const float2 ok = *pk, ov = *pv;
                nk.x += ok.x;
                nk.y += ok.y;
                nv.x += ov.x;
                nv.y += ov.y;
            }
            *pk = nk;
            *pv = nv;
        }
    }
}

// ------------------------------------------------------------------ host side

size_t attn_bwd_workspace_floats(int B, int n_units, int Hq)
{
    return 2 * static_cast<size_t>(B) * n_units * Hq;
}

static size_t dq_smem(int D, int G)
{
    return static_cast<size_t>(4) * (D / 64) * BWD_KEYS * 128 + 2 * G * D * 4 + 16 + 1024;
}

static size_t dkv_smem(int D)
{
    return static_cast<size_t>(D / 64) * (2 * BWD_KEYS * 128 + 3 * BWD_ROWS * 128) + 3 * BWD_ROWS * 4 + 1024;
}

template <int D, int G, bool COPY>
static cudaError_t launch_attn_bwd_t(const AttnBwdParams &p, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(p.B) * p.n_units * p.Hq;
    cudaError_t e = cudaMemsetAsync(p.dalpha, 0, sizeof(float) * p.Hq * D, stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(p.dbeta, 0, sizeof(float) * p.Hq * D, stream);
    if (e != cudaSuccess)
        return e;
    if (rows > 0) {
        attn_bwd_d_kernel<D><<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, stream>>>(p.o, p.dO, p.Drow,
                                                                                                rows);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        const size_t s1 = dq_smem(D, G);
        auto k1 = attn_bwd_dq_kernel<D, G, COPY>;
        if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s1))) !=
            cudaSuccess)
            return e;
        constexpr int UNITS = BWD_ROWS / G;
        dim3 g1((p.n_units + UNITS - 1) / UNITS, p.B * p.Hkv);
        k1<<<g1, 128, s1, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    // dk/dv also runs without query rows: it writes (or keeps) zeros
    const size_t s2 = dkv_smem(D);
    auto k2 = attn_bwd_dkv_kernel<D, G, COPY>;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s2))) !=
        cudaSuccess)
        return e;
    dim3 g2((p.T_kv + BWD_KEYS - 1) / BWD_KEYS, p.B * p.Hkv);
    k2<<<g2, 128, s2, stream>>>(p);
    return cudaGetLastError();
}

template <bool COPY>
static cudaError_t dispatch_attn_bwd(int D, int G, const AttnBwdParams &p, cudaStream_t stream)
{
#define ORTHROS_BWD_CASE(DD, GG) \
    if (D == DD && G == GG)      \
        return launch_attn_bwd_t<DD, GG, COPY>(p, stream);
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

cudaError_t launch_attn_bwd(int D, int G, const AttnBwdParams &p, cudaStream_t stream)
{
    return p.pos ? dispatch_attn_bwd<true>(D, G, p, stream) : dispatch_attn_bwd<false>(D, G, p, stream);
}

}  // namespace orthros
