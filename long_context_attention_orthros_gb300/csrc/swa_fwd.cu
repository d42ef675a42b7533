// swa_fwd.cu -- base-stream causal sliding-window attention, Eq. (4) of
// "Orthros: Phase-Aware Heterogeneous Attention" (Sec. 2.3 of the close-reading
// notes), with the base scale-offset q = Q_raw * alpha + beta (Sec. 3.1) fused
// into the query load.
//
// Work decomposition
//   A tile is 128 query rows = TOK tokens x G query heads that share one KV head
//   (G = Hq / Hkv, TOK = 128 / G).  Row r of a tile is (token r / G, head r % G),
//   which is exactly the order in which a 4-D TMA box {64, G, TOK, 1} lands in
//   shared memory, so every K/V byte staged for the tile serves all G heads.
//   Keys are staged in blocks of 32 rows.  Tile n of a (batch, KV head) stream
//   needs key blocks kb_lo(n) .. kb_hi(n) (the band max(0, t-w+1) .. t of its
//   tokens); consecutive tiles share all but one of those blocks.
//
//   The grid is persistent (one CTA per SM).  Each CTA walks a contiguous range
//   of tiles; one producer warp streams Q tiles (double buffered) and K/V
//   blocks (ring of STAGES slots) with TMA, and keeps each K/V block resident
//   for as long as any later tile of the range still needs it, so K and V
//   leave HBM once.  Eight consumer warps own 16 rows each and run a
//   flash-style online softmax over 16-key chunks with warp MMAs, skipping
//   chunks that lie outside all of their rows' windows.  The output tile is
//   staged in shared memory and written back with a TMA store.
//
//   When the window is so wide that a tile's band does not fit in the ring,
//   blocks are streamed once per tile instead (same code, no reuse).
#include "common.cuh"
#include "kernels.cuh"
#include "xattn.cuh"

namespace orthros {

template <int D, int G>
struct SwaCfg {
    static constexpr int ROWS = 128;
    static constexpr int TOK = ROWS / G;
    static constexpr int KB = 32;  // keys per staged block
    static constexpr int SLABS = D / 64;
    static constexpr int STAGES = 8;
    static constexpr int CWARPS = 8;
    static constexpr int THREADS = (CWARPS + 1) * 32;
    static constexpr int Q_BYTES = ROWS * D * 2;
    static constexpr int Q_SLAB = ROWS * 128;
    static constexpr int KV_BYTES = KB * D * 2;  // one of K or V for one block
    static constexpr int KV_SLAB = KB * 128;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int RING_OFF = 0;
    static constexpr int Q_OFF = RING_OFF + STAGES * STAGE_BYTES;
    static constexpr int O_OFF = Q_OFF + 2 * Q_BYTES;
    static constexpr int BAR_OFF = O_OFF + Q_BYTES;
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int SMEM = BAR_OFF + NBARS * 8 + 1024;  // + alignment slack
};

__device__ __forceinline__ int swa_kb_lo(int n, int TOK, int window, int KB)
{
    const int t = n * TOK - window + 1;
    return t > 0 ? t / KB : 0;
}

__device__ __forceinline__ int swa_kb_hi(int n, int TOK, int T, int KB)
{
    int t = n * TOK + TOK - 1;
    if (t > T - 1)
        t = T - 1;
    return t / KB;
}

template <int D, int G>
__global__ void __launch_bounds__(SwaCfg<D, G>::THREADS, 1)
    swa_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                   const SwaParams p)
{
    using C = SwaCfg<D, G>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_s + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *full = bars;                 // [STAGES] K/V block landed
    uint64_t *empty = bars + C::STAGES;    // [STAGES] K/V block released by all consumers
    uint64_t *qfull = bars + 2 * C::STAGES;      // [2]
    uint64_t *qempty = bars + 2 * C::STAGES + 2; // [2]
    uint64_t *osync = bars + 2 * C::STAGES + 4;  // consumer-warp rendezvous around the O stage

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::CWARPS);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], C::CWARPS);
        }
        mbar_init(osync, C::CWARPS);
        fence_barrier_init();
    }
    __syncthreads();

    const long long gt_begin = p.total_tiles * blockIdx.x / gridDim.x;
    const long long gt_end = p.total_tiles * (blockIdx.x + 1) / gridDim.x;
    const int tps = p.tiles_per_stream;

    if (warp == C::CWARPS) {
        // ------------------------------------------------------------ producer
        if (lane != 0)
            return;
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        long long load_idx = 0, q_idx = 0;
        bool ok = true;
        auto load_block = [&](int b, int g, int kb) -> bool {
            const int s = static_cast<int>(load_idx % C::STAGES);
            if (load_idx >= C::STAGES &&
                !mbar_wait(&empty[s], static_cast<uint32_t>(((load_idx / C::STAGES) - 1) & 1)))
                return false;
            uint8_t *dst = smem + C::RING_OFF + s * C::STAGE_BYTES;
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
            for (int sl = 0; sl < C::SLABS; ++sl) {
                tma_load_4d(dst + sl * C::KV_SLAB, &kmap, &full[s], sl * 64, g, kb * C::KB, b);
                tma_load_4d(dst + C::KV_BYTES + sl * C::KV_SLAB, &vmap, &full[s], sl * 64, g,
                            kb * C::KB, b);
            }
            ++load_idx;
            return true;
        };
        auto load_q = [&](int b, int g, int n) -> bool {
            const int s = static_cast<int>(q_idx & 1);
            if (q_idx >= 2 && !mbar_wait(&qempty[s], static_cast<uint32_t>(((q_idx >> 1) - 1) & 1)))
                return false;
            uint8_t *dst = smem + C::Q_OFF + s * C::Q_BYTES;
            mbar_arrive_expect_tx(&qfull[s], C::Q_BYTES);
#pragma unroll
            for (int sl = 0; sl < C::SLABS; ++sl)
                tma_load_4d(dst + sl * C::Q_SLAB, &qmap, &qfull[s], sl * 64, g * G, n * C::TOK, b);
            ++q_idx;
            return true;
        };
        for (long long gt = gt_begin; gt < gt_end && ok;) {
            const int stream = static_cast<int>(gt / tps);
            // absolute tile indices: the launched row range starts at tile p.n_base
            const int n0r = static_cast<int>(gt % tps);
            const int n0 = p.n_base + n0r;
            const int n1 = p.n_base + static_cast<int>((tps < n0r + (gt_end - gt) ? (long long)tps : n0r + (gt_end - gt)));
            const int b = stream / p.Hkv, g = stream % p.Hkv;
            int next_kb = swa_kb_lo(n0, C::TOK, p.window, C::KB);
            for (int n = n0; n < n1 && ok; ++n) {
                ok = load_q(b, g, n);
                const int hi = swa_kb_hi(n, C::TOK, p.T, C::KB);
                int kb = p.reuse ? next_kb : swa_kb_lo(n, C::TOK, p.window, C::KB);
                for (; kb <= hi && ok; ++kb)
                    ok = load_block(b, g, kb);
                next_kb = kb;
            }
            gt += n1 - n0;
        }
        if (!ok)
            record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int R0 = warp * 16;        // first tile row of this warp
    const int gr = lane >> 2;        // fragment row (and row + 8)
    const int qd = (lane & 3) * 2;   // fragment column pair
    const int tokA_off = (R0 + gr) / G;
    const int tokB_off = (R0 + gr + 8) / G;
    const int tok_min_off = R0 / G, tok_max_off = (R0 + 15) / G;
    const int ld_row = (lane & 7) + (((lane >> 3) & 1) << 3);  // ldmatrix row (A and V^T)
    const int ld_hi = lane >> 4;                                // ldmatrix second column chunk
    const int kld_row = (lane & 7) + ((lane >> 4) << 3);        // ldmatrix row for K (B operand)
    const int kld_hi = (lane >> 3) & 1;
    const float NEG_INF = -__int_as_float(0x7f800000);

    long long load_idx = 0, q_idx = 0;
    bool ok = true;
    uint32_t osync_phase = 0;
    // bounded rendezvous of the consumer warps (an mbarrier, so a stuck peer cannot hang us)
    auto consumer_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(osync);
        const bool r = mbar_wait(osync, osync_phase & 1u);
        ++osync_phase;
        return r;
    };
    for (long long gt = gt_begin; gt < gt_end && ok;) {
        const int stream = static_cast<int>(gt / tps);
        const int n0r = static_cast<int>(gt % tps);
        const int n0 = p.n_base + n0r;
        const int n1 = p.n_base + static_cast<int>((tps < n0r + (gt_end - gt) ? (long long)tps : n0r + (gt_end - gt)));
        const int b = stream / p.Hkv, g = stream % p.Hkv;
        const int hA = g * G + (gr % G), hB = g * G + ((gr + 8) % G);
        const long long seg_base = load_idx;  // ring index of block kb_lo(n0) in reuse mode
        const int seg_kb0 = swa_kb_lo(n0, C::TOK, p.window, C::KB);
        for (int n = n0; n < n1 && ok; ++n) {
            const int t0 = n * C::TOK;
            // ---- Q fragments with the fused scale-offset
            const int qs = static_cast<int>(q_idx & 1);
            if (!mbar_wait(&qfull[qs], static_cast<uint32_t>((q_idx >> 1) & 1))) {
                ok = false;
                break;
            }
            uint32_t qa[D / 16][4], ql[D / 16][4];  // scaled query: bf16 high part and residual
            const uint32_t qbase = sbase + C::Q_OFF + qs * C::Q_BYTES;
#pragma unroll
            for (int kt = 0; kt < D / 16; ++kt) {
                const uint32_t a = qbase + (kt * 16 / 64) * C::Q_SLAB +
                                   sw128_offset(R0 + ld_row, ((kt * 16) % 64) / 8 + ld_hi);
                ldsm_x4(a, qa[kt][0], qa[kt][1], qa[kt][2], qa[kt][3]);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&qempty[qs]);
            ++q_idx;
#pragma unroll
            for (int kt = 0; kt < D / 16; ++kt) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int h = (r & 1) ? hB : hA;
                    const int dd = kt * 16 + qd + ((r & 2) ? 8 : 0);
                    const float2 al = __ldg(reinterpret_cast<const float2 *>(p.alpha + h * D + dd));
                    const float2 be = __ldg(reinterpret_cast<const float2 *>(p.beta + h * D + dd));
                    const float2 x = unpack_bf16x2(qa[kt][r]);
                    split_q_pair(fmaf(x.x, al.x, be.x) * p.qscale, fmaf(x.y, al.y, be.y) * p.qscale,
                                 qa[kt][r], ql[kt][r]);
                }
            }

            float o[D / 8][4];
#pragma unroll
            for (int i = 0; i < D / 8; ++i)
                o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            float mA = NEG_INF, mB = NEG_INF, lA = 0.f, lB = 0.f;
            const int tA = t0 + tokA_off, tB = t0 + tokB_off;
            const int tmin = t0 + tok_min_off, tmax = t0 + tok_max_off;

            const int kb_lo = swa_kb_lo(n, C::TOK, p.window, C::KB);
            const int kb_hi = swa_kb_hi(n, C::TOK, p.T, C::KB);
            for (int kb = kb_lo; kb <= kb_hi; ++kb) {
                const long long idx = p.reuse ? seg_base + (kb - seg_kb0) : load_idx + (kb - kb_lo);
                const int s = static_cast<int>(idx % C::STAGES);
                if (!mbar_wait(&full[s], static_cast<uint32_t>((idx / C::STAGES) & 1))) {
                    ok = false;
                    break;
                }
                const uint32_t kbase = sbase + C::RING_OFF + s * C::STAGE_BYTES;
                const uint32_t vbase = kbase + C::KV_BYTES;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int j0 = kb * C::KB + c * 16;
                    if (j0 > tmax || j0 + 15 < tmin - p.window + 1)
                        continue;  // chunk outside every row's window (warp-uniform)
                    float sacc[2][4];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
                    for (int kt = 0; kt < D / 16; ++kt) {
                        uint32_t b0, b1, b2, b3;
                        const uint32_t a = kbase + (kt * 16 / 64) * C::KV_SLAB +
                                           sw128_offset(c * 16 + kld_row, ((kt * 16) % 64) / 8 + kld_hi);
                        ldsm_x4(a, b0, b1, b2, b3);
                        mma_16816(sacc[0], qa[kt], b0, b1);
                        mma_16816(sacc[1], qa[kt], b2, b3);
                        mma_16816(sacc[0], ql[kt], b0, b1);
                        mma_16816(sacc[1], ql[kt], b2, b3);
                    }
                    const bool full_chunk = (j0 >= 0) && (j0 + 15 <= tmin) && (j0 > tmax - p.window);
                    if (!full_chunk) {
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = j0 + i * 8 + qd + (e & 1);
                                const int t = (e & 2) ? tB : tA;
                                if (!(j <= t && j > t - p.window && j >= 0))
                                    sacc[i][e] = NEG_INF;
                            }
                    }
                    float cmA = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
                    float cmB = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
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
                        pr[i][0] = fast_exp2(sacc[i][0] - uA);
                        pr[i][1] = fast_exp2(sacc[i][1] - uA);
                        pr[i][2] = fast_exp2(sacc[i][2] - uB);
                        pr[i][3] = fast_exp2(sacc[i][3] - uB);
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
                        const uint32_t a = vbase + (dp * 16 / 64) * C::KV_SLAB +
                                           sw128_offset(c * 16 + ld_row, ((dp * 16) % 64) / 8 + ld_hi);
                        ldsm_x4_trans(a, v0, v1, v2, v3);
                        mma_16816(o[2 * dp], pa, v0, v1);
                        mma_16816(o[2 * dp + 1], pa, v2, v3);
                    }
                }
                if (!p.reuse) {
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&empty[s]);
                }
            }
            if (!ok)
                break;
            if (p.reuse) {
                // release blocks no later tile of this segment needs
                const int rel_hi = (n + 1 < n1) ? swa_kb_lo(n + 1, C::TOK, p.window, C::KB) - 1
                                                : swa_kb_hi(n1 - 1, C::TOK, p.T, C::KB);
                __syncwarp();
                if (lane == 0)
                    for (int kb = kb_lo; kb <= rel_hi; ++kb)
                        mbar_arrive(&empty[static_cast<int>((seg_base + (kb - seg_kb0)) % C::STAGES)]);
            } else {
                load_idx += kb_hi - kb_lo + 1;
            }

            // ---- epilogue: normalise, stage as bf16 (128-byte swizzle), TMA store
            lA += __shfl_xor_sync(0xffffffffu, lA, 1);
            lA += __shfl_xor_sync(0xffffffffu, lA, 2);
            lB += __shfl_xor_sync(0xffffffffu, lB, 1);
            lB += __shfl_xor_sync(0xffffffffu, lB, 2);
            const float iA = lA > 0.f ? 1.f / lA : 0.f;
            const float iB = lB > 0.f ? 1.f / lB : 0.f;
            if (p.lse != nullptr && (lane & 3) == 0) {  // the rows' log-sum-exp, natural log
                if (tA < p.T && lA > 0.f)
                    p.lse[(static_cast<long long>(b) * p.T + tA) * p.Hq + hA] = (mA + __log2f(lA)) * 0.6931471805599453f;
                if (tB < p.T && lB > 0.f)
                    p.lse[(static_cast<long long>(b) * p.T + tB) * p.Hq + hB] = (mB + __log2f(lB)) * 0.6931471805599453f;
            }
            if (threadIdx.x == 0)
                bulk_wait_read_all();  // previous tile's store has finished reading the stage
            if (!consumer_sync()) {
                ok = false;
                break;
            }
            uint8_t *ost = smem + C::O_OFF;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                const int dcol = i * 8 + qd;
                const int sl = dcol / 64, ch = (dcol % 64) / 8;
                *reinterpret_cast<uint32_t *>(ost + sl * C::Q_SLAB + sw128_offset(R0 + gr, ch) + qd * 2) =
                    pack_bf16x2(o[i][0] * iA, o[i][1] * iA);
                *reinterpret_cast<uint32_t *>(ost + sl * C::Q_SLAB + sw128_offset(R0 + gr + 8, ch) + qd * 2) =
                    pack_bf16x2(o[i][2] * iB, o[i][3] * iB);
            }
            fence_proxy_async_smem();
            if (!consumer_sync()) {
                ok = false;
                break;
            }
            if (threadIdx.x == 0) {
#pragma unroll
                for (int sl = 0; sl < C::SLABS; ++sl)
                    tma_store_4d(&omap, ost + sl * C::Q_SLAB, sl * 64, g * G, t0, b);
                bulk_commit();
            }
        }
        if (p.reuse)
            load_idx = seg_base + (swa_kb_hi(n1 - 1, C::TOK, p.T, C::KB) - seg_kb0 + 1);
        gt += n1 - n0;
    }
    if (threadIdx.x == 0)
        bulk_wait_all();
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------------ host launch

template <int D, int G>
static cudaError_t launch_swa_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const SwaParams &p, int num_sms,
                                cudaStream_t stream)
{
    using C = SwaCfg<D, G>;
    auto kern = swa_fwd_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    long long grid = p.total_tiles < num_sms ? p.total_tiles : num_sms;
    if (grid < 1)
        grid = 1;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(q, k, v, o, p);
    return cudaGetLastError();
}

cudaError_t launch_swa(int D, int G, const CUtensorMap &q, const CUtensorMap &k,
                       const CUtensorMap &v, const CUtensorMap &o, SwaParams p, int num_sms,
                       cudaStream_t stream)
{
    const int TOK = 128 / G, KB = 32, STAGES = 8;
    // the row range [row_begin, row_end) as whole tiles (row_begin is a multiple of 128)
    p.n_base = p.row_begin / TOK;
    p.tiles_per_stream = (p.row_end + TOK - 1) / TOK - p.n_base;
    // widest band of key blocks any tile can need (worst-case alignment)
    const long long band = (static_cast<long long>(p.window) - 1 + TOK + KB - 1) / KB + 1;
    p.reuse = band <= STAGES ? 1 : 0;
    p.total_tiles *= p.tiles_per_stream;
    // tensor-memory kernel whenever a tile's whole band fits its ring and tensor memory
    if (swa_tc_supported(D, G, p.window))
        return launch_swa_tc(D, G, q, k, v, o, p, num_sms, stream);
#define ORTHROS_SWA_CASE(DD, GG) \
    if (D == DD && G == GG)      \
        return launch_swa_t<DD, GG>(q, k, v, o, p, num_sms, stream);
    ORTHROS_SWA_CASE(128, 1)
    ORTHROS_SWA_CASE(128, 2)
    ORTHROS_SWA_CASE(128, 4)
    ORTHROS_SWA_CASE(128, 8)
    ORTHROS_SWA_CASE(128, 16)
    ORTHROS_SWA_CASE(64, 1)
    ORTHROS_SWA_CASE(64, 2)
    ORTHROS_SWA_CASE(64, 4)
    ORTHROS_SWA_CASE(64, 8)
    ORTHROS_SWA_CASE(64, 16)
#undef ORTHROS_SWA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace orthros
