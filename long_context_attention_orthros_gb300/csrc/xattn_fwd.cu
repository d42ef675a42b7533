// xattn_fwd.cu -- output-copy full causal cross-attention, Eq. (5) of
// "Orthros: Phase-Aware Heterogeneous Attention" (Sec. 2.3 / 2.4 of the
// close-reading notes), with the copy scale-offset q' = Q'_raw * alpha' + beta'
// fused into the query load.
//
// A copy i at original position pos_i attends over base keys 0 .. pos_i of its
// own sequence; the mask uses pos_i, never the copy's slot in memory (copies may
// be appended after the base tokens, Algorithm 2).  Query rows of one KV head are
// grouped: row r of a (batch, KV head) pair is (copy r / G, head r % G), so each
// K/V byte staged in shared memory serves every query head that reads it (GQA).
//
// Split-KV: grid (split, row tile, batch * KV head).  A CTA streams the keys
// [split * chunk, min((split + 1) * chunk, kmax + 1)) of its KV head through a
// 3-stage TMA ring (64-key blocks, 128-byte swizzle) filled by one producer
// warp; kmax is the largest position among its rows.  Four consumer warps run
// the online softmax with warp MMAs:
//   * at most 8 rows (T_out * G <= 8, e.g. one copy of G = 4 heads): the rows on
//     the MMA's N side and 16 keys on M (half the MMAs of a 16-row tile); each
//     warp takes one 16-key chunk of every block and the four warps merge their
//     results in shared memory (one partial per CTA);
//   * up to 16 rows: all four warps share the same 16 rows and take every
//     fourth 16-key chunk of a block (4 partial results per CTA);
//   * many rows: each warp owns 16 rows and walks every chunk.
// Partials are unnormalised (max, sum, o[d]) per row; a second kernel merges the
// partials of a row with a warp-shuffle log-sum-exp reduction.  When a row has a
// single partial the first kernel writes the output directly.
#include "kernels.cuh"
#include "xattn.cuh"

namespace orthros {

template <int D>
struct XCfg {
    static constexpr int KB = 64;
    static constexpr int SLAB = KB * 128;
    static constexpr int KV_BYTES = KB * D * 2;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int STAGES = 3;
    static constexpr int CWARPS = 4;
    static constexpr int THREADS = (CWARPS + 1) * 32;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int MISC_OFF = BAR_OFF + 2 * STAGES * 8;
    static constexpr int SMEM = MISC_OFF + 64 * 4 + 1024;
};

template <int D, int WK>
__global__ void __launch_bounds__(XCfg<D>::THREADS)
    xattn_partial_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const XattnParams p)
{
    using C = XCfg<D>;
    constexpr int RPC = 16 * (C::CWARPS / WK);  // query rows per CTA
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_s + pad;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    int *s_pos = reinterpret_cast<int *>(smem + C::MISC_OFF);  // [RPC], -1 = masked row

    const int split = blockIdx.x, rt = blockIdx.y, bh = blockIdx.z;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int row0 = rt * RPC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x < RPC) {
        const int r = row0 + threadIdx.x;
        int ps = -1;
        if (r < p.R) {
            ps = p.pos[static_cast<long long>(b) * p.T_out + r / p.G];
            if (ps < 0 || ps >= p.T_kv) {
                if (split == 0 && r % p.G == 0)
                    record_error(p.dev_err, ORTHROS_DEVERR_POSITION);
                ps = -1;
            }
        }
        s_pos[threadIdx.x] = ps;
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
    for (int i = 0; i < RPC; ++i)
        kmax = max(kmax, s_pos[i]);
    const int js = split * p.chunk;
    const int je = min(js + p.chunk, kmax + 1);
    const int nblk = je > js ? (je - js + C::KB - 1) / C::KB : 0;

    if (warp == C::CWARPS) {
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
                tma_load_4d(dst + sl * C::SLAB, &kmap, &full[s], sl * 64, g, js + i * C::KB, b);
                tma_load_4d(dst + C::KV_BYTES + sl * C::SLAB, &vmap, &full[s], sl * 64, g,
                            js + i * C::KB, b);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int rg = warp / WK, kl = warp % WK;
    const int gr = lane >> 2, qd = (lane & 3) * 2;
    const int rA = rg * 16 + gr, rB = rA + 8;
    // padding rows (beyond R) borrow kmax so they never force the masked path;
    // their results are never written.  Rows with a bad position keep -1.
    auto lim_of = [&](int r) { return (row0 + r < p.R) ? s_pos[r] : kmax; };
    const int limA = lim_of(rA), limB = lim_of(rB);
    int pmin = 0x7fffffff, pmax = -1;
    for (int i = 0; i < 16; ++i) {
        const int l = lim_of(rg * 16 + i);
        pmin = min(pmin, l);
        pmax = max(pmax, l);
    }

    WarpRows16<D> st;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = (r & 1) ? rB : rA;
            const int grow = row0 + row;
            const int dcol = kt * 16 + qd + ((r & 2) ? 8 : 0);
            uint32_t hi = 0, lo = 0;
            if (grow < p.R && s_pos[row] >= 0) {
                const int h = g * p.G + grow % p.G;
                const orthros_bf16 *qrow =
                    p.qc + b * p.qc_bstride + (static_cast<long long>(grow / p.G) * p.Hq + h) * D;
                load_q_pair(qrow, p.alpha_c + h * D, p.beta_c + h * D, dcol, p.qscale, hi, lo);
            }
            st.qa[kt][r] = hi;
            st.ql[kt][r] = lo;
        }
    st.reset();

    bool ok = true;
    for (int i = 0; i < nblk && ok; ++i) {
        const int s = i % C::STAGES;
        if (!mbar_wait(&full[s], static_cast<uint32_t>((i / C::STAGES) & 1))) {
            ok = false;
            break;
        }
        const uint32_t kbase = sbase + s * C::STAGE_BYTES;
#pragma unroll
        for (int c = kl; c < 4; c += WK) {
            const int j0 = js + i * C::KB + c * 16;
            if (j0 > pmax)
                continue;
            st.step(kbase, C::SLAB, kbase + C::KV_BYTES, C::SLAB, c * 16, j0, limA, limB, j0 + 15 <= pmin);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[s]);
    }
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);

    st.finish_sums();
    const int BH = p.B * p.Hkv;
    const int part = split * WK + kl;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int row = half ? rB : rA;
        const int grow = row0 + row;
        if (grow >= p.R)
            continue;
        const float m = half ? st.mB : st.mA;
        const float l = half ? st.lB : st.lA;
        if (p.direct) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int h = g * p.G + grow % p.G;
            if (p.lse != nullptr && (lane & 3) == 0)
                p.lse[(static_cast<long long>(b) * p.T_out + grow / p.G) * p.Hq + h] =
                    l > 0.f ? (m + __log2f(l)) * kLn2F : -__int_as_float(0x7f800000);
            orthros_bf16 *orow =
                p.oc + b * p.oc_bstride + (static_cast<long long>(grow / p.G) * p.Hq + h) * D;
#pragma unroll
            for (int i = 0; i < D / 8; ++i)
                *reinterpret_cast<uint32_t *>(orow + i * 8 + qd) =
                    pack_bf16x2(st.o[i][half * 2] * inv, st.o[i][half * 2 + 1] * inv);
        } else {
            const long long slot = (static_cast<long long>(part) * BH + bh) * p.R + grow;
            float *po = p.part_o + slot * D;
#pragma unroll
            for (int i = 0; i < D / 8; ++i)
                *reinterpret_cast<float2 *>(po + i * 8 + qd) =
                    make_float2(st.o[i][half * 2], st.o[i][half * 2 + 1]);
            if ((lane & 3) == 0)
                p.part_ml[slot] = make_float2(m, l);
        }
    }
}

// At most 8 rows of one (batch, KV head): grid (split, 1, batch * KV head).  The rows sit on the
// MMA's N side (WarpKeys16: S^T = K q^T, O^T += V^T P^T), warp w takes keys 16 w .. 16 w + 15 of
// every 64-key block, and the four warps' (max, sum, o) are merged in shared memory (the ring is
// free once every block has been consumed) into one partial per CTA, or the output when the CTA
// is the row's only split.
template <int D>
__global__ void __launch_bounds__(XCfg<D>::THREADS)
    xattn_partial_keys_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                              const XattnParams p)
{
    using C = XCfg<D>;
    constexpr int RMAX = 8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_s + pad;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    int *s_pos = reinterpret_cast<int *>(smem + C::MISC_OFF);  // [RMAX], -1 = masked row

    const int split = blockIdx.x, bh = blockIdx.z;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x < RMAX) {
        const int r = threadIdx.x;
        int ps = -1;
        if (r < p.R) {
            ps = p.pos[static_cast<long long>(b) * p.T_out + r / p.G];
            if (ps < 0 || ps >= p.T_kv) {
                if (split == 0 && r % p.G == 0)
                    record_error(p.dev_err, ORTHROS_DEVERR_POSITION);
                ps = -1;
            }
        }
        s_pos[r] = ps;
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
    const int js = split * p.chunk;
    const int je = min(js + p.chunk, kmax + 1);
    const int nblk = je > js ? (je - js + C::KB - 1) / C::KB : 0;

    if (warp == C::CWARPS) {
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
                tma_load_4d(dst + sl * C::SLAB, &kmap, &full[s], sl * 64, g, js + i * C::KB, b);
                tma_load_4d(dst + C::KV_BYTES + sl * C::SLAB, &vmap, &full[s], sl * 64, g,
                            js + i * C::KB, b);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // q^T fragments hold row lane / 4; the lane keeps rows 2 (lane % 4) + {0, 1}.  Padding rows
    // (beyond R) borrow kmax so they never force the masked path; their results are never
    // written.  Rows with a bad position keep -1 (every key masked).
    WarpKeys16<D, 1, false> st;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int row = lane >> 2;
            const int dcol = kt * 16 + 2 * (lane & 3) + 8 * hf;
            uint32_t hi = 0, lo = 0;
            if (row < p.R && s_pos[row] >= 0) {
                const int h = g * p.G + row % p.G;
                const orthros_bf16 *qrow = p.qc + b * p.qc_bstride + (static_cast<long long>(row / p.G) * p.Hq + h) * D;
                load_q_pair(qrow, p.alpha_c + h * D, p.beta_c + h * D, dcol, p.qscale, hi, lo);
            }
            st.qb[0][kt][hf] = hi;
            st.ql[0][kt][hf] = lo;
        }
    st.reset();
    auto lim_of = [&](int r) { return r < p.R ? s_pos[r] : kmax; };
    int lim[1][2];
    lim[0][0] = lim_of(2 * (lane & 3));
    lim[0][1] = lim_of(2 * (lane & 3) + 1);
    int pmin = 0x7fffffff, pmax = -1;
    for (int i = 0; i < RMAX; ++i) {
        pmin = min(pmin, lim_of(i));
        pmax = max(pmax, lim_of(i));
    }

    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
        const int s = i % C::STAGES;
        if (!mbar_wait(&full[s], static_cast<uint32_t>((i / C::STAGES) & 1))) {
            ok = false;
            break;
        }
        const uint32_t kbase = sbase + s * C::STAGE_BYTES;
        const int j0 = js + i * C::KB + warp * 16;
        if (j0 <= pmax)
            st.step(kbase, C::SLAB, kbase + C::KV_BYTES, C::SLAB, warp * 16, j0, lim, j0 + 15 <= pmin);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[s]);
    }
    if (!ok && lane == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    st.finish_sums();

    // the four warps' results, each scaled to the CTA's max, summed through shared memory
    constexpr int CT = C::CWARPS * 32;
    float *ms = reinterpret_cast<float *>(smem);  // [CWARPS][RMAX] max
    float *ls = ms + C::CWARPS * RMAX;            // [CWARPS][RMAX] sum
    float *os = ls + C::CWARPS * RMAX;            // [CWARPS][RMAX][D] output
    named_barrier(3, CT);  // every warp is past its last block: the ring may be overwritten
#pragma unroll
    for (int r2 = 0; r2 < 2; ++r2)
        if ((lane >> 2) == 0) {
            ms[warp * RMAX + 2 * lane + r2] = st.m[0][r2];
            ls[warp * RMAX + 2 * lane + r2] = st.l[0][r2];
        }
    named_barrier(3, CT);
    const float NEG_INF = -__int_as_float(0x7f800000);
#pragma unroll
    for (int r2 = 0; r2 < 2; ++r2) {
        const int row = 2 * (lane & 3) + r2;
        float M = NEG_INF;
#pragma unroll
        for (int w = 0; w < C::CWARPS; ++w)
            M = fmaxf(M, ms[w * RMAX + row]);
        const float f = (M == NEG_INF || st.m[0][r2] == NEG_INF) ? 0.f : fast_exp2(st.m[0][r2] - M);
        float *po = os + (warp * RMAX + row) * D + (lane >> 2);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            po[16 * mt] = st.o[0][mt][r2] * f;
            po[16 * mt + 8] = st.o[0][mt][2 + r2] * f;
        }
    }
    named_barrier(3, CT);
    const int BH = p.B * p.Hkv;
    const int tid = threadIdx.x;
    for (int i = tid; i < p.R * (D / 2); i += CT) {  // two columns per thread and step
        const int row = i / (D / 2), c = 2 * (i % (D / 2));
        float M = NEG_INF, L = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int w = 0; w < C::CWARPS; ++w)
            M = fmaxf(M, ms[w * RMAX + row]);
#pragma unroll
        for (int w = 0; w < C::CWARPS; ++w) {
            if (ms[w * RMAX + row] != NEG_INF)
                L += ls[w * RMAX + row] * fast_exp2(ms[w * RMAX + row] - M);
            a0 += os[(w * RMAX + row) * D + c];
            a1 += os[(w * RMAX + row) * D + c + 1];
        }
        const int h = g * p.G + row % p.G, copy = row / p.G;
        if (p.direct) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
            *reinterpret_cast<uint32_t *>(p.oc + b * p.oc_bstride + (static_cast<long long>(copy) * p.Hq + h) * D + c) =
                pack_bf16x2(a0 * inv, a1 * inv);
            if (c == 0 && p.lse != nullptr)
                p.lse[(static_cast<long long>(b) * p.T_out + copy) * p.Hq + h] =
                    L > 0.f ? (M + __log2f(L)) * kLn2F : NEG_INF;
        } else {
            const long long slot = (static_cast<long long>(split) * BH + bh) * p.R + row;
            *reinterpret_cast<float2 *>(p.part_o + slot * D + c) = make_float2(a0, a1);
            if (c == 0)
                p.part_ml[slot] = make_float2(M, L);
        }
    }
}

// The same work as xattn_partial_keys_kernel on a fixed number of CTAs that walk the (split,
// batch * KV head) items, for a copies' pass that runs beside the persistent SWA kernel on the
// SMs it leaves: a CTA takes more than half of an SM's shared memory, so however the two grids
// are dispatched the pass holds at most gridDim.x SMs.  Each CTA runs two independent lanes of
// one producer warp and four consumer warps, each lane with its own ring and its own scratch
// for the warps' merge (so the next item's blocks load while an item is merged).
template <int D>
struct XpCfg {
    using X = XCfg<D>;
    static constexpr int RMAX = 8;
    static constexpr int LANE_THREADS = X::THREADS;                     // 4 consumer warps + producer
    static constexpr int THREADS = 2 * LANE_THREADS;
    static constexpr int SCR_OFF = X::STAGES * X::STAGE_BYTES;         // [CWARPS][RMAX] max, sum; [CWARPS][RMAX][D] o
    static constexpr int SCR_BYTES = X::CWARPS * RMAX * (2 + D) * 4;
    static constexpr int BAR_OFF = SCR_OFF + SCR_BYTES;
    static constexpr int LANE_BYTES = (BAR_OFF + 2 * X::STAGES * 8 + 1023) / 1024 * 1024;
    static constexpr int SMEM_USED = 2 * LANE_BYTES + 1024;
    static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;  // one CTA per SM
    static_assert(SMEM <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(XpCfg<D>::THREADS, 1)
    xattn_partial_keys_persist_kernel(const __grid_constant__ CUtensorMap kmap,
                                      const __grid_constant__ CUtensorMap vmap, const XattnParams p)
{
    using C = XCfg<D>;
    using P = XpCfg<D>;
    constexpr int RMAX = P::RMAX;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
    const int L = threadIdx.x / P::LANE_THREADS, lt = threadIdx.x % P::LANE_THREADS;
    const int lw = lt >> 5, lane = lt & 31;
    uint8_t *smem = smem_raw + pad + L * P::LANE_BYTES;
    const uint32_t sbase = raw_s + pad + L * P::LANE_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + P::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    if (lt == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::CWARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int BH = p.B * p.Hkv;
    const long long n_items = static_cast<long long>(p.splits) * BH;
    const long long w_step = 2LL * gridDim.x;
    // an item's key blocks: keys split * chunk .. up to the largest valid position of its rows
    auto item_keys = [&](long long w, int &split, int &b, int &g, int &kmax, int &js, int &nblk) {
        split = static_cast<int>(w % p.splits);
        const int bh = static_cast<int>(w / p.splits);
        b = bh / p.Hkv;
        g = bh % p.Hkv;
        kmax = -1;
        for (int r = 0; r < p.R; ++r) {
            const int ps = __ldg(p.pos + static_cast<long long>(b) * p.T_out + r / p.G);
            if (ps >= 0 && ps < p.T_kv)
                kmax = max(kmax, ps);
        }
        js = split * p.chunk;
        const int je = min(js + p.chunk, kmax + 1);
        nblk = je > js ? (je - js + C::KB - 1) / C::KB : 0;
    };

    if (lw == C::CWARPS) {
        // ------------------------------------------------------------------ producer of lane L
        if (lane != 0)
            return;
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        long long i = 0;  // blocks loaded by this lane over all its items
        for (long long w = 2LL * blockIdx.x + L; w < n_items; w += w_step) {
            int split, b, g, kmax, js, nblk;
            item_keys(w, split, b, g, kmax, js, nblk);
            for (int j = 0; j < nblk; ++j, ++i) {
                const int s = static_cast<int>(i % C::STAGES);
                if (i >= C::STAGES && !mbar_wait(&empty[s], static_cast<uint32_t>(((i / C::STAGES) - 1) & 1))) {
                    record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
                    return;
                }
                uint8_t *dst = smem + s * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
                for (int sl = 0; sl < D / 64; ++sl) {
                    tma_load_4d(dst + sl * C::SLAB, &kmap, &full[s], sl * 64, g, js + j * C::KB, b);
                    tma_load_4d(dst + C::KV_BYTES + sl * C::SLAB, &vmap, &full[s], sl * 64, g, js + j * C::KB, b);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers of lane L
    // every consumer warp passes the same named barriers for every item, whatever happens to
    // its waits (a timed-out wait only stops its work), so none is left waiting at a barrier
    constexpr int CT = C::CWARPS * 32;
    const int bar_id = 3 + L;
    float *ms = reinterpret_cast<float *>(smem + P::SCR_OFF);  // [CWARPS][RMAX] max
    float *ls = ms + C::CWARPS * RMAX;                           // [CWARPS][RMAX] sum
    float *os = ls + C::CWARPS * RMAX;                           // [CWARPS][RMAX][D] output
    const float NEG_INF = -__int_as_float(0x7f800000);
    bool ok = true;
    long long i = 0;
    for (long long w = 2LL * blockIdx.x + L; w < n_items; w += w_step) {
        int split, b, g, kmax, js, nblk;
        item_keys(w, split, b, g, kmax, js, nblk);
        const int bh = b * p.Hkv + g;
        // row r's last key (-1: a bad position, every key masked); padding rows borrow kmax
        auto lim_of = [&](int r) {
            if (r >= p.R)
                return kmax;
            const int ps = __ldg(p.pos + static_cast<long long>(b) * p.T_out + r / p.G);
            return (ps >= 0 && ps < p.T_kv) ? ps : -1;
        };
        WarpKeys16<D, 1, false> st;
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int row = lane >> 2;
                const int dcol = kt * 16 + 2 * (lane & 3) + 8 * hf;
                uint32_t hi = 0, lo = 0;
                if (row < p.R && lim_of(row) >= 0) {
                    const int h = g * p.G + row % p.G;
                    const orthros_bf16 *qrow =
                        p.qc + b * p.qc_bstride + (static_cast<long long>(row / p.G) * p.Hq + h) * D;
                    load_q_pair(qrow, p.alpha_c + h * D, p.beta_c + h * D, dcol, p.qscale, hi, lo);
                }
                st.qb[0][kt][hf] = hi;
                st.ql[0][kt][hf] = lo;
            }
        st.reset();
        int lim[1][2];
        lim[0][0] = lim_of(2 * (lane & 3));
        lim[0][1] = lim_of(2 * (lane & 3) + 1);
        int pmin = 0x7fffffff, pmax = -1;
        for (int r = 0; r < RMAX; ++r) {
            pmin = min(pmin, lim_of(r));
            pmax = max(pmax, lim_of(r));
        }
        for (int j = 0; j < nblk; ++j, ++i) {
            const int s = static_cast<int>(i % C::STAGES);
            if (ok && !mbar_wait(&full[s], static_cast<uint32_t>((i / C::STAGES) & 1)))
                ok = false;
            const uint32_t kbase = sbase + s * C::STAGE_BYTES;
            const int j0 = js + j * C::KB + lw * 16;
            if (ok && j0 <= pmax)
                st.step(kbase, C::SLAB, kbase + C::KV_BYTES, C::SLAB, lw * 16, j0, lim, j0 + 15 <= pmin);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
        }
        st.finish_sums();
        named_barrier(bar_id, CT);  // the previous item's merge has been read: the scratch is free
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2)
            if ((lane >> 2) == 0) {
                ms[lw * RMAX + 2 * lane + r2] = st.m[0][r2];
                ls[lw * RMAX + 2 * lane + r2] = st.l[0][r2];
            }
        named_barrier(bar_id, CT);
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2) {
            const int row = 2 * (lane & 3) + r2;
            float M = NEG_INF;
#pragma unroll
            for (int q = 0; q < C::CWARPS; ++q)
                M = fmaxf(M, ms[q * RMAX + row]);
            const float f = (M == NEG_INF || st.m[0][r2] == NEG_INF) ? 0.f : fast_exp2(st.m[0][r2] - M);
            float *po = os + (lw * RMAX + row) * D + (lane >> 2);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                po[16 * mt] = st.o[0][mt][r2] * f;
                po[16 * mt + 8] = st.o[0][mt][2 + r2] * f;
            }
        }
        named_barrier(bar_id, CT);
        for (int x = lt; x < p.R * (D / 2); x += CT) {  // two columns per thread and step
            const int row = x / (D / 2), c = 2 * (x % (D / 2));
            float M = NEG_INF, Ls = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int q = 0; q < C::CWARPS; ++q)
                M = fmaxf(M, ms[q * RMAX + row]);
#pragma unroll
            for (int q = 0; q < C::CWARPS; ++q) {
                if (ms[q * RMAX + row] != NEG_INF)
                    Ls += ls[q * RMAX + row] * fast_exp2(ms[q * RMAX + row] - M);
                a0 += os[(q * RMAX + row) * D + c];
                a1 += os[(q * RMAX + row) * D + c + 1];
            }
            const int h = g * p.G + row % p.G, copy = row / p.G;
            if (p.direct) {
                const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
                *reinterpret_cast<uint32_t *>(p.oc + b * p.oc_bstride + (static_cast<long long>(copy) * p.Hq + h) * D +
                                              c) = pack_bf16x2(a0 * inv, a1 * inv);
                if (c == 0 && p.lse != nullptr)
                    p.lse[(static_cast<long long>(b) * p.T_out + copy) * p.Hq + h] =
                        Ls > 0.f ? (M + __log2f(Ls)) * kLn2F : NEG_INF;
            } else {
                const long long slot = (static_cast<long long>(split) * BH + bh) * p.R + row;
                *reinterpret_cast<float2 *>(p.part_o + slot * D + c) = make_float2(a0, a1);
                if (c == 0)
                    p.part_ml[slot] = make_float2(M, Ls);
            }
        }
    }
    if (!ok && lt == 0)
        record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
}

// One warp per output row: merge the row's partial (max, sum, o) triples.
template <int D>
__global__ void __launch_bounds__(128) xattn_combine_kernel(const XattnParams p)
{
    // one block per output row (b, copy i, head h); its four warps split the partials
    const long long row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = static_cast<int>(row / (static_cast<long long>(p.T_out) * p.Hq));
    const int rem = static_cast<int>(row % (static_cast<long long>(p.T_out) * p.Hq));
    const int i = rem / p.Hq, h = rem % p.Hq;
    const int g = h / p.G;
    const int bh = b * p.Hkv + g;
    const int r = i * p.G + h % p.G;
    const int BH = p.B * p.Hkv;
    const float NEG_INF = -__int_as_float(0x7f800000);
    __shared__ float red_ml[4];
    __shared__ float red_o[4][D];
    auto ml_at = [&](int q) { return __ldcg(&p.part_ml[(static_cast<long long>(q) * BH + bh) * p.R + r]); };

    // the row's overall max M (log2 units) and sum L over the non-empty partials
    float M = NEG_INF;
    for (int q = threadIdx.x; q < p.n_part; q += 128) {
        const float2 ml = ml_at(q);
        if (ml.y > 0.f)
            M = fmaxf(M, ml.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0)
        red_ml[warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red_ml[0], red_ml[1]), fmaxf(red_ml[2], red_ml[3]));
    __syncthreads();
    float L = 0.f;
    for (int q = threadIdx.x; q < p.n_part; q += 128) {
        const float2 ml = ml_at(q);
        if (ml.y > 0.f)
            L += ml.y * fast_exp2(ml.x - M);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0)
        red_ml[warp] = L;
    __syncthreads();
    L = (red_ml[0] + red_ml[1]) + (red_ml[2] + red_ml[3]);

    // sum of exp2(m_q - M) * o_q: warp w takes partials w, w + 4, ...; independent loads
    constexpr int E = D / 32;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        acc[e] = 0.f;
#pragma unroll 4
    for (int q = warp; q < p.n_part; q += 4) {
        const long long slot = (static_cast<long long>(q) * BH + bh) * p.R + r;
        const float2 ml = __ldcg(&p.part_ml[slot]);
        const float w = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
        const float *po = p.part_o + slot * D + lane * E;
        if constexpr (E == 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(po));
            // an empty partial may hold anything; its weight must not meet a NaN
            if (ml.y > 0.f) {
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            }
        } else {
            const float2 v = __ldcg(reinterpret_cast<const float2 *>(po));
            if (ml.y > 0.f) {
                acc[0] += w * v.x;
                acc[1] += w * v.y;
            }
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
        red_o[warp][lane * E + e] = acc[e];
    __syncthreads();
    if (warp != 0)
        return;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (p.lse != nullptr && lane == 0)
        p.lse[row] = L > 0.f ? (M + __log2f(L)) * kLn2F : NEG_INF;
    orthros_bf16 *orow = p.oc + b * p.oc_bstride + (static_cast<long long>(i) * p.Hq + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        const int c = lane * E + e;
        const float x0 = (red_o[0][c] + red_o[1][c]) + (red_o[2][c] + red_o[3][c]);
        const float x1 = (red_o[0][c + 1] + red_o[1][c + 1]) + (red_o[2][c + 1] + red_o[3][c + 1]);
        *reinterpret_cast<uint32_t *>(orow + e) = pack_bf16x2(x0 * inv, x1 * inv);
    }
}

// ------------------------------------------------------------------ host side

struct XattnPlan {
    int WK, RPC, row_tiles, splits, chunk, n_part, direct, keys;
};

// Deterministic split plan (also used by the workspace-size query): aim for about
// two co-resident CTAs per SM of a 152-SM part in a single wave.
XattnPlan xattn_plan(int B, int T_out, int T_kv, int Hq, int Hkv)
{
    XattnPlan pl{};
    const int G = Hq / Hkv;
    const long long R = static_cast<long long>(T_out) * G;
    pl.WK = R <= 16 ? 4 : 1;
    pl.RPC = 16 * (4 / pl.WK);
    pl.row_tiles = static_cast<int>((R + pl.RPC - 1) / pl.RPC);
    const long long target = 304;
    const long long base = static_cast<long long>(B) * Hkv * pl.row_tiles;
    long long splits = (target + base - 1) / base;
    const long long max_splits = (T_kv + 255) / 256;  // at least 256 keys per split
    if (splits > max_splits)
        splits = max_splits;
    if (splits < 1)
        splits = 1;
    long long chunk = (T_kv + splits - 1) / splits;
    chunk = (chunk + 63) / 64 * 64;
    splits = (T_kv + chunk - 1) / chunk;
    pl.splits = static_cast<int>(splits);
    pl.chunk = static_cast<int>(chunk);
    pl.keys = R <= 8 ? 1 : 0;  // rows on the MMA's N side, one partial per CTA
    pl.n_part = pl.keys ? pl.splits : pl.splits * pl.WK;
    pl.direct = pl.n_part == 1 ? 1 : 0;
    return pl;
}

size_t xattn_workspace_bytes(int B, int T_out, int T_kv, int Hq, int Hkv, int D)
{
    // many copies run on the tensor-memory kernel, which keeps no partials
    if (xattn_tc_supported(D, Hq / Hkv, T_out))
        return 256;
    const XattnPlan pl = xattn_plan(B, T_out, T_kv, Hq, Hkv);
    if (pl.direct)
        return 256;
    const size_t rows = static_cast<size_t>(pl.n_part) * B * Hkv * T_out * (Hq / Hkv);
    const size_t o_bytes = (rows * D * sizeof(float) + 255) / 256 * 256;
    return o_bytes + (rows * sizeof(float2) + 255) / 256 * 256;
}

template <int D, int WK>
static cudaError_t launch_partial(const CUtensorMap &k, const CUtensorMap &v, const XattnParams &p,
                                  cudaStream_t stream)
{
    auto kern = xattn_partial_kernel<D, WK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, XCfg<D>::SMEM);
    if (e != cudaSuccess)
        return e;
    dim3 grid(p.splits, p.row_tiles, p.B * p.Hkv);
    kern<<<grid, XCfg<D>::THREADS, XCfg<D>::SMEM, stream>>>(k, v, p);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_partial_keys_persist(const CUtensorMap &k, const CUtensorMap &v, const XattnParams &p,
                                               int ctas, cudaStream_t stream)
{
    auto kern = xattn_partial_keys_persist_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, XpCfg<D>::SMEM);
    if (e != cudaSuccess)
        return e;
    kern<<<static_cast<unsigned>(ctas), XpCfg<D>::THREADS, XpCfg<D>::SMEM, stream>>>(k, v, p);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_partial_keys(const CUtensorMap &k, const CUtensorMap &v, const XattnParams &p,
                                       cudaStream_t stream)
{
    auto kern = xattn_partial_keys_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, XCfg<D>::SMEM);
    if (e != cudaSuccess)
        return e;
    dim3 grid(p.splits, 1, p.B * p.Hkv);
    kern<<<grid, XCfg<D>::THREADS, XCfg<D>::SMEM, stream>>>(k, v, p);
    return cudaGetLastError();
}

cudaError_t launch_xattn(int D, const CUtensorMap &k, const CUtensorMap &v, XattnParams p,
                         void *workspace, cudaStream_t stream, int ctas)
{
    const XattnPlan pl = xattn_plan(p.B, p.T_out, p.T_kv, p.Hq, p.Hkv);
    p.G = p.Hq / p.Hkv;
    p.R = p.T_out * p.G;
    p.row_tiles = pl.row_tiles;
    p.splits = pl.splits;
    p.chunk = pl.chunk;
    p.n_part = pl.n_part;
    p.direct = pl.direct;
    if (!pl.direct) {
        const size_t rows = static_cast<size_t>(pl.n_part) * p.B * p.Hkv * p.R;
        const size_t o_bytes = (rows * D * sizeof(float) + 255) / 256 * 256;
        p.part_o = static_cast<float *>(workspace);
        p.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) + o_bytes);
    }
    cudaError_t e;
    if (pl.keys && ctas > 0)  // on at most `ctas` SMs, beside the SWA kernel
        e = D == 128 ? launch_partial_keys_persist<128>(k, v, p, ctas, stream)
                     : launch_partial_keys_persist<64>(k, v, p, ctas, stream);
    else if (pl.keys)
        e = D == 128 ? launch_partial_keys<128>(k, v, p, stream) : launch_partial_keys<64>(k, v, p, stream);
    else if (D == 128)
        e = pl.WK == 4 ? launch_partial<128, 4>(k, v, p, stream) : launch_partial<128, 1>(k, v, p, stream);
    else
        e = pl.WK == 4 ? launch_partial<64, 4>(k, v, p, stream) : launch_partial<64, 1>(k, v, p, stream);
    if (e != cudaSuccess || pl.direct)
        return e;
    return launch_xattn_combine(D, p, stream);
}

cudaError_t launch_xattn_combine(int D, const XattnParams &p, cudaStream_t stream)
{
    const unsigned blocks = static_cast<unsigned>(static_cast<long long>(p.B) * p.T_out * p.Hq);
    if (blocks == 0)
        return cudaSuccess;
    if (D == 128)
        xattn_combine_kernel<128><<<blocks, 128, 0, stream>>>(p);
    else
        xattn_combine_kernel<64><<<blocks, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace orthros
