// xattn_tc.cu -- output-copy full causal cross-attention, Eq. (5) of "Orthros:
// Phase-Aware Heterogeneous Attention", for many copies per sequence (SFT answer
// spans, and every position in PT mode, Sec. 3.2), on the 5th-generation tensor
// cores (tcgen05 + tensor memory).  The copy scale-offset q' = Q'_raw * alpha' +
// beta' (Sec. 3.1) is applied once per tile in shared memory.
//
// A CTA owns 256 copy rows of one (batch, KV head): tiles A and B of 128 rows =
// 128 / G copies x the G query heads of the KV head, in the order a 4-D TMA box
// lands them (row = copy * G + head).  It streams the keys 0 .. max(pos) of its
// rows in blocks of 64 through a four-stage ring (slab-major, so the two slots of
// a pair are adjacent), each pair of blocks serving both tiles:
//   S_t = q_t K^T   (one N = 128 product per K step over the pair's 128 keys;
//                    fp16: q rounded once after scale-offset, softmax scale and
//                    log2(e); K converted from bf16 in shared memory, a key row
//                    whose largest |k| reaches 65520 scaled by an exact 2^-e_j
//                    first and its logits multiplied back by 2^e_j), fp32 in TMEM;
//   online softmax per row with the row's own causal limit (key <= pos), P as
//   bf16 over S; the running max is raised only when it grows by more than 8 (in
//   log2 units), so the rescale of O is rare and P stays <= 256 (exact scaling);
//   O_t += P V      (bf16, fp32 accumulation in TMEM);
// and finally o' = O / l rounded to bf16.  Each tile has one 128-column S buffer;
// the two tiles take turns on the tensor pipe (S_A, S_B, then per pair P V of A,
// S_A of the next pair, P V of B, S_B of the next pair), so one tile's MMAs run
// while the other's softmax works.  The softmax takes a pair as two 64-column
// halves; when the second half raises the running max, the first half's P is
// rescaled in place.  Rows whose position is outside [0, T_kv) get zeros and
// ORTHROS_DEVERR_POSITION.
//
// Roles (512 threads, one CTA per SM):
//   warp 0        TMA producer: the two raw query tiles, K/V blocks
//   warp 1        allocates tensor memory; lane 0 issues every tcgen05.mma
//   warps 2-3     convert each landed K block to fp16 (with warps 12-15)
//   warps 4-7     softmax and epilogue of tile A (TMEM lanes = rows)
//   warps 8-11    the same for tile B
//   warps 12-15   query preparation of both tiles, then K conversion
// Tensor memory: S of tile t at 128 t; O_A at 256, O_B at 256 + D.
// Every mbarrier wait is bounded; a timeout records ORTHROS_DEVERR_TIMEOUT and
// all roles drain to the common exit, where tensor memory is released.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace orthros {

template <int D>
struct XtCfg {
    static constexpr int ROWS = 128;           // rows of one tile
    static constexpr int KB = XATTN_TC_KEYS;   // keys per block (= the K/V boxes' height)
    static constexpr int SLABS = D / 64;
    static constexpr int STAGES = 4;
    static constexpr int KSLOT = KB * 128;     // one 64-wide slab of one block
    static constexpr int SLAB_STRIDE = STAGES * KSLOT;  // slab-major ring: a slab holds every slot
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + SLABS * SLAB_STRIDE;
    static constexpr int Q_OFF = V_OFF + SLABS * SLAB_STRIDE;
    static constexpr int Q_SLAB = ROWS * 128;
    static constexpr int Q_BYTES = SLABS * Q_SLAB;
    static constexpr int POS_OFF = Q_OFF + 2 * Q_BYTES;   // int [256]: row limits
    static constexpr int RED_OFF = POS_OFF + 256 * 4;     // int [16]: per-warp maxima
    static constexpr int KEXP_OFF = RED_OFF + 16 * 4;     // int8 [STAGES][KB]: key row shift e_j
    static constexpr int KFLAG_OFF = KEXP_OFF + STAGES * KB;  // uint8 [STAGES][8]: converter warp w shifted rows
    static constexpr int BAR_OFF = KFLAG_OFF + STAGES * 8;
    static constexpr int NBARS = 3 * STAGES + 16;
    static constexpr int HOLD_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = HOLD_OFF + 16 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static constexpr uint32_t TM_S = 0;        // + 128 * tile
    static constexpr uint32_t TM_O = 256;      // + D * tile
    static constexpr int CPR = D / 8;          // 16-byte chunks per query row
    static constexpr int RPP = 128 / CPR;      // rows one pass of 128 threads covers
    static constexpr int CONV_THREADS = 192;   // warps 2-3 and 12-15
};

template <int D, int G>
__global__ void __launch_bounds__(512, 1)
    xattn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const XattnParams p)
{
    using C = XtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_s + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *full = bars;                   // [STAGES] K/V block landed
    uint64_t *kconv = bars + C::STAGES;      // [STAGES] K block converted
    uint64_t *empty = bars + 2 * C::STAGES;  // [STAGES] block released (MMA commit)
    uint64_t *qfull = bars + 3 * C::STAGES;  // [2] raw query tile landed
    uint64_t *qt_full = qfull + 2;           // [2] query tile prepared
    uint64_t *s_full = qfull + 4;            // [tile] S of a pair of blocks complete
    uint64_t *p_full = qfull + 8;            // [tile] P written (and O rescaled if needed)
    uint64_t *o_done = qfull + 12;           // [tile] O += P V of a pair complete (one phase per pair)
    uint64_t *o_final = qfull + 14;          // [tile] O += P V of the last pair complete
    int *s_pos = reinterpret_cast<int *>(smem + C::POS_OFF);
    int *s_red = reinterpret_cast<int *>(smem + C::RED_OFF);
    int8_t *kexp = reinterpret_cast<int8_t *>(smem + C::KEXP_OFF);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::HOLD_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int R = p.T_out * G;
    const int row_base = pair * 256;  // first row of tile A within the (b, KV head) rows

    // ---- row limits (key <= pos of the row's copy) and the CTA's key range
    int lim = -1;
    if (threadIdx.x < 256) {
        const int row = row_base + threadIdx.x;
        if (row < R) {
            const int ps = p.pos[static_cast<long long>(b) * p.T_out + row / G];
            if (ps >= 0 && ps < p.T_kv)
                lim = ps;
            else if (row % G == 0)
                record_error(p.dev_err, ORTHROS_DEVERR_POSITION);
        }
        s_pos[threadIdx.x] = lim;
    }
    const int wmax = __reduce_max_sync(0xffffffffu, lim);
    if (lane == 0)
        s_red[warp] = wmax;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&kconv[s], C::CONV_THREADS / 32);
            mbar_init(&empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&qfull[t], 1);
            mbar_init(&qt_full[t], 4);
            mbar_init(&o_done[t], 1);
            mbar_init(&o_final[t], 1);
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 4);
        }
        for (int s = 0; s < C::STAGES; ++s)
            reinterpret_cast<uint64_t *>(smem + C::KFLAG_OFF)[s] = 0;
        fence_barrier_init();
    }
    if (warp == 1)
        tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;
    int kmax = -1;
#pragma unroll
    for (int w = 0; w < 8; ++w)
        kmax = max(kmax, s_red[w]);
    const int nkb = kmax < 0 ? 0 : kmax / C::KB + 1;  // key blocks of this CTA
    const int npair = (nkb + 1) / 2;                   // pairs of blocks: one S product each

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0 && nkb > 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            for (int t = 0; t < 2; ++t) {
                mbar_arrive_expect_tx(&qfull[t], C::Q_BYTES);
#pragma unroll
                for (int sl = 0; sl < C::SLABS; ++sl)
                    tma_load_4d(smem + C::Q_OFF + t * C::Q_BYTES + sl * C::Q_SLAB, &qmap, &qfull[t], sl * 64, g * G,
                                (row_base + t * 128) / G, b);
            }
            for (int j = 0; j < 2 * npair; ++j) {
                const int s = j % C::STAGES;
                if (j >= C::STAGES && !mbar_wait(&empty[s], static_cast<uint32_t>(((j / C::STAGES) - 1) & 1))) {
                    record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], 2 * C::SLABS * C::KSLOT);
#pragma unroll
                for (int sl = 0; sl < C::SLABS; ++sl) {
                    tma_load_4d(smem + C::K_OFF + sl * C::SLAB_STRIDE + s * C::KSLOT, &kmap, &full[s], sl * 64, g,
                                j * C::KB, b);
                    tma_load_4d(smem + C::V_OFF + sl * C::SLAB_STRIDE + s * C::KSLOT, &vmap, &full[s], sl * 64, g,
                                j * C::KB, b);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        // Pair pp = key blocks 2 pp, 2 pp + 1 (ring slots 2 pp mod 4 and the next one, adjacent in
        // every slab): S_t = q_t K^T is one N = 128 product per K step into tile t's single S
        // buffer, and O_t += P V eight K steps of 16 keys.  Order S_A(0) S_B(0), then per pair
        // PV_A(pp) S_A(pp+1) PV_B(pp) S_B(pp+1): S_t(pp+1) overwrites the P that PV_t(pp) reads,
        // so it waits for that PV to complete, while the other tile's work keeps the pipe busy.
        if (lane == 0 && npair > 0) {
            constexpr uint32_t IDESC_QK = umma_idesc(128, 2 * C::KB, false, false);
            constexpr uint32_t IDESC_PV = umma_idesc(128, D, true, true);
            bool ok = mbar_wait(&qt_full[0], 0) && mbar_wait(&qt_full[1], 0);
            auto issue_s = [&](int t, int pp) -> bool {
                const int s0 = (2 * pp) % C::STAGES;
                const uint32_t ph = static_cast<uint32_t>(((2 * pp) / C::STAGES) & 1);
                if (t == 0)  // the pair's blocks landed and converted
                    for (int h = 0; h < 2; ++h)
                        if (!(mbar_wait(&full[s0 + h], ph) && mbar_wait(&kconv[s0 + h], ph)))
                            return false;
                if (pp >= 1 && !mbar_wait(&o_done[t], static_cast<uint32_t>((pp - 1) & 1)))
                    return false;
                tc_fence_after();
                const uint64_t kdesc = umma_desc_sw128(sbase + C::K_OFF + s0 * C::KSLOT, 16, 1024);
                const uint64_t qdesc = umma_desc_sw128(sbase + C::Q_OFF + t * C::Q_BYTES, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = static_cast<uint32_t>((kk >> 2) * C::SLAB_STRIDE + (kk & 3) * 32) >> 4;
                    const uint32_t qoff = static_cast<uint32_t>((kk >> 2) * C::Q_SLAB + (kk & 3) * 32) >> 4;
                    umma_ss(tbase + C::TM_S + 128 * t, qdesc + qoff, kdesc + koff, IDESC_QK, kk != 0);
                }
                umma_commit(&s_full[t]);
                return true;
            };
            auto issue_pv = [&](int t, int pp) -> bool {
                if (!mbar_wait(&p_full[t], static_cast<uint32_t>(pp & 1)))
                    return false;
                tc_fence_after();
                const int s0 = (2 * pp) % C::STAGES;
                const uint64_t vdesc = umma_desc_sw128(sbase + C::V_OFF + s0 * C::KSLOT, C::SLAB_STRIDE, 1024);
#pragma unroll
                for (int kk = 0; kk < 2 * C::KB / 16; ++kk)
                    umma_ts(tbase + C::TM_O + D * t, tbase + C::TM_S + 128 * t + 8 * kk,
                            vdesc + static_cast<uint64_t>(kk * (2048 >> 4)), IDESC_PV, (pp > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&o_done[t]);
                if (pp == npair - 1)
                    umma_commit(&o_final[t]);  // the epilogue's own barrier (o_done may run ahead of it)
                return true;
            };
            ok = ok && issue_s(0, 0) && issue_s(1, 0);
            for (int pp = 0; pp < npair && ok; ++pp) {
                ok = issue_pv(0, pp) && (pp + 1 >= npair || issue_s(0, pp + 1)) && issue_pv(1, pp);
                if (!ok)
                    break;
                umma_commit(&empty[(2 * pp) % C::STAGES]);  // both tiles' S and PV of the pair are done
                umma_commit(&empty[(2 * pp) % C::STAGES + 1]);
                ok = pp + 1 >= npair || issue_s(1, pp + 1);
            }
            if (!ok)
                record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
        }
    } else if (warp < 4 || warp >= 12) {
        // ------------------------------------------------------------------ query prep + K converters
        bool ok = true, bad = false;
        if (warp >= 12 && nkb > 0) {
            const int tid = threadIdx.x - 384;  // 0..127
            const int cr = tid % C::CPR, row0 = tid / C::CPR;
            const int sl = cr / 8, c8 = cr % 8;
            float as[2][8], bsv[2][8];
#pragma unroll
            for (int hsel = 0; hsel < 2; ++hsel) {
                const int h = g * G + (row0 + hsel * C::RPP) % G;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    as[hsel][e] = __ldg(p.alpha_c + h * D + 8 * cr + e) * p.qscale;
                    bsv[hsel][e] = __ldg(p.beta_c + h * D + 8 * cr + e) * p.qscale;
                }
            }
            for (int t = 0; t < 2 && ok; ++t) {
                if (!(ok = mbar_wait(&qfull[t], 0)))
                    break;
                uint8_t *qb = smem + C::Q_OFF + t * C::Q_BYTES + sl * C::Q_SLAB;
                float amax = 0.f;
#pragma unroll 4
                for (int jr = 0; jr < 128 / C::RPP; ++jr) {
                    const int row = row0 + jr * C::RPP;
                    const int hs = ((jr * C::RPP) % G == 0) ? 0 : 1;
                    uint4 *ptr = reinterpret_cast<uint4 *>(qb + sw128_offset(row, c8));
                    const uint4 raw = *ptr;
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                    uint32_t o4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 qq = ffma2(unpack_bf16x2(w[e]), make_float2(as[hs][2 * e], as[hs][2 * e + 1]),
                                                make_float2(bsv[hs][2 * e], bsv[hs][2 * e + 1]));
                        amax = fmax3(amax, fabsf(qq.x), fabsf(qq.y));
                        __half2 hv = __floats2half2_rn(qq.x, qq.y);
                        o4[e] = *reinterpret_cast<uint32_t *>(&hv);
                    }
                    *ptr = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                }
                bad |= !(amax < 65504.f);
                fence_proxy_async_smem();  // the MMA reads q through the async proxy
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&qt_full[t]);
            }
        }
        // K conversion: 8 consecutive lanes per key row (its 16-byte chunk c8 in every slab), the
        // (row, c8) pairs dealt out cid, cid + 192, cid + 384 (warp-uniform: 192 and 128 are
        // multiples of 32)
        const int cid = warp < 4 ? threadIdx.x - 64 : threadIdx.x - 384 + 64;  // 0..191
        const int cw = cid >> 5;                                                // converter warp 0..5
        constexpr int PAIRS = C::KB * 8;
        static_assert(C::CONV_THREADS % 32 == 0 && (C::KB * 8) % 32 == 0 && C::CONV_THREADS / 8 == 24,
                      "rows of a converter warp: (cid / 8) + 24 it");
        for (int j = 0; j < 2 * npair && ok; ++j) {
            const int s = j % C::STAGES;
            if (!(ok = mbar_wait(&full[s], static_cast<uint32_t>((j / C::STAGES) & 1))))
                break;
            uint8_t *blk = smem + C::K_OFF + s * C::KSLOT;
            // common case: every chunk below 65520 converts as is; when a chunk of the warp's rows
            // reaches it, the warp shifts those rows instead (rare)
            constexpr int ITS = (PAIRS + C::CONV_THREADS - 1) / C::CONV_THREADS;
            const int nrows = cid + (ITS - 1) * C::CONV_THREADS < PAIRS ? ITS : ITS - 1;  // warp-uniform
            uint4 u[ITS][C::SLABS];
            uint32_t kept = 0;
#pragma unroll
            for (int it = 0; it < ITS; ++it)
                if (it < nrows) {
#pragma unroll
                    for (int sl = 0; sl < C::SLABS; ++sl) {
                        u[it][sl] = *reinterpret_cast<const uint4 *>(blk + sl * C::SLAB_STRIDE +
                                                                     ((cid >> 3) + 24 * it) * 128 + (cid & 7) * 16);
                        kept |= (bf16x8_absmax(u[it][sl]) < 65520.f ? 0u : 1u) << (it * C::SLABS + sl);
                    }
                }
            const bool wany = __any_sync(0xffffffffu, kept != 0);
            if (!wany) {
#pragma unroll
                for (int it = 0; it < ITS; ++it)
                    if (it < nrows) {
#pragma unroll
                        for (int sl = 0; sl < C::SLABS; ++sl)
                            *reinterpret_cast<uint4 *>(blk + sl * C::SLAB_STRIDE + ((cid >> 3) + 24 * it) * 128 +
                                                       (cid & 7) * 16) = k_to_fp16(u[it][sl]);
                    }
            } else {
                shift_key_rows<C::SLABS>(blk, C::SLAB_STRIDE, 0, cid >> 3, C::CONV_THREADS / 8, nrows, cid & 7,
                                         kexp + s * C::KB, bad);
            }
            if (lane == 0)
                smem[C::KFLAG_OFF + s * 8 + cw] = wany ? 1 : 0;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&kconv[s]);
        }
        if (bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
        if (!ok && lane == 0)
            record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    } else {
        // ------------------------------------------------------------------ softmax + epilogue
        const int t = (warp - 4) >> 2;  // tile
        const int rw = warp & 3;
        const int r = rw * 32 + lane;   // row of the tile = tensor-memory lane
        const int row = row_base + t * 128 + r;
        const int pr = s_pos[t * 128 + r];
        const uint32_t s_lane = tbase + (static_cast<uint32_t>(rw * 32) << 16) + C::TM_S + 128 * t;
        const uint32_t o_col = tbase + (static_cast<uint32_t>(rw * 32) << 16) + C::TM_O + D * t;
        const float NEG_INF = -__int_as_float(0x7f800000);
        float m = NEG_INF, l = 0.f;
        bool ok = true, range_bad = false;
        // pair pp: the two 64-column halves of S_t in turn (half hh = key block 2 pp + hh), each with
        // the lazily raised running max; P of half hh goes to columns 32 hh .. 32 hh + 31 as bf16
        for (int pp = 0; pp < npair && ok; ++pp) {
            if (!(ok = mbar_wait(&s_full[t], static_cast<uint32_t>(pp & 1))))
                break;
            tc_fence_after();
            float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll 1
            for (int hh = 0; hh < 2 && ok; ++hh) {
                const int j = 2 * pp + hh;
                const int ks = j % C::STAGES;
                const uint32_t s_col = s_lane + 64 * hh;
                const int k0 = j * C::KB;
                const bool whole = __all_sync(0xffffffffu, k0 + C::KB - 1 <= pr);
                const int nvalid = pr - k0;  // column c is a valid key iff c <= nvalid
                uint32_t va[32], vb[32];
                tmem_ld32(s_col, va);
                tmem_ld32(s_col + 32, vb);
                // the block's shift flags: its conversion barrier completed before its S was issued,
                // so this non-blocking test succeeds and orders the flag read after the converters'
                // writes
                const uint32_t kph = static_cast<uint32_t>((j / C::STAGES) & 1);
                const bool conv_seen = mbar_test_wait(&kconv[ks], kph);
                const uint64_t kf = *reinterpret_cast<const volatile uint64_t *>(smem + C::KFLAG_OFF + ks * 8);
                tmem_wait_ld();
                if (!conv_seen || kf != 0) {
                    if (!(ok = mbar_wait(&kconv[ks], kph)))
                        break;
                    const uint64_t kf2 = *reinterpret_cast<const volatile uint64_t *>(smem + C::KFLAG_OFF + ks * 8);
                    uint32_t kw = 0;  // one bit per converter warp that shifted rows of this block
#pragma unroll
                    for (int cw = 0; cw < C::CONV_THREADS / 32; ++cw)
                        kw |= (((kf2 >> (8 * cw)) & 0xffu) ? 1u : 0u) << cw;
                    if (kw != 0) {  // logits of shifted key rows times 2^e_j (rare), in tensor memory
                        unshift_chunk32(s_col, kexp + ks * C::KB, 0, kw, 24, 4, range_bad);
                        unshift_chunk32(s_col + 32, kexp + ks * C::KB, 32, kw, 24, 4, range_bad);
                        tmem_ld32(s_col, va);
                        tmem_ld32(s_col + 32, vb);
                        tmem_wait_ld();
                    }
                }
                if (!whole) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        if (e > nvalid)
                            va[e] = __float_as_uint(NEG_INF);
                        if (32 + e > nvalid)
                            vb[e] = __float_as_uint(NEG_INF);
                    }
                }
                float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(va[e]), __uint_as_float(va[e + 1]));
                    m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(vb[e]), __uint_as_float(vb[e + 1]));
                }
                const float mb = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                // raise the running max only when it grows by more than 2^8 (P stays <= 256)
                const bool raise = mb > m + 8.f;
                if (__any_sync(0xffffffffu, raise)) {
                    const float f = raise ? fast_exp2(m - mb) : 1.f;  // m = -inf before the first key: f = 0
                    if (pp > 0) {
                        // O holds the pairs before pp (S_t of this pair waited for their P V)
                        if (!(ok = mbar_wait(&o_done[t], static_cast<uint32_t>((pp - 1) & 1))))
                            break;
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < D; c += 32) {
                            uint32_t w[32];
                            tmem_ld32(o_col + c, w);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                w[e] = __float_as_uint(__uint_as_float(w[e]) * f);
                            tmem_st32(o_col + c, w);
                        }
                    }
                    if (hh == 1) {  // P of the first half was taken against the old max: scale it too
                        tmem_wait_st();
                        uint32_t w[32];
                        tmem_ld32(s_lane, w);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float2 pq = unpack_bf16x2(w[e]);
                            w[e] = pack_bf16x2(pq.x * f, pq.y * f);
                        }
                        tmem_st32(s_lane, w);
                        l2[0].x *= f;
                        l2[0].y *= f;
                        l2[1].x *= f;
                        l2[1].y *= f;
                    }
                    if (raise) {
                        l *= f;
                        m = mb;
                    }
                }
                const float uo = (m == NEG_INF) ? 0.f : m;
                const float2 nu = make_float2(-uo, -uo);
                // P = exp2(S - m) as bf16 over columns 32 hh .. 32 hh + 31 of the S buffer, row sum
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    const uint32_t *v = hq ? vb : va;
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 d = fadd2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), nu);
                        const float2 pp2 = make_float2(fast_exp2(d.x), fast_exp2(d.y));
                        l2[e & 1] = fadd2(l2[e & 1], pp2);
                        pw[e] = pack_bf16x2(pp2.x, pp2.y);
                    }
                    tmem_st16(s_lane + 32 * hh + 16 * hq, pw);
                }
            }
            if (!ok)
                break;
            l += (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[t]);
        }
        // ---- epilogue: O / l -> bf16 -> the copy's output row (and its log-sum-exp)
        const bool store = row < R;
        if (store && p.lse != nullptr && ok)
            p.lse[(static_cast<long long>(b) * p.T_out + row / G) * p.Hq + g * G + row % G] =
                l > 0.f ? (m + __log2f(l)) * kLn2F : -__int_as_float(0x7f800000);
        orthros_bf16 *orow = p.oc + b * p.oc_bstride +
                             (static_cast<long long>(row / G) * p.Hq + g * G + row % G) * D;
        const bool o32 = ((reinterpret_cast<uintptr_t>(p.oc) | static_cast<uintptr_t>(p.oc_bstride * 2)) & 31u) == 0;
        if (ok && nkb > 0) {
            if (!(ok = mbar_wait(&o_final[t], 0))) {
                record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
            } else {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const float2 il = make_float2(inv, inv);
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t v[32];
                    tmem_ld32(o_col + c, v);
                    tmem_wait_ld();
                    uint4 w[4];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 y = fmul2(
                                make_float2(__uint_as_float(v[8 * c4 + 2 * e]), __uint_as_float(v[8 * c4 + 2 * e + 1])), il);
                            pk[e] = pack_bf16x2(y.x, y.y);
                        }
                        w[c4] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    if (store) {
                        if (o32) {
                            st_global_v8(orow + c, w[0], w[1]);
                            st_global_v8(orow + c + 16, w[2], w[3]);
                        } else {
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4)
                                *reinterpret_cast<uint4 *>(orow + c + 8 * c4) = w[c4];
                        }
                    }
                }
            }
        } else if (store && nkb == 0) {
            // no valid key anywhere in this CTA (every position rejected): zero rows
#pragma unroll 1
            for (int c = 0; c < D; c += 8)
                *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (range_bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
        if (!ok && lane == 0)
            record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    }

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

template <int D, int G>
static cudaError_t launch_xattn_tc_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                     const XattnParams &p, cudaStream_t stream)
{
    using C = XtCfg<D>;
    auto kern = xattn_tc_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    const long long R = static_cast<long long>(p.T_out) * G;
    dim3 grid(static_cast<unsigned>((R + 255) / 256), static_cast<unsigned>(p.B * p.Hkv));
    kern<<<grid, 512, C::SMEM, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

bool xattn_tc_supported(int D, int G, int T_out)
{
    return (D == 64 || D == 128) && G >= 2 && G <= 16 && static_cast<long long>(T_out) * G >= 256;
}

cudaError_t launch_xattn_tc(int D, int G, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                            const XattnParams &p, cudaStream_t stream)
{
#define ORTHROS_XT_CASE(DD, GG) \
    if (D == DD && G == GG)     \
        return launch_xattn_tc_t<DD, GG>(q, k, v, p, stream);
    ORTHROS_XT_CASE(128, 2)
    ORTHROS_XT_CASE(128, 4)
    ORTHROS_XT_CASE(128, 8)
    ORTHROS_XT_CASE(128, 16)
    ORTHROS_XT_CASE(64, 2)
    ORTHROS_XT_CASE(64, 4)
    ORTHROS_XT_CASE(64, 8)
    ORTHROS_XT_CASE(64, 16)
#undef ORTHROS_XT_CASE
    return cudaErrorInvalidValue;
}

}  // namespace orthros
