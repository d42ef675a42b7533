// swa_tc.cu -- base-stream sliding-window attention, Eq. (4) of "Orthros:
// Phase-Aware Heterogeneous Attention" (Sec. 2.3 of the close-reading notes),
// with the base scale-offset q = Q_raw * alpha + beta (Sec. 3.1) fused into the
// query load, on the 5th-generation tensor cores (tcgen05 + tensor memory).
//
// Tiles are those of swa_fwd.cu: 128 query rows = TOK tokens x G heads sharing
// one KV head, row r = (token r / G, head r % G) as a 4-D TMA box lands it.  A
// persistent CTA walks consecutive tiles of a (batch, KV head) stream and keeps
// each 32-key K/V block resident in a ring for every tile of its band, so K and
// V leave HBM once.  The band of a tile (at most NB blocks) is one MMA of
// N = 32 * blocks per k-step: the K ring carries NB - 1 mirror slots after its
// last slot (the producer writes blocks of the first NB - 1 slots twice), so a
// band that starts anywhere in the ring is contiguous.
//
// Arithmetic:
//   S = q K^T in fp16 (q rounded once to fp16 after scale-offset, softmax scale
//       and log2(e); K converted from bf16 to fp16 in shared memory: a key row
//       whose largest |k| reaches 65520 (beyond fp16) is first scaled by an exact
//       power of two 2^-e_j into [2^14, 2^15), and the softmax multiplies that
//       key's logits by 2^e_j, so every finite bf16 key is taken), fp32
//       accumulation;
//   P = exp2(S - rowmax) over the whole band at once (the band fits in tensor
//       memory, so there is no online rescaling), stored as bf16 over S;
//   O = P V in bf16 with fp32 accumulation; o = O / rowsum rounded to bf16.
//
// Roles (512 threads, one CTA per SM):
//   warp 0        TMA producer: raw Q tiles (double buffered), K/V blocks
//   warp 1        allocates tensor memory; lane 0 issues every tcgen05.mma
//   warps 2-3     convert each landed K block to fp16 in place
//   warps 4-7     softmax + epilogue of even tiles (S buffer 0), one thread per
//                 row / tensor-memory lane; the epilogue stores O / l as bf16
//                 straight from registers to global memory
//   warps 8-11    the same for odd tiles (S buffer 1)
//   warps 12-15   query preparation in place in shared memory (bf16 -> scaled fp16)
// S = q K^T reads q and K from shared memory; O = P V reads P from tensor
// memory.  Tensor memory: S/P buffers [0, 2 * 32 * NB), O at column 384.
// Every mbarrier wait is bounded; a timeout records ORTHROS_DEVERR_TIMEOUT and
// all roles drain to the common exit, where tensor memory is released.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace orthros {

template <int D>
struct TcCfg {
    static constexpr int ROWS = 128;
    static constexpr int KB = 32;
    static constexpr int SLABS = D / 64;
    static constexpr int NB = D == 128 ? 5 : 6;  // most blocks a tile's band may span
    static constexpr int STAGES = 8;
    static constexpr int MIRROR = NB - 1;
    static constexpr int THREADS = 512;
    static constexpr int SLOT = KB * 128;                   // one slot of one slab array
    static constexpr int K_SLAB = (STAGES + MIRROR) * SLOT;  // one K slab array (with mirrors)
    static constexpr int V_SLAB = STAGES * SLOT;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + SLABS * K_SLAB;
    static constexpr int Q_OFF = V_OFF + SLABS * V_SLAB;
    static constexpr int Q_SLAB = ROWS * 128;
    static constexpr int Q_BYTES = SLABS * Q_SLAB;  // one of two query buffers
    static constexpr int BAR_OFF = Q_OFF + 2 * Q_BYTES;
    static constexpr int NBARS = 3 * STAGES + 13;
    static constexpr int KEXP_OFF = BAR_OFF + NBARS * 8;      // int8 [STAGES][KB]: key row shift e_j
    static constexpr int KFLAG_OFF = KEXP_OFF + STAGES * KB;  // uint8 [2 warps][8]: slot holds shifted rows
    static constexpr int KBAND_OFF = KFLAG_OFF + 16;          // uint32 [2]: shifted blocks of a tile's band
    static constexpr int HOLD_OFF = KBAND_OFF + 8;            // tensor-memory base address
    static constexpr int SMEM = HOLD_OFF + 16 + 1024;         // + alignment slack
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(STAGES <= 8, "one flag byte per slot in a 64-bit word");
    static constexpr uint32_t TM_SSTRIDE = 32 * NB;
    static constexpr uint32_t TM_O = 384;
    static constexpr uint32_t TM_COLS = 512;
    static_assert(2 * TM_SSTRIDE <= TM_O && TM_O + D <= TM_COLS, "tensor memory budget");
    static constexpr int CPR = D / 8;      // 16-byte chunks per query row
    static constexpr int RPP = 128 / CPR;  // rows one pass of 128 threads covers
};

__device__ __forceinline__ int tc_kb_lo(int n, int TOK, int window)
{
    const int t = n * TOK - window + 1;
    return t > 0 ? t / 32 : 0;
}

__device__ __forceinline__ int tc_kb_hi(int n, int TOK, int T)
{
    int t = n * TOK + TOK - 1;
    if (t > T - 1)
        t = T - 1;
    return t / 32;
}

// RANGE: the launch covers a row range that may start mid-sequence (tile base n_base > 0)
// LSE: also store each row's log-sum-exp (p.lse); a separate instance, so that the
// inference path carries no trace of it
template <int D, int G, bool RANGE, bool LSE>
__global__ void __launch_bounds__(512, 1)
    swa_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const SwaParams p)
{
    using C = TcCfg<D>;
    constexpr int TOK = 128 / G;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_s + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *full = bars;                   // [STAGES] block landed (TMA)
    uint64_t *kconv = bars + C::STAGES;      // [STAGES] K block converted to fp16
    uint64_t *empty = bars + 2 * C::STAGES;  // [STAGES] block released (MMA commit)
    uint64_t *qfull = bars + 3 * C::STAGES;  // [2] raw Q tile landed
    uint64_t *qt_full = qfull + 2;           // [2] q prepared in place
    uint64_t *s_full = qfull + 4;            // [2] S = q K^T complete
    uint64_t *p_full = qfull + 6;            // [2] P written over S
    uint64_t *o_full = qfull + 8;            // [2] O = P V complete (by the parity of the tile)
    uint64_t *o_free = qfull + 10;           // O read out of tensor memory
    uint64_t *kinfo = qfull + 11;            // [2] the band's shift word of S buffer u written
    int8_t *kexp = reinterpret_cast<int8_t *>(smem + C::KEXP_OFF);
    volatile uint32_t *kband = reinterpret_cast<volatile uint32_t *>(smem + C::KBAND_OFF);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::HOLD_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&kconv[s], 2);
            mbar_init(&empty[s], 1);
        }
        reinterpret_cast<uint64_t *>(smem + C::KFLAG_OFF)[0] = 0;
        reinterpret_cast<uint64_t *>(smem + C::KFLAG_OFF)[1] = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qt_full[i], 4);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
        }
        mbar_init(&o_full[0], 1);
        mbar_init(&o_full[1], 1);
        mbar_init(o_free, 4);
        mbar_init(&kinfo[0], 1);
        mbar_init(&kinfo[1], 1);
        tmem_holder[1] = static_cast<uint32_t>(p.n_base);
        fence_barrier_init();
    }
    if (warp == 1)
        tmem_alloc(tmem_holder, C::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;

    const long long gt_begin = p.total_tiles * blockIdx.x / gridDim.x;
    const long long gt_end = p.total_tiles * (blockIdx.x + 1) / gridDim.x;
    const int tps = p.tiles_per_stream;
    // the tile sequence of this CTA, in segments of consecutive tiles of one stream; tile
    // indices are absolute (the launched row range starts at tile n_base).  n_base is read
    // from shared memory where a segment starts, so no role keeps it in a register.
    const volatile int *n_base_s = reinterpret_cast<const volatile int *>(tmem_holder + 1);
    auto n_base = [&]() { return RANGE ? *n_base_s : 0; };
    auto seg_begin = [&](long long gt) { return n_base() + static_cast<int>(gt % tps); };
    auto seg_end = [&](long long gt, int n0) {
        const long long lim = n0 + (gt_end - gt);
        const int end = n_base() + tps;
        return static_cast<int>(lim < end ? lim : end);
    };

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            bool ok = true;
            long long load_idx = 0;
            int it = 0;
            for (long long gt = gt_begin; gt < gt_end && ok;) {
                const int stream = static_cast<int>(gt / tps), n0 = seg_begin(gt);
                const int n1 = seg_end(gt, n0);
                const int b = stream / p.Hkv, g = stream % p.Hkv;
                int next_kb = tc_kb_lo(n0, TOK, p.window);
                for (int n = n0; n < n1 && ok; ++n, ++it) {
                    const int qb = it & 1;
                    // query buffer qb is free once QK of tile it-2 has read it
                    if (it >= 2 && !mbar_wait(&s_full[qb], static_cast<uint32_t>(((it - 2) >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&qfull[qb], C::Q_BYTES);
#pragma unroll
                    for (int sl = 0; sl < C::SLABS; ++sl)
                        tma_load_4d(smem + C::Q_OFF + qb * C::Q_BYTES + sl * C::Q_SLAB, &qmap, &qfull[qb], sl * 64,
                                    g * G, n * TOK, b);
                    const int hi = tc_kb_hi(n, TOK, p.T);
                    for (; next_kb <= hi && ok; ++next_kb, ++load_idx) {
                        const int s = static_cast<int>(load_idx % C::STAGES);
                        if (load_idx >= C::STAGES &&
                            !mbar_wait(&empty[s], static_cast<uint32_t>(((load_idx / C::STAGES) - 1) & 1))) {
                            ok = false;
                            break;
                        }
                        const bool mirror = s < C::MIRROR;
                        mbar_arrive_expect_tx(&full[s], C::SLABS * C::SLOT * (mirror ? 3 : 2));
#pragma unroll
                        for (int sl = 0; sl < C::SLABS; ++sl) {
                            uint8_t *kdst = smem + C::K_OFF + sl * C::K_SLAB;
                            tma_load_4d(kdst + s * C::SLOT, &kmap, &full[s], sl * 64, g, next_kb * C::KB, b);
                            if (mirror)
                                tma_load_4d(kdst + (s + C::STAGES) * C::SLOT, &kmap, &full[s], sl * 64, g,
                                            next_kb * C::KB, b);
                            tma_load_4d(smem + C::V_OFF + sl * C::V_SLAB + s * C::SLOT, &vmap, &full[s], sl * 64,
                                        g, next_kb * C::KB, b);
                        }
                    }
                }
                gt += n1 - n0;
            }
            if (!ok)
                record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t IDESC_PV = umma_idesc(128, D, true, true);
            // ring position (count of K/V blocks loaded before) of the current stream segment's first block
            int seg_base = 0, seg_kb0 = 0, seg = -1, last_khi = -1, waited = -1;
            // the previous tile, whose PV is issued after this tile's QK
            bool have_prev = false;
            int p_nb = 0, p_klo = 0, p_seg = -1, p_idx0 = 0;
            int n = static_cast<int>(gt_begin % tps) - 1;  // relative to the range; na = n + p.n_base
            // O = P V for tile pit; the first `rel` blocks of its band go back to the ring
            auto issue_pv = [&](int pit, int rel) -> bool {
                const int pbuf = pit & 1;
                ok = mbar_wait(&p_full[pbuf], static_cast<uint32_t>((pit >> 1) & 1)) &&
                     (pit < 1 || mbar_wait(o_free, static_cast<uint32_t>((pit - 1) & 1)));
                if (!ok)
                    return false;
                tc_fence_after();
                const uint32_t s_col = tbase + pbuf * C::TM_SSTRIDE;
#pragma unroll 1
                for (int j = 0; j < p_nb; ++j) {
                    const uint32_t vslot = sbase + C::V_OFF + static_cast<uint32_t>((p_idx0 + j) % C::STAGES) * C::SLOT;
                    const uint64_t vdesc = umma_desc_sw128(vslot, C::V_SLAB, 1024);
                    umma_ts(tbase + C::TM_O, s_col + 16 * j, vdesc, IDESC_PV, j != 0);
                    umma_ts(tbase + C::TM_O, s_col + 16 * j + 8, vdesc + (2048 >> 4), IDESC_PV, 1);
                }
                umma_commit(&o_full[pbuf]);
#pragma unroll 1
                for (int r = 0; r < rel; ++r)
                    umma_commit(&empty[(p_idx0 + r) % C::STAGES]);
                return true;
            };
            // one pass per tile, plus a last pass for the PV of the last tile
            for (long long gt = gt_begin, it = 0; ok; ++gt, ++it) {
                const bool have = gt < gt_end;
                int klo = 0, nb = 0, idx0 = 0;
                if (have) {
                    if (++n == tps || gt == gt_begin) {  // a new stream segment
                        if (n == tps)
                            n = 0;
                        if (seg >= 0)
                            seg_base += last_khi - seg_kb0 + 1;
                        ++seg;
                        seg_kb0 = tc_kb_lo(n + n_base(), TOK, p.window);
                    }
                    const int na = n + n_base();  // absolute tile index
                    klo = tc_kb_lo(na, TOK, p.window);
                    last_khi = tc_kb_hi(na, TOK, p.T);
                    nb = last_khi - klo + 1;
                    idx0 = seg_base + (klo - seg_kb0);
                    // a new segment's first band (a row range that starts mid-sequence) may not fit
                    // the ring next to the previous segment's last band: release that tile first
                    if (have_prev && p_seg != seg && p_nb + nb > C::STAGES) {
                        if (!issue_pv(static_cast<int>(it - 1), p_nb))
                            break;
                        have_prev = false;
                    }
                    const int buf = static_cast<int>(it & 1);
                    // ---- S[buf] = q K^T for tile `it`
                    ok = mbar_wait(&qt_full[buf], static_cast<uint32_t>((it >> 1) & 1));
                    if (ok && it >= 2)  // PV(it-2) has read P from S[buf]
                        ok = mbar_wait(&o_full[buf], static_cast<uint32_t>(((it - 2) >> 1) & 1));
#pragma unroll 1
                    for (int idx = max(waited + 1, idx0); idx < idx0 + nb && ok; ++idx) {
                        const uint32_t ph = static_cast<uint32_t>((idx / C::STAGES) & 1);
                        ok = mbar_wait(&full[idx % C::STAGES], ph) && mbar_wait(&kconv[idx % C::STAGES], ph);
                        waited = idx;
                    }
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t slot0 = static_cast<uint32_t>(idx0 % C::STAGES);
                    const uint64_t kdesc = umma_desc_sw128(sbase + C::K_OFF + slot0 * C::SLOT, 16, 1024);
                    const uint64_t qdesc = umma_desc_sw128(sbase + C::Q_OFF + buf * C::Q_BYTES, 16, 1024);
                    const uint32_t idesc = umma_idesc(128, 32 * nb, false, false);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = static_cast<uint32_t>((kk >> 2) * C::K_SLAB + (kk & 3) * 32) >> 4;
                        const uint32_t qoff = static_cast<uint32_t>((kk >> 2) * C::Q_SLAB + (kk & 3) * 32) >> 4;
                        umma_ss(tbase + buf * C::TM_SSTRIDE, qdesc + qoff, kdesc + koff, idesc, kk != 0);
                    }
                    umma_commit(&s_full[buf]);
                    // which blocks of the band hold shifted key rows (the converters' flags, seen
                    // through the kconv waits above), for the softmax of this tile
                    const volatile uint64_t *kf = reinterpret_cast<const volatile uint64_t *>(smem + C::KFLAG_OFF);
                    const uint64_t f0 = kf[0], f1 = kf[1];
                    uint32_t smask = 0;  // bits 2 j, 2 j + 1: band block j holds shifted rows of converter warp 0, 1
                    if ((f0 | f1) != 0) {
#pragma unroll 1
                        for (int j = 0; j < nb; ++j) {
                            const int sh = 8 * ((idx0 + j) % C::STAGES);
                            smask |= (((f0 >> sh) & 0xffu) ? 1u : 0u) << (2 * j);
                            smask |= (((f1 >> sh) & 0xffu) ? 1u : 0u) << (2 * j + 1);
                        }
                    }
                    kband[buf] = smask | (slot0 << 16);
                    mbar_arrive(&kinfo[buf]);
                }
                // ---- O = P V for the previous tile: within a segment it keeps the blocks this tile
                // still uses; at a segment change or after the last tile it releases its whole band
                if (have_prev && !issue_pv(static_cast<int>(it - 1), (have && p_seg == seg) ? klo - p_klo : p_nb))
                    break;
                if (!have)
                    break;
                have_prev = true;
                p_nb = nb;
                p_klo = klo;
                p_seg = seg;
                p_idx0 = idx0;
            }
            if (!ok)
                record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------------ K converters
        // 8 lanes per key row (the row's 16-byte chunk c8 in every slab), rows rsub + 4 NCW i
        constexpr int NCW = 2;            // converter warps
        const int ct = threadIdx.x - 64;  // 0 .. 63
        const int c8 = ct & 7, rsub = ct >> 3;
        constexpr int ROWS_T = C::KB / (4 * NCW);  // key rows per thread and block
        uint8_t *kflag = smem + C::KFLAG_OFF + (warp - 2) * 8;
        bool ok = true, bad = false;
        long long idx = 0;
        for (long long gt = gt_begin; gt < gt_end && ok;) {
            const int n0 = seg_begin(gt);
            const int n1 = seg_end(gt, n0);
            const int nload = tc_kb_hi(n1 - 1, TOK, p.T) - tc_kb_lo(n0, TOK, p.window) + 1;
            for (int i = 0; i < nload; ++i, ++idx) {
                const int s = static_cast<int>(idx % C::STAGES);
                if (!mbar_wait(&full[s], static_cast<uint32_t>((idx / C::STAGES) & 1))) {
                    ok = false;
                    break;
                }
                // common case: every chunk below 65520 converts as is; when a chunk of the warp's
                // rows reaches it, the warp shifts those rows instead (rare)
                // common case: every chunk below 65520 converts as is, in passes of up to four rows
                // per lane (loads of a pass in flight together); when a chunk of the warp's rows
                // reaches 65520 the warp shifts its rows instead (rare)
                constexpr int RP = ROWS_T < 4 ? ROWS_T : 4;
                bool block_any = false;
                int r_bad = 0;  // first row (of this lane's) of the pass that found a value beyond fp16
#pragma unroll 1
                for (int r0 = 0; r0 < ROWS_T && !block_any; r0 += RP) {
                    uint4 u[RP][C::SLABS];
                    uint32_t kept = 0;
#pragma unroll
                    for (int r = 0; r < RP; ++r)
#pragma unroll
                        for (int sl = 0; sl < C::SLABS; ++sl) {
                            u[r][sl] = *reinterpret_cast<const uint4 *>(smem + C::K_OFF + sl * C::K_SLAB + s * C::SLOT +
                                                                        (rsub + 4 * NCW * (r0 + r)) * 128 + c8 * 16);
                            kept |= (bf16x8_absmax(u[r][sl]) < 65520.f ? 0u : 1u) << (r * C::SLABS + sl);
                        }
                    block_any = __any_sync(0xffffffffu, kept != 0);
                    r_bad = r0;
                    if (!block_any) {
#pragma unroll
                        for (int r = 0; r < RP; ++r)
#pragma unroll
                            for (int sl = 0; sl < C::SLABS; ++sl) {
                                uint8_t *dst = smem + C::K_OFF + sl * C::K_SLAB + s * C::SLOT +
                                               (rsub + 4 * NCW * (r0 + r)) * 128 + c8 * 16;
                                const uint4 h = k_to_fp16(u[r][sl]);
                                *reinterpret_cast<uint4 *>(dst) = h;
                                if (s < C::MIRROR)
                                    *reinterpret_cast<uint4 *>(dst + C::STAGES * C::SLOT) = h;
                            }
                    }
                }
                if (block_any) {
                    // rows of the passes before r_bad are converted and hold nothing beyond fp16;
                    // the rest, still bf16, take the per-row shift
                    if (c8 == 0)
                        for (int r = 0; r < r_bad; ++r)
                            kexp[s * C::KB + rsub + 4 * NCW * r] = 0;
                    shift_key_rows<C::SLABS>(smem + C::K_OFF + s * C::SLOT, C::K_SLAB,
                                             s < C::MIRROR ? C::STAGES * C::SLOT : 0, rsub + 4 * NCW * r_bad, 4 * NCW,
                                             ROWS_T - r_bad, c8, kexp + s * C::KB, bad);
                }
                if (lane == 0)
                    kflag[s] = block_any ? 1 : 0;
                fence_proxy_async_smem();  // the MMA reads the converted block through the async proxy
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&kconv[s]);
            }
            gt += n1 - n0;
        }
        if (bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
        if (!ok && lane == 0)
            record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    } else if (warp < 12) {
        // ------------------------------------------------------------------ softmax (two warpgroups)
        const int wg = (warp - 4) >> 2;  // 0: even tiles / S buffer 0, 1: odd tiles / S buffer 1
        const int rw = warp & 3;
        const int r = rw * 32 + lane;
        const int ti = r / G;
        const uint32_t s_col = tbase + (static_cast<uint32_t>(rw * 32) << 16) + wg * C::TM_SSTRIDE;
        const uint32_t o_lane = tbase + (static_cast<uint32_t>(rw * 32) << 16) + C::TM_O;
        const float NEG_INF = -__int_as_float(0x7f800000);
        // rows can be written as whole 32-byte sectors when the output is 32-byte aligned
        const bool o32 = ((reinterpret_cast<uintptr_t>(p.o) | static_cast<uintptr_t>(p.o_bstride * 2)) & 31u) == 0;
        bool ok = true, range_bad = false;
        int it = 0;
        // this warpgroup's epilogue for its tile `eit`: O / l -> bf16 -> global memory
        auto epilogue = [&](int eit, int eb, int eg, int en, float inv_l) -> bool {
            if (!mbar_wait(&o_full[wg], static_cast<uint32_t>((eit >> 1) & 1)))
                return false;
            tc_fence_after();
            const int token = en * TOK + ti;
            const bool valid = token < p.T;
            orthros_bf16 *orow =
                p.o + eb * p.o_bstride + (static_cast<long long>(token) * p.Hq + eg * G + r % G) * D;
            uint32_t v[2][32];
            tmem_ld32(o_lane, v[0]);
            tmem_wait_ld();
#pragma unroll
            for (int cq = 0; cq < D / 32; ++cq) {
                if (cq + 1 < D / 32)
                    tmem_ld32(o_lane + 32 * (cq + 1), v[(cq + 1) & 1]);
                uint4 w[4];
                const float2 il = make_float2(inv_l, inv_l);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint32_t *x = &v[cq & 1][8 * c4];
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 y = fmul2(make_float2(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1])), il);
                        pk[e] = pack_bf16x2(y.x, y.y);
                    }
                    w[c4] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                tmem_wait_ld();
                if (cq == D / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(o_free);
                }
                if (valid) {
                    if (o32) {
                        st_global_v8(orow + 32 * cq, w[0], w[1]);
                        st_global_v8(orow + 32 * cq + 16, w[2], w[3]);
                    } else {
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
                            *reinterpret_cast<uint4 *>(orow + 32 * cq + 8 * c4) = w[c4];
                    }
                }
            }
            return true;
        };
        for (long long gt = gt_begin; gt < gt_end && ok;) {
            const int n0 = seg_begin(gt);
            const int n1 = seg_end(gt, n0);
            const int stream_b = static_cast<int>(gt / tps) / p.Hkv, stream_g = static_cast<int>(gt / tps) % p.Hkv;
            for (int n = n0; n < n1; ++n, ++it) {
                if ((it & 1) != wg)
                    continue;
                const int klo = tc_kb_lo(n, TOK, p.window), khi = tc_kb_hi(n, TOK, p.T);
                const int nb = khi - klo + 1;
                const int bs = klo * 32;
                const int t = n * TOK + ti;
                const int lo_key = max(0, t - p.window + 1), hi_key = min(t, p.T - 1);
                if (!mbar_wait(&s_full[wg], static_cast<uint32_t>((it >> 1) & 1)) ||
                    !mbar_wait(&kinfo[wg], static_cast<uint32_t>((it >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // blocks of the band whose key rows were shifted into fp16 range (almost always none)
                const uint32_t band = kband[wg];
                const uint32_t smask = band & 0xffffu;
                const int slot0 = static_cast<int>(band >> 16);
                // keys of this row: lo_key .. hi_key; a key is valid iff 0 <= key - lo_key <= span
                int lo = lo_key, span = hi_key - lo_key;
                if (span < 0) {
                    lo = -(1 << 29);  // empty row: every key fails the test below
                    span = 0;
                }
                const unsigned uspan = static_cast<unsigned>(span);
                // chunks whose keys are inside the window of every row of this warp need no mask
                unsigned inner = 0;
                for (int q = 0; q < nb; ++q) {
                    const int key0 = bs + 32 * q;
                    if (__all_sync(0xffffffffu, key0 >= lo_key && key0 + 31 <= hi_key))
                        inner |= 1u << q;
                }
                // logits of shifted key rows times 2^e_j (rare): rewritten in tensor memory first
#pragma unroll 1
                for (int q = 0; q < nb && smask != 0; ++q) {
                    const uint32_t wm = (smask >> (2 * q)) & 3u;
                    if (wm != 0)
                        unshift_chunk32(s_col + 32 * q, kexp + ((slot0 + q) % C::STAGES) * C::KB, 0, wm, 8, 4,
                                        range_bad);
                }
                // The band is read in 16-column halves, the next half's load in flight while the
                // current one is processed (tcgen05.wait::ld waits for every load of the thread).
                // Row max of one half into m4; a half of a chunk that needs the mask is masked here
                // and written back, so the exponent pass needs no mask
                auto half_max = [&](uint32_t (&v)[16], int hq, float (&m4)[4]) {
                    if (!(inner >> (hq >> 1) & 1u)) {
                        const int k0 = bs + 16 * hq - lo;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (static_cast<unsigned>(k0 + e) > uspan)
                                v[e] = __float_as_uint(NEG_INF);
                        tmem_st16(s_col + 16 * hq, v);
                    }
#pragma unroll
                    for (int e = 0; e < 16; e += 2)
                        m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
                };
                // P = exp2(S - mu) of one half as 8 bf16 pairs (written over S columns already read);
                // row sums into l2
                auto half_exp = [&](const uint32_t (&v)[16], float2 nmu, float2 (&l2)[2], int hq) {
                    uint32_t pw[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 d = fadd2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), nmu);
                        const float2 pp = make_float2(fast_exp2(d.x), fast_exp2(d.y));
                        l2[e & 1] = fadd2(l2[e & 1], pp);
                        pw[e] = pack_bf16x2(pp.x, pp.y);
                    }
                    tmem_st8(s_col + 8 * hq, pw);
                };
                const int nh = 2 * nb;
                uint32_t va[16], vb[16];
                // pass 1: row max over the band
                float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
                tmem_ld16(s_col, va);
                tmem_wait_ld();
#pragma unroll 1
                for (int hq = 0; hq < nh; hq += 2) {
                    tmem_ld16(s_col + 16 * (hq + 1), vb);
                    half_max(va, hq, m4);
                    tmem_wait_ld();
                    if (hq + 2 < nh)
                        tmem_ld16(s_col + 16 * (hq + 2), va);
                    half_max(vb, hq + 1, m4);
                    if (hq + 2 < nh)
                        tmem_wait_ld();
                }
                tmem_wait_st();
                const float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                const float mu = (m == NEG_INF) ? 0.f : m;
                const float2 nmu = make_float2(-mu, -mu);
                // pass 2: P = exp2(S - max) as bf16 over S, row sum
                float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                tmem_ld16(s_col, va);
                tmem_wait_ld();
#pragma unroll 1
                for (int hq = 0; hq < nh; hq += 2) {
                    tmem_ld16(s_col + 16 * (hq + 1), vb);
                    half_exp(va, nmu, l2, hq);
                    tmem_wait_ld();
                    if (hq + 2 < nh)
                        tmem_ld16(s_col + 16 * (hq + 2), va);
                    half_exp(vb, nmu, l2, hq + 1);
                    if (hq + 2 < nh)
                        tmem_wait_ld();
                }
                const float l4[4] = {l2[0].x, l2[0].y, l2[1].x, l2[1].y};
                const float l0 = l4[0] + l4[1], l1 = l4[2] + l4[3];
                const float l = l0 + l1;
                if (LSE && t < p.T && l > 0.f)  // the row's log-sum-exp, natural log
                    p.lse[(static_cast<long long>(stream_b) * p.T + t) * p.Hq + stream_g * G + r % G] =
                        (mu + __log2f(l)) * 0.6931471805599453f;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[wg]);
                // this warpgroup also writes its tile's output once O = P V is done
                if (!epilogue(it, stream_b, stream_g, n, l > 0.f ? 1.f / l : 0.f)) {
                    ok = false;
                    break;
                }
            }
            gt += n1 - n0;
        }
        if (range_bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
        if (!ok && lane == 0)
            record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    } else {
        // ------------------------------------------------------------------ query preparation
        const int tid = threadIdx.x - 384;  // 0..127
        const int cr = tid % C::CPR;        // this thread's 16-byte chunk within a query row
        const int row0 = tid / C::CPR;      // first row it prepares; then every RPP-th row
        const int sl = cr / 8, c8 = cr % 8;
        bool ok = true, bad = false;
        int it = 0;
        for (long long gt = gt_begin; gt < gt_end && ok;) {
            const int stream = static_cast<int>(gt / tps), n0 = seg_begin(gt);
            const int n1 = seg_end(gt, n0);
            const int g = stream % p.Hkv;
            // alpha * scale and beta * scale for this thread's columns; its rows alternate
            // between at most two heads (G divides 2 * RPP)
            float as[2][8], bsv[2][8];
#pragma unroll
            for (int hsel = 0; hsel < 2; ++hsel) {
                const int h = g * G + (row0 + hsel * C::RPP) % G;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    as[hsel][e] = __ldg(p.alpha + h * D + 8 * cr + e) * p.qscale;
                    bsv[hsel][e] = __ldg(p.beta + h * D + 8 * cr + e) * p.qscale;
                }
            }
            for (int n = n0; n < n1 && ok; ++n, ++it) {
                const int buf = it & 1;
                if (!mbar_wait(&qfull[buf], static_cast<uint32_t>((it >> 1) & 1))) {
                    ok = false;
                    break;
                }
                uint8_t *qb = smem + C::Q_OFF + buf * C::Q_BYTES + sl * C::Q_SLAB;
                float amax = 0.f;
#pragma unroll 4
                for (int j = 0; j < C::CPR; ++j) {
                    const int row = row0 + j * C::RPP;
                    const int hs = ((j * C::RPP) % G == 0) ? 0 : 1;  // which of the two heads
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
                    mbar_arrive(&qt_full[buf]);
            }
            gt += n1 - n0;
        }
        if (bad)
            record_error(p.dev_err, ORTHROS_DEVERR_RANGE);
        if (!ok && lane == 0)
            record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
    }

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TM_COLS);
    }
}

template <int D, int G>
static cudaError_t launch_swa_tc_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                   const SwaParams &p, int num_sms, cudaStream_t stream)
{
    using C = TcCfg<D>;
    // the log-sum-exp is asked for on full calls only (row_begin = 0)
    if (p.lse != nullptr && p.n_base > 0)
        return cudaErrorInvalidValue;
    auto kern = p.lse != nullptr ? swa_tc_kernel<D, G, false, true>
                                 : (p.n_base > 0 ? swa_tc_kernel<D, G, true, false> : swa_tc_kernel<D, G, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    long long grid = p.total_tiles < num_sms ? p.total_tiles : num_sms;
    if (grid < 1)
        grid = 1;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

// Can the tensor-memory kernel run this (head dim, grouping, window)?  A tile's
// band must fit NB blocks (tensor memory, mirror slots), and the ring must hold
// the band of one tile plus the blocks the next tile adds.
bool swa_tc_supported(int D, int G, int window)
{
    if (G < 2 || G > 16 || (D != 64 && D != 128))
        return false;
    const long long TOK = 128 / G;
    const int NB = D == 128 ? TcCfg<128>::NB : TcCfg<64>::NB;
    // exact widest band over tile alignments (far from the sequence start)
    const long long base = (static_cast<long long>(window) / TOK + 64) * TOK * 32;
    long long widest = 0;
    for (long long n = base / TOK; n < base / TOK + 64; ++n) {
        const long long t0 = n * TOK;
        const long long lo = (t0 - window + 1) / 32, hi = (t0 + TOK - 1) / 32;
        widest = hi - lo + 1 > widest ? hi - lo + 1 : widest;
    }
    const long long advance = (TOK + 31) / 32;
    return widest <= NB && widest + advance <= TcCfg<128>::STAGES;
}

cudaError_t launch_swa_tc(int D, int G, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                          const CUtensorMap &o, const SwaParams &p, int num_sms, cudaStream_t stream)
{
    (void)o;  // rows are stored straight from registers (p.o)
#define ORTHROS_TC_CASE(DD, GG) \
    if (D == DD && G == GG)     \
        return launch_swa_tc_t<DD, GG>(q, k, v, p, num_sms, stream);
    ORTHROS_TC_CASE(128, 2)
    ORTHROS_TC_CASE(128, 4)
    ORTHROS_TC_CASE(128, 8)
    ORTHROS_TC_CASE(128, 16)
    ORTHROS_TC_CASE(64, 2)
    ORTHROS_TC_CASE(64, 4)
    ORTHROS_TC_CASE(64, 8)
    ORTHROS_TC_CASE(64, 16)
#undef ORTHROS_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace orthros
