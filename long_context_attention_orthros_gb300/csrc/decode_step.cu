// decode_step.cu -- one fused decode step of "Orthros: Phase-Aware Heterogeneous
// Attention" (Sec. 3.2 decode mode, T_in = 0 and T_out = 1 per step; the
// [A, B, C] -> D, D' example of Sec. 2.4): per sequence b with p = cache_len[b],
//   append k_new / v_new at cache row p,
//   o  = Eq. (4) for the new base token over rows max(0, p-w+1) .. p,
//   oc = Eq. (5) for its output copy over rows 0 .. p,
//   cache_len[b] = p + 1.
//
// One launch, grid (nsplit + 1, B * Hkv):
//   * split CTAs (x < nsplit) stream whole 64-key blocks of the old cache rows
//     [0, 64 * floor(p / 64)) through a TMA ring and produce partial softmax
//     results for the copy's G query heads (GQA: one K/V pass serves all G);
//   * the tail CTA (x == nsplit) handles the rest with plain loads: the ragged
//     rows 64 * floor(p / 64) .. p-1 plus the new row (taken from k_new / v_new,
//     never read back from the cache) for the copy, the base token's window,
//     and the append itself;
//   * each split CTA merges its four warps' partial results in shared memory and
//     writes one partial; the last CTA of each (b, KV head) to finish merges the
//     partials (an atomic arrival counter, no spin-wait), loading all of their
//     weights first so that the partial outputs stream in with several loads in
//     flight, and the last group of each sequence bumps cache_len.  Counters are
//     left at zero for the next step.
// Rows at or beyond the old cache_len are never read from memory.
#include "kernels.cuh"
#include "xattn.cuh"

namespace orthros {

template <int D>
struct DCfg {
    static constexpr int KB = 64;
    static constexpr int SLAB = KB * 128;
    static constexpr int KV_BYTES = KB * D * 2;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int STAGES = 3;
    static constexpr int CWARPS = 4;
    static constexpr int CTHREADS = CWARPS * 32;
    static constexpr int THREADS = CTHREADS + 32;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int SMEM = BAR_OFF + 2 * STAGES * 8 + 64 + 1024;
};

// Tail-CTA helper (128 threads): softmax attention of G query rows q_s[G][D]
// (scaled into log2 units) over keys lo .. p of one KV head, where rows < p come
// from the cache and row p from k_new / v_new.  Leaves the unnormalised result in
// acc (thread t < D holds column t of every row), and m_s / l_s per row.
template <int D, int G>
__device__ void tail_attend(const float *q_s, float *logit_s, float *m_s, float *l_s, float *corr_s,
                            const orthros_bf16 *kc, const orthros_bf16 *vc, long long row_stride,
                            const orthros_bf16 *knew, const orthros_bf16 *vnew, int lo, int p,
                            float (&acc)[G])
{
    constexpr int NT = 128;
    const int t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31;
    const float NEG_INF = -__int_as_float(0x7f800000);
    if (t < G) {
        m_s[t] = NEG_INF;
        l_s[t] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < G; ++r)
        acc[r] = 0.f;
    named_barrier(1, NT);
    for (int c0 = lo; c0 <= p; c0 += NT) {
        const int j = c0 + t;
        if (j <= p) {
            const orthros_bf16 *krow = (j == p) ? knew : kc + j * row_stride;
            float kf[D];
#pragma unroll
            for (int e = 0; e < D; e += 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(krow + e);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = unpack_bf16x2(w[q]);
                    kf[e + 2 * q] = f.x;
                    kf[e + 2 * q + 1] = f.y;
                }
            }
#pragma unroll
            for (int r = 0; r < G; ++r) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < D; ++e)
                    s = fmaf(q_s[r * D + e], kf[e], s);
                logit_s[r * NT + t] = s;
            }
        } else {
#pragma unroll
            for (int r = 0; r < G; ++r)
                logit_s[r * NT + t] = NEG_INF;
        }
        named_barrier(1, NT);
        // per-row online update (warp w handles rows w, w + 4, ...)
        for (int r = warp; r < G; r += 4) {
            float cm = NEG_INF;
            for (int i = lane; i < NT; i += 32)
                cm = fmaxf(cm, logit_s[r * NT + i]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
            const float mo = m_s[r];
            const float mn = fmaxf(mo, cm);  // finite: every chunk holds a valid key
            float sum = 0.f;
            for (int i = lane; i < NT; i += 32) {
                const float pr = fast_exp2(logit_s[r * NT + i] - mn);
                logit_s[r * NT + i] = pr;
                sum += pr;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (lane == 0) {
                const float corr = fast_exp2(mo - mn);
                corr_s[r] = corr;
                l_s[r] = l_s[r] * corr + sum;
                m_s[r] = mn;
            }
        }
        named_barrier(1, NT);
        if (t < D) {
            const int jn = min(NT, p - c0 + 1);
#pragma unroll
            for (int r = 0; r < G; ++r)
                acc[r] *= corr_s[r];
            for (int i = 0; i < jn; ++i) {
                const int jj = c0 + i;
                const orthros_bf16 *vrow = (jj == p) ? vnew : vc + jj * row_stride;
                const float v = __uint_as_float(static_cast<uint32_t>(vrow[t]) << 16);
#pragma unroll
                for (int r = 0; r < G; ++r)
                    acc[r] = fmaf(logit_s[r * NT + i], v, acc[r]);
            }
        }
        named_barrier(1, NT);
    }
}

template <int D, int G>
__global__ void __launch_bounds__(DCfg<D>::THREADS)
    decode_step_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const DecodeParams p)
{
    using C = DCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_s + pad;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    int *s_flag = reinterpret_cast<int *>(smem + C::BAR_OFF + 2 * C::STAGES * 8);

    // Launched as a programmatic dependent of the previous kernel on the stream (the previous
    // step, say): the next step's grid may be launched as soon as every CTA of this one has
    // started, and this grid touches nothing the previous one wrote (cache_len, the cache, the
    // partials' workspace) before that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int x = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.Hkv, g = bh % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pcur = p.cache_len[b];
    const bool cache_full = pcur < 0 || pcur >= p.L_max;
    const int nfull = cache_full ? 0 : (pcur / C::KB) * C::KB;  // keys in whole blocks
    int chunk = (nfull + p.nsplit - 1) / p.nsplit;
    chunk = (chunk + C::KB - 1) / C::KB * C::KB;
    const int js = x * chunk;
    const int je = min(js + chunk, nfull);
    const int nblk = (x < p.nsplit && je > js) ? (je - js) / C::KB : 0;
    const long long row_stride = static_cast<long long>(p.Hkv) * D;
    const orthros_bf16 *kc = p.k_cache + (static_cast<long long>(b) * p.L_max * p.Hkv + g) * D;
    const orthros_bf16 *vc = p.v_cache + (static_cast<long long>(b) * p.L_max * p.Hkv + g) * D;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::CWARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == C::CWARPS) {
        // producer (split CTAs only)
        if (lane != 0 || nblk == 0)
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

    const int BH = p.B * p.Hkv;
    float *part_o = p.part_o + static_cast<long long>(bh) * p.n_part * G * D;
    float2 *part_ml = p.part_ml + static_cast<long long>(bh) * p.n_part * G;

    if (x < p.nsplit) {
        // ------------------------------------------------ split CTA: copy rows
        // the G copy rows of this KV head on the MMA's N side (keys on M): q^T fragments
        // hold row 8 nt + lane / 4; the lane keeps rows 8 nt + 2 (lane % 4) + {0, 1}
        constexpr int NT = (G + 7) / 8;
        WarpKeys16<D, NT, false> st;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int kt = 0; kt < D / 16; ++kt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int row = 8 * nt + (lane >> 2);
                    const int dcol = kt * 16 + 2 * (lane & 3) + 8 * hf;
                    uint32_t hi = 0, lo = 0;
                    if (row < G && !cache_full) {
                        const int h = g * G + row;
                        load_q_pair(p.qc_new + (static_cast<long long>(b) * p.Hq + h) * D, p.alpha_c + h * D,
                                    p.beta_c + h * D, dcol, p.qscale, hi, lo);
                    }
                    st.qb[nt][kt][hf] = hi;
                    st.ql[nt][kt][hf] = lo;
                }
        st.reset();
        int lim[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            lim[nt][0] = lim[nt][1] = 0x7fffffff;
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            const int s = i % C::STAGES;
            if (!mbar_wait(&full[s], static_cast<uint32_t>((i / C::STAGES) & 1))) {
                ok = false;
                break;
            }
            const uint32_t kbase = sbase + s * C::STAGE_BYTES;
            // every key of a whole block is below p: no mask (padding rows are never written)
            st.step(kbase, C::SLAB, kbase + C::KV_BYTES, C::SLAB, warp * 16, js + i * C::KB + warp * 16, lim, true);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
        }
        if (!ok && lane == 0)
            record_error(p.dev_err, ORTHROS_DEVERR_TIMEOUT);
        st.finish_sums();
        // one partial per CTA: the four warps' results merged in shared memory (the ring is free:
        // every block has been consumed)
        float *ms = reinterpret_cast<float *>(smem);  // [CWARPS][G] max
        float *ls = ms + C::CWARPS * G;               // [CWARPS][G] sum
        float *os = ls + C::CWARPS * G;               // [CWARPS][G][D] output, scaled to the CTA's max
        named_barrier(3, C::CTHREADS);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int row = 8 * nt + 2 * (lane & 3) + r2;
                if (row < G && (lane >> 2) == 0) {
                    ms[warp * G + row] = st.m[nt][r2];
                    ls[warp * G + row] = st.l[nt][r2];
                }
            }
        named_barrier(3, C::CTHREADS);
        const float NEG_INF = -__int_as_float(0x7f800000);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int row = 8 * nt + 2 * (lane & 3) + r2;
                if (row >= G)
                    continue;
                float M = NEG_INF;
#pragma unroll
                for (int w = 0; w < C::CWARPS; ++w)
                    M = fmaxf(M, ms[w * G + row]);
                const float f = (M == NEG_INF || st.m[nt][r2] == NEG_INF) ? 0.f : fast_exp2(st.m[nt][r2] - M);
                float *po = os + (warp * G + row) * D + (lane >> 2);
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    po[16 * mt] = st.o[nt][mt][r2] * f;
                    po[16 * mt + 8] = st.o[nt][mt][2 + r2] * f;
                }
            }
        named_barrier(3, C::CTHREADS);
        for (int i = threadIdx.x; i < G * D; i += C::CTHREADS) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < C::CWARPS; ++w)
                a += os[w * G * D + i];
            part_o[static_cast<long long>(x) * G * D + i] = a;
        }
        if (threadIdx.x < G) {
            const int row = threadIdx.x;
            float M = NEG_INF, L = 0.f;
#pragma unroll
            for (int w = 0; w < C::CWARPS; ++w)
                M = fmaxf(M, ms[w * G + row]);
#pragma unroll
            for (int w = 0; w < C::CWARPS; ++w)
                if (ms[w * G + row] != NEG_INF)
                    L += ls[w * G + row] * fast_exp2(ms[w * G + row] - M);
            part_ml[static_cast<long long>(x) * G + row] = make_float2(M, L);
        }
    } else {
        // ------------------------------------------------ tail CTA
        float *q_s = reinterpret_cast<float *>(smem);          // [G][D]
        float *logit_s = q_s + G * D;                          // [G][128]
        float *m_s = logit_s + G * 128;                        // [G]
        float *l_s = m_s + G;
        float *corr_s = l_s + G;
        const int t = threadIdx.x;
        if (cache_full) {
            if (g == 0 && t == 0)
                record_error(p.dev_err, ORTHROS_DEVERR_CACHE_FULL);
            for (int i = t; i < G * D; i += C::CTHREADS) {
                const int h = g * G + i / D;
                p.o[(static_cast<long long>(b) * p.Hq + h) * D + i % D] = 0;
            }
        } else {
            const orthros_bf16 *knew = p.k_new + (static_cast<long long>(b) * p.Hkv + g) * D;
            const orthros_bf16 *vnew = p.v_new + (static_cast<long long>(b) * p.Hkv + g) * D;
            float acc[G];
            // (1) the copy over the ragged rows nfull .. p-1 and the new row p
            for (int i = t; i < G * D; i += C::CTHREADS) {
                const int h = g * G + i / D, e = i % D;
                const float x0 = __uint_as_float(
                    static_cast<uint32_t>(p.qc_new[(static_cast<long long>(b) * p.Hq + h) * D + e]) << 16);
                q_s[i] = fmaf(x0, p.alpha_c[h * D + e], p.beta_c[h * D + e]) * p.qscale;
            }
            tail_attend<D, G>(q_s, logit_s, m_s, l_s, corr_s, kc, vc, row_stride, knew, vnew, nfull, pcur, acc);
            const int part = p.nsplit;
            if (t < D) {
#pragma unroll
                for (int r = 0; r < G; ++r)
                    part_o[(static_cast<long long>(part) * G + r) * D + t] = acc[r];
            }
            if (t < G)
                part_ml[static_cast<long long>(part) * G + t] = make_float2(m_s[t], l_s[t]);
            named_barrier(1, C::CTHREADS);
            // (2) the base token over its window max(0, p-w+1) .. p
            for (int i = t; i < G * D; i += C::CTHREADS) {
                const int h = g * G + i / D, e = i % D;
                const float x0 = __uint_as_float(
                    static_cast<uint32_t>(p.q_new[(static_cast<long long>(b) * p.Hq + h) * D + e]) << 16);
                q_s[i] = fmaf(x0, p.alpha[h * D + e], p.beta[h * D + e]) * p.qscale;
            }
            const int lo = pcur - p.window + 1 > 0 ? pcur - p.window + 1 : 0;
            tail_attend<D, G>(q_s, logit_s, m_s, l_s, corr_s, kc, vc, row_stride, knew, vnew, lo, pcur, acc);
            if (t < D) {
#pragma unroll
                for (int r = 0; r < G; ++r) {
                    const int h = g * G + r;
                    const float v = l_s[r] > 0.f ? acc[r] / l_s[r] : 0.f;
                    p.o[(static_cast<long long>(b) * p.Hq + h) * D + t] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                }
            }
            // (3) append the new base token's K/V (the copy writes nothing)
            if (t < D / 8) {
                reinterpret_cast<uint4 *>(p.k_cache + ((static_cast<long long>(b) * p.L_max + pcur) * p.Hkv + g) * D)[t] =
                    reinterpret_cast<const uint4 *>(knew)[t];
                reinterpret_cast<uint4 *>(p.v_cache + ((static_cast<long long>(b) * p.L_max + pcur) * p.Hkv + g) * D)[t] =
                    reinterpret_cast<const uint4 *>(vnew)[t];
            }
        }
    }

    // ---------------------------------------------------- arrival and merge
    __threadfence();
    named_barrier(2, C::CTHREADS);
    if (threadIdx.x == 0)
        s_flag[0] = (atomicAdd(&p.cnt_bh[bh], 1) == p.nsplit) ? 1 : 0;
    named_barrier(2, C::CTHREADS);
    if (!s_flag[0])
        return;
    __threadfence();
    const float NEG_INF = -__int_as_float(0x7f800000);
    float *w_s = reinterpret_cast<float *>(smem);  // [G][n_part] partial weights (this CTA's work is done)
    for (int r = warp; r < G; r += C::CWARPS) {
        const int h = g * G + r;
        orthros_bf16 *orow = p.oc + (static_cast<long long>(b) * p.Hq + h) * D;
        if (cache_full) {
            for (int e = lane; e < D; e += 32)
                orow[e] = 0;
            continue;
        }
        // the partials' weights exp2(m - M), all loaded at once (lane q, q + 32, ...)
        float M = NEG_INF;
        for (int q = lane; q < p.n_part; q += 32) {
            const float2 ml = __ldcg(&part_ml[static_cast<long long>(q) * G + r]);
            if (ml.y > 0.f)
                M = fmaxf(M, ml.x);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
        for (int q = lane; q < p.n_part; q += 32) {
            const float2 ml = __ldcg(&part_ml[static_cast<long long>(q) * G + r]);
            const float w = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
            w_s[r * p.n_part + q] = w;
            L += ml.y > 0.f ? ml.y * w : 0.f;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            L += __shfl_xor_sync(0xffffffffu, L, off);
        __syncwarp();
        // the weighted sum of the partial outputs: independent loads, several in flight
        constexpr int E = D / 32;
        float a[E];
#pragma unroll
        for (int e = 0; e < E; ++e)
            a[e] = 0.f;
#pragma unroll 8
        for (int q = 0; q < p.n_part; ++q) {
            const float w = w_s[r * p.n_part + q];
            const float *po = part_o + (static_cast<long long>(q) * G + r) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e)
                a[e] = fmaf(w, __ldcg(po + e), a[e]);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<uint32_t *>(orow + lane * E + e) = pack_bf16x2(a[e] * inv, a[e + 1] * inv);
    }
    if (threadIdx.x == 0) {
        p.cnt_bh[bh] = 0;
        __threadfence();
        if (atomicAdd(&p.cnt_b[b], 1) == p.Hkv - 1) {
            if (!cache_full)
                p.cache_len[b] = pcur + 1;
            p.cnt_b[b] = 0;
        }
    }
    (void)BH;
}

// ------------------------------------------------------------------ host side

int decode_nsplit(int B, int L_max, int Hkv)
{
    const long long BH = static_cast<long long>(B) * Hkv;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 148;
    // two CTAs fit an SM (shared memory): the split and tail CTAs of every (b, KV head) in one wave
    long long ns = 2LL * sms / BH - 1;
    const long long by_len = (static_cast<long long>(L_max) + 1023) / 1024;
    if (ns > by_len)
        ns = by_len;
    if (ns < 1)
        ns = 1;
    return static_cast<int>(ns);
}

size_t decode_workspace_bytes(int B, int L_max, int Hq, int Hkv, int D)
{
    const int G = Hq / Hkv;
    const int ns = decode_nsplit(B, L_max, Hkv);
    const size_t n_part = static_cast<size_t>(ns) + 1;
    const size_t BH = static_cast<size_t>(B) * Hkv;
    const size_t o_bytes = (BH * n_part * G * D * sizeof(float) + 255) / 256 * 256;
    const size_t ml_bytes = (BH * n_part * G * sizeof(float2) + 255) / 256 * 256;
    const size_t cnt_bytes = ((BH + B) * sizeof(int) + 255) / 256 * 256;
    return o_bytes + ml_bytes + cnt_bytes;
}

template <int D, int G>
static cudaError_t launch_decode_t(const CUtensorMap &k, const CUtensorMap &v, const DecodeParams &p,
                                   cudaStream_t stream)
{
    auto kern = decode_step_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<D>::SMEM);
    if (e != cudaSuccess)
        return e;
    // programmatic dependent launch: the grid is set up while the previous kernel on the stream
    // finishes (its CTAs wait for it before their first access; see the kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nsplit + 1, p.B * p.Hkv);
    cfg.blockDim = dim3(DCfg<D>::THREADS);
    cfg.dynamicSmemBytes = DCfg<D>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, k, v, p);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_decode(int D, const CUtensorMap &k, const CUtensorMap &v, DecodeParams p,
                          void *workspace, cudaStream_t stream)
{
    const int G = p.Hq / p.Hkv;
    p.nsplit = decode_nsplit(p.B, p.L_max, p.Hkv);
    p.n_part = p.nsplit + 1;  // one per split CTA and the tail
    const size_t BH = static_cast<size_t>(p.B) * p.Hkv;
    const size_t o_bytes = (BH * p.n_part * G * D * sizeof(float) + 255) / 256 * 256;
    const size_t ml_bytes = (BH * p.n_part * G * sizeof(float2) + 255) / 256 * 256;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.part_o = reinterpret_cast<float *>(ws);
    p.part_ml = reinterpret_cast<float2 *>(ws + o_bytes);
    p.cnt_bh = reinterpret_cast<int *>(ws + o_bytes + ml_bytes);
    p.cnt_b = p.cnt_bh + BH;
#define ORTHROS_DEC_CASE(DD, GG) \
    if (D == DD && G == GG)      \
        return launch_decode_t<DD, GG>(k, v, p, stream);
    ORTHROS_DEC_CASE(128, 1)
    ORTHROS_DEC_CASE(128, 2)
    ORTHROS_DEC_CASE(128, 4)
    ORTHROS_DEC_CASE(128, 8)
    ORTHROS_DEC_CASE(128, 16)
    ORTHROS_DEC_CASE(64, 1)
    ORTHROS_DEC_CASE(64, 2)
    ORTHROS_DEC_CASE(64, 4)
    ORTHROS_DEC_CASE(64, 8)
    ORTHROS_DEC_CASE(64, 16)
#undef ORTHROS_DEC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace orthros
