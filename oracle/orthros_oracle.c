/*
 * orthros_oracle.c -- plain, slow, fp64 CPU statement of the Orthros per-layer
 * attention operator.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle: only the test
 * suite, the package's smoke check and the benchmark's CPU-baseline / reference
 * arm load it.  It shares no code, header or table with the CUDA path.
 *
 * What it follows (Orthros: Phase-Aware Heterogeneous Attention, read through
 * the close-reading notes of arXiv 2610.13735; the display equations did not
 * survive extraction, so the formulas are restated from the surrounding prose):
 *
 *  - Sec. 3.1 / symbol table: the base stream and the output copies share W_Q;
 *    each stream applies its own 1 x d scale-offset to the projected query,
 *      q_t  = (x_t  W_Q) * alpha  + beta      (base stream)
 *      q'_t = (x'_t W_Q) * alpha' + beta'     (output copies)
 *    The operator receives Q_raw = x W_Q already projected (bf16), alpha/beta as
 *    fp32 [Hq, d] (one 1 x d vector per query head).
 *  - Eq. (4): every base position t attends with softmax over the window
 *    W_t = {max(1, t-w+1) .. t} (1-based; here 0-based {max(0, t-w+1) .. t}).
 *  - Eq. (5): a copy at original position t attends over all base keys j <= t.
 *    Copies read only base K/V and never write K/V (Sec. 3.1-3.2 dependency
 *    isolation); the mask uses the copy's original position, not its physical
 *    slot when copies are appended (Algorithm 2).
 *  - Sec. 3.2 decode: each step appends the new base token's K/V to the cache,
 *    then the base token attends over its window and the copy at the same
 *    position over the whole cache (the [A,B,C] -> D, D' teaching example).
 *  - Softmax logits are (q . k) * scale with scale = 1/sqrt(d) (standard scaled
 *    dot-product attention; the printed formula is not legible).
 *  - GQA: query head h reads KV head h / (Hq / Hkv) (contiguous groups).
 *
 * Everything is computed in double precision from the exactly widened bf16
 * inputs; nothing is rounded.  No blocking, fusion or reordering beyond the
 * definition: each output row is an independent max-subtracted softmax.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the calling thread's later parallel regions (timing only; no effect on values). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* q[e] = bf16(q_raw[e]) * alpha[e] + beta[e]  (the stream's scale-offset) */
static void scale_offset_row(const uint16_t *q_raw, const float *alpha, const float *beta,
                             int d, double *q)
{
    for (int e = 0; e < d; ++e)
        q[e] = bf16_to_double(q_raw[e]) * (double)alpha[e] + (double)beta[e];
}

/*
 * Softmax attention of one query row q[d] over key rows j = lo..hi (inclusive)
 * of one KV head.  key(j) = kv_k + j * kv_row_stride, likewise for values.
 * out[d] = sum_j p_j v_j,  p_j = exp(s_j - max s) / sum exp(s - max s),
 * s_j = scale * (q . k_j).  `logit` is scratch of at least hi-lo+1 doubles.
 */
static void attend(const double *q, const uint16_t *kv_k, const uint16_t *kv_v,
                   int64_t kv_row_stride, int64_t lo, int64_t hi, int d, double scale,
                   double *logit, double *out)
{
    double m = -INFINITY;
    for (int64_t j = lo; j <= hi; ++j) {
        const uint16_t *kj = kv_k + j * kv_row_stride;
        double s = 0.0;
        for (int e = 0; e < d; ++e)
            s += q[e] * bf16_to_double(kj[e]);
        s *= scale;
        logit[j - lo] = s;
        if (s > m)
            m = s;
    }
    for (int e = 0; e < d; ++e)
        out[e] = 0.0;
    double den = 0.0;
    for (int64_t j = lo; j <= hi; ++j) {
        const double p = exp(logit[j - lo] - m);
        const uint16_t *vj = kv_v + j * kv_row_stride;
        den += p;
        for (int e = 0; e < d; ++e)
            out[e] += p * bf16_to_double(vj[e]);
    }
    for (int e = 0; e < d; ++e)
        out[e] /= den;
}

static int shapes_ok(int B, int T, int Hq, int Hkv, int d)
{
    return B >= 1 && T >= 1 && Hq >= 1 && Hkv >= 1 && d >= 1 && Hq % Hkv == 0;
}

/*
 * Base stream, Eq. (4), at the listed rows (b_idx[r], t_idx[r]) for all Hq heads.
 * q_raw: bf16 [B, T, Hq, d]; k, v: bf16 [B, T, Hkv, d]; alpha, beta: fp32 [Hq, d];
 * o: fp64 [n, Hq, d].  Returns 0, or -1 on a bad argument.
 */
int oracle_swa_rows(const uint16_t *q_raw, const uint16_t *k, const uint16_t *v,
                    const float *alpha, const float *beta, double *o,
                    int B, int T, int Hq, int Hkv, int d, int window, double scale,
                    const int32_t *b_idx, const int32_t *t_idx, int n)
{
    if (!shapes_ok(B, T, Hq, Hkv, d) || window < 1 || n < 0)
        return -1;
    for (int r = 0; r < n; ++r)
        if (b_idx[r] < 0 || b_idx[r] >= B || t_idx[r] < 0 || t_idx[r] >= T)
            return -1;
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * d;
    int bad = 0;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *logit = (double *)malloc(sizeof(double) * (size_t)window);
        if (!q || !logit) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t job = 0; job < (int64_t)n * Hq; ++job) {
                const int r = (int)(job / Hq), h = (int)(job % Hq);
                const int64_t b = b_idx[r], t = t_idx[r];
                const int g = h / group;
                const int64_t lo = t - window + 1 > 0 ? t - window + 1 : 0;
                scale_offset_row(q_raw + ((b * T + t) * Hq + h) * d, alpha + (int64_t)h * d,
                                 beta + (int64_t)h * d, d, q);
                const uint16_t *kb = k + (b * T * Hkv + g) * d;
                const uint16_t *vb = v + (b * T * Hkv + g) * d;
                attend(q, kb, vb, kv_row, lo, t, d, scale, logit,
                       o + ((int64_t)r * Hq + h) * d);
            }
        }
        free(q);
        free(logit);
    }
    return bad ? -2 : 0;
}

/* Base stream, Eq. (4), at every position: o fp64 [B, T, Hq, d]. */
int oracle_swa(const uint16_t *q_raw, const uint16_t *k, const uint16_t *v,
               const float *alpha, const float *beta, double *o,
               int B, int T, int Hq, int Hkv, int d, int window, double scale)
{
    if (!shapes_ok(B, T, Hq, Hkv, d) || window < 1)
        return -1;
    int32_t *bi = (int32_t *)malloc(sizeof(int32_t) * (size_t)B * T);
    int32_t *ti = (int32_t *)malloc(sizeof(int32_t) * (size_t)B * T);
    if (!bi || !ti) {
        free(bi);
        free(ti);
        return -2;
    }
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            bi[(int64_t)b * T + t] = b;
            ti[(int64_t)b * T + t] = t;
        }
    int rc = oracle_swa_rows(q_raw, k, v, alpha, beta, o, B, T, Hq, Hkv, d, window, scale,
                             bi, ti, B * T);
    free(bi);
    free(ti);
    return rc;
}

/*
 * Output copies, Eq. (5): copy i of sequence b sits at original position
 * pos[b, i] and attends over base keys 0..pos[b, i] of that sequence.
 * qc_raw: bf16 [B, T_out, Hq, d]; pos: int32 [B, T_out]; k, v: bf16 [B, T_kv, Hkv, d];
 * oc: fp64 [B, T_out, Hq, d].  Returns 0, or -1 on a bad argument or position.
 */
int oracle_xattn(const uint16_t *qc_raw, const int32_t *pos, const uint16_t *k,
                 const uint16_t *v, const float *alpha_c, const float *beta_c, double *oc,
                 int B, int T_out, int T_kv, int Hq, int Hkv, int d, double scale)
{
    if (!shapes_ok(B, T_kv, Hq, Hkv, d) || T_out < 0)
        return -1;
    for (int64_t i = 0; i < (int64_t)B * T_out; ++i)
        if (pos[i] < 0 || pos[i] >= T_kv)
            return -1;
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * d;
    int bad = 0;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *logit = (double *)malloc(sizeof(double) * (size_t)T_kv);
        if (!q || !logit) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t job = 0; job < (int64_t)B * T_out * Hq; ++job) {
                const int64_t bi = job / Hq; /* flattened (b, i) */
                const int h = (int)(job % Hq);
                const int64_t b = bi / T_out;
                const int g = h / group;
                scale_offset_row(qc_raw + (bi * Hq + h) * d, alpha_c + (int64_t)h * d,
                                 beta_c + (int64_t)h * d, d, q);
                const uint16_t *kb = k + (b * T_kv * Hkv + g) * d;
                const uint16_t *vb = v + (b * T_kv * Hkv + g) * d;
                attend(q, kb, vb, kv_row, 0, pos[bi], d, scale, logit, oc + (bi * Hq + h) * d);
            }
        }
        free(q);
        free(logit);
    }
    return bad ? -2 : 0;
}

/*
 * One decode step (Sec. 3.2, T_in = 0, T_out = 1): for every sequence b with
 * p = cache_len[b], first append k_new[b], v_new[b] at cache row p (the new base
 * token's K/V), then
 *   o[b]  = SWA of q_new[b]  over cache rows max(0, p-w+1) .. p   (Eq. 4)
 *   oc[b] = attention of qc_new[b] over cache rows 0 .. p          (Eq. 5)
 * and finally cache_len[b] = p + 1.  The copy writes nothing to the cache.
 * q_new, qc_new: bf16 [B, Hq, d]; k_new, v_new: bf16 [B, Hkv, d];
 * k_cache, v_cache: bf16 [B, L_max, Hkv, d] (updated); o, oc: fp64 [B, Hq, d].
 */
int oracle_decode_step(const uint16_t *q_new, const uint16_t *qc_new, const uint16_t *k_new,
                       const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache,
                       int32_t *cache_len, int L_max, const float *alpha, const float *beta,
                       const float *alpha_c, const float *beta_c, double *o, double *oc,
                       int B, int Hq, int Hkv, int d, int window, double scale)
{
    if (!shapes_ok(B, L_max, Hq, Hkv, d) || window < 1)
        return -1;
    for (int b = 0; b < B; ++b)
        if (cache_len[b] < 0 || cache_len[b] >= L_max)
            return -1;
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * d;
    /* append first: the new token is part of its own window and of the copy's history */
    for (int b = 0; b < B; ++b) {
        const int64_t p = cache_len[b];
        memcpy(k_cache + ((int64_t)b * L_max + p) * kv_row, k_new + (int64_t)b * kv_row,
               sizeof(uint16_t) * (size_t)kv_row);
        memcpy(v_cache + ((int64_t)b * L_max + p) * kv_row, v_new + (int64_t)b * kv_row,
               sizeof(uint16_t) * (size_t)kv_row);
    }
    int bad = 0;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *logit = (double *)malloc(sizeof(double) * (size_t)L_max);
        if (!q || !logit) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t job = 0; job < (int64_t)B * Hq * 2; ++job) {
                const int copy = (int)(job & 1);
                const int64_t bh = job >> 1;
                const int64_t b = bh / Hq;
                const int h = (int)(bh % Hq);
                const int g = h / group;
                const int64_t p = cache_len[b];
                const uint16_t *kb = k_cache + (b * L_max * Hkv + g) * d;
                const uint16_t *vb = v_cache + (b * L_max * Hkv + g) * d;
                if (!copy) {
                    scale_offset_row(q_new + bh * d, alpha + (int64_t)h * d,
                                     beta + (int64_t)h * d, d, q);
                    const int64_t lo = p - window + 1 > 0 ? p - window + 1 : 0;
                    attend(q, kb, vb, kv_row, lo, p, d, scale, logit, o + bh * d);
                } else {
                    scale_offset_row(qc_new + bh * d, alpha_c + (int64_t)h * d,
                                     beta_c + (int64_t)h * d, d, q);
                    attend(q, kb, vb, kv_row, 0, p, d, scale, logit, oc + bh * d);
                }
            }
        }
        free(q);
        free(logit);
    }
    for (int b = 0; b < B; ++b)
        cache_len[b] += 1;
    return bad ? -2 : 0;
}

/*
 * Gradient of the base stream, Eq. (4) with its scale-offset, for a loss L whose
 * gradient with respect to the output o is dO (bf16 [B, T, Hq, d]).  Per row
 * (b, t, h) with window keys j = lo..t:
 *   p_j  = softmax_j(s_j),  s_j = scale * (q . k_j),  q = q_raw * alpha + beta
 *   dp_j = dO . v_j,  D = sum_j p_j dp_j,  ds_j = p_j (dp_j - D)
 *   dq   = scale * sum_j ds_j k_j,   dk_j += scale * ds_j q,   dv_j += p_j dO
 * and through the scale-offset: dq_raw = dq * alpha, dalpha += q_raw * dq,
 * dbeta += dq (summed over every row of the head).
 * Outputs (fp64, overwritten): dq_raw [B, T, Hq, d]; dk, dv [B, T, Hkv, d];
 * dalpha, dbeta [Hq, d].  Each KV head is one parallel job, so every output
 * element has a single writer.  Returns 0, or -1 on a bad argument.
 */
int oracle_swa_bwd(const uint16_t *q_raw, const uint16_t *k, const uint16_t *v,
                   const float *alpha, const float *beta, const uint16_t *dO,
                   double *dq_raw, double *dk, double *dv, double *dalpha, double *dbeta,
                   int B, int T, int Hq, int Hkv, int d, int window, double scale)
{
    if (!shapes_ok(B, T, Hq, Hkv, d) || window < 1)
        return -1;
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * d;
    memset(dq_raw, 0, sizeof(double) * (size_t)B * T * Hq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * T * Hkv * d);
    memset(dv, 0, sizeof(double) * (size_t)B * T * Hkv * d);
    memset(dalpha, 0, sizeof(double) * (size_t)Hq * d);
    memset(dbeta, 0, sizeof(double) * (size_t)Hq * d);
    int bad = 0;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *dq = (double *)malloc(sizeof(double) * (size_t)d);
        double *p = (double *)malloc(sizeof(double) * (size_t)window);
        double *dp = (double *)malloc(sizeof(double) * (size_t)window);
        if (!q || !dq || !p || !dp) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int g = 0; g < Hkv; ++g)
                for (int64_t b = 0; b < B; ++b)
                    for (int64_t t = 0; t < T; ++t)
                        for (int hh = 0; hh < group; ++hh) {
                            const int h = g * group + hh;
                            const int64_t lo = t - window + 1 > 0 ? t - window + 1 : 0;
                            const int64_t n = t - lo + 1;
                            const uint16_t *xr = q_raw + ((b * T + t) * Hq + h) * d;
                            const uint16_t *gr = dO + ((b * T + t) * Hq + h) * d;
                            const uint16_t *kb = k + (b * T * Hkv + g) * d;
                            const uint16_t *vb = v + (b * T * Hkv + g) * d;
                            scale_offset_row(xr, alpha + (int64_t)h * d, beta + (int64_t)h * d, d, q);
                            /* forward probabilities over the window */
                            double m = -INFINITY;
                            for (int64_t j = 0; j < n; ++j) {
                                const uint16_t *kj = kb + (lo + j) * kv_row;
                                double s = 0.0;
                                for (int e = 0; e < d; ++e)
                                    s += q[e] * bf16_to_double(kj[e]);
                                p[j] = s * scale;
                                if (p[j] > m)
                                    m = p[j];
                            }
                            double den = 0.0;
                            for (int64_t j = 0; j < n; ++j) {
                                p[j] = exp(p[j] - m);
                                den += p[j];
                            }
                            /* dp_j = dO . v_j and D = sum_j p_j dp_j */
                            double D = 0.0;
                            for (int64_t j = 0; j < n; ++j) {
                                p[j] /= den;
                                const uint16_t *vj = vb + (lo + j) * kv_row;
                                double acc = 0.0;
                                for (int e = 0; e < d; ++e)
                                    acc += bf16_to_double(gr[e]) * bf16_to_double(vj[e]);
                                dp[j] = acc;
                                D += p[j] * acc;
                            }
                            for (int e = 0; e < d; ++e)
                                dq[e] = 0.0;
                            for (int64_t j = 0; j < n; ++j) {
                                const double ds = p[j] * (dp[j] - D);
                                const uint16_t *kj = kb + (lo + j) * kv_row;
                                double *dkj = dk + ((b * T + lo + j) * Hkv + g) * d;
                                double *dvj = dv + ((b * T + lo + j) * Hkv + g) * d;
                                for (int e = 0; e < d; ++e) {
                                    dq[e] += scale * ds * bf16_to_double(kj[e]);
                                    dkj[e] += scale * ds * q[e];
                                    dvj[e] += p[j] * bf16_to_double(gr[e]);
                                }
                            }
                            double *dxr = dq_raw + ((b * T + t) * Hq + h) * d;
                            for (int e = 0; e < d; ++e) {
                                dxr[e] = dq[e] * (double)alpha[(int64_t)h * d + e];
                                dalpha[(int64_t)h * d + e] += bf16_to_double(xr[e]) * dq[e];
                                dbeta[(int64_t)h * d + e] += dq[e];
                            }
                        }
        }
        free(q);
        free(dq);
        free(p);
        free(dp);
    }
    return bad ? -2 : 0;
}

/*
 * Gradient of the output copies, Eq. (5) with the copies' scale-offset, for a
 * loss whose gradient with respect to the copy outputs oc is dOc (bf16
 * [B, T_out, Hq, d]).  Copy i of sequence b sits at original position
 * p = pos[b, i] and attends base keys j = 0..p; with q' = qc_raw * alpha_c + beta_c:
 *   p_j = softmax_j(scale * q' . k_j),  dp_j = dOc . v_j,  D = sum_j p_j dp_j,
 *   ds_j = p_j (dp_j - D),  dq' = scale * sum_j ds_j k_j,
 *   dk_j += scale * ds_j q',  dv_j += p_j dOc,
 *   dqc_raw = dq' * alpha_c,  dalpha_c += qc_raw * dq',  dbeta_c += dq'.
 * The copies' gradient reaches only base K/V (copies own no K/V).  Outputs
 * (fp64, overwritten): dqc_raw [B, T_out, Hq, d]; dk, dv [B, T_kv, Hkv, d] (the
 * copies' share only: a training step adds it to the base stream's);
 * dalpha_c, dbeta_c [Hq, d].  One parallel job per KV head.  Returns 0, or -1
 * on a bad argument or position.
 */
int oracle_xattn_bwd(const uint16_t *qc_raw, const int32_t *pos, const uint16_t *k,
                     const uint16_t *v, const float *alpha_c, const float *beta_c,
                     const uint16_t *dOc, double *dqc_raw, double *dk, double *dv,
                     double *dalpha_c, double *dbeta_c, int B, int T_out, int T_kv, int Hq,
                     int Hkv, int d, double scale)
{
    if (!shapes_ok(B, T_kv, Hq, Hkv, d) || T_out < 0)
        return -1;
    for (int64_t i = 0; i < (int64_t)B * T_out; ++i)
        if (pos[i] < 0 || pos[i] >= T_kv)
            return -1;
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * d;
    memset(dqc_raw, 0, sizeof(double) * (size_t)B * T_out * Hq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * T_kv * Hkv * d);
    memset(dv, 0, sizeof(double) * (size_t)B * T_kv * Hkv * d);
    memset(dalpha_c, 0, sizeof(double) * (size_t)Hq * d);
    memset(dbeta_c, 0, sizeof(double) * (size_t)Hq * d);
    int bad = 0;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *dq = (double *)malloc(sizeof(double) * (size_t)d);
        double *p = (double *)malloc(sizeof(double) * (size_t)T_kv);
        double *dp = (double *)malloc(sizeof(double) * (size_t)T_kv);
        if (!q || !dq || !p || !dp) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int g = 0; g < Hkv; ++g)
                for (int64_t b = 0; b < B; ++b)
                    for (int64_t i = 0; i < T_out; ++i)
                        for (int hh = 0; hh < group; ++hh) {
                            const int h = g * group + hh;
                            const int64_t n = (int64_t)pos[b * T_out + i] + 1; /* keys 0..pos */
                            const uint16_t *xr = qc_raw + ((b * T_out + i) * Hq + h) * d;
                            const uint16_t *gr = dOc + ((b * T_out + i) * Hq + h) * d;
                            const uint16_t *kb = k + (b * T_kv * Hkv + g) * d;
                            const uint16_t *vb = v + (b * T_kv * Hkv + g) * d;
                            scale_offset_row(xr, alpha_c + (int64_t)h * d, beta_c + (int64_t)h * d, d, q);
                            double m = -INFINITY;
                            for (int64_t j = 0; j < n; ++j) {
                                const uint16_t *kj = kb + j * kv_row;
                                double s = 0.0;
                                for (int e = 0; e < d; ++e)
                                    s += q[e] * bf16_to_double(kj[e]);
                                p[j] = s * scale;
                                if (p[j] > m)
                                    m = p[j];
                            }
                            double den = 0.0;
                            for (int64_t j = 0; j < n; ++j) {
                                p[j] = exp(p[j] - m);
                                den += p[j];
                            }
                            double D = 0.0;
                            for (int64_t j = 0; j < n; ++j) {
                                p[j] /= den;
                                const uint16_t *vj = vb + j * kv_row;
                                double acc = 0.0;
                                for (int e = 0; e < d; ++e)
                                    acc += bf16_to_double(gr[e]) * bf16_to_double(vj[e]);
                                dp[j] = acc;
                                D += p[j] * acc;
                            }
                            for (int e = 0; e < d; ++e)
                                dq[e] = 0.0;
                            for (int64_t j = 0; j < n; ++j) {
                                const double ds = p[j] * (dp[j] - D);
                                const uint16_t *kj = kb + j * kv_row;
                                double *dkj = dk + ((b * T_kv + j) * Hkv + g) * d;
                                double *dvj = dv + ((b * T_kv + j) * Hkv + g) * d;
                                for (int e = 0; e < d; ++e) {
                                    dq[e] += scale * ds * bf16_to_double(kj[e]);
                                    dkj[e] += scale * ds * q[e];
                                    dvj[e] += p[j] * bf16_to_double(gr[e]);
                                }
                            }
                            double *dxr = dqc_raw + ((b * T_out + i) * Hq + h) * d;
                            for (int e = 0; e < d; ++e) {
                                dxr[e] = dq[e] * (double)alpha_c[(int64_t)h * d + e];
                                dalpha_c[(int64_t)h * d + e] += bf16_to_double(xr[e]) * dq[e];
                                dbeta_c[(int64_t)h * d + e] += dq[e];
                            }
                        }
        }
        free(q);
        free(dq);
        free(p);
        free(dp);
    }
    return bad ? -2 : 0;
}

/*
 * Each base row's log-sum-exp, Eq. (4): lse[b, t, h] = ln sum_{j in W_t} exp(scale * q_t . k_j)
 * with q_t = q_raw * alpha + beta, the normaliser of the row's softmax (the quantity a
 * training forward keeps for the gradient).  lse: fp64 [B, T, Hq].  Returns 0, or -1 on a
 * bad argument.
 */
int oracle_swa_lse(const uint16_t *q_raw, const uint16_t *k, const float *alpha, const float *beta,
                   double *lse, int B, int T, int Hq, int Hkv, int d, int window, double scale)
{
    if (!shapes_ok(B, T, Hq, Hkv, d) || window < 1)
        return -1;
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * d;
    int bad = 0;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *s = (double *)malloc(sizeof(double) * (size_t)window);
        if (!q || !s) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t job = 0; job < (int64_t)B * T * Hq; ++job) {
                const int64_t bt = job / Hq, t = bt % T, b = bt / T;
                const int h = (int)(job % Hq);
                const int64_t lo = t - window + 1 > 0 ? t - window + 1 : 0;
                const uint16_t *kb = k + (b * T * Hkv + h / group) * d;
                scale_offset_row(q_raw + job * d, alpha + (int64_t)h * d, beta + (int64_t)h * d, d, q);
                double m = -INFINITY;
                for (int64_t j = lo; j <= t; ++j) {
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e)
                        acc += q[e] * bf16_to_double(kb[j * kv_row + e]);
                    s[j - lo] = acc * scale;
                    if (s[j - lo] > m)
                        m = s[j - lo];
                }
                double sum = 0.0;
                for (int64_t j = lo; j <= t; ++j)
                    sum += exp(s[j - lo] - m);
                lse[job] = m + log(sum);
            }
        }
        free(q);
        free(s);
    }
    return bad ? -2 : 0;
}

/*
 * Each copy row's log-sum-exp, Eq. (5): lse[b, i, h] = ln sum_{0 <= j <= pos[b, i]}
 * exp(scale * q'_i . k_j) with q'_i = qc_raw * alpha_c + beta_c, the normaliser of the
 * copy's softmax over the base keys up to its original position.  lse: fp64 [B, T_out, Hq].
 * Returns 0, or -1 on a bad argument (a position outside [0, T_kv)).
 */
int oracle_xattn_lse(const uint16_t *qc_raw, const int32_t *pos, const uint16_t *k, const float *alpha_c,
                     const float *beta_c, double *lse, int B, int T_out, int T_kv, int Hq, int Hkv, int d,
                     double scale)
{
    if (!shapes_ok(B, T_kv, Hq, Hkv, d) || T_out < 0)
        return -1;
    for (int64_t i = 0; i < (int64_t)B * T_out; ++i)
        if (pos[i] < 0 || pos[i] >= T_kv)
            return -1;
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * d;
    int bad = 0;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *s = (double *)malloc(sizeof(double) * (size_t)T_kv);
        if (!q || !s) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t job = 0; job < (int64_t)B * T_out * Hq; ++job) {
                const int64_t bi = job / Hq, b = bi / T_out;
                const int h = (int)(job % Hq);
                const uint16_t *kb = k + (b * T_kv * Hkv + h / group) * d;
                scale_offset_row(qc_raw + job * d, alpha_c + (int64_t)h * d, beta_c + (int64_t)h * d, d, q);
                double m = -INFINITY;
                for (int64_t j = 0; j <= pos[bi]; ++j) {
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e)
                        acc += q[e] * bf16_to_double(kb[j * kv_row + e]);
                    s[j] = acc * scale;
                    if (s[j] > m)
                        m = s[j];
                }
                double sum = 0.0;
                for (int64_t j = 0; j <= pos[bi]; ++j)
                    sum += exp(s[j] - m);
                lse[job] = m + log(sum);
            }
        }
        free(q);
        free(s);
    }
    return bad ? -2 : 0;
}
