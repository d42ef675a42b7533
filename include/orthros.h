/*
 * orthros.h -- C ABI of the Orthros per-layer attention operator on one GB300
 * (sm_103a).
 *
 * The operator (Orthros: Phase-Aware Heterogeneous Attention, arXiv 2610.13735;
 * close-reading notes Sec. 2.1-2.5 with Fig. 1, Eqs. (4)-(5), Algorithms 1-2):
 *
 *   base stream   q_t  = Q_raw[t]  * alpha  + beta        (scale-offset, Sec. 3.1)
 *                 o_t  = softmax_{j in W_t}(scale * q_t . k_j) v_j,
 *                 W_t  = {max(0, t-w+1) .. t}              (Eq. 4, 0-based)
 *   output copy   q'_i = Q'_raw[i] * alpha' + beta'
 *                 o'_i = softmax_{j <= pos_i}(scale * q'_i . k_j) v_j   (Eq. 5)
 *
 * K and V are produced by the base stream only; copies never write K/V
 * (dependency isolation, Sec. 2.4).  pos_i is the copy's ORIGINAL position,
 * whatever slot the copy occupies in memory (Algorithm 2 appends copies at the
 * tensor tail).  Query head h reads KV head h / (Hq / Hkv).
 *
 * Conventions shared by every entry point
 *  - bf16 tensors are passed as pointers to raw bf16 bits (orthros_bf16) in
 *    device memory, token-major [B, T, H, d] with d contiguous.  Each tensor
 *    takes a batch stride in ELEMENTS (0 = dense, i.e. T*H*d); within a batch
 *    the layout is dense.  A non-zero batch stride lets Q_raw and Q'_raw live in
 *    one [B, T+T_out, Hq, d] buffer (copies appended after the base tokens).
 *    Base addresses must be 16-byte aligned and batch strides multiples of 8.
 *  - alpha, beta, alpha', beta' are fp32 [Hq, d] device arrays (one 1 x d
 *    vector per query head).
 *  - scale multiplies the logit q . k (pass 1/sqrt(d) for the standard
 *    scaling); it is applied after the scale-offset.
 *  - Supported: d in {64, 128}; Hq % Hkv == 0 with Hq / Hkv <= 16; window >= 1.
 *  - stream is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream; the returned status reports host-side
 *    argument checks and launch errors only.
 *  - Ownership: the caller owns every buffer (inputs, outputs, KV cache,
 *    workspace).  The library keeps no per-call state and never allocates
 *    device memory at run time (the one fixed array behind
 *    orthros_xattn_fwd_noalloc is part of the loaded module).  Outputs must not
 *    alias inputs.
 *  - dev_err (optional, may be NULL) is an int32 in device memory.  A kernel
 *    that meets bad data it cannot reject on the host (a copy position outside
 *    [0, T_kv), a full KV cache) ORs an ORTHROS_DEVERR_* bit into it, writes
 *    zeros for the affected outputs and carries on; nothing traps.
 *  - No C++ exception crosses this boundary.
 */
#ifndef ORTHROS_H
#define ORTHROS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t orthros_bf16; /* raw bf16 bits */

typedef enum {
    ORTHROS_OK = 0,
    ORTHROS_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer or stride */
    ORTHROS_ERR_UNSUPPORTED = 2, /* d, head grouping or device not supported */
    ORTHROS_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the size query asks */
    ORTHROS_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed */
} orthros_status;

/* bits ORed into *dev_err by kernels */
#define ORTHROS_DEVERR_POSITION 1   /* a copy position outside [0, T_kv) */
#define ORTHROS_DEVERR_CACHE_FULL 2 /* decode: cache_len[b] + 1 > L_max */
#define ORTHROS_DEVERR_TIMEOUT 4    /* an internal pipeline wait gave up after ~2 s (a bug) */
#define ORTHROS_DEVERR_RANGE 8      /* an infinite key, a scaled query (or gradient dS) beyond fp16, or a logit beyond fp32 */

/* Human-readable name of a status code (static string, never NULL). */
const char *orthros_status_string(orthros_status s);

/* Library version as 10000*major + 100*minor + patch. */
int orthros_version(void);

/*
 * Base-stream causal sliding-window attention, Eq. (4), with the base
 * scale-offset fused into the query load (Sec. 3.1).
 *
 *   q_raw  [B, T, Hq, d]  bf16  (batch stride q_bstride elements, 0 = T*Hq*d)
 *   k, v   [B, T, Hkv, d] bf16  (batch stride kv_bstride, 0 = T*Hkv*d)
 *   alpha, beta [Hq, d] fp32
 *   o      [B, T, Hq, d]  bf16  output (batch stride o_bstride, 0 = T*Hq*d)
 *
 * Every row t of every sequence attends to keys max(0, t-window+1) .. t of its
 * own sequence.  window >= T gives plain causal attention.  Accumulation and
 * softmax are fp32.  q . k is taken with at least 11 significant bits of the
 * scaled query: in fp16 on the tensor-memory path (q rounded once to fp16, K
 * converted from bf16; a key row whose largest |k| reaches 65520 is converted as
 * k * 2^-e with its largest element in [2^14, 2^15) and its logits multiplied back
 * by 2^e in fp32, so every finite key is taken; an infinite key, a scaled |q| >=
 * 65504 or a logit beyond fp32 sets ORTHROS_DEVERR_RANGE), or as a bf16 high part
 * plus residual on the path used for windows too wide for tensor memory.  The
 * softmax weights enter P V as
 * bf16; o is rounded to bf16 (nearest even).
 */
orthros_status orthros_swa_fwd(const orthros_bf16 *q_raw, const orthros_bf16 *k,
                               const orthros_bf16 *v, const float *alpha, const float *beta,
                               orthros_bf16 *o, int B, int T, int Hq, int Hkv, int d,
                               int window, float scale, int64_t q_bstride, int64_t kv_bstride,
                               int64_t o_bstride, int32_t *dev_err, void *stream);

/*
 * orthros_swa_fwd for output rows row_begin .. row_end-1 of every sequence only
 * (chunked prefill; the paper has no counterpart): those rows of o get exactly
 * what orthros_swa_fwd writes there, and no other row of o is written.  Rows
 * read their keys from row max(0, t-window+1), so a chunk needs the K/V rows
 * max(0, row_begin-window+1) .. row_end-1 and the q_raw rows of the chunk in
 * place; the rest of the buffers is not read.  row_begin must be a multiple of
 * 128 and row_end a multiple of 128 or T; 0 <= row_begin <= row_end <= T
 * (row_begin == row_end is a no-op).  Other arguments as orthros_swa_fwd.
 */
orthros_status orthros_swa_fwd_rows(const orthros_bf16 *q_raw, const orthros_bf16 *k,
                                    const orthros_bf16 *v, const float *alpha, const float *beta,
                                    orthros_bf16 *o, int B, int T, int Hq, int Hkv, int d,
                                    int window, float scale, int64_t q_bstride,
                                    int64_t kv_bstride, int64_t o_bstride, int row_begin,
                                    int row_end, int32_t *dev_err, void *stream);

/*
 * orthros_swa_fwd that also writes, for training, each row's log-sum-exp:
 *   lse[b, t, h] = ln sum_{j in W_t} exp(scale * q_t . k_j)      (fp32 [B, T, Hq], dense)
 * the normaliser of the row's softmax, which orthros_swa_bwd can take instead of
 * recomputing it.  lse must be 16-byte aligned; other arguments as orthros_swa_fwd.
 */
orthros_status orthros_swa_fwd_lse(const orthros_bf16 *q_raw, const orthros_bf16 *k,
                                   const orthros_bf16 *v, const float *alpha, const float *beta,
                                   orthros_bf16 *o, float *lse, int B, int T, int Hq, int Hkv, int d,
                                   int window, float scale, int64_t q_bstride, int64_t kv_bstride,
                                   int64_t o_bstride, int32_t *dev_err, void *stream);

/*
 * Bytes of device workspace orthros_xattn_fwd needs for these sizes
 * (split-KV partial results).  Many copies per KV head (T_out * Hq/Hkv >= 256)
 * run on a kernel that keeps no partials, and few copies whose rows all fit one
 * partial need none: both get the 256-byte minimum.  Returns 0 for invalid
 * sizes.
 */
size_t orthros_xattn_workspace_size(int B, int T_out, int T_kv, int Hq, int Hkv, int d);

/*
 * Output-copy full causal cross-attention, Eq. (5), with the copy
 * scale-offset fused into the query load.
 *
 *   qc_raw [B, T_out, Hq, d] bf16 (batch stride qc_bstride, 0 = T_out*Hq*d)
 *   pos    [B, T_out] int32 device, the copies' ORIGINAL positions, any order,
 *          duplicates allowed, each in [0, T_kv)
 *   k, v   [B, T_kv, Hkv, d] bf16 base-stream K/V (batch stride kv_bstride)
 *   alpha_c, beta_c [Hq, d] fp32
 *   oc     [B, T_out, Hq, d] bf16 output (batch stride oc_bstride)
 *   workspace: device buffer of at least orthros_xattn_workspace_size(...)
 *          bytes, 256-byte aligned, contents need not be initialised.
 *
 * Split-KV: the key range of each KV head is cut into chunks streamed by
 * separate CTAs (query heads of one KV head share each K/V load); partial
 * (max, sum, unnormalised output) triples are merged by a log-sum-exp
 * combine kernel.  Two kernel launches.  A copy whose position is out of
 * range gets a zero output and sets ORTHROS_DEVERR_POSITION.  T_out == 0 is a
 * no-op.
 */
orthros_status orthros_xattn_fwd(const orthros_bf16 *qc_raw, const int32_t *pos,
                                 const orthros_bf16 *k, const orthros_bf16 *v,
                                 const float *alpha_c, const float *beta_c, orthros_bf16 *oc,
                                 int B, int T_out, int T_kv, int Hq, int Hkv, int d, float scale,
                                 int64_t qc_bstride, int64_t kv_bstride, int64_t oc_bstride,
                                 void *workspace, size_t ws_bytes, int32_t *dev_err,
                                 void *stream);

/*
 * orthros_xattn_fwd that also writes, for training, each copy row's log-sum-exp:
 *   lse[b, i, h] = ln sum_{0 <= j <= pos[b, i]} exp(scale * q'_i . k_j)
 * (fp32 [B, T_out, Hq], dense; -inf for a copy whose position is out of range),
 * the normaliser of the copy's softmax, which orthros_xattn_bwd can take instead
 * of recomputing it.  lse must be 16-byte aligned; other arguments as
 * orthros_xattn_fwd.
 */
orthros_status orthros_xattn_fwd_lse(const orthros_bf16 *qc_raw, const int32_t *pos,
                                     const orthros_bf16 *k, const orthros_bf16 *v,
                                     const float *alpha_c, const float *beta_c, orthros_bf16 *oc,
                                     float *lse, int B, int T_out, int T_kv, int Hq, int Hkv, int d,
                                     float scale, int64_t qc_bstride, int64_t kv_bstride,
                                     int64_t oc_bstride, void *workspace, size_t ws_bytes,
                                     int32_t *dev_err, void *stream);

/*
 * Bytes of device workspace orthros_prefill_fwd needs for these sizes (that of
 * the copies' cross-attention).  Returns 0 for invalid sizes.
 */
size_t orthros_prefill_workspace_size(int B, int T, int T_out, int Hq, int Hkv, int d);

/*
 * One prefill layer in one call (the paper has no counterpart; a convenience):
 * Eq. (4) for the base stream and Eq. (5) for T_out output copies over the base
 * K/V up to their original positions (Sec. 3.2, prefill mode), with the results
 * and error behaviour of orthros_swa_fwd and orthros_xattn_fwd with T_kv = T
 * (bit for bit).  For at most 8 copy rows per KV head (T_out * Hq / Hkv <= 8,
 * e.g. one copy per sequence) the copies' kernels run on a second stream of the
 * library's own, forked from and joined back into `stream` with events, while
 * the SWA kernel, which is bound by its MMA issue, holds fewer SMs: the copies'
 * pass, bound by HBM, runs on exactly the SMs left to it (one CTA per SM) and
 * uses the spare bandwidth (three kernel launches; the copies' kernel reads K/V
 * a second time).  Work queued on `stream` after the call runs after both.  For
 * more copies the two run one after the other on `stream`.  Capturable in a CUDA
 * graph.  A variant that attended the copies inside the SWA pass, reading K/V
 * once, measured no faster on GB300: the extra work in the SWA kernel cost as
 * much time as the second read saves.
 *
 *   q_raw, k, v, alpha, beta, o, window, q_bstride, kv_bstride, o_bstride:
 *          as orthros_swa_fwd
 *   qc_raw, pos, alpha_c, beta_c, oc, qc_bstride, oc_bstride: as
 *          orthros_xattn_fwd with T_kv = T (qc_raw may point into the q_raw
 *          buffer, after the base tokens)
 *   workspace: orthros_prefill_workspace_size(...) bytes, 256-byte aligned,
 *          contents need not be initialised (unused when T_out == 0).
 */
orthros_status orthros_prefill_fwd(const orthros_bf16 *q_raw, const orthros_bf16 *k,
                                   const orthros_bf16 *v, const float *alpha, const float *beta,
                                   orthros_bf16 *o, const orthros_bf16 *qc_raw,
                                   const int32_t *pos, const float *alpha_c, const float *beta_c,
                                   orthros_bf16 *oc, int B, int T, int T_out, int Hq, int Hkv,
                                   int d, int window, float scale, int64_t q_bstride,
                                   int64_t kv_bstride, int64_t o_bstride, int64_t qc_bstride,
                                   int64_t oc_bstride, void *workspace, size_t ws_bytes,
                                   int32_t *dev_err, void *stream);

/*
 * orthros_xattn_fwd without a workspace argument, for callers that cannot
 * allocate device memory (the paper has no counterpart; this is a deployment
 * convenience).  Such callers include plug-ins whose host runtime owns all
 * device memory and forbids allocation on the hot path, and latency-bound loops
 * that must never call cudaMalloc, which can block on the device and fail once
 * memory is fragmented or capped.
 *
 * Same arguments, layouts, results and status codes as orthros_xattn_fwd
 * (bits identical for the same inputs: the same kernels run).  The split-KV
 * partials live in a fixed file-scope device array of
 * ORTHROS_XATTN_NOALLOC_MAX_BYTES that every GPU loading this library holds
 * until the process exits; nothing is allocated per call.  Sizes for which
 * orthros_xattn_workspace_size(...) exceeds that maximum are rejected with
 * ORTHROS_ERR_WORKSPACE before anything runs.  All calls share the array, so
 * calls that overlap on the GPU race on it; order them (one stream, or events).
 * The array's device address is looked up on the first call made on each
 * device; make that first call before any stream capture begins.
 */
#define ORTHROS_XATTN_NOALLOC_MAX_BYTES (8u << 20)
orthros_status orthros_xattn_fwd_noalloc(const orthros_bf16 *qc_raw, const int32_t *pos,
                                         const orthros_bf16 *k, const orthros_bf16 *v,
                                         const float *alpha_c, const float *beta_c,
                                         orthros_bf16 *oc, int B, int T_out, int T_kv, int Hq,
                                         int Hkv, int d, float scale, int64_t qc_bstride,
                                         int64_t kv_bstride, int64_t oc_bstride, int32_t *dev_err,
                                         void *stream);

/*
 * Bytes of device workspace orthros_decode_step needs.  The workspace must be
 * zero-filled once before its first use (e.g. cudaMemset); every step leaves
 * its counters at zero again, so it can be reused step after step (but not by
 * two steps in flight at once).  Returns 0 for invalid sizes.
 */
size_t orthros_decode_workspace_size(int B, int L_max, int Hq, int Hkv, int d);

/*
 * One decode step (Sec. 3.2, decode mode: T_in = 0, T_out = 1 per step): a new
 * base token and its output copy at the same original position p = cache_len[b].
 * In one kernel launch, for every sequence b:
 *   1. k_new[b], v_new[b] are written to cache row p (KV-cache append);
 *   2. o[b]  = Eq. (4) for q_new[b]  over cache rows max(0, p-window+1) .. p;
 *   3. oc[b] = Eq. (5) for qc_new[b] over cache rows 0 .. p (the whole cache,
 *      including the new token);
 *   4. cache_len[b] = p + 1.
 * The copy never writes the cache.  Rows at or beyond the old cache_len are
 * never read from memory (the new row is taken from k_new / v_new).
 *
 *   q_new, qc_new [B, Hq, d] bf16; k_new, v_new [B, Hkv, d] bf16
 *   k_cache, v_cache [B, L_max, Hkv, d] bf16 (updated in place)
 *   cache_len [B] int32 device (updated in place); each must be < L_max
 *   o, oc [B, Hq, d] bf16 outputs
 *   workspace: orthros_decode_workspace_size(...) bytes, zeroed before first use.
 * A sequence whose cache is full gets zero outputs, no append, no increment,
 * and sets ORTHROS_DEVERR_CACHE_FULL.
 */
orthros_status orthros_decode_step(const orthros_bf16 *q_new, const orthros_bf16 *qc_new,
                                   const orthros_bf16 *k_new, const orthros_bf16 *v_new,
                                   orthros_bf16 *k_cache, orthros_bf16 *v_cache,
                                   int32_t *cache_len, int L_max, const float *alpha,
                                   const float *beta, const float *alpha_c, const float *beta_c,
                                   orthros_bf16 *o, orthros_bf16 *oc, int B, int Hq, int Hkv,
                                   int d, int window, float scale, void *workspace,
                                   size_t ws_bytes, int32_t *dev_err, void *stream);

/*
 * Bytes of device workspace orthros_swa_bwd needs: two fp32 values per query
 * row (the row's log-sum-exp and dO . o) and fp16 copies of K and of the
 * scale-offset q.  Returns 0 for invalid sizes.
 */
size_t orthros_swa_bwd_workspace_size(int B, int T, int Hq, int Hkv, int d);

/*
 * Gradient of the base stream (Eq. (4) with its scale-offset, Sec. 3.1), for
 * the training modes of Sec. 3.2.  Given the forward inputs, the forward
 * output o (as orthros_swa_fwd wrote it) and the output gradient dO, with
 * p_tj the softmax weight of key j for row t and q_t = Q_raw[t]*alpha+beta:
 *   dp_tj = dO_t . v_j,  D_t = dO_t . o_t,  ds_tj = p_tj (dp_tj - D_t)
 *   dq_t  = scale * sum_j ds_tj k_j         dq_raw_t = dq_t * alpha
 *   dk_j  = scale * sum_t ds_tj q_t         dv_j = sum_t p_tj dO_t
 *   dalpha = sum_t Q_raw[t] * dq_t          dbeta = sum_t dq_t   (per head, over B and T)
 * summed over every query head of a KV head for dk, dv.
 *
 *   q_raw, o, dO [B, T, Hq, d] bf16, dense; k, v [B, T, Hkv, d] bf16, dense
 *   alpha, beta [Hq, d] fp32
 *   lse: NULL, or the forward's per-row log-sum-exp (orthros_swa_fwd_lse), which
 *        saves the dq kernel its first pass over the keys
 *   dq_raw [B, T, Hq, d], dk, dv [B, T, Hkv, d], dalpha, dbeta [Hq, d]: fp32
 *   outputs, every element written (dalpha and dbeta are zeroed first)
 *   workspace: orthros_swa_bwd_workspace_size(...) bytes, 16-byte aligned.
 * Products take fp32 accumulation.  q . k on tensor memory is fp16: K converted
 * from bf16 into the workspace (key rows beyond fp16 shifted by a power of two, as
 * on the forward's tensor-memory path, with the row shifts kept in the workspace)
 * and q rounded once to fp16 (|q| >= 65504 sets ORTHROS_DEVERR_RANGE); the dq
 * kernel used without lse (warp MMAs) takes q as
 * a bf16 high part plus residual.  P is rounded to bf16 before it multiplies
 * dO; dS is rounded to bf16 before it multiplies K (dq) and to fp16 before it
 * multiplies the fp16 q (dk; |dS| >= 65504 sets ORTHROS_DEVERR_RANGE).  The
 * key-band dq (below) takes dS in fp16 against the fp16 K, times 2^e for a key
 * row shifted by 2^-e (|dS 2^e| >= 65504 sets ORTHROS_DEVERR_RANGE).
 * Launches: the fp16 copy of K; one pass over the query rows for the fp16 q,
 * D_t and a given lse in log2 units; dq (rows on the MMA's M side: with lse a
 * persistent tensor-memory kernel, which for Hq / Hkv in {4, 8} and windows
 * whose row tile sees at most five 32-key blocks takes each tile's key band
 * in one product and sums dalpha, dbeta itself, else a column sum follows;
 * without lse a two-pass warp-MMA kernel that stores each row's log-sum-exp),
 * then dk and dv (keys on the M side, tensor memory, no atomics).  dq, dk, dv have one writer per element;
 * dalpha, dbeta are summed with atomics.  dev_err (optional) as elsewhere.
 * Supported: d in {64, 128}; Hq / Hkv in {1, 2, 4, 8, 16}; any window >= 1.
 * Outputs must not alias inputs.
 */
orthros_status orthros_swa_bwd(const orthros_bf16 *q_raw, const orthros_bf16 *k,
                               const orthros_bf16 *v, const float *alpha, const float *beta,
                               const orthros_bf16 *o, const orthros_bf16 *dO, const float *lse,
                               float *dq_raw, float *dk, float *dv, float *dalpha, float *dbeta,
                               int B, int T,
                               int Hq, int Hkv, int d, int window, float scale, void *workspace,
                               size_t ws_bytes, int32_t *dev_err, void *stream);

/*
 * Bytes of device workspace orthros_xattn_bwd needs (two fp32 values per copy
 * row, fp16 copies of K and of the copies' scale-offset q, and per-split row
 * partials of the split dq path).  Returns 0 for invalid sizes.
 */
size_t orthros_xattn_bwd_workspace_size(int B, int T_out, int T_kv, int Hq, int Hkv, int d);

/*
 * Gradient of the output copies (Eq. (5) with the copies' scale-offset), the
 * second half of a training step's attention gradient.  With p_ij the weight of
 * base key j (0 <= j <= pos_i) for copy row i and q'_i = Q'_raw[i]*alpha'+beta':
 *   dp_ij = dOc_i . v_j,  D_i = dOc_i . oc_i,  ds_ij = p_ij (dp_ij - D_i)
 *   dq'_i = scale * sum_j ds_ij k_j         dqc_raw_i = dq'_i * alpha'
 *   dk_j  = scale * sum_i ds_ij q'_i        dv_j = sum_i p_ij dOc_i
 *   dalpha' = sum_i Q'_raw[i] * dq'_i       dbeta' = sum_i dq'_i
 * Copies own no K/V, so their gradient reaches the base K and V only: with
 * accumulate != 0 the copies' share is ADDED to dk and dv (e.g. after
 * orthros_swa_bwd filled them); with accumulate == 0 they are overwritten.
 *
 *   qc_raw, oc, dOc [B, T_out, Hq, d] bf16, dense; pos [B, T_out] int32
 *   k, v [B, T_kv, Hkv, d] bf16, dense; alpha_c, beta_c [Hq, d] fp32
 *   lse: NULL, or the forward's per-copy-row log-sum-exp (orthros_xattn_fwd_lse),
 *        which saves the dq kernel its first pass over the keys
 *   dqc_raw [B, T_out, Hq, d], dk, dv [B, T_kv, Hkv, d], dalpha_c, dbeta_c
 *   [Hq, d]: fp32 outputs (dalpha_c and dbeta_c are zeroed first)
 *   workspace: orthros_xattn_bwd_workspace_size(...) bytes, 16-byte aligned.
 * A copy whose position is outside [0, T_kv) gets a zero row of dqc_raw,
 * contributes nothing, and sets ORTHROS_DEVERR_POSITION in *dev_err.
 * Arithmetic and launches as orthros_swa_bwd, with the dq kernel on tensor
 * memory in two passes (the first finds each copy row's log-sum-exp; skipped
 * when lse is given); when one 128-row tile per (batch, KV head) holds every
 * copy, its key range is split over many CTAs (without lse: per-split maxima
 * and sums and a combine first; then per-split dq added up).  With lse and at
 * most 8 copy rows per KV head (T_out * Hq / Hkv <= 8) the dq runs on warp MMAs
 * instead, q . k with q as a bf16 high part plus residual against the bf16 K
 * (no fp16 K, no key shifts), dS rounded to bf16, the keys split over CTAs and
 * each split's dq, dalpha_c, dbeta_c added with atomics.
 * T_out == 0 leaves dk, dv as they are (accumulate) or zero.  Outputs must not
 * alias inputs.
 */
orthros_status orthros_xattn_bwd(const orthros_bf16 *qc_raw, const int32_t *pos,
                                 const orthros_bf16 *k, const orthros_bf16 *v,
                                 const float *alpha_c, const float *beta_c,
                                 const orthros_bf16 *oc, const orthros_bf16 *dOc, const float *lse,
                                 float *dqc_raw, float *dk, float *dv, float *dalpha_c,
                                 float *dbeta_c, int B, int T_out, int T_kv, int Hq, int Hkv,
                                 int d, float scale, int accumulate, void *workspace,
                                 size_t ws_bytes, int32_t *dev_err, void *stream);

/*
 * Bytes of device workspace orthros_attn_bwd needs: the regions of
 * orthros_swa_bwd and orthros_xattn_bwd, with one fp16 copy of K for both.
 * Returns 0 for invalid sizes.
 */
size_t orthros_attn_bwd_workspace_size(int B, int T, int T_out, int Hq, int Hkv, int d);

/*
 * A layer's whole attention gradient in one call: orthros_swa_bwd of the base
 * stream and orthros_xattn_bwd of the output copies (over the same K, V;
 * T_kv = T), with the same arguments, meanings and arithmetic, except that
 *   dk, dv  get the sum of both streams' shares, written once (not added to
 *           what the buffers held);
 *   lse, lsec  are each stream's forward log-sum-exp (orthros_swa_fwd_lse,
 *           orthros_xattn_fwd_lse) or NULL;
 *   one fp16 copy of K serves both streams, and one dk/dv launch takes, for
 *   each block of 128 keys, the base rows and then the copy rows that see it.
 * T_out == 0 is allowed (qc_raw, pos, oc, dOc, lsec and dqc_raw are then not
 * read; dalpha_c and dbeta_c are zeroed).  workspace:
 * orthros_attn_bwd_workspace_size(...) bytes, 16-byte aligned.  Outputs must
 * not alias inputs.
 */
orthros_status orthros_attn_bwd(const orthros_bf16 *q_raw, const orthros_bf16 *k,
                                const orthros_bf16 *v, const float *alpha, const float *beta,
                                const orthros_bf16 *o, const orthros_bf16 *dO, const float *lse,
                                const orthros_bf16 *qc_raw, const int32_t *pos,
                                const float *alpha_c, const float *beta_c, const orthros_bf16 *oc,
                                const orthros_bf16 *dOc, const float *lsec, float *dq_raw,
                                float *dk, float *dv, float *dalpha, float *dbeta, float *dqc_raw,
                                float *dalpha_c, float *dbeta_c, int B, int T, int T_out, int Hq,
                                int Hkv, int d, int window, float scale, void *workspace,
                                size_t ws_bytes, int32_t *dev_err, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ORTHROS_H */
