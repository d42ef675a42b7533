// kernels.cuh -- launch parameters and host launchers of the Orthros kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/orthros.h"

namespace orthros {

struct SwaParams {
    const float *alpha;
    const float *beta;
    orthros_bf16 *o;       // output (the tensor-memory kernel stores rows directly)
    long long o_bstride;   // elements between batches of o
    int Hq;
    int32_t *dev_err;
    int T, Hkv, window;
    float qscale;          // softmax scale * log2(e), folded into the query
    int tiles_per_stream;  // tiles of the launched row range, set by the launcher
    int n_base;            // index of the range's first tile (rows n_base * TOK ..), set by the launcher
    int row_begin, row_end;  // output rows of each sequence to compute (row_begin a multiple of 128)
    long long total_tiles; // B * Hkv on input; B * Hkv * tiles_per_stream after launch set-up
    int reuse;             // 1: keep K/V blocks resident across consecutive tiles (set by launcher)
    float *lse;            // optional [B, T, Hq]: natural log of each row's sum of exp(scale q . k)
    int B;
};

struct XattnParams {
    const orthros_bf16 *qc;
    const int32_t *pos;
    const float *alpha_c;
    const float *beta_c;
    float *part_o;     // [n_part][B*Hkv][R][D]
    float2 *part_ml;   // [n_part][B*Hkv][R]  (max in log2 units, sum)
    orthros_bf16 *oc;
    float *lse;        // optional: each copy row's log-sum-exp, natural log, [B, T_out, Hq] (-inf: no key)
    int32_t *dev_err;
    long long qc_bstride, oc_bstride;
    int B, T_out, T_kv, Hq, Hkv, G, R, row_tiles, splits, chunk, n_part, direct;
    float qscale;
};

struct DecodeParams {
    const orthros_bf16 *q_new, *qc_new, *k_new, *v_new;
    orthros_bf16 *k_cache, *v_cache;
    int32_t *cache_len;
    const float *alpha, *beta, *alpha_c, *beta_c;
    orthros_bf16 *o, *oc;
    float *part_o;    // [B*Hkv][n_part][G][D]
    float2 *part_ml;  // [B*Hkv][n_part][G]
    int *cnt_bh;      // [B*Hkv]
    int *cnt_b;       // [B]
    int32_t *dev_err;
    int B, Hq, Hkv, L_max, window, nsplit, n_part;
    float qscale;
};

// gradient of the base stream (Eq. 4) or of the output copies (Eq. 5), each with its
// scale-offset.  Query rows are "units" (base tokens, or copies) x heads, dense
// [B, n_units, Hq, d]; K/V dense [B, T_kv, Hkv, d].  A unit's position is the token
// itself (pos == nullptr) or pos[b * n_units + u]; it sees keys pos-window+1 .. pos.
struct AttnBwdParams {
    const orthros_bf16 *q, *k, *v, *o, *dO;  // q raw, the forward output o, its gradient dO
    const float *alpha, *beta;
    const int32_t *pos;                      // copies' original positions, or nullptr (base)
    const float *lse_in;                     // optional [B*n_units*Hq] natural-log lse from the forward
    float *dq, *dk, *dv, *dalpha, *dbeta;    // dq = gradient of q raw; dalpha / dbeta zeroed first
    float *lse, *Drow;                       // workspace [B*n_units*Hq] each: log2-sum-exp, dO . o
    uint16_t *k16;                           // workspace: K as fp16 [B, T_kv, Hkv, d]
    uint16_t *q16;                           // workspace: q = x alpha + beta as fp16 [B, n_units, Hq, d]
    // workspace, written with k16: each key row's shift e (k16 holds k * 2^-e; e != 0 only for a
    // row whose largest |k| reaches 65520) as int8 [B*Hkv][nkb * 64], and per 64-key block
    // whether any row of it is shifted, uint8 [B*Hkv][nkb]
    int8_t *kexp;
    uint8_t *kflag;
    int nkb;                                 // 64-key blocks of T_kv
    int32_t *dev_err;
    int B, n_units, T_kv, Hq, Hkv, window;   // window = T_kv for the copies
    int accumulate;                          // add to dk, dv instead of overwriting them
    float scale;
    // few copy rows over a long key range: the tensor-memory dq kernel splits the keys of its
    // row tile over blockIdx.z (set by the launcher): mode 1 writes per-split (max, sum) of
    // each row, a combine kernel makes the log-sum-exp, mode 2 adds each split's dq
    int split_mode, splits;
    float2 *part_ml;                         // workspace [B*Hkv][splits][128]
};

// workspace: lse, D (fp32 per query row), then at 256-byte boundaries the fp16 copy of K, the
// key rows' shifts and the 64-key blocks' shift flags
size_t attn_bwd_workspace_bytes(int B, int n_units, int T_kv, int Hkv, int Hq, int D);
size_t attn_bwd_kexp_offset(int B, int n_units, int T_kv, int Hkv, int Hq, int D);
size_t attn_bwd_kflag_offset(int B, int n_units, int T_kv, int Hkv, int Hq, int D);
int attn_bwd_key_blocks(int T_kv);
size_t attn_bwd_k16_offset(int B, int n_units, int Hq);
// extra workspace of the copies' gradient: per-split row partials of the split dq path
constexpr int ATTN_BWD_MAX_SPLITS = 64;
size_t attn_bwd_split_bytes(int B, int Hkv);
// maps of the tensor-memory kernels: [0], [1] the fp16 q (p.q16) and dO with boxes of
// 64 x G heads x 64/G units, [2], [3] V and the fp16 copy of K (p.k16) with boxes of
// 64 x 1 x 128 keys (dK/dV); [4], [5] q raw and dO with boxes of 64 x G x 128/G, [6..8] K, V
// and the fp16 K with boxes of 64 x 1 x 64 (dQ); [9] the fp16 q with boxes of 64 x G x 128/G;
// [10], [11] the fp16 K and V with boxes of 64 x 1 x 32 (the base stream's band dQ)
constexpr int ATTN_BWD_MAPS = 13;
cudaError_t launch_attn_bwd(int D, int G, const AttnBwdParams &p, const CUtensorMap *maps, cudaStream_t stream);
// a layer's gradient, both streams: p the base stream, pc the copies (pc.k16 = p.k16; maps and
// mapsc as above for each stream, mapsc's fp16-K maps over p.k16); dK / dV written once
cudaError_t launch_attn_bwd_layer(int D, int G, const AttnBwdParams &p, const AttnBwdParams &pc,
                                  const CUtensorMap *maps, const CUtensorMap *mapsc, cudaStream_t stream);

cudaError_t launch_swa(int D, int G, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const CUtensorMap &o, SwaParams p, int num_sms, cudaStream_t stream);
bool swa_tc_supported(int D, int G, int window);
cudaError_t launch_swa_tc(int D, int G, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                          const CUtensorMap &o, const SwaParams &p, int num_sms, cudaStream_t stream);

size_t xattn_workspace_bytes(int B, int T_out, int T_kv, int Hq, int Hkv, int D);
// ctas > 0: at most 8 copy rows per (batch, KV head) run on exactly `ctas` CTAs of one SM each
cudaError_t launch_xattn(int D, const CUtensorMap &k, const CUtensorMap &v, XattnParams p, void *workspace,
                         cudaStream_t stream, int ctas = 0);
// merge split partials [n_part][B*Hkv][R][D] into the copy outputs
cudaError_t launch_xattn_combine(int D, const XattnParams &p, cudaStream_t stream);
// many copies per (batch, KV head) (T_out * G >= 256): tcgen05 flash kernel over key blocks of
// XATTN_TC_KEYS (the K/V tensor maps' box height)
constexpr int XATTN_TC_KEYS = 64;
bool xattn_tc_supported(int D, int G, int T_out);
cudaError_t launch_xattn_tc(int D, int G, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                            const XattnParams &p, cudaStream_t stream);

size_t decode_workspace_bytes(int B, int L_max, int Hq, int Hkv, int D);
cudaError_t launch_decode(int D, const CUtensorMap &k, const CUtensorMap &v, DecodeParams p, void *workspace,
                          cudaStream_t stream);

}  // namespace orthros
