// orthros_api.cu -- the C ABI (include/orthros.h): host-side argument checks,
// TMA descriptor set-up and kernel dispatch.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "kernels.cuh"

namespace {

using orthros::DecodeParams;
using orthros::SwaParams;
using orthros::XattnParams;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 4-D bf16 view {d, H, T, B} of a token-major tensor, 128-byte swizzled boxes of
// {64, box_h, box_t, 1}.  Out-of-range boxes read zeros.
bool make_map(CUtensorMap *m, const void *base, int d, int H, long long T, int B, long long bstride_elems,
              int box_h, int box_t)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                             static_cast<cuuint64_t>(bstride_elems) * 2};
    cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_h), static_cast<cuuint32_t>(box_t), 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool heads_ok(int Hq, int Hkv)
{
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
        return false;
    const int G = Hq / Hkv;
    return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
}

// A batch stride: 0 selects the dense value; otherwise at least dense and a multiple of 8.
bool resolve_bstride(long long &s, long long dense)
{
    if (s == 0) {
        s = dense;
        return true;
    }
    return s >= dense && s % 8 == 0;
}

const float kLog2e = 1.4426950408889634f;

// tensor maps of the gradient's kernels: for dK/dV, the fp16 q and dO in rounds of 64 rows
// (64/G units x G heads), V and the fp16 K in blocks of 128 keys; for dQ, raw q and dO in
// tiles of 128 rows, K, V and the fp16 K in blocks of 64 keys, the fp16 q in tiles of 128
// rows (the base stream's persistent dQ), and the fp16 K and V in blocks of 32 keys (its band)
// 4-D fp32 view {d, H, T, B} of a dense token-major tensor, 128-byte swizzled boxes of
// {32, box_h, box_t, 1} (stores clip at the tensor's edges).
bool make_map_f32(CUtensorMap *m, const void *base, int d, int H, long long T, int B, int box_h, int box_t)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(H) * d * 4,
                             static_cast<cuuint64_t>(T) * H * d * 4};
    cuuint32_t box[4] = {32u, static_cast<cuuint32_t>(box_h), static_cast<cuuint32_t>(box_t), 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// m[12]: the fp32 dq_raw output of the stream (the band dq kernel stores it by TMA); a copy of
// m[9] when dq is null (never used then)
bool bwd_maps(CUtensorMap *m, const void *q, const void *dO, const void *k, const void *v, const void *k16,
              const void *q16, int d, int Hq, int Hkv, int n_units, int T_kv, int B, const void *dq)
{
    const int G = Hq / Hkv;
    const long long qs = static_cast<long long>(n_units) * Hq * d, ks = static_cast<long long>(T_kv) * Hkv * d;
    return make_map(&m[0], q16, d, Hq, n_units, B, qs, G, 64 / G) &&
           make_map(&m[1], dO, d, Hq, n_units, B, qs, G, 64 / G) &&
           make_map(&m[2], v, d, Hkv, T_kv, B, ks, 1, 128) && make_map(&m[3], k16, d, Hkv, T_kv, B, ks, 1, 128) &&
           make_map(&m[4], q, d, Hq, n_units, B, qs, G, 128 / G) &&
           make_map(&m[5], dO, d, Hq, n_units, B, qs, G, 128 / G) && make_map(&m[6], k, d, Hkv, T_kv, B, ks, 1, 64) &&
           make_map(&m[7], v, d, Hkv, T_kv, B, ks, 1, 64) && make_map(&m[8], k16, d, Hkv, T_kv, B, ks, 1, 64) &&
           make_map(&m[9], q16, d, Hq, n_units, B, qs, G, 128 / G) &&
           make_map(&m[10], k16, d, Hkv, T_kv, B, ks, 1, 32) && make_map(&m[11], v, d, Hkv, T_kv, B, ks, 1, 32) &&
           (dq != nullptr && n_units > 0 ? make_map_f32(&m[12], dq, d, Hq, n_units, B, G, 128 / G)
                                         : (m[12] = m[9], true));
}

}  // namespace

extern "C" {

const char *orthros_status_string(orthros_status s)
{
    switch (s) {
    case ORTHROS_OK:
        return "ok";
    case ORTHROS_ERR_INVALID_ARG:
        return "invalid argument";
    case ORTHROS_ERR_UNSUPPORTED:
        return "unsupported configuration";
    case ORTHROS_ERR_WORKSPACE:
        return "workspace missing or too small";
    case ORTHROS_ERR_CUDA:
        return "CUDA error";
    }
    return "unknown status";
}

int orthros_version(void) { return 100; }

}  // extern "C"

namespace {

// Checks the arguments of a base-stream call and fills its tensor maps and parameters.  Returns
// ORTHROS_OK with *empty set when there is no row to compute.
orthros_status swa_setup(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                         const float *alpha, const float *beta, orthros_bf16 *o, float *lse, int B, int T, int Hq,
                         int Hkv, int d, int window, float scale, int64_t q_bstride, int64_t kv_bstride,
                         int64_t o_bstride, int row_begin, int row_end, int32_t *dev_err, CUtensorMap *maps,
                         SwaParams &p, bool *empty)
{
    *empty = false;
    if (!aligned16(q_raw) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) || !aligned16(beta) ||
        !aligned16(o) || B < 1 || T < 1 || window < 1 || !std::isfinite(scale))
        return ORTHROS_ERR_INVALID_ARG;
    if (row_begin < 0 || row_end > T || row_begin > row_end || row_begin % 128 != 0 ||
        (row_end % 128 != 0 && row_end != T))
        return ORTHROS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return ORTHROS_ERR_UNSUPPORTED;
    if (row_begin == row_end) {
        *empty = true;
        return ORTHROS_OK;
    }
    long long qs = q_bstride, ks = kv_bstride, os = o_bstride;
    if (!resolve_bstride(qs, static_cast<long long>(T) * Hq * d) ||
        !resolve_bstride(ks, static_cast<long long>(T) * Hkv * d) ||
        !resolve_bstride(os, static_cast<long long>(T) * Hq * d))
        return ORTHROS_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    const int TOK = 128 / G;
    if (!make_map(&maps[0], q_raw, d, Hq, T, B, qs, G, TOK) || !make_map(&maps[1], k, d, Hkv, T, B, ks, 1, 32) ||
        !make_map(&maps[2], v, d, Hkv, T, B, ks, 1, 32) || !make_map(&maps[3], o, d, Hq, T, B, os, G, TOK))
        return ORTHROS_ERR_CUDA;
    p = SwaParams{};
    p.alpha = alpha;
    p.beta = beta;
    p.o = o;
    p.o_bstride = os;
    p.Hq = Hq;
    p.dev_err = dev_err;
    p.T = T;
    p.Hkv = Hkv;
    p.window = window;
    p.qscale = scale * kLog2e;
    p.total_tiles = static_cast<long long>(B) * Hkv;
    p.row_begin = row_begin;
    p.row_end = row_end;
    p.lse = lse;
    p.B = B;
    return ORTHROS_OK;
}

orthros_status swa_fwd_impl(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                            const float *alpha, const float *beta, orthros_bf16 *o, float *lse, int B, int T, int Hq,
                            int Hkv, int d, int window, float scale, int64_t q_bstride, int64_t kv_bstride,
                            int64_t o_bstride, int row_begin, int row_end, int32_t *dev_err, void *stream,
                            int sm_reserve = 0)
{
    CUtensorMap maps[4];
    SwaParams p;
    bool empty = false;
    const orthros_status st = swa_setup(q_raw, k, v, alpha, beta, o, lse, B, T, Hq, Hkv, d, window, scale, q_bstride,
                                        kv_bstride, o_bstride, row_begin, row_end, dev_err, maps, p, &empty);
    if (st != ORTHROS_OK || empty)
        return st;
    const int sms = num_sms() - sm_reserve;  // the persistent kernel's CTAs
    if (sms <= 0)
        return ORTHROS_ERR_CUDA;
    const cudaError_t e =
        orthros::launch_swa(d, Hq / Hkv, maps[0], maps[1], maps[2], maps[3], p, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ORTHROS_OK : ORTHROS_ERR_CUDA;
}

}  // namespace

extern "C" {

orthros_status orthros_swa_fwd_rows(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                                    const float *alpha, const float *beta, orthros_bf16 *o, int B, int T, int Hq,
                                    int Hkv, int d, int window, float scale, int64_t q_bstride, int64_t kv_bstride,
                                    int64_t o_bstride, int row_begin, int row_end, int32_t *dev_err, void *stream)
{
    return swa_fwd_impl(q_raw, k, v, alpha, beta, o, nullptr, B, T, Hq, Hkv, d, window, scale, q_bstride, kv_bstride,
                        o_bstride, row_begin, row_end, dev_err, stream);
}

orthros_status orthros_swa_fwd_lse(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                                   const float *alpha, const float *beta, orthros_bf16 *o, float *lse, int B, int T,
                                   int Hq, int Hkv, int d, int window, float scale, int64_t q_bstride,
                                   int64_t kv_bstride, int64_t o_bstride, int32_t *dev_err, void *stream)
{
    if (!aligned16(lse))
        return ORTHROS_ERR_INVALID_ARG;
    return swa_fwd_impl(q_raw, k, v, alpha, beta, o, lse, B, T, Hq, Hkv, d, window, scale, q_bstride, kv_bstride,
                        o_bstride, 0, T, dev_err, stream);
}

orthros_status orthros_swa_fwd(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                               const float *alpha, const float *beta, orthros_bf16 *o, int B, int T, int Hq,
                               int Hkv, int d, int window, float scale, int64_t q_bstride, int64_t kv_bstride,
                               int64_t o_bstride, int32_t *dev_err, void *stream)
{
    return orthros_swa_fwd_rows(q_raw, k, v, alpha, beta, o, B, T, Hq, Hkv, d, window, scale, q_bstride, kv_bstride,
                                o_bstride, 0, T < 1 ? 0 : T, dev_err, stream);
}

size_t orthros_xattn_workspace_size(int B, int T_out, int T_kv, int Hq, int Hkv, int d)
{
    if (B < 1 || T_out < 0 || T_kv < 1 || (d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return 0;
    if (T_out == 0)
        return 256;
    return orthros::xattn_workspace_bytes(B, T_out, T_kv, Hq, Hkv, d);
}

}  // extern "C"

namespace {

orthros_status xattn_fwd_impl(const orthros_bf16 *qc_raw, const int32_t *pos, const orthros_bf16 *k,
                              const orthros_bf16 *v, const float *alpha_c, const float *beta_c, orthros_bf16 *oc,
                              float *lse, int B, int T_out, int T_kv, int Hq, int Hkv, int d, float scale,
                              int64_t qc_bstride, int64_t kv_bstride, int64_t oc_bstride, void *workspace,
                              size_t ws_bytes, int32_t *dev_err, void *stream, int ctas = 0)
{
    if (B < 1 || T_out < 0 || T_kv < 1 || !std::isfinite(scale))
        return ORTHROS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return ORTHROS_ERR_UNSUPPORTED;
    if (T_out == 0)
        return ORTHROS_OK;
    if (!aligned16(qc_raw) || !pos || !aligned16(k) || !aligned16(v) || !aligned16(alpha_c) ||
        !aligned16(beta_c) || !aligned16(oc))
        return ORTHROS_ERR_INVALID_ARG;
    long long qs = qc_bstride, ks = kv_bstride, os = oc_bstride;
    if (!resolve_bstride(qs, static_cast<long long>(T_out) * Hq * d) ||
        !resolve_bstride(ks, static_cast<long long>(T_kv) * Hkv * d) ||
        !resolve_bstride(os, static_cast<long long>(T_out) * Hq * d))
        return ORTHROS_ERR_INVALID_ARG;
    const size_t need = orthros::xattn_workspace_bytes(B, T_out, T_kv, Hq, Hkv, d);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ORTHROS_ERR_WORKSPACE;
    XattnParams p{};
    p.qc = qc_raw;
    p.pos = pos;
    p.alpha_c = alpha_c;
    p.beta_c = beta_c;
    p.oc = oc;
    p.lse = lse;
    p.dev_err = dev_err;
    p.qc_bstride = qs;
    p.oc_bstride = os;
    p.B = B;
    p.T_out = T_out;
    p.T_kv = T_kv;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.qscale = scale * kLog2e;
    const int G = Hq / Hkv;
    CUtensorMap mq, mk, mv;
    cudaError_t e;
    if (orthros::xattn_tc_supported(d, G, T_out)) {
        // many copies: tensor-memory flash kernel, 128-row query tiles, K/V blocks of XATTN_TC_KEYS
        p.G = G;
        p.R = T_out * G;
        constexpr int KB = orthros::XATTN_TC_KEYS;
        if (!make_map(&mq, qc_raw, d, Hq, T_out, B, qs, G, 128 / G) || !make_map(&mk, k, d, Hkv, T_kv, B, ks, 1, KB) ||
            !make_map(&mv, v, d, Hkv, T_kv, B, ks, 1, KB))
            return ORTHROS_ERR_CUDA;
        e = orthros::launch_xattn_tc(d, G, mq, mk, mv, p, static_cast<cudaStream_t>(stream));
    } else {
        if (!make_map(&mk, k, d, Hkv, T_kv, B, ks, 1, 64) || !make_map(&mv, v, d, Hkv, T_kv, B, ks, 1, 64))
            return ORTHROS_ERR_CUDA;
        e = orthros::launch_xattn(d, mk, mv, p, workspace, static_cast<cudaStream_t>(stream), ctas);
    }
    return e == cudaSuccess ? ORTHROS_OK : ORTHROS_ERR_CUDA;
}

}  // namespace

extern "C" {

orthros_status orthros_xattn_fwd(const orthros_bf16 *qc_raw, const int32_t *pos, const orthros_bf16 *k,
                                 const orthros_bf16 *v, const float *alpha_c, const float *beta_c,
                                 orthros_bf16 *oc, int B, int T_out, int T_kv, int Hq, int Hkv, int d, float scale,
                                 int64_t qc_bstride, int64_t kv_bstride, int64_t oc_bstride, void *workspace,
                                 size_t ws_bytes, int32_t *dev_err, void *stream)
{
    return xattn_fwd_impl(qc_raw, pos, k, v, alpha_c, beta_c, oc, nullptr, B, T_out, T_kv, Hq, Hkv, d, scale,
                          qc_bstride, kv_bstride, oc_bstride, workspace, ws_bytes, dev_err, stream);
}

orthros_status orthros_xattn_fwd_lse(const orthros_bf16 *qc_raw, const int32_t *pos, const orthros_bf16 *k,
                                     const orthros_bf16 *v, const float *alpha_c, const float *beta_c,
                                     orthros_bf16 *oc, float *lse, int B, int T_out, int T_kv, int Hq, int Hkv, int d,
                                     float scale, int64_t qc_bstride, int64_t kv_bstride, int64_t oc_bstride,
                                     void *workspace, size_t ws_bytes, int32_t *dev_err, void *stream)
{
    if (T_out > 0 && !aligned16(lse))
        return ORTHROS_ERR_INVALID_ARG;
    return xattn_fwd_impl(qc_raw, pos, k, v, alpha_c, beta_c, oc, lse, B, T_out, T_kv, Hq, Hkv, d, scale, qc_bstride,
                          kv_bstride, oc_bstride, workspace, ws_bytes, dev_err, stream);
}

size_t orthros_prefill_workspace_size(int B, int T, int T_out, int Hq, int Hkv, int d)
{
    if (B < 1 || T < 1 || T_out < 0 || (d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return 0;
    return T_out == 0 ? 256 : orthros::xattn_workspace_bytes(B, T_out, T, Hq, Hkv, d);
}

}  // extern "C"

namespace {

// The stream on which orthros_prefill_fwd runs the copies' pass beside the SWA kernel: one per
// device, created on first use and kept for the life of the process.
cudaStream_t copy_stream()
{
    static std::mutex mu;
    static cudaStream_t streams[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (streams[dev] == nullptr && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
        streams[dev] = nullptr;
    return streams[dev];
}

// SMs that the persistent SWA kernel leaves to the copies' split-KV pass so that the two, run at
// once, end together: SMs shared in proportion to each pass's bytes over its per-SM rate.  On a
// GB300 the SWA kernel (bound by its MMA issue) moves about 37 GB/s per SM and the split-KV pass
// about twice that once the SWA kernel holds the other SMs.
int copy_sm_reserve(int sms, int B, int T, int Hq, int Hkv, int d)
{
    const double swa_bytes = 2.0 * B * T * (2.0 * Hq + 2.0 * Hkv) * d;  // q, o, K, V
    const double copy_bytes = 2.0 * B * T * 2.0 * Hkv * d;              // K, V up to the last position
    const double c = (copy_bytes / 2.0) / swa_bytes;
    const int x = static_cast<int>(std::lround(sms * c / (1.0 + c)));
    return x < 2 ? 0 : (x > sms / 4 ? sms / 4 : x);
}

}  // namespace

extern "C" {

orthros_status orthros_prefill_fwd(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                                   const float *alpha, const float *beta, orthros_bf16 *o, const orthros_bf16 *qc_raw,
                                   const int32_t *pos, const float *alpha_c, const float *beta_c, orthros_bf16 *oc,
                                   int B, int T, int T_out, int Hq, int Hkv, int d, int window, float scale,
                                   int64_t q_bstride, int64_t kv_bstride, int64_t o_bstride, int64_t qc_bstride,
                                   int64_t oc_bstride, void *workspace, size_t ws_bytes, int32_t *dev_err,
                                   void *stream)
{
    if (T_out < 0)
        return ORTHROS_ERR_INVALID_ARG;
    if (T_out > 0 && (!workspace || ws_bytes < orthros_prefill_workspace_size(B, T, T_out, Hq, Hkv, d)))
        return ORTHROS_ERR_WORKSPACE;
    // At most 8 copy rows per KV head (the split-KV pass with the rows on the MMA's N side, bound
    // by HBM) run on a second stream while the SWA kernel, bound by its MMA issue and holding
    // fewer SMs, runs on the caller's; the caller's stream waits for both.  The copies' kernel
    // then has exactly as many CTAs as SMs left to it, each too large to share an SM, so it
    // cannot take SWA's SMs whichever grid is dispatched first.  Otherwise the two run one
    // after the other on the caller's stream.
    const int sms = num_sms();
    const bool overlap = T_out > 0 && (d == 64 || d == 128) && heads_ok(Hq, Hkv) &&
                         static_cast<long long>(T_out) * (Hq / Hkv) <= 8 && sms > 0;
    const int reserve = overlap ? copy_sm_reserve(sms, B, T, Hq, Hkv, d) : 0;
    cudaStream_t cs = reserve > 0 ? copy_stream() : nullptr;
    if (cs == nullptr) {
        const orthros_status st = orthros_swa_fwd(q_raw, k, v, alpha, beta, o, B, T, Hq, Hkv, d, window, scale,
                                                  q_bstride, kv_bstride, o_bstride, dev_err, stream);
        if (st != ORTHROS_OK || T_out == 0)
            return st;
        return orthros_xattn_fwd(qc_raw, pos, k, v, alpha_c, beta_c, oc, B, T_out, T, Hq, Hkv, d, scale, qc_bstride,
                                 kv_bstride, oc_bstride, workspace, ws_bytes, dev_err, stream);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t fork = nullptr, join = nullptr;
    if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
        if (fork)
            cudaEventDestroy(fork);
        return ORTHROS_ERR_CUDA;
    }
    orthros_status st = ORTHROS_ERR_CUDA;
    if (cudaEventRecord(fork, s) == cudaSuccess && cudaStreamWaitEvent(cs, fork, 0) == cudaSuccess) {
        // the SWA kernel is launched first so that its persistent CTAs take their SMs first
        st = swa_fwd_impl(q_raw, k, v, alpha, beta, o, nullptr, B, T, Hq, Hkv, d, window, scale, q_bstride,
                          kv_bstride, o_bstride, 0, T < 1 ? 0 : T, dev_err, stream, reserve);
        if (st == ORTHROS_OK)
            st = xattn_fwd_impl(qc_raw, pos, k, v, alpha_c, beta_c, oc, nullptr, B, T_out, T, Hq, Hkv, d, scale,
                                qc_bstride, kv_bstride, oc_bstride, workspace, ws_bytes, dev_err, cs, reserve);
        // the caller's stream waits for whatever the copy stream was given
        if ((cudaEventRecord(join, cs) != cudaSuccess || cudaStreamWaitEvent(s, join, 0) != cudaSuccess) &&
            st == ORTHROS_OK)
            st = ORTHROS_ERR_CUDA;
    }
    cudaEventDestroy(fork);
    cudaEventDestroy(join);
    return st;
}

size_t orthros_decode_workspace_size(int B, int L_max, int Hq, int Hkv, int d)
{
    if (B < 1 || L_max < 1 || (d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return 0;
    return orthros::decode_workspace_bytes(B, L_max, Hq, Hkv, d);
}

orthros_status orthros_decode_step(const orthros_bf16 *q_new, const orthros_bf16 *qc_new,
                                   const orthros_bf16 *k_new, const orthros_bf16 *v_new, orthros_bf16 *k_cache,
                                   orthros_bf16 *v_cache, int32_t *cache_len, int L_max, const float *alpha,
                                   const float *beta, const float *alpha_c, const float *beta_c, orthros_bf16 *o,
                                   orthros_bf16 *oc, int B, int Hq, int Hkv, int d, int window, float scale,
                                   void *workspace, size_t ws_bytes, int32_t *dev_err, void *stream)
{
    if (!aligned16(q_new) || !aligned16(qc_new) || !aligned16(k_new) || !aligned16(v_new) ||
        !aligned16(k_cache) || !aligned16(v_cache) || !cache_len || !aligned16(alpha) || !aligned16(beta) ||
        !aligned16(alpha_c) || !aligned16(beta_c) || !aligned16(o) || !aligned16(oc) || B < 1 || L_max < 1 ||
        window < 1 || !std::isfinite(scale))
        return ORTHROS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return ORTHROS_ERR_UNSUPPORTED;
    const size_t need = orthros::decode_workspace_bytes(B, L_max, Hq, Hkv, d);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ORTHROS_ERR_WORKSPACE;
    CUtensorMap mk, mv;
    const long long cs = static_cast<long long>(L_max) * Hkv * d;
    if (!make_map(&mk, k_cache, d, Hkv, L_max, B, cs, 1, 64) || !make_map(&mv, v_cache, d, Hkv, L_max, B, cs, 1, 64))
        return ORTHROS_ERR_CUDA;
    DecodeParams p{};
    p.q_new = q_new;
    p.qc_new = qc_new;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.cache_len = cache_len;
    p.alpha = alpha;
    p.beta = beta;
    p.alpha_c = alpha_c;
    p.beta_c = beta_c;
    p.o = o;
    p.oc = oc;
    p.dev_err = dev_err;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.L_max = L_max;
    p.window = window;
    p.qscale = scale * kLog2e;
    const cudaError_t e = orthros::launch_decode(d, mk, mv, p, workspace, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ORTHROS_OK : ORTHROS_ERR_CUDA;
}

size_t orthros_swa_bwd_workspace_size(int B, int T, int Hq, int Hkv, int d)
{
    if (B < 1 || T < 1 || (d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return 0;
    // + the fp16 q of the persistent dq kernel (used when the forward's lse is given)
    return orthros::attn_bwd_workspace_bytes(B, T, T, Hkv, Hq, d) + 2 * static_cast<size_t>(B) * T * Hq * d;
}

orthros_status orthros_swa_bwd(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                               const float *alpha, const float *beta, const orthros_bf16 *o, const orthros_bf16 *dO,
                               const float *lse, float *dq_raw, float *dk, float *dv, float *dalpha, float *dbeta,
                               int B, int T, int Hq, int Hkv, int d, int window, float scale, void *workspace,
                               size_t ws_bytes, int32_t *dev_err, void *stream)
{
    if (!aligned16(q_raw) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) || !aligned16(beta) ||
        !aligned16(o) || !aligned16(dO) || !aligned16(dq_raw) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(dalpha) || !aligned16(dbeta) || B < 1 || T < 1 || window < 1 || !std::isfinite(scale))
        return ORTHROS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return ORTHROS_ERR_UNSUPPORTED;
    const size_t need = orthros_swa_bwd_workspace_size(B, T, Hq, Hkv, d);
    if (!aligned16(workspace) || ws_bytes < need)
        return ORTHROS_ERR_WORKSPACE;
    orthros::AttnBwdParams p{};
    p.q = q_raw;
    p.k = k;
    p.v = v;
    p.o = o;
    p.dO = dO;
    p.alpha = alpha;
    p.beta = beta;
    p.pos = nullptr;
    p.lse_in = lse;
    p.dq = dq_raw;
    p.dk = dk;
    p.dv = dv;
    p.dalpha = dalpha;
    p.dbeta = dbeta;
    p.lse = static_cast<float *>(workspace);
    p.Drow = p.lse + static_cast<size_t>(B) * T * Hq;
    p.k16 = reinterpret_cast<uint16_t *>(static_cast<char *>(workspace) + orthros::attn_bwd_k16_offset(B, T, Hq));
    p.kexp = reinterpret_cast<int8_t *>(static_cast<char *>(workspace) + orthros::attn_bwd_kexp_offset(B, T, T, Hkv, Hq, d));
    p.kflag = reinterpret_cast<uint8_t *>(static_cast<char *>(workspace) +
                                          orthros::attn_bwd_kflag_offset(B, T, T, Hkv, Hq, d));
    p.nkb = orthros::attn_bwd_key_blocks(T);
    p.q16 = reinterpret_cast<uint16_t *>(static_cast<char *>(workspace) +
                                         orthros::attn_bwd_workspace_bytes(B, T, T, Hkv, Hq, d));
    p.dev_err = dev_err;
    p.B = B;
    p.n_units = T;
    p.T_kv = T;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = window;
    p.accumulate = 0;
    p.scale = scale;
    CUtensorMap maps[orthros::ATTN_BWD_MAPS];
    if (!bwd_maps(maps, q_raw, dO, k, v, p.k16, p.q16, d, Hq, Hkv, T, T, B, dq_raw))
        return ORTHROS_ERR_CUDA;
    const cudaError_t e = orthros::launch_attn_bwd(d, Hq / Hkv, p, maps, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ORTHROS_OK : ORTHROS_ERR_CUDA;
}

size_t orthros_xattn_bwd_workspace_size(int B, int T_out, int T_kv, int Hq, int Hkv, int d)
{
    if (B < 1 || T_out < 0 || T_kv < 1 || (d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return 0;
    return orthros::attn_bwd_workspace_bytes(B, T_out, T_kv, Hkv, Hq, d) + orthros::attn_bwd_split_bytes(B, Hkv) +
           2 * static_cast<size_t>(B) * T_out * Hq * d;  // the copies' fp16 q
}

orthros_status orthros_xattn_bwd(const orthros_bf16 *qc_raw, const int32_t *pos, const orthros_bf16 *k,
                                 const orthros_bf16 *v, const float *alpha_c, const float *beta_c,
                                 const orthros_bf16 *oc, const orthros_bf16 *dOc, const float *lse, float *dqc_raw,
                                 float *dk, float *dv,
                                 float *dalpha_c, float *dbeta_c, int B, int T_out, int T_kv, int Hq, int Hkv, int d,
                                 float scale, int accumulate, void *workspace, size_t ws_bytes, int32_t *dev_err,
                                 void *stream)
{
    if ((T_out > 0 && (!aligned16(qc_raw) || !pos || !aligned16(oc) || !aligned16(dOc) || !aligned16(dqc_raw) ||
                       (lse != nullptr && !aligned16(lse)))) ||
        !aligned16(k) || !aligned16(v) || !aligned16(alpha_c) || !aligned16(beta_c) || !aligned16(dk) ||
        !aligned16(dv) || !aligned16(dalpha_c) || !aligned16(dbeta_c) || B < 1 || T_out < 0 || T_kv < 1 ||
        !std::isfinite(scale))
        return ORTHROS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return ORTHROS_ERR_UNSUPPORTED;
    const size_t need = orthros_xattn_bwd_workspace_size(B, T_out, T_kv, Hq, Hkv, d);
    if (!aligned16(workspace) || ws_bytes < need)
        return ORTHROS_ERR_WORKSPACE;
    orthros::AttnBwdParams p{};
    p.q = qc_raw;
    p.k = k;
    p.v = v;
    p.o = oc;
    p.dO = dOc;
    p.alpha = alpha_c;
    p.beta = beta_c;
    p.pos = pos ? pos : reinterpret_cast<const int32_t *>(workspace);  // T_out == 0: never read
    p.lse_in = T_out > 0 ? lse : nullptr;
    p.dq = dqc_raw;
    p.dk = dk;
    p.dv = dv;
    p.dalpha = dalpha_c;
    p.dbeta = dbeta_c;
    p.lse = static_cast<float *>(workspace);
    p.Drow = p.lse + static_cast<size_t>(B) * T_out * Hq;
    p.k16 = reinterpret_cast<uint16_t *>(static_cast<char *>(workspace) + orthros::attn_bwd_k16_offset(B, T_out, Hq));
    p.kexp = reinterpret_cast<int8_t *>(static_cast<char *>(workspace) +
                                        orthros::attn_bwd_kexp_offset(B, T_out, T_kv, Hkv, Hq, d));
    p.kflag = reinterpret_cast<uint8_t *>(static_cast<char *>(workspace) +
                                          orthros::attn_bwd_kflag_offset(B, T_out, T_kv, Hkv, Hq, d));
    p.nkb = orthros::attn_bwd_key_blocks(T_kv);
    p.part_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                           orthros::attn_bwd_workspace_bytes(B, T_out, T_kv, Hkv, Hq, d));
    p.q16 = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(p.part_ml) + orthros::attn_bwd_split_bytes(B, Hkv));
    p.dev_err = dev_err;
    p.B = B;
    p.n_units = T_out;
    p.T_kv = T_kv;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = T_kv;
    p.accumulate = accumulate ? 1 : 0;
    p.scale = scale;
    CUtensorMap maps[orthros::ATTN_BWD_MAPS];
    if (!bwd_maps(maps, T_out > 0 ? qc_raw : k, T_out > 0 ? dOc : k, k, v, p.k16, T_out > 0 ? p.q16 : p.k16, d, Hq, Hkv,
                  T_out > 0 ? T_out : 1, T_kv, B, nullptr))
        return ORTHROS_ERR_CUDA;
    const cudaError_t e = orthros::launch_attn_bwd(d, Hq / Hkv, p, maps, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ORTHROS_OK : ORTHROS_ERR_CUDA;
}

size_t orthros_attn_bwd_workspace_size(int B, int T, int T_out, int Hq, int Hkv, int d)
{
    if (B < 1 || T < 1 || T_out < 0 || (d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return 0;
    // the base stream's region (rows, fp16 K, fp16 q), then the copies' (rows, split partials, fp16 q)
    const size_t base = (orthros_swa_bwd_workspace_size(B, T, Hq, Hkv, d) + 255) & ~static_cast<size_t>(255);
    return base + orthros::attn_bwd_k16_offset(B, T_out, Hq) + orthros::attn_bwd_split_bytes(B, Hkv) +
           2 * static_cast<size_t>(B) * T_out * Hq * d;
}

orthros_status orthros_attn_bwd(const orthros_bf16 *q_raw, const orthros_bf16 *k, const orthros_bf16 *v,
                                const float *alpha, const float *beta, const orthros_bf16 *o, const orthros_bf16 *dO,
                                const float *lse, const orthros_bf16 *qc_raw, const int32_t *pos,
                                const float *alpha_c, const float *beta_c, const orthros_bf16 *oc,
                                const orthros_bf16 *dOc, const float *lsec, float *dq_raw, float *dk, float *dv,
                                float *dalpha, float *dbeta, float *dqc_raw, float *dalpha_c, float *dbeta_c, int B,
                                int T, int T_out, int Hq, int Hkv, int d, int window, float scale, void *workspace,
                                size_t ws_bytes, int32_t *dev_err, void *stream)
{
    if (!aligned16(q_raw) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) || !aligned16(beta) ||
        !aligned16(o) || !aligned16(dO) || !aligned16(dq_raw) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(dalpha) || !aligned16(dbeta) || (lse != nullptr && !aligned16(lse)) || !aligned16(alpha_c) ||
        !aligned16(beta_c) || !aligned16(dalpha_c) || !aligned16(dbeta_c) || B < 1 || T < 1 || T_out < 0 ||
        window < 1 || !std::isfinite(scale))
        return ORTHROS_ERR_INVALID_ARG;
    if (T_out > 0 && (!aligned16(qc_raw) || !pos || !aligned16(oc) || !aligned16(dOc) || !aligned16(dqc_raw) ||
                      (lsec != nullptr && !aligned16(lsec))))
        return ORTHROS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || !heads_ok(Hq, Hkv))
        return ORTHROS_ERR_UNSUPPORTED;
    const size_t need = orthros_attn_bwd_workspace_size(B, T, T_out, Hq, Hkv, d);
    if (!aligned16(workspace) || ws_bytes < need)
        return ORTHROS_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    orthros::AttnBwdParams p{};
    p.q = q_raw;
    p.k = k;
    p.v = v;
    p.o = o;
    p.dO = dO;
    p.alpha = alpha;
    p.beta = beta;
    p.pos = nullptr;
    p.lse_in = lse;
    p.dq = dq_raw;
    p.dk = dk;
    p.dv = dv;
    p.dalpha = dalpha;
    p.dbeta = dbeta;
    p.lse = reinterpret_cast<float *>(ws);
    p.Drow = p.lse + static_cast<size_t>(B) * T * Hq;
    p.k16 = reinterpret_cast<uint16_t *>(ws + orthros::attn_bwd_k16_offset(B, T, Hq));
    p.kexp = reinterpret_cast<int8_t *>(ws + orthros::attn_bwd_kexp_offset(B, T, T, Hkv, Hq, d));
    p.kflag = reinterpret_cast<uint8_t *>(ws + orthros::attn_bwd_kflag_offset(B, T, T, Hkv, Hq, d));
    p.nkb = orthros::attn_bwd_key_blocks(T);
    p.q16 = reinterpret_cast<uint16_t *>(ws + orthros::attn_bwd_workspace_bytes(B, T, T, Hkv, Hq, d));
    p.dev_err = dev_err;
    p.B = B;
    p.n_units = T;
    p.T_kv = T;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = window;
    p.accumulate = 0;
    p.scale = scale;

    char *wc = ws + ((orthros_swa_bwd_workspace_size(B, T, Hq, Hkv, d) + 255) & ~static_cast<size_t>(255));
    orthros::AttnBwdParams pc = p;
    pc.q = qc_raw;
    pc.o = oc;
    pc.dO = dOc;
    pc.alpha = alpha_c;
    pc.beta = beta_c;
    pc.pos = T_out > 0 ? pos : reinterpret_cast<const int32_t *>(ws);  // T_out == 0: never read
    pc.lse_in = T_out > 0 ? lsec : nullptr;
    pc.dq = dqc_raw;
    pc.dalpha = dalpha_c;
    pc.dbeta = dbeta_c;
    pc.lse = reinterpret_cast<float *>(wc);
    pc.Drow = pc.lse + static_cast<size_t>(B) * T_out * Hq;
    pc.part_ml = reinterpret_cast<float2 *>(wc + orthros::attn_bwd_k16_offset(B, T_out, Hq));
    pc.q16 = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(pc.part_ml) + orthros::attn_bwd_split_bytes(B, Hkv));
    pc.n_units = T_out;
    pc.window = T;  // a copy at position P sees keys 0..P
    CUtensorMap maps[orthros::ATTN_BWD_MAPS], mapsc[orthros::ATTN_BWD_MAPS];
    if (!bwd_maps(maps, q_raw, dO, k, v, p.k16, p.q16, d, Hq, Hkv, T, T, B, dq_raw) ||
        !bwd_maps(mapsc, T_out > 0 ? qc_raw : k, T_out > 0 ? dOc : k, k, v, p.k16, T_out > 0 ? pc.q16 : p.k16, d, Hq,
                  Hkv, T_out > 0 ? T_out : 1, T, B, nullptr))
        return ORTHROS_ERR_CUDA;
    const cudaError_t e =
        orthros::launch_attn_bwd_layer(d, Hq / Hkv, p, pc, maps, mapsc, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ORTHROS_OK : ORTHROS_ERR_CUDA;
}

}  // extern "C"
