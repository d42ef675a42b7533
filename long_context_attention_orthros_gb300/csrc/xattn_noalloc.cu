// xattn_noalloc.cu -- orthros_xattn_fwd_noalloc: the output-copy cross-attention
// for callers that cannot allocate device memory themselves.
//
// Some callers have no way to obtain a workspace: a plug-in hosted by another
// runtime that owns every byte of device memory and forbids allocation on its
// hot path, or a latency-bound loop that must never call cudaMalloc (it can
// block on the device and can fail once memory is fragmented or capped).  This
// entry point therefore keeps the split-KV partial results in a fixed,
// file-scope device array instead of a caller-provided workspace, and calls
// no allocating routine at all.
//
// The array costs ORTHROS_XATTN_NOALLOC_MAX_BYTES of device memory on every GPU
// that loads this library, for as long as the process lives.  All calls share
// it: two calls whose kernels overlap on the GPU (different streams, or
// different host threads, without ordering between them) race on it and give
// wrong results.  Each call overwrites every partial it later reads, so nothing
// in the array needs to start at zero.
//
// In host code the array's name is only a host-side stand-in, never a device
// address.  The device address is looked up with cudaGetSymbolAddress once per
// device, by the first call made while that device is current; make that first
// call before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.cuh"

static __device__ __align__(256) unsigned char g_xattn_scratch[ORTHROS_XATTN_NOALLOC_MAX_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_xattn_scratch on the current device (looked up once per device).
void *scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_xattn_scratch) != cudaSuccess || !ptr)
            return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" orthros_status orthros_xattn_fwd_noalloc(const orthros_bf16 *qc_raw, const int32_t *pos,
                                                    const orthros_bf16 *k, const orthros_bf16 *v,
                                                    const float *alpha_c, const float *beta_c, orthros_bf16 *oc,
                                                    int B, int T_out, int T_kv, int Hq, int Hkv, int d,
                                                    float scale, int64_t qc_bstride, int64_t kv_bstride,
                                                    int64_t oc_bstride, int32_t *dev_err, void *stream)
{
    const size_t need = orthros_xattn_workspace_size(B, T_out, T_kv, Hq, Hkv, d);
    if (need == 0)  // sizes, head dimension or grouping refused: the same status orthros_xattn_fwd gives
        return orthros_xattn_fwd(qc_raw, pos, k, v, alpha_c, beta_c, oc, B, T_out, T_kv, Hq, Hkv, d, scale,
                                 qc_bstride, kv_bstride, oc_bstride, nullptr, 0, dev_err, stream);
    if (need > ORTHROS_XATTN_NOALLOC_MAX_BYTES)
        return ORTHROS_ERR_WORKSPACE;  // these sizes need more scratch than the fixed array holds
    void *scratch = scratch_on_current_device();
    if (!scratch)
        return ORTHROS_ERR_CUDA;
    return orthros_xattn_fwd(qc_raw, pos, k, v, alpha_c, beta_c, oc, B, T_out, T_kv, Hq, Hkv, d, scale,
                             qc_bstride, kv_bstride, oc_bstride, scratch, ORTHROS_XATTN_NOALLOC_MAX_BYTES,
                             dev_err, stream);
}
