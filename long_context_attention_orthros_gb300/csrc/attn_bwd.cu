// attn_bwd.cu -- host side of the gradients of "Orthros: Phase-Aware Heterogeneous Attention"
// (the base stream, Eq. (4), and the output copies, Eq. (5), each with its scale-offset):
// the workspace layout and the dispatch on the head dimension.  The kernels and their launch
// order are in attn_bwd.cuh, instantiated per head dimension in attn_bwd_d128.cu and
// attn_bwd_d64.cu.
#include "kernels.cuh"

namespace orthros {

cudaError_t attn_bwd_launch_d128(int G, const AttnBwdParams &p, const CUtensorMap *maps, cudaStream_t stream);
cudaError_t attn_bwd_launch_d64(int G, const AttnBwdParams &p, const CUtensorMap *maps, cudaStream_t stream);
cudaError_t attn_bwd_layer_d128(int G, const AttnBwdParams &p, const AttnBwdParams &pc, const CUtensorMap *maps,
                               const CUtensorMap *mapsc, cudaStream_t stream);
cudaError_t attn_bwd_layer_d64(int G, const AttnBwdParams &p, const AttnBwdParams &pc, const CUtensorMap *maps,
                              const CUtensorMap *mapsc, cudaStream_t stream);

static size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

int attn_bwd_key_blocks(int T_kv) { return (T_kv + 63) / 64; }

size_t attn_bwd_kexp_offset(int B, int n_units, int T_kv, int Hkv, int Hq, int D)
{
    return attn_bwd_k16_offset(B, n_units, Hq) + round256(2 * static_cast<size_t>(B) * T_kv * Hkv * D);
}

size_t attn_bwd_kflag_offset(int B, int n_units, int T_kv, int Hkv, int Hq, int D)
{
    return attn_bwd_kexp_offset(B, n_units, T_kv, Hkv, Hq, D) +
           round256(static_cast<size_t>(B) * Hkv * attn_bwd_key_blocks(T_kv) * 64);
}

size_t attn_bwd_workspace_bytes(int B, int n_units, int T_kv, int Hkv, int Hq, int D)
{
    return attn_bwd_kflag_offset(B, n_units, T_kv, Hkv, Hq, D) +
           round256(static_cast<size_t>(B) * Hkv * attn_bwd_key_blocks(T_kv));
}

size_t attn_bwd_split_bytes(int B, int Hkv)
{
    return static_cast<size_t>(B) * Hkv * ATTN_BWD_MAX_SPLITS * 128 * sizeof(float2);
}

size_t attn_bwd_k16_offset(int B, int n_units, int Hq)
{
    return (8 * static_cast<size_t>(B) * n_units * Hq + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_attn_bwd(int D, int G, const AttnBwdParams &p, const CUtensorMap *maps, cudaStream_t stream)
{
    if (D == 128)
        return attn_bwd_launch_d128(G, p, maps, stream);
    if (D == 64)
        return attn_bwd_launch_d64(G, p, maps, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_bwd_layer(int D, int G, const AttnBwdParams &p, const AttnBwdParams &pc,
                                  const CUtensorMap *maps, const CUtensorMap *mapsc, cudaStream_t stream)
{
    if (D == 128)
        return attn_bwd_layer_d128(G, p, pc, maps, mapsc, stream);
    if (D == 64)
        return attn_bwd_layer_d64(G, p, pc, maps, mapsc, stream);
    return cudaErrorInvalidValue;
}

}  // namespace orthros
