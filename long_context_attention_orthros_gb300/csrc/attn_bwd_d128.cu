// attn_bwd_d128.cu -- the gradient's kernels and launches (attn_bwd.cuh) instantiated for head
// dimension 128.
#include "attn_bwd.cuh"

namespace orthros {

cudaError_t attn_bwd_launch_d128(int G, const AttnBwdParams &p, const CUtensorMap *maps, cudaStream_t stream)
{
    return attn_bwd_dispatch<128>(G, p, maps, stream);
}

cudaError_t attn_bwd_layer_d128(int G, const AttnBwdParams &p, const AttnBwdParams &pc, const CUtensorMap *maps,
                              const CUtensorMap *mapsc, cudaStream_t stream)
{
    return attn_bwd_layer_dispatch<128>(G, p, pc, maps, mapsc, stream);
}

}  // namespace orthros
