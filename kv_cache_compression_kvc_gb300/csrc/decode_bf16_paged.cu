// decode_bf16_paged.cu -- bf16-storage instantiations of the decode attention kernel over a paged cache.
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_bf16_paged(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<__nv_bfloat16, kDecodePaged>(p, D, G, stream);
}
}  // namespace kvc
