// decode_f32_paged.cu -- fp32-storage instantiations of the decode attention kernel over a paged cache.
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_f32_paged(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<float, kDecodePaged>(p, D, G, stream);
}
}  // namespace kvc
