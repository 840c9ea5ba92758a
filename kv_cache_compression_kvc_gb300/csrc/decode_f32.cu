// decode_f32.cu -- fp32-storage instantiations of the decode attention kernel.
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_f32(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<float, kDecodePlain>(p, D, G, stream);
}
}  // namespace kvc
