// decode_f32_rope.cu -- fp32-storage instantiations of the decode attention kernel with RoPE at in-cache positions.
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_f32_rope(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<float, kDecodeRope>(p, D, G, stream);
}
}  // namespace kvc
