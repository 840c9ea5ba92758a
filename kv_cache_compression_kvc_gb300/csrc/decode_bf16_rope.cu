// decode_bf16_rope.cu -- bf16-storage instantiations of the decode attention kernel with RoPE at in-cache positions.
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_bf16_rope(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<__nv_bfloat16, kDecodeRope>(p, D, G, stream);
}
}  // namespace kvc
