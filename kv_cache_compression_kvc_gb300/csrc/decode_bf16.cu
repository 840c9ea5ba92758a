// decode_bf16.cu -- bf16-storage instantiations of the decode attention kernel.
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_bf16(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<__nv_bfloat16, kDecodePlain>(p, D, G, stream);
}
}  // namespace kvc
