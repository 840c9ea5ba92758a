// decode_bf16_alibi.cu -- bf16-storage instantiations of the decode attention kernel with ALiBi at in-cache positions.
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_bf16_alibi(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<__nv_bfloat16, kDecodeAlibi>(p, D, G, stream);
}
}  // namespace kvc
