// decode_bf16_duo.cu -- bf16-storage instantiations of the decode attention kernel for DuoAttention (full and ring caches in one launch).
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_bf16_duo(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<__nv_bfloat16, kDecodeDuo>(p, D, G, stream);
}
}  // namespace kvc
