// decode_f32_duo.cu -- fp32-storage instantiations of the decode attention kernel for DuoAttention (full and ring caches in one launch).
#include "decode_attn.cuh"

namespace kvc {
cudaError_t launch_decode_attn_f32_duo(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
    return launch_decode_variant<float, kDecodeDuo>(p, D, G, stream);
}
}  // namespace kvc
