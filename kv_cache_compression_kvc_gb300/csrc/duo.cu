// duo.cu -- appending a token to DuoAttention's two caches ("Compressão e Poda Dinâmica de KV
// Cache", section "Decomposição funcional com o DuoAttention": retrieval heads keep the full
// cache, streaming heads a constant buffer of attention sinks and recent tokens).
//
// One warp per (batch, KV head) row of the new token: a retrieval head's row goes to the tail of
// its full cache (slot len, then len + 1); a streaming head's row goes to the slot of text
// position t in its sink + ring layout (slot t for t < S, else S + (t - S) mod (W + 1)).  The
// head map sends model KV head kh to its retrieval index or its streaming index.
#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int kDuoAppendWarps = 4;

__global__ void __launch_bounds__(kDuoAppendWarps * 32) duo_append_kernel(const DuoAppendParams p)
{
    const int row = blockIdx.x * kDuoAppendWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();                                 // lengths and t may come from the previous kernel
    if (row >= p.B * p.Hkv) return;
    const int b = row / p.Hkv, kh = row % p.Hkv;
    const int idx = p.index_of[kh];             // retrieval index, or n_ret + streaming index
    const bool ret = idx < p.n_ret;
    char *kd, *vd;
    if (ret) {
        const int pr = b * p.n_ret + idx;
        const int len = p.len[pr];
        __syncwarp();                           // every lane has read len before lane 0 bumps it
        if (len < 0 || len >= p.cap) {
            if (lane == 0) record_code(p.dev_code, len < 0 ? 5 : 1);
            return;
        }
        if (lane == 0) p.len[pr] = len + 1;
        const size_t off = ((size_t)b * p.sb + (size_t)idx * p.sh + (size_t)len * p.ss) * p.eb;
        kd = static_cast<char *>(p.k) + off;
        vd = static_cast<char *>(p.v) + off;
    } else {
        const int64_t t = *p.t;
        if (t < 0) {
            if (lane == 0) record_code(p.dev_code, 4);
            return;
        }
        const int slot = t < p.S ? (int)t : p.S + (int)((t - p.S) % (int64_t)(p.W + 1));
        const int is = idx - p.n_ret;
        const size_t off = ((size_t)b * p.sb2 + (size_t)is * p.sh2 + (size_t)slot * p.ss2) * p.eb;
        kd = static_cast<char *>(p.k2) + off;
        vd = static_cast<char *>(p.v2) + off;
    }
    const int row_bytes = p.D * p.eb;
    const char *kn = static_cast<const char *>(p.k_new) + (size_t)row * row_bytes;
    const char *vn = static_cast<const char *>(p.v_new) + (size_t)row * row_bytes;
    for (int c = lane * 16; c < row_bytes; c += 32 * 16) {
        const uint4 kx = __ldg(reinterpret_cast<const uint4 *>(kn + c));
        const uint4 vx = __ldg(reinterpret_cast<const uint4 *>(vn + c));
        *reinterpret_cast<uint4 *>(kd + c) = kx;
        *reinterpret_cast<uint4 *>(vd + c) = vx;
    }
}

}  // namespace

cudaError_t launch_duo_append(const DuoAppendParams &p, cudaStream_t stream)
{
    const int rows = p.B * p.Hkv;
    if (rows == 0) return cudaSuccess;
    return launch_pdl(duo_append_kernel, dim3((unsigned)((rows + kDuoAppendWarps - 1) / kDuoAppendWarps)),
                      dim3(kDuoAppendWarps * 32), 0, stream, p);
}

}  // namespace kvc
