// decode_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// kvc_decode_attn needs a caller-provided workspace for the partial softmax states of its
// split-slot schedule.  Some callers have no way to provide one: a host engine that plans all
// device memory at start-up and refuses allocations afterwards, a plugin running inside another
// framework's stream capture (where a cudaMalloc would break the capture), or a process whose
// memory pool is fixed by an external budget.  This entry point serves them: its scratch lives
// in a file-scope device array that the library's module owns, so no call allocates, frees or
// asks a library to allocate.
//
// Consequences a caller must know:
//   - The array is kKvcNoAllocScratchBytes bytes on every GPU where this library's module is
//     loaded, held until the process exits.  Problems whose workspace would exceed it are
//     rejected with KVC_ERR_WORKSPACE before anything is launched.
//   - All calls share the array and it keeps whatever the previous call left in it.  Every call
//     first clears, on its own stream, the part that must start at zero (the per-head tickets).
//     Calls that can overlap on the GPU (different streams without ordering between them) race
//     on the array and give undefined results: order them on one stream.
//   - The host-side name of the array is only a stand-in for the device symbol.  Its device
//     address is looked up with cudaGetSymbolAddress once per device, by the first call made
//     while that device is current, and cached.  Make that first call before any stream capture
//     on that device.
#include <cstdio>
#include <mutex>

#include "../../include/kvc.h"
#include "internal.h"

namespace {

constexpr size_t kKvcNoAllocScratchBytes = 8u << 20;   // 8 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kKvcNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDev] = {};

kvc_status noalloc_fail(kvc_status st, const char *what, cudaError_t e)
{
    char buf[256];
    snprintf(buf, sizeof(buf), "kvc_decode_attn_noalloc: %s: %s", what, cudaGetErrorString(e));
    kvc::set_last_error(buf);
    return st;
}

}  // namespace

extern "C" kvc_status kvc_decode_attn_noalloc(const void *q, int32_t n_heads_q,
                                              const kvc_cache *cache, const int32_t *len,
                                              int32_t n_valid, const kvc_rope *rope, float scale,
                                              float *out, float *logits, int64_t logits_stride,
                                              float *lse, void *stream)
{
    if (cache == nullptr || n_heads_q <= 0 || cache->batch <= 0 || cache->n_heads_kv <= 0 ||
        cache->cap < 0)
        return kvc_decode_attn(q, n_heads_q, cache, len, n_valid, rope, scale, out, logits,
                               logits_stride, lse, nullptr, 0, stream);   // reports the error
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(KVC_ERR_CUDA, "cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDev)
        return noalloc_fail(KVC_ERR_CUDA, "device ordinal out of range", cudaErrorInvalidDevice);
    int n_sm = 0;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return noalloc_fail(KVC_ERR_CUDA, "cudaDeviceGetAttribute", e);
    const kvc::DecodePlan pl = kvc::decode_plan(cache->batch, n_heads_q, cache->n_heads_kv,
                                                cache->d_head, cache->cap, n_sm);
    if (pl.bytes > kKvcNoAllocScratchBytes) {
        char buf[256];
        snprintf(buf, sizeof(buf),
                 "kvc_decode_attn_noalloc: this problem needs %zu bytes of scratch; the "
                 "library's fixed scratch holds %zu (use kvc_decode_attn with a workspace)",
                 pl.bytes, kKvcNoAllocScratchBytes);
        kvc::set_last_error(buf);
        return KVC_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (g_scratch_ptr[dev] == nullptr) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess) return noalloc_fail(KVC_ERR_CUDA, "cudaGetSymbolAddress", e);
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.bytes > 0) {
        // the tickets must start at zero whatever an earlier call left behind
        e = cudaMemsetAsync(static_cast<char *>(scratch) + pl.off_cnt, 0,
                            pl.bytes - pl.off_cnt, s);
        if (e != cudaSuccess) return noalloc_fail(KVC_ERR_CUDA, "cudaMemsetAsync", e);
    }
    return kvc_decode_attn(q, n_heads_q, cache, len, n_valid, rope, scale, out, logits,
                           logits_stride, lse, scratch, kKvcNoAllocScratchBytes, stream);
}
