// common.cuh -- small device helpers shared by libkvc's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvc {

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;
// Finite "minus infinity" for running maxima: exp2(x - kNegBig) never produces NaN.
constexpr float kNegBig = -1.0e30f;

__device__ __forceinline__ void record_code(int32_t *code, int32_t c)
{
    if (code != nullptr) atomicCAS(code, 0, c);
}

// bf16 stored in the low / high half of a 32-bit word (element 2i in the low half).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Streaming 16/8-byte global loads that do not allocate in L1 (each KV byte is read once).
__device__ __forceinline__ uint4 ld_stream_16(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_stream_8(const void *p)
{
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

// A vector of VW consecutive elements of type T held as raw 32-bit words.
template <typename T, int VW>
struct RawVec;

template <>
struct RawVec<float, 4> {
    uint4 w;
    __device__ __forceinline__ void load(const float *p) { w = ld_stream_16(p); }
    __device__ __forceinline__ void zero() { w = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ void to_float(float *f) const
    {
        f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
        f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
    }
};
template <>
struct RawVec<__nv_bfloat16, 8> {
    uint4 w;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { w = ld_stream_16(p); }
    __device__ __forceinline__ void zero() { w = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ void to_float(float *f) const
    {
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
        f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
    }
};
template <>
struct RawVec<__nv_bfloat16, 4> {
    uint2 w;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { w = ld_stream_8(p); }
    __device__ __forceinline__ void zero() { w = make_uint2(0, 0); }
    __device__ __forceinline__ void to_float(float *f) const
    {
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    }
};

// Plain (cached) load of VW elements of T into floats: used for small, reused operands.
template <typename T, int VW>
__device__ __forceinline__ void load_cached(const T *p, float *f)
{
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < VW; i += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(p + i);
            f[i] = x.x; f[i + 1] = x.y; f[i + 2] = x.z; f[i + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < VW; i += 2) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(p + i);
            f[i] = bf16_lo(w); f[i + 1] = bf16_hi(w);
        }
    }
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---- mbarriers, bulk copies (PTX) ---------------------------------------------------------------
// Waits are bounded: after kMbarSpinLimit failed polls the thread gives up, so a kernel can
// never hang on a lost arrival.  mbar_wait records KVC_DEV_TIMEOUT and returns as if the phase
// had completed; mbar_wait_ok only reports the outcome, for kernels that then stop issuing
// work and wait (again bounded) for their own copies in flight before they exit.
constexpr uint32_t kMbarSpinLimit = 1u << 22;
constexpr int kDevCodeTimeout = 7;           // KVC_DEV_TIMEOUT
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, int32_t *code)
{
    for (uint32_t it = 0; it < kMbarSpinLimit; ++it)
        if (mbar_try_wait(bar, parity)) return;
    record_code(code, kDevCodeTimeout);
}
// true once the phase with the given parity has completed; false after `limit` failed polls
__device__ __forceinline__ bool mbar_wait_ok(uint32_t bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// The same wait for a block that may be aborting: when the first poll fails it keeps polling
// but also gives up as soon as another thread of the block has raised *abort (checked every
// 64 polls, off the fast path), so after one wait has run out the others end quickly.
__device__ __forceinline__ bool mbar_wait_abortable(uint32_t bar, uint32_t parity, uint32_t limit,
                                                    const volatile int *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    for (uint32_t it = 1; it < limit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u && *abort != 0) return false;
    }
    return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// ---- programmatic dependent launch -----------------------------------------------------------
// A kernel launched with programmatic stream serialization may start while the previous kernel
// in the stream is still finishing.  It must call pdl_wait() before it reads anything that kernel
// may have written; pdl_trigger() lets the next kernel in the stream start its own prologue.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Release / acquire ticket on a pair's counter (one thread, after a block barrier): the block's
// partial state is visible to whichever block takes the last ticket.
__device__ __forceinline__ int ticket_acq_rel(int *p)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


// ---- split-slot decode: merge of the partial softmax states of one (batch, KV head) pair -------
// Called by all NT threads of the last block to finish pair q.  Partial state s of head g is
// (m, l) at ws_ml[((q*max_seg + s)*G + g)*2] and o[0..D) at ws_o[((q*max_seg + s)*G + g)*D]
// (m in log2 units, o not yet divided by l).  The merge reads nseg * G * (D + 2) floats that sit
// in L2, so its cost is latency: one warp per head reduces the (m, l) pairs with shuffles and
// leaves the weights 2^(m_s - M) / L in `scratch`; then each thread owns 16-byte chunks of the
// output and sums them over the segments with UNR independent loads in flight.  When the
// output has fewer chunks than threads, H thread subsets split the segments and add their
// sums through shared memory.  scratch: n_scratch floats; a pair that needs more than that
// takes the plain loop.
template <int G, int D, int NT>
__device__ __noinline__ void merge_pair_partials(const float *ws_o, const float *ws_ml,
                                                    int max_seg, int q, int nseg, float *out,
                                                    float *lse, int rows0, float *scratch,
                                                    int n_scratch)
{
    static_assert(D % 4 == 0, "16-byte output chunks");
    constexpr int NWARP = NT / 32;
    constexpr int NCH = G * D / 4;                        // 16-byte chunks of the output
    constexpr int H_RAW = NT / NCH;
    constexpr int H = H_RAW < 1 ? 1 : (H_RAW > 8 ? 8 : H_RAW);   // segment subsets
    constexpr int CPT = (NCH + NT - 1) / NT;              // chunks per thread (H == 1)
    constexpr int UNR = CPT >= 8 ? 1 : 8 / CPT;           // segments per batch of loads
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t base = (size_t)q * max_seg * G;          // state (s, g) is base + s*G + g
    if (nseg * G + (H - 1) * G * D > n_scratch) {
        for (int i = threadIdx.x; i < G * D; i += NT) {
            const int g = i / D, d = i % D;
            float M = kNegBig;
            for (int s = 0; s < nseg; ++s) M = fmaxf(M, __ldcg(&ws_ml[(base + s * G + g) * 2]));
            float L = 0.f, O = 0.f;
            for (int s = 0; s < nseg; ++s) {
                const size_t slot = base + s * G + g;
                const float c = ex2(__ldcg(&ws_ml[slot * 2]) - M);
                L += __ldcg(&ws_ml[slot * 2 + 1]) * c;
                O += __ldcg(&ws_o[slot * D + d]) * c;
            }
            out[(size_t)(rows0 + g) * D + d] = L > 0.f ? O / L : 0.f;
            if (d == 0 && lse != nullptr)
                lse[rows0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        return;
    }
    float *w = scratch;                                   // [nseg][G] weights
    float *part = scratch + nseg * G;                     // [H-1][NCH][4] subset sums
    for (int g = warp; g < G; g += NWARP) {
        const float *ml = ws_ml + (base + g) * 2;         // segment s at ml[s * 2G]
        float m0 = kNegBig, l0 = 0.f;
        if (lane < nseg) {
            m0 = __ldcg(ml + (size_t)lane * 2 * G);
            l0 = __ldcg(ml + (size_t)lane * 2 * G + 1);
        }
        float M = m0;
        for (int s = lane + 32; s < nseg; s += 32) M = fmaxf(M, __ldcg(ml + (size_t)s * 2 * G));
        M = warp_max(M);
        float L = 0.f;
        if (lane < nseg) {
            const float c = ex2(m0 - M);
            w[lane * G + g] = c;
            L = l0 * c;
        }
        for (int s = lane + 32; s < nseg; s += 32) {
            const float c = ex2(__ldcg(ml + (size_t)s * 2 * G) - M);
            w[s * G + g] = c;
            L += __ldcg(ml + (size_t)s * 2 * G + 1) * c;
        }
        L = warp_sum(L);
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int s = lane; s < nseg; s += 32) w[s * G + g] *= inv;
        if (lane == 0 && lse != nullptr)
            lse[rows0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    const int h = H > 1 ? (int)threadIdx.x / NCH : 0;     // segment subset of this thread
    float4 acc[CPT];
    int chunk[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        chunk[k] = H > 1 ? (int)threadIdx.x % NCH : (int)threadIdx.x + k * NT;
    }
    const bool active = h < H;
    const size_t seg_stride = (size_t)G * D / 4;          // float4 units between segments
    const float4 *src = reinterpret_cast<const float4 *>(ws_o) + base * (D / 4);
    if (active) {
        for (int s0 = h; s0 < nseg; s0 += H * UNR) {
            float4 v[CPT][UNR];
#pragma unroll
            for (int k = 0; k < CPT; ++k)
#pragma unroll
                for (int u = 0; u < UNR; ++u) {
                    const int s = s0 + u * H;
                    v[k][u] = (chunk[k] < NCH && s < nseg)
                                  ? __ldcg(src + (size_t)s * seg_stride + chunk[k])
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int g = chunk[k] * 4 / D;
#pragma unroll
                for (int u = 0; u < UNR; ++u) {
                    const int s = s0 + u * H;
                    const float c = s < nseg ? w[s * G + g] : 0.f;
                    acc[k].x = fmaf(c, v[k][u].x, acc[k].x);
                    acc[k].y = fmaf(c, v[k][u].y, acc[k].y);
                    acc[k].z = fmaf(c, v[k][u].z, acc[k].z);
                    acc[k].w = fmaf(c, v[k][u].w, acc[k].w);
                }
            }
        }
    }
    if (H > 1) {
        if (active && h > 0) {
            float *dst = part + ((size_t)(h - 1) * NCH + chunk[0]) * 4;
            dst[0] = acc[0].x;
            dst[1] = acc[0].y;
            dst[2] = acc[0].z;
            dst[3] = acc[0].w;
        }
        __syncthreads();
        if (h == 0) {
#pragma unroll
            for (int j = 1; j < H; ++j) {
                const float *pj = part + ((size_t)(j - 1) * NCH + chunk[0]) * 4;
                acc[0].x += pj[0];
                acc[0].y += pj[1];
                acc[0].z += pj[2];
                acc[0].w += pj[3];
            }
        }
    }
    if (h == 0) {
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            if (chunk[k] >= NCH) continue;
            float *o = out + (size_t)rows0 * D + (size_t)chunk[k] * 4;
            o[0] = acc[k].x;
            o[1] = acc[k].y;
            o[2] = acc[k].z;
            o[3] = acc[k].w;
        }
    }
}
}  // namespace kvc
