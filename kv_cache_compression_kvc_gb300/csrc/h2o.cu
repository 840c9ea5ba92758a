// h2o.cu -- H2O score accumulation and eviction ("Compressão e Poda Dinâmica de KV Cache",
// section "Heavy-Hitter Oracle (H2O) e a esparsidade de cauda pesada").
//
// Per decode step and (batch, head): s_j += alpha_j with alpha_j = exp(logit_j - lse) taken
// from the decode kernel's logits; then, if the cache holds more than the budget, the token
// with the smallest s among those outside the recent quota (pos <= t - L_local) is evicted --
// equal scores evict the larger position -- and its slot becomes the next token's slot
// (in-place compaction by slot reuse: no row moves).  One warp per row; the argmin is a warp
// reduction over (s, pos, slot).
#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

// true if candidate a (score sa, position pa) should be evicted rather than b.
__device__ __forceinline__ bool evict_before(float sa, int pa, float sb, int pb)
{
    return sa < sb || (sa == sb && pa > pb);
}

__global__ void h2o_accumulate_evict_kernel(const H2OParams p)
{
    const int row = (int)((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.rows) return;
    const int64_t t = *p.t;
    const float *lg = p.logits + (size_t)row * p.logits_stride;
    float *s = p.score + (size_t)row * p.stride;
    const int32_t *pos = p.pos + (size_t)row * p.stride;
    const float lse = p.lse[row];
    const int64_t limit = t - p.L_local;

    float best_s = INFINITY;
    int best_p = -1, best_j = -1;
    for (int j = lane; j < p.n_slots; j += 32) {
        const float sj = s[j] + expf(lg[j] - lse);
        s[j] = sj;
        const int pj = pos[j];
        if ((int64_t)pj <= limit &&
            (best_j < 0 || evict_before(sj, pj, best_s, best_p))) {
            best_s = sj; best_p = pj; best_j = j;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, best_s, o);
        const int op = __shfl_xor_sync(0xffffffffu, best_p, o);
        const int oj = __shfl_xor_sync(0xffffffffu, best_j, o);
        if (oj >= 0 && (best_j < 0 || evict_before(os, op, best_s, best_p))) {
            best_s = os; best_p = op; best_j = oj;
        }
    }
    if (lane == 0 && p.n_slots > p.budget) {
        if (best_j < 0) record_code(p.dev_code, 6 /* KVC_DEV_NO_CANDIDATE */);
        else p.free_slot[row] = best_j;
    }
}

__global__ void gather_scores_kernel(const float *s_full, int64_t s_stride, const int32_t *idx,
                                     int64_t idx_stride, int rows, int n_keep, float *out)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)rows * n_keep) return;
    const int r = (int)(i / n_keep), j = (int)(i % n_keep);
    out[(size_t)r * n_keep + j] = s_full[(size_t)r * s_stride + idx[(size_t)r * idx_stride + j]];
}

}  // namespace

cudaError_t launch_h2o_accumulate_evict(const H2OParams &p, cudaStream_t stream)
{
    if (p.rows == 0) return cudaSuccess;
    const int threads = 128;
    const long long blocks = ((long long)p.rows * 32 + threads - 1) / threads;
    h2o_accumulate_evict_kernel<<<(unsigned)blocks, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gather_scores(const float *s_full, int64_t s_stride, const int32_t *idx,
                                 int64_t idx_stride, int rows, int n_keep, float *out,
                                 cudaStream_t stream)
{
    const long long total = (long long)rows * n_keep;
    if (total == 0) return cudaSuccess;
    gather_scores_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(
        s_full, s_stride, idx, idx_stride, rows, n_keep, out);
    return cudaGetLastError();
}

}  // namespace kvc
