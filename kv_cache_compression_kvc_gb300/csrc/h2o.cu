// h2o.cu -- H2O score accumulation and eviction ("Compressão e Poda Dinâmica de KV Cache",
// section "Heavy-Hitter Oracle (H2O) e a esparsidade de cauda pesada").
//
// Per decode step and (batch, head): s_j += alpha_j with alpha_j = exp(logit_j - lse) taken
// from the decode kernel's logits; then, if the cache holds more than the budget, the token
// with the smallest s among those outside the recent quota (pos <= t - L_local) is evicted --
// equal scores evict the larger position -- and its slot becomes the next token's slot
// (in-place compaction by slot reuse: no row moves).  One block of H2O_THREADS per row: each
// thread updates a strided set of slots with its loads batched (H2O_BATCH in flight), keeps its
// own best candidate, and the block reduces (s, pos, slot) with shuffles and one shared-memory
// step.  The order (lower s first, then larger pos) is total since positions are distinct, so
// the result does not depend on how the reduction is split.
//
// Grouped-query caches (G query heads per KV head): a row is evicted for the whole group, so
// its score adds the attention of all G heads, s_j += sum_g exp(logit_{g,j} - lse_g), the terms
// taken in head order.  The query heads of KV row r are rows r*G .. r*G + G - 1 of the logits
// and lse.  One instance per group size the decode supports (2, 4, 6, 8) issues the loads of
// all G heads together; another G takes a generic instance; one head keeps its own.
#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

// true if candidate a (score sa, position pa) should be evicted rather than b.
__device__ __forceinline__ bool evict_before(float sa, int pa, float sb, int pb)
{
    return sa < sb || (sa == sb && pa > pb);
}

constexpr int H2O_THREADS = 128;
constexpr int H2O_BATCH = 4;

// folds candidate (os, op, oj) into (bs, bp, bj); oj < 0 is "no candidate"
__device__ __forceinline__ void h2o_fold(float &bs, int &bp, int &bj, float os, int op, int oj)
{
    if (oj >= 0 && (bj < 0 || evict_before(os, op, bs, bp))) {
        bs = os;
        bp = op;
        bj = oj;
    }
}

// GT: 1 one head; 2..8 that group size; 0 any group size (p.G)
template <int GT>
__global__ void __launch_bounds__(H2O_THREADS) h2o_accumulate_evict_kernel(const H2OParams p)
{
    constexpr bool GROUPED = GT != 1;
    __shared__ float w_s[H2O_THREADS / 32];
    __shared__ int w_p[H2O_THREADS / 32], w_j[H2O_THREADS / 32];
    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();                                 // logits and lse come from the decode kernel
    const int64_t t = *p.t;
    const int G = GT == 0 ? p.G : GT;
    const float *__restrict__ lg = p.logits + (size_t)row * G * p.logits_stride;
    float *__restrict__ s = p.score + (size_t)row * p.stride;
    const int32_t *__restrict__ pos = p.pos + (size_t)row * p.stride;
    const float lse = p.lse[(size_t)row * G];
    const int64_t limit = t - p.L_local;
    const int n = p.n_slots;
    float lse_g[GT > 1 ? GT : 1];               // the group's log-sum-exps (head 0 is lse)
    if constexpr (GT > 1) {
#pragma unroll
        for (int g = 1; g < GT; ++g) lse_g[g] = p.lse[(size_t)row * GT + g];
    }

    float best_s = INFINITY;
    int best_p = -1, best_j = -1;
    for (int j0 = tid; j0 < n; j0 += H2O_THREADS * H2O_BATCH) {
        float sv[H2O_BATCH], lv[H2O_BATCH];
        int pv[H2O_BATCH];
#pragma unroll
        for (int u = 0; u < H2O_BATCH; ++u) {
            const int j = j0 + u * H2O_THREADS;
            lv[u] = 0.f;
            if (j < n) {
                sv[u] = s[j];
                lv[u] = __ldg(lg + j);
                pv[u] = __ldg(pos + j);
            }
        }
        if constexpr (GT > 1) {
            // every head's logits in flight at once, then the terms in head order
            float lx[GT - 1][H2O_BATCH];
#pragma unroll
            for (int g = 1; g < GT; ++g)
#pragma unroll
                for (int u = 0; u < H2O_BATCH; ++u) {
                    const int j = j0 + u * H2O_THREADS;
                    lx[g - 1][u] = j < n ? __ldg(lg + (size_t)g * p.logits_stride + j) : 0.f;
                }
#pragma unroll
            for (int u = 0; u < H2O_BATCH; ++u) {
                float acc = expf(lv[u] - lse);
#pragma unroll
                for (int g = 1; g < GT; ++g) acc += expf(lx[g - 1][u] - lse_g[g]);
                lv[u] = acc;
            }
        } else if constexpr (GT == 0) {
            // the group's other heads, in head order after head 0
            for (int g = 1; g < G; ++g) {
                const float *__restrict__ lgg = lg + (size_t)g * p.logits_stride;
                const float lse_g = p.lse[(size_t)row * G + g];
#pragma unroll
                for (int u = 0; u < H2O_BATCH; ++u) {
                    const int j = j0 + u * H2O_THREADS;
                    if (j < n) lv[u] = g == 1 ? expf(lv[u] - lse) + expf(__ldg(lgg + j) - lse_g)
                                              : lv[u] + expf(__ldg(lgg + j) - lse_g);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < H2O_BATCH; ++u) {
            const int j = j0 + u * H2O_THREADS;
            if (j < n) {
                const float sj = sv[u] + ((GROUPED && G > 1) ? lv[u] : expf(lv[u] - lse));
                s[j] = sj;
                if ((int64_t)pv[u] <= limit) h2o_fold(best_s, best_p, best_j, sj, pv[u], j);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, best_s, o);
        const int op = __shfl_xor_sync(0xffffffffu, best_p, o);
        const int oj = __shfl_xor_sync(0xffffffffu, best_j, o);
        h2o_fold(best_s, best_p, best_j, os, op, oj);
    }
    if (lane == 0) {
        w_s[warp] = best_s;
        w_p[warp] = best_p;
        w_j[warp] = best_j;
    }
    __syncthreads();
    if (tid == 0 && n > p.budget) {
        for (int w = 1; w < H2O_THREADS / 32; ++w) h2o_fold(best_s, best_p, best_j, w_s[w], w_p[w], w_j[w]);
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

// Grouped-query prompt scores: query heads kh*G + g (member g of every group) copied into a
// contiguous [B][Hkv][N][D] buffer, so the one-head scoring runs on them unchanged.
__global__ void group_member_copy_kernel(const char *__restrict__ q, char *__restrict__ dst,
                                         int Hkv, int G, int g, int N, int row_bytes,
                                         long long n_vec)
{
    const int vpr = row_bytes / 16;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / vpr;
        const int c = (int)(i - r * vpr);
        const long long bk = r / N;              // b * Hkv + kh
        const int n = (int)(r - bk * N);
        const long long src_row = (bk * G + g) * N + n;
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(q + src_row * row_bytes) + c);
        reinterpret_cast<uint4 *>(dst + r * row_bytes)[c] = x;
    }
}

// acc += x, element by element (the group's members added in head order)
__global__ void add_rows_kernel(float *__restrict__ acc, const float *__restrict__ x, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        acc[i] += x[i];
}

}  // namespace

cudaError_t launch_h2o_accumulate_evict(const H2OParams &p, cudaStream_t stream)
{
    if (p.rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)p.rows), block(H2O_THREADS);
    switch (p.G) {
    case 1: return launch_pdl(h2o_accumulate_evict_kernel<1>, grid, block, 0, stream, p);
    case 2: return launch_pdl(h2o_accumulate_evict_kernel<2>, grid, block, 0, stream, p);
    case 4: return launch_pdl(h2o_accumulate_evict_kernel<4>, grid, block, 0, stream, p);
    case 6: return launch_pdl(h2o_accumulate_evict_kernel<6>, grid, block, 0, stream, p);
    case 8: return launch_pdl(h2o_accumulate_evict_kernel<8>, grid, block, 0, stream, p);
    default: return launch_pdl(h2o_accumulate_evict_kernel<0>, grid, block, 0, stream, p);
    }
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

cudaError_t launch_group_member_copy(const void *q, void *dst, int B, int Hkv, int G, int g, int N,
                                     int row_bytes, cudaStream_t stream)
{
    const long long n_vec = (long long)B * Hkv * N * (row_bytes / 16);
    if (n_vec == 0) return cudaSuccess;
    const long long blocks = (n_vec + 255) / 256;
    group_member_copy_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(
        static_cast<const char *>(q), static_cast<char *>(dst), Hkv, G, g, N, row_bytes, n_vec);
    return cudaGetLastError();
}

cudaError_t launch_add_rows(float *acc, const float *x, long long n, cudaStream_t stream)
{
    if (n == 0) return cudaSuccess;
    const long long blocks = (n + 255) / 256;
    add_rows_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(acc, x, n);
    return cudaGetLastError();
}

}  // namespace kvc
