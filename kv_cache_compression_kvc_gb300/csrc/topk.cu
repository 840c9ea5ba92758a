// topk.cu -- exact per-row top-k with the lowest-index tie rule, indices emitted ascending.
//
// SnapKV step 4 ("Compressão e Poda Dinâmica de KV Cache", "SnapKV e a seleção de contexto no
// prefill": keep the positions with the largest pooled score, per KV head) and H2O's prompt
// compression (keep the K_HH largest accumulated scores).  Equal scores keep the lower index;
// kept indices keep their original order, followed by `tail` always-kept indices n .. n+tail-1
// (the SnapKV observation window, or H2O's recent quota).
//
// One 1024-thread block per row.  Scores are mapped to order-preserving 32-bit keys (staged in
// shared memory when the row fits).  A min/max pass finds the highest bit in which the row's
// keys differ, so the radix passes skip the bits every key shares (scores of one row sit in a
// few octaves); then 8-bit radix passes with one private shared-memory histogram per warp find
// the exact key T of the k-th largest and how many keys equal to T are still to be taken.  A
// last pair of passes emits, in index order, every key > T plus the first `need` keys == T:
// each warp owns a contiguous segment, counts its keeps with ballots, a block scan gives each
// warp its output offset.
#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int TK_THREADS = 1024;
constexpr int TK_WARPS = TK_THREADS / 32;

__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int TK_SMEM_KEYS = 40 * 1024;   // rows up to this many keys are staged in smem

__global__ void __launch_bounds__(TK_THREADS)
topk_rows_kernel(const float *score, int64_t score_stride, int n, int k, int tail, int32_t *idx,
                 int64_t idx_stride)
{
    __shared__ uint32_t whist[TK_WARPS][256];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t sh_bin, sh_above, sh_lo, sh_hi;
    __shared__ uint32_t w_gt[TK_WARPS], w_eq[TK_WARPS];
    __shared__ uint32_t w_keep_before[TK_WARPS], w_eq_before[TK_WARPS];
    extern __shared__ uint32_t skeys[];

    const float *s = score + (size_t)blockIdx.x * score_stride;
    int32_t *out = idx + (size_t)blockIdx.x * idx_stride;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int j = tid; j < tail; j += TK_THREADS) out[k + j] = n + j;
    if (k <= 0) return;
    if (k >= n) {
        for (int j = tid; j < n; j += TK_THREADS) out[j] = j;
        return;
    }
    const bool staged = n <= TK_SMEM_KEYS;
    auto key_at = [&](int i) -> uint32_t { return staged ? skeys[i] : order_key(s[i]); };

    // ---- stage the keys, find their range ---------------------------------------------------
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int i = tid; i < n; i += TK_THREADS) {
        const uint32_t u = order_key(s[i]);
        if (staged) skeys[i] = u;
        lo = min(lo, u);
        hi = max(hi, u);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (tid == 0) { sh_lo = 0xffffffffu; sh_hi = 0u; }
    __syncthreads();
    if (lane == 0) { atomicMin(&sh_lo, lo); atomicMax(&sh_hi, hi); }
    __syncthreads();
    lo = sh_lo;
    hi = sh_hi;
    const uint32_t diff = lo ^ hi;
    const int top = diff ? 31 - __clz(diff) : -1;   // highest bit where keys differ

    // ---- radix select of the k-th largest key over the differing bits ------------------------
    // bits every key shares (all 32 when the keys are all equal, top = -1)
    const uint32_t shared_mask = top < 0 ? 0xffffffffu : (top >= 31 ? 0u : ~((2u << top) - 1u));
    uint32_t prefix = hi & shared_mask;
    uint32_t mask = shared_mask;
    uint32_t need = (uint32_t)k;   // still to take among keys matching the prefix
    for (int t = top; t >= 0; t -= 8) {
        const int shift = t >= 7 ? t - 7 : 0;
        const uint32_t dmask = (2u << (t - shift)) - 1u;   // digit of bits shift .. t
        for (int j = tid; j < TK_WARPS * 256; j += TK_THREADS) (&whist[0][0])[j] = 0;
        __syncthreads();
        uint32_t *mine = whist[warp];
        for (int i = tid; i < n; i += TK_THREADS) {
            const uint32_t u = key_at(i);
            if ((u & mask) == prefix) atomicAdd(&mine[(u >> shift) & dmask], 1u);
        }
        __syncthreads();
        for (int j = tid; j < 256; j += TK_THREADS) {
            uint32_t c = 0;
#pragma unroll 8
            for (int w = 0; w < TK_WARPS; ++w) c += whist[w][j];
            hist[j] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // lane L owns bins 8L .. 8L+7; count of keys in bins above lane L's range
            uint32_t c[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { c[j] = hist[lane * 8 + j]; tot += c[j]; }
            uint32_t incl = tot;   // suffix (inclusive) sum over lanes >= lane
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t x = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += x;
            }
            uint32_t cum = incl - tot;  // keys in bins above 8L+7
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                if (cum < need && cum + c[j] >= need) {
                    sh_bin = (uint32_t)(lane * 8 + j);
                    sh_above = cum;
                }
                cum += c[j];
            }
        }
        __syncthreads();
        prefix |= sh_bin << shift;
        mask |= dmask << shift;
        need -= sh_above;
        __syncthreads();
    }
    const uint32_t T = prefix;   // every bit fixed: the exact k-th largest key

    // ---- counts per warp segment ------------------------------------------------------------
    const int seg = ((n + TK_WARPS - 1) / TK_WARPS + 31) & ~31;
    const int beg = warp * seg;
    const int end = min(beg + seg, n);
    uint32_t gt = 0, eq = 0;
    for (int i0 = beg; i0 < end; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t u = i < end ? key_at(i) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, i < end && u > T));
        eq += __popc(__ballot_sync(0xffffffffu, i < end && u == T));
    }
    if (lane == 0) { w_gt[warp] = gt; w_eq[warp] = eq; }
    __syncthreads();
    if (tid == 0) {
        uint32_t eq_run = 0, keep_run = 0;
        for (int w = 0; w < TK_WARPS; ++w) {
            w_eq_before[w] = eq_run;
            w_keep_before[w] = keep_run;
            const uint32_t eq_take =
                eq_run >= need ? 0u : (w_eq[w] < need - eq_run ? w_eq[w] : need - eq_run);
            keep_run += w_gt[w] + eq_take;
            eq_run += w_eq[w];
        }
    }
    __syncthreads();

    // ---- emit in index order -----------------------------------------------------------------
    uint32_t eq_seen = w_eq_before[warp];
    uint32_t written = w_keep_before[warp];
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int i0 = beg; i0 < end; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t u = i < end ? key_at(i) : 0u;
        const bool is_eq = i < end && u == T;
        const uint32_t eq_ballot = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t eq_rank = eq_seen + __popc(eq_ballot & lt_mask);
        const bool keep = (i < end) && (u > T || (is_eq && eq_rank < need));
        const uint32_t keep_ballot = __ballot_sync(0xffffffffu, keep);
        if (keep) out[written + __popc(keep_ballot & lt_mask)] = i;
        written += __popc(keep_ballot);
        eq_seen += __popc(eq_ballot);
    }
}

__global__ void iota_rows_kernel(int32_t *idx, int64_t idx_stride, int rows, int n)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)rows * n) return;
    idx[(size_t)(i / n) * idx_stride + (size_t)(i % n)] = (int32_t)(i % n);
}

}  // namespace

cudaError_t launch_topk_rows(const float *score, int64_t score_stride, int rows, int n, int k,
                             int tail, int32_t *idx, int64_t idx_stride, cudaStream_t stream)
{
    if (rows == 0) return cudaSuccess;
    const int dyn = n <= TK_SMEM_KEYS ? n * (int)sizeof(uint32_t) : 0;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             TK_SMEM_KEYS * (int)sizeof(uint32_t));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    topk_rows_kernel<<<rows, TK_THREADS, dyn, stream>>>(score, score_stride, n, k, tail, idx,
                                                         idx_stride);
    return cudaGetLastError();
}

cudaError_t launch_iota_rows(int32_t *idx, int64_t idx_stride, int rows, int n,
                             cudaStream_t stream)
{
    const long long total = (long long)rows * n;
    if (total == 0) return cudaSuccess;
    iota_rows_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(idx, idx_stride, rows,
                                                                          n);
    return cudaGetLastError();
}

}  // namespace kvc
