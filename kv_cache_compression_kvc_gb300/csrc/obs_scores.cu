// obs_scores.cu -- observation-window attention scores on CUDA cores (fp32 FMA).
//
// SnapKV steps 1-2 ("Compressão e Poda Dinâmica de KV Cache", "SnapKV e a seleção de contexto
// no prefill"): the last L_obs prompt queries of each query head attend causally to the
// prompt keys; the attention each key receives is averaged over the window.  The same kernels
// compute H2O's prompt scores (section "Heavy-Hitter Oracle (H2O)...": s_j = sum_t alpha_t,j)
// with the window covering the whole prompt and a plain sum.
//
// Softmax needs each row's normaliser before any column can be summed, so there are two
// passes over the keys:
//   pass 1: per (row tile, key chunk) block, the running max and sum of exp2 of every row
//           over the chunk's keys; a merge kernel turns the chunk states into log2-sum-exp;
//   pass 2: per (key tile) block, every row's probability exp2(l - lse) is recomputed and
//           summed down the columns, one query head at a time, in a fixed order (the column
//           sums are bit-reproducible).
// Tiles: 32 rows (never crossing a head) x 64 keys, head dimension in slices of 32, operands
// staged in shared memory as fp32; 256 threads, each 2 rows x 4 keys.
// This is the path for fp32 inputs; bf16 inputs of supported shapes use the tensor-core
// kernel in obs_scores_tc.cu.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int RT = 32;    // rows per tile
constexpr int KT = 64;    // keys per tile
constexpr int DS = 32;    // head-dim slice
constexpr int NT = 256;   // threads

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Logits of a 32-row x 64-key tile (base-2 scaled).  Rows w0 .. w0+31 of query head gq (rows
// past L_obs are zero); keys k0 .. k0+63 (keys past N are zero).  Thread (tx, ty) gets rows
// 2*ty + {0,1} and keys tx + 16*{0..3}.
template <typename T>
__device__ __forceinline__ void tile_logits(const ScoreParams &p, const T *qh, const T *kbh,
                                            int w0, int k0, float (&Qs)[RT][DS + 1],
                                            float (&Ks)[KT][DS + 1], float (&acc)[2][4])
{
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int d0 = 0; d0 < p.D; d0 += DS) {
        // stage: Q 32x32 (4 per thread), K 64x32 (8 per thread)
#pragma unroll
        for (int e = 0; e < (RT * DS) / NT; ++e) {
            const int idx = tid + e * NT;
            const int r = idx / DS, d = idx % DS;
            const int w = w0 + r;
            Qs[r][d] = (w < p.L_obs) ? to_f(qh[(size_t)w * p.D + d0 + d]) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < (KT * DS) / NT; ++e) {
            const int idx = tid + e * NT;
            const int r = idx / DS, d = idx % DS;
            const int key = k0 + r;
            Ks[r][d] = (key < p.N) ? to_f(kbh[(size_t)key * p.ss + d0 + d]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int d = 0; d < DS; ++d) {
            const float q0 = Qs[2 * ty][d], q1 = Qs[2 * ty + 1][d];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float kv = Ks[tx + 16 * j][d];
                acc[0][j] = fmaf(q0, kv, acc[0][j]);
                acc[1][j] = fmaf(q1, kv, acc[1][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] *= p.scale_log2;
}

// Pass 1: grid (G * row_blocks, n_chunks, B*Hkv).
template <typename T>
__global__ void __launch_bounds__(NT) rowstats_kernel(const ScoreParams p)
{
    __shared__ float Qs[RT][DS + 1];
    __shared__ float Ks[KT][DS + 1];
    const int row_blocks = (p.L_obs + RT - 1) / RT;
    const int g = blockIdx.x / row_blocks;
    const int w0 = (blockIdx.x % row_blocks) * RT;
    const int chunk_id = blockIdx.y;
    const int bkh = blockIdx.z;
    const int b = bkh / p.Hkv, kh = bkh % p.Hkv;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int R = p.G * p.L_obs;

    const T *qh = static_cast<const T *>(p.q) +
                  ((size_t)(b * p.Hq + kh * p.G + g) * p.L_obs) * p.D;
    const T *kbh = static_cast<const T *>(p.k) + (size_t)b * p.sb + (size_t)kh * p.sh;

    const int first_pos = p.N - p.L_obs;               // text position of window row 0
    const int max_pos = first_pos + min(w0 + RT, p.L_obs) - 1;
    const int c_begin = chunk_id * p.chunk;
    const int c_end = min(min(c_begin + p.chunk, p.N), max_pos + 1);

    float m_run[2] = {kNegBig, kNegBig}, z_run[2] = {0.f, 0.f};
    for (int k0 = c_begin; k0 < c_end; k0 += KT) {
        float acc[2][4];
        tile_logits<T>(p, qh, kbh, w0, k0, Qs, Ks, acc);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int pos = first_pos + w0 + 2 * ty + i;
            float mx = kNegBig;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = k0 + tx + 16 * j;
                if (key >= c_end || key > pos) acc[i][j] = -INFINITY;
                mx = fmaxf(mx, acc[i][j]);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_new = fmaxf(m_run[i], mx);
            float z = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) z += exp2f(acc[i][j] - m_new);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            z_run[i] = z_run[i] * exp2f(m_run[i] - m_new) + z;
            m_run[i] = m_new;
        }
    }
    if (tx == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int w = w0 + 2 * ty + i;
            if (w < p.L_obs) {
                const int r = g * p.L_obs + w;
                float *dst = p.row_ml + (((size_t)bkh * p.n_chunks + chunk_id) * R + r) * 2;
                dst[0] = m_run[i];
                dst[1] = z_run[i];
            }
        }
    }
}

// Merge the chunk states of every row: lse2 = M + log2(sum_c z_c * 2^(m_c - M)).
__global__ void rowlse_kernel(const ScoreParams p)
{
    const int R = p.G * p.L_obs;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)p.B * p.Hkv * R) return;
    const long long bkh = i / R;
    const int r = (int)(i % R);
    float M = kNegBig;
    for (int c = 0; c < p.n_chunks; ++c)
        M = fmaxf(M, p.row_ml[((bkh * p.n_chunks + c) * R + r) * 2]);
    float Z = 0.f;
    for (int c = 0; c < p.n_chunks; ++c) {
        const float *s = p.row_ml + ((bkh * p.n_chunks + c) * R + r) * 2;
        Z += s[1] * exp2f(s[0] - M);
    }
    p.row_lse2[bkh * R + r] = M + log2f(Z);
}

// Pass 2: grid (key tiles over n_cols, B*Hkv).
template <typename T>
__global__ void __launch_bounds__(NT) colsum_kernel(const ScoreParams p)
{
    __shared__ float Qs[RT][DS + 1];
    __shared__ float Ks[KT][DS + 1];
    __shared__ float red[16][KT + 1];
    const int k0 = blockIdx.x * KT;
    const int bkh = blockIdx.y;
    const int b = bkh / p.Hkv, kh = bkh % p.Hkv;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int R = p.G * p.L_obs;
    const int first_pos = p.N - p.L_obs;
    const T *kbh = static_cast<const T *>(p.k) + (size_t)b * p.sb + (size_t)kh * p.sh;
    const float *lse_b = p.row_lse2 + (size_t)bkh * R;

    // window rows whose position reaches this key tile: first_pos + w >= k0
    int w_first = k0 - first_pos;
    w_first = w_first < 0 ? 0 : (w_first / RT) * RT;

    for (int g = 0; g < p.G; ++g) {
        const T *qh = static_cast<const T *>(p.q) +
                      ((size_t)(b * p.Hq + kh * p.G + g) * p.L_obs) * p.D;
        float col = 0.f;   // held by threads tid < KT: column k0 + tid
        for (int w0 = w_first; w0 < p.L_obs; w0 += RT) {
            float acc[2][4];
            tile_logits<T>(p, qh, kbh, w0, k0, Qs, Ks, acc);
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int w = w0 + 2 * ty + i;
                if (w >= p.L_obs) continue;
                const int pos = first_pos + w;
                const float lse2 = lse_b[g * p.L_obs + w];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int key = k0 + tx + 16 * j;
                    if (key <= pos && key < p.N) part[j] += exp2f(acc[i][j] - lse2);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) red[ty][tx + 16 * j] = part[j];
            __syncthreads();
            if (tid < KT) {
                float s = 0.f;
#pragma unroll
                for (int y = 0; y < 16; ++y) s += red[y][tid];
                col += s;
            }
            __syncthreads();
        }
        if (tid < KT && k0 + tid < p.n_cols)
            p.s_out[(size_t)(b * p.Hq + kh * p.G + g) * p.n_cols + k0 + tid] = col * p.col_mult;
    }
}

// Pool (kernel pool_k, stride 1, zero padding, divisor pool_k) then max over the G heads.
// Every pooled sum adds s[i-r] .. s[i+r] left to right in fp32 (terms outside the prefix are
// zeros, and adding +0 leaves a non-negative sum unchanged) and divides by pool_k with an IEEE
// division: a fixed arithmetic order, so a reader can replay it exactly.  Each thread produces
// POOL_RUN consecutive outputs from one window of loads (a sliding window over the row).
constexpr int POOL_RUN = 8;
constexpr int POOL_MAXK = 15;

template <int PK>
__global__ void pool_groupmax_kernel(const float *s, int64_t s_row_stride, float *score, int BH,
                                     int G, int n)
{
    constexpr int r = (PK - 1) / 2;
    constexpr int WIN = POOL_RUN + PK - 1;
    const int runs = (n + POOL_RUN - 1) / POOL_RUN;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (long long)BH * runs) return;
    const int bh = (int)(t / runs);
    const int i0 = (int)(t % runs) * POOL_RUN;
    float best[POOL_RUN];
#pragma unroll
    for (int u = 0; u < POOL_RUN; ++u) best[u] = -INFINITY;
    for (int g = 0; g < G; ++g) {
        const float *sg = s + (size_t)(bh * G + g) * s_row_stride;
        float win[WIN];
#pragma unroll
        for (int j = 0; j < WIN; ++j) {
            const int idx = i0 - r + j;
            win[j] = (idx >= 0 && idx < n) ? sg[idx] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < POOL_RUN; ++u) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < PK; ++j) acc = __fadd_rn(acc, win[u + j]);
            best[u] = fmaxf(best[u], __fdiv_rn(acc, (float)PK));
        }
    }
#pragma unroll
    for (int u = 0; u < POOL_RUN; ++u)
        if (i0 + u < n) score[(size_t)bh * n + i0 + u] = best[u];
}

}  // namespace

ScorePlan score_plan(int B, int Hkv, int G, int N, int L_obs, int n_sm, size_t base_off)
{
    // Pass 1 splits the keys into n_chunks chunks of whole 128-key tiles so that about four
    // blocks per SM are in flight (counted in 128-row tiles, the tensor-core kernel's unit;
    // the CUDA-core kernel, which uses smaller row tiles, then simply has more blocks).
    constexpr int KTILE = 128;
    ScorePlan pl;
    const int R = G * L_obs;
    const long long mtiles = (R + KTILE - 1) / KTILE;
    const long long pairs = (long long)B * Hkv;
    const long long base = pairs * mtiles;
    const long long want = 4LL * (n_sm > 0 ? n_sm : 152);
    const long long key_tiles = (N + KTILE - 1) / KTILE;
    long long n_chunks = (want + base - 1) / base;
    if (n_chunks > key_tiles) n_chunks = key_tiles;
    if (n_chunks < 1) n_chunks = 1;
    long long chunk_tiles = (key_tiles + n_chunks - 1) / n_chunks;
    if (chunk_tiles < 1) chunk_tiles = 1;
    n_chunks = (key_tiles + chunk_tiles - 1) / chunk_tiles;
    if (n_chunks < 1) n_chunks = 1;
    pl.n_chunks = (int)n_chunks;
    pl.chunk = (int)(chunk_tiles * KTILE);
    auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
    pl.off_ml = align(base_off);
    pl.off_lse = align(pl.off_ml + (size_t)pairs * n_chunks * R * 2 * sizeof(float));
    pl.bytes = align(pl.off_lse + (size_t)pairs * (mtiles * KTILE) * sizeof(float));
    return pl;
}

cudaError_t launch_obs_scores(const ScoreParams &p, int dtype, cudaStream_t stream)
{
    const int row_blocks = (p.L_obs + RT - 1) / RT;
    dim3 g1(p.G * row_blocks, p.n_chunks, p.B * p.Hkv);
    if (dtype == 0) rowstats_kernel<float><<<g1, NT, 0, stream>>>(p);
    else rowstats_kernel<__nv_bfloat16><<<g1, NT, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.Hkv * p.G * p.L_obs;
    rowlse_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.n_cols <= 0) return cudaSuccess;
    dim3 g2((p.n_cols + KT - 1) / KT, p.B * p.Hkv);
    if (dtype == 0) colsum_kernel<float><<<g2, NT, 0, stream>>>(p);
    else colsum_kernel<__nv_bfloat16><<<g2, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pool_groupmax(const float *s, int64_t s_row_stride, float *score, int BH,
                                 int G, int n, int pool_k, cudaStream_t stream)
{
    const long long total = (long long)BH * ((n + POOL_RUN - 1) / POOL_RUN);
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + 255) / 256);
    switch (pool_k) {
#define KVC_POOL_CASE(PK) \
    case PK: pool_groupmax_kernel<PK><<<blocks, 256, 0, stream>>>(s, s_row_stride, score, BH, G, n); break;
    KVC_POOL_CASE(1) KVC_POOL_CASE(3) KVC_POOL_CASE(5) KVC_POOL_CASE(7)
    KVC_POOL_CASE(9) KVC_POOL_CASE(11) KVC_POOL_CASE(13) KVC_POOL_CASE(15)
#undef KVC_POOL_CASE
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kvc
