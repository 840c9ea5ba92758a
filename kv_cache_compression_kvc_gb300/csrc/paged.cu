// paged.cu -- block-level eviction over page tables ("Compressão e Poda Dinâmica de KV Cache",
// section "Implementação prática em vLLM e SGLang": the cache is allocated in blocks of 16 or 32
// tokens reached through a page table; a block is rated by the sum of its tokens' importance,
// Score(block) = sum over t in the block of s_t; when memory runs out the lowest-scoring blocks
// leave the page table and return to the free pool with no copy of their contents).
//
// State per layer: a pool of physical blocks K/V [Hkv][n_pool][bs][D] (head-major: one head's
// blocks share a region); per sequence b a page
// table (physical ids in logical order), its block count, its token count and one score per
// table entry; a stack of free physical ids shared by the sequences.
//
// paged_append_kernel (one block per sequence): the new token goes to the last block at offset
// len % bs; when that is 0 a block is popped from the free stack first and appended to the
// table with score 0.  Pops from several sequences in one launch take distinct stack entries
// (atomicSub on the stack top), so which sequence gets which free id depends on timing; the
// logical cache does not.
//
// block_accumulate_kernel (one thread block per (table entry, sequence)): the entry's score
// grows by the attention this step's query heads gave its tokens, alpha = exp(logit - lse) from
// the decode kernel's logits (indexed by logical slot), summed in a fixed order (threads over
// (head, offset) pairs, then a shuffle tree), so results do not depend on timing.  Many short
// blocks, so that the update, which runs beside the next layer's decode, never holds an SM for
// long.
//
// block_release_kernel (one warp per sequence): if the sequence holds more than budget_blocks
// blocks, the lowest-scoring block outside the recent_blocks newest is released (equal scores
// release the newer one): the table and scores after it shift down by one entry, the token
// count drops by bs, and its physical id is pushed onto the free stack (atomicAdd on the stack
// top; pushes and pops never share a launch).
#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int kAppendThreads = 128;
constexpr int kEvictThreads = 128;
constexpr int kPickThreads = 256;
constexpr int kDevBadLength = 5;
constexpr int kDevNoCandidate = 6;
constexpr int kDevBadBlock = 9;
constexpr int kDevPoolEmpty = 10;
constexpr int kDevPoolOverflow = 11;

__global__ void __launch_bounds__(kAppendThreads) paged_append_kernel(const PagedParams p,
                                                                      int row_bytes)
{
    __shared__ int s_blk, s_off;
    const int b = blockIdx.x;
    pdl_trigger();
    pdl_wait();                                 // lengths and tables may come from the previous kernel
    if (threadIdx.x == 0) {
        const int n = p.len[b], nb = p.n_blocks[b];
        int blk = -1, off = 0;
        if (n < 0 || n >= p.max_blocks * p.bs || nb != (n + p.bs - 1) / p.bs) {
            record_code(p.dev_code, kDevBadLength);
        } else {
            const int lb = n / p.bs;
            off = n - lb * p.bs;
            int32_t *row_tab = p.table + (size_t)b * p.max_blocks;
            if (off == 0) {                     // the last block is full: open a new one
                const int old = atomicSub(p.free_top, 1);
                if (old <= 0 || old > p.free_cap) {
                    atomicAdd(p.free_top, 1);
                    record_code(p.dev_code, kDevPoolEmpty);
                } else {
                    const int id = p.free_ids[old - 1];
                    if (id < 0 || id >= p.n_pool) {
                        record_code(p.dev_code, kDevBadBlock);
                    } else {
                        blk = id;
                        row_tab[lb] = id;
                        p.score[(size_t)b * p.max_blocks + lb] = 0.f;
                        p.n_blocks[b] = lb + 1;
                    }
                }
            } else {
                const int id = row_tab[lb];
                if (id < 0 || id >= p.n_pool) record_code(p.dev_code, kDevBadBlock);
                else blk = id;
            }
            if (blk >= 0) {
                p.len[b] = n + 1;
                if (p.pos != nullptr && p.t != nullptr) p.pos[(size_t)blk * p.bs + off] = (int32_t)*p.t;
            }
        }
        s_blk = blk;
        s_off = off;
    }
    __syncthreads();
    const int blk = s_blk, off = s_off;
    if (blk < 0) return;
    // Hkv rows of K and of V, 16-byte vectors
    const int vpr = row_bytes / 16;
    const int total = p.Hkv * vpr;
    const char *kn = static_cast<const char *>(p.k_new) + (size_t)b * p.Hkv * row_bytes;
    const char *vn = static_cast<const char *>(p.v_new) + (size_t)b * p.Hkv * row_bytes;
    char *kd = static_cast<char *>(p.k);
    char *vd = static_cast<char *>(p.v);
    for (int i = threadIdx.x; i < total; i += kAppendThreads) {
        const int h = i / vpr, c = i - h * vpr;
        const size_t dst = ((((size_t)h * p.n_pool + blk) * p.bs + off) * row_bytes) + (size_t)c * 16;
        const size_t src = (size_t)h * row_bytes + (size_t)c * 16;
        const uint4 kx = __ldg(reinterpret_cast<const uint4 *>(kn + src));
        const uint4 vx = __ldg(reinterpret_cast<const uint4 *>(vn + src));
        *reinterpret_cast<uint4 *>(kd + dst) = kx;
        *reinterpret_cast<uint4 *>(vd + dst) = vx;
    }
}

// true if block a (score sa, index ia) is released rather than b: lower score, then newer
__device__ __forceinline__ bool release_before(float sa, int ia, float sb, int ib)
{
    return sa < sb || (sa == sb && ia > ib);
}

// n (tokens) and nb (blocks) of sequence b agree with each other and with the table size
__device__ __forceinline__ bool lengths_ok(const PagedParams &p, int n, int nb)
{
    return n >= 0 && nb >= 0 && nb <= p.max_blocks && n <= nb * p.bs &&
           (nb == 0 || n > (nb - 1) * p.bs);
}

// Accumulation: one thread block per (logical block i, sequence b); its threads take the
// (head, offset) terms of block i in order and the block sums them with a fixed tree, so each
// score gets the same bits whatever the timing.
__global__ void __launch_bounds__(kEvictThreads) block_accumulate_kernel(const PagedParams p)
{
    constexpr int NW = kEvictThreads / 32;
    __shared__ float s_part[NW];
    const int i = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();                                 // logits and lse come from the decode kernel
    const int n = p.len[b], nb = p.n_blocks[b];
    if (!lengths_ok(p, n, nb)) {
        if (i == 0 && tid == 0) record_code(p.dev_code, kDevBadLength);
        return;
    }
    if (i >= nb) return;
    const int fill = min(p.bs, n - i * p.bs);
    const float *lg0 = p.logits + (size_t)b * p.Hq * p.logits_stride + (size_t)i * p.bs;
    const float *lse = p.lse + (size_t)b * p.Hq;
    const int terms = p.Hq * p.bs;
    float part = 0.f;
#pragma unroll 4
    for (int x = tid; x < terms; x += kEvictThreads) {
        const int h = x / p.bs, off = x - h * p.bs;
        if (off < fill)
            part += expf(__ldg(lg0 + (size_t)h * p.logits_stride + off) - __ldg(lse + h));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) s_part[warp] = part;
    __syncthreads();
    if (tid == 0) {
        float tot = s_part[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) tot += s_part[w];
        p.score[(size_t)b * p.max_blocks + i] += tot;
    }
}

// Release: one warp per sequence, after the accumulation of every block has finished.
__global__ void __launch_bounds__(32) block_release_kernel(const PagedParams p)
{
    const int b = blockIdx.x, lane = threadIdx.x;
    pdl_trigger();
    pdl_wait();                                 // the scores of this step are complete
    const int n = p.len[b], nb = p.n_blocks[b];
    if (!lengths_ok(p, n, nb) || nb <= p.budget_blocks) {
        if (lane == 0 && p.released != nullptr) p.released[b] = -1;
        return;
    }
    float *sc = p.score + (size_t)b * p.max_blocks;
    int32_t *row_tab = p.table + (size_t)b * p.max_blocks;
    // the lowest score among blocks 0 .. nb - recent - 1 (equal scores: the newer)
    const int n_cand = nb - p.recent_blocks;
    float best = INFINITY;
    int bi = -1;
    for (int i = lane; i < n_cand; i += 32) {
        const float v = sc[i];
        if (bi < 0 || release_before(v, i, best, bi)) {
            best = v;
            bi = i;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi >= 0 && (bi < 0 || release_before(ov, oi, best, bi))) {
            best = ov;
            bi = oi;
        }
    }
    if (lane == 0 && p.released != nullptr) p.released[b] = bi;
    if (bi < 0) {
        if (lane == 0) record_code(p.dev_code, kDevNoCandidate);
        return;
    }
    const int phys = row_tab[bi];
    // the entries after the victim move down one place, 32 at a time in ascending order (a
    // chunk's reads lie above every index an earlier chunk wrote)
    for (int c = bi; c < nb - 1; c += 32) {
        const int j = c + lane;
        int32_t id = 0;
        float v = 0.f;
        if (j < nb - 1) {
            id = row_tab[j + 1];
            v = sc[j + 1];
        }
        __syncwarp();
        if (j < nb - 1) {
            row_tab[j] = id;
            sc[j] = v;
        }
        __syncwarp();
    }
    if (lane == 0) {
        p.n_blocks[b] = nb - 1;
        p.len[b] = n - p.bs;
        const int slot = atomicAdd(p.free_top, 1);
        if (slot < 0 || slot >= p.free_cap) {
            atomicSub(p.free_top, 1);
            record_code(p.dev_code, kDevPoolOverflow);
        } else {
            p.free_ids[slot] = phys;
        }
    }
}

// ---- the prompt: one-shot compression to budget_blocks blocks ----------------------------
// Score of prompt block i of sequence b: the sum over the H heads and its tokens of the
// prompt's per-token scores, in a fixed order (threads over (head, offset), shuffle tree).
__global__ void __launch_bounds__(kEvictThreads) block_prompt_score_kernel(const BlockPromptParams p)
{
    constexpr int NW = kEvictThreads / 32;
    __shared__ float s_part[NW];
    const int i = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();                                 // the scores may come from the previous kernel
    const int fill = min(p.bs, p.N - i * p.bs);
    const float *s0 = p.s + (size_t)b * p.H * p.s_stride + (size_t)i * p.bs;
    float part = 0.f;
    for (int x = tid; x < p.H * p.bs; x += kEvictThreads) {
        const int h = x / p.bs, off = x - h * p.bs;
        if (off < fill) part += __ldg(s0 + (size_t)h * p.s_stride + off);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) s_part[warp] = part;
    __syncthreads();
    if (tid == 0) {
        float tot = s_part[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) tot += s_part[w];
        p.ws_score[(size_t)b * p.nblk + i] = tot;
    }
}

// Selection: block i < n_old is kept when fewer than k_old older blocks outrank it (a higher
// score, or an equal score and a lower index); the recent blocks always.  The kept blocks take
// consecutive table entries in ascending order and one contiguous range of free ids.
__global__ void __launch_bounds__(kPickThreads) block_prompt_pick_kernel(const BlockPromptParams p)
{
    __shared__ int s_keep[kPickThreads];
    __shared__ int s_base, s_ok;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    const float *sc = p.ws_score + (size_t)b * p.nblk;
    const int recent = min(p.recent_blocks, p.nblk);
    const int n_old = p.nblk - recent;
    const int k_old = p.nblk <= p.budget_blocks ? n_old : p.budget_blocks - recent;
    const int n_keep = k_old + recent;
    if (tid == 0) {
        s_ok = 1;
        if (p.n_blocks[b] != 0) {               // the table must start empty
            record_code(p.dev_code, kDevBadLength);
            s_ok = 0;
        } else {
            const int old = atomicSub(p.free_top, n_keep);
            if (old < n_keep || old > p.free_cap) {
                atomicAdd(p.free_top, n_keep);
                record_code(p.dev_code, kDevPoolEmpty);
                s_ok = 0;
            } else {
                s_base = old - n_keep;
            }
        }
    }
    __syncthreads();
    if (!s_ok) return;
    int written = 0;                            // entries before this chunk of blocks
    for (int c0 = 0; c0 < p.nblk; c0 += kPickThreads) {
        const int i = c0 + tid;
        int keep = 0;
        if (i < p.nblk) {
            if (i >= n_old || k_old >= n_old) {
                keep = 1;
            } else {
                const float v = sc[i];
                int rank = 0;
                for (int j = 0; j < n_old && rank < k_old; ++j) {
                    const float u = sc[j];
                    rank += (u > v || (u == v && j < i)) ? 1 : 0;
                }
                keep = rank < k_old;
            }
        }
        s_keep[tid] = keep;
        __syncthreads();
        // exclusive scan of the flags, in thread order (the chunk is at most kPickThreads)
        int before = written;
        for (int j = 0; j < tid; ++j) before += s_keep[j];
        if (keep) {
            const int id = p.free_ids[s_base + before];
            p.table[(size_t)b * p.max_blocks + before] = id;
            p.score[(size_t)b * p.max_blocks + before] = sc[i];
            p.ws_src[(size_t)b * p.budget_blocks + before] = i;
        }
        int total = 0;
        for (int j = 0; j < kPickThreads; ++j) total += s_keep[j];
        written += total;
        __syncthreads();
    }
    if (tid == 0) {
        p.n_blocks[b] = n_keep;
        p.len[b] = (n_keep - 1) * p.bs + (p.N - (p.nblk - 1) * p.bs);   // the newest may be partial
    }
}

// Copy: kept block e of sequence b, head h -> its pool block, the tokens of K and V.
__global__ void __launch_bounds__(kAppendThreads) block_prompt_gather_kernel(const BlockPromptParams p)
{
    const int e = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
    pdl_trigger();
    pdl_wait();
    if (e >= p.n_blocks[b]) return;
    const int src_blk = p.ws_src[(size_t)b * p.budget_blocks + e];
    const int phys = p.table[(size_t)b * p.max_blocks + e];
    if (src_blk < 0 || src_blk >= p.nblk || phys < 0 || phys >= p.n_pool) {
        if (threadIdx.x == 0) record_code(p.dev_code, kDevBadBlock);
        return;
    }
    const int fill = min(p.bs, p.N - src_blk * p.bs);
    const int vpr = p.row_bytes / 16;
    for (int x = threadIdx.x; x < fill * vpr; x += kAppendThreads) {
        const int r = x / vpr, c = x - r * vpr;
        const size_t src = ((size_t)b * p.sb + (size_t)h * p.sh + (size_t)(src_blk * p.bs + r) * p.ss) *
                               (size_t)p.eb + (size_t)c * 16;
        const size_t dst = (((size_t)h * p.n_pool + phys) * p.bs + r) * (size_t)p.row_bytes +
                           (size_t)c * 16;
        const uint4 kx = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(p.pk) + src));
        const uint4 vx = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(p.pv) + src));
        *reinterpret_cast<uint4 *>(static_cast<char *>(p.k) + dst) = kx;
        *reinterpret_cast<uint4 *>(static_cast<char *>(p.v) + dst) = vx;
    }
}

}  // namespace

cudaError_t launch_paged_append(const PagedParams &p, int elem_bytes, cudaStream_t stream)
{
    if (p.B == 0) return cudaSuccess;
    return launch_pdl(paged_append_kernel, dim3((unsigned)p.B), dim3(kAppendThreads), 0, stream,
                      p, p.D * elem_bytes);
}

cudaError_t launch_block_accumulate_evict(const PagedParams &p, cudaStream_t stream)
{
    if (p.B == 0) return cudaSuccess;
    cudaError_t e = launch_pdl(block_accumulate_kernel, dim3((unsigned)p.max_blocks, (unsigned)p.B),
                               dim3(kEvictThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(block_release_kernel, dim3((unsigned)p.B), dim3(32), 0, stream, p);
}

cudaError_t launch_block_prompt_select(const BlockPromptParams &p, cudaStream_t stream)
{
    if (p.B == 0 || p.nblk == 0) return cudaSuccess;
    cudaError_t e = launch_pdl(block_prompt_score_kernel, dim3((unsigned)p.nblk, (unsigned)p.B),
                               dim3(kEvictThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    e = launch_pdl(block_prompt_pick_kernel, dim3((unsigned)p.B), dim3(kPickThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(block_prompt_gather_kernel,
                      dim3((unsigned)p.budget_blocks, (unsigned)p.B, (unsigned)p.H),
                      dim3(kAppendThreads), 0, stream, p);
}

}  // namespace kvc
