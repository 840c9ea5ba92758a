// internal.h -- launch-parameter structs and launcher declarations shared by libkvc's own
// translation units.  Not part of the public ABI (include/kvc.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace kvc {

// ------------------------------------------------------------------------------------------
// Decode attention (split over slots, log-sum-exp merge by the last block of each KV head).
// Launches `kernel` with programmatic stream serialization: its prologue may overlap the end of
// the previous kernel in the stream; the kernel calls pdl_wait() before reading its inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DecodeParams {
    const void *q;
    const void *k;
    const void *v;
    int64_t sb, sh, ss;          // cache strides, elements
    int32_t B, Hq, Hkv, cap;
    const int32_t *len;          // device [B*Hkv] or nullptr
    int32_t n_valid;             // used when len == nullptr
    // RoPE / StreamingLLM layout (rope != 0)
    int32_t rope, S, W;
    const int64_t *t;
    const float *cos_sin;        // [n_pos][2][D/2]: cosines then sines per distance
    int32_t n_pos;               // rows of cos_sin
    const float *alibi;          // ALiBi slopes per query head [Hq] (same layout as RoPE) or null
    // paged cache: K/V pool [Hkv][n_pool][bs][D]; len is per sequence [B]; cap = max_blocks*bs
    const int32_t *table;        // [B][max_blocks] physical block of each logical block
    int32_t max_blocks, bs, n_pool;
    // DuoAttention: pairs 0 .. B*n_ret-1 are retrieval heads over k/v ([B][n_ret][cap][D], len
    // per pair or n_valid); pairs B*n_ret .. are streaming heads over the ring caches k2/v2
    // ([B][n_str][ring_cap][D]) with min(*t + 1, ring_cap) valid slots.  head_of maps retrieval
    // index r (then n_ret + streaming index s) to the model's KV head.
    int32_t n_ret, n_str, NT2, ring_cap;
    const void *k2;
    const void *v2;
    int64_t sb2, sh2;
    uint8_t head_of[256];
    int32_t kv_settled;          // cache slots and lengths final before the previous launch began
    int32_t balance;             // split the tiles by the lengths (not by capacity)
    uint32_t spin_limit;         // polls before a bounded wait gives up (0: the default)
    int32_t starve;              // test hook: issue no cache loads, so the first wait runs out
    float scale_log2;            // scale * log2(e)
    float *out;                  // [B][Hq][D]
    float *logits;               // nullable, [B*Hq][logits_stride]
    int64_t logits_stride;
    float *lse;                  // nullable, [B*Hq]
    // persistent schedule: P = B*Hkv pairs of NT tiles each, split evenly over the blocks
    int32_t P, NT, max_seg, n_sm;
    float *ws_o;                 // [P][max_seg][G][D] partial weighted values
    float *ws_ml;                // [P][max_seg][G][2] partial (max, sum)
    int32_t *ws_cnt;             // [P] tickets, zero between calls
    int32_t *dev_code;
};

struct DecodePlan {
    int32_t max_seg;             // blocks that can share one (batch, KV head) pair
    size_t off_o, off_ml, off_cnt, bytes;
};

// seg_pairs: pairs of the longest kind (0: all B*Hkv pairs are alike); a pair's tiles meet at
// most C / seg_pairs + 2 blocks.
DecodePlan decode_plan(int B, int Hq, int Hkv, int D, int cap, int n_sm, int seg_pairs = 0);
// Sets the calling thread's kvc_last_error() message.
void set_last_error(const char *msg);
cudaError_t launch_decode_attn_f32(const DecodeParams &p, int D, int G, cudaStream_t stream);
cudaError_t launch_decode_attn_bf16(const DecodeParams &p, int D, int G, cudaStream_t stream);
// Tensor-core grouped-query decode (bf16, no RoPE, group 2..8).  Sets *used = false, launching
// nothing, when the case is not covered (the CUDA-core kernel then runs).
cudaError_t launch_decode_attn_mma(const DecodeParams &p, int D, int G, cudaStream_t stream,
                                   bool *used);
cudaError_t launch_decode_attn_f32_rope(const DecodeParams &p, int D, int G, cudaStream_t stream);
cudaError_t launch_decode_attn_bf16_rope(const DecodeParams &p, int D, int G,
                                         cudaStream_t stream);
cudaError_t launch_decode_attn_f32_paged(const DecodeParams &p, int D, int G, cudaStream_t stream);
cudaError_t launch_decode_attn_bf16_paged(const DecodeParams &p, int D, int G,
                                          cudaStream_t stream);
cudaError_t launch_decode_attn_f32_duo(const DecodeParams &p, int D, int G, cudaStream_t stream);
cudaError_t launch_decode_attn_bf16_duo(const DecodeParams &p, int D, int G, cudaStream_t stream);
cudaError_t launch_decode_attn_f32_alibi(const DecodeParams &p, int D, int G, cudaStream_t stream);
cudaError_t launch_decode_attn_bf16_alibi(const DecodeParams &p, int D, int G,
                                          cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// Append, gather, position advance.
struct AppendParams {
    void *k;
    void *v;
    int64_t sb, sh, ss;
    int32_t B, H, cap, D;
    int32_t policy;
    const void *k_new;
    const void *v_new;
    const int64_t *t;
    int32_t *len;
    int32_t S, W;
    const int32_t *free_slot;
    int32_t *pos;
    int64_t pos_stride;
    float *score;
    int64_t score_stride;
    int32_t *dev_code;
};
cudaError_t launch_append(const AppendParams &p, int elem_bytes, cudaStream_t stream);

struct GatherParams {
    const void *sk;
    const void *sv;
    int64_t s_sb, s_sh, s_ss;
    int32_t s_cap;
    void *dk;
    void *dv;
    int64_t d_sb, d_sh, d_ss;
    int32_t B, H, D;
    const int32_t *idx;
    int64_t idx_stride;
    int32_t n_keep;
    int32_t *pos_dst;
    int64_t pos_stride;
    int32_t *len_dst;
    int32_t *dev_code;
};
cudaError_t launch_gather(const GatherParams &p, int elem_bytes, cudaStream_t stream);
cudaError_t launch_position_advance(int64_t *t, int64_t delta, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// Observation-window scoring (SnapKV steps 1-2; H2O prompt column sums).
// Rows r = g*L_obs + w of KV head kh are the window queries of q-head kh*G+g; the query at
// window index w sits at text position N - L_obs + w and sees keys 0 .. N - L_obs + w.
struct ScoreParams {
    const void *q;               // [B][Hq][L_obs][D] contiguous
    const void *k;               // prompt keys (cache strides)
    int64_t sb, sh, ss;
    int32_t B, Hq, Hkv, G, D, N, L_obs;
    float scale_log2;            // scale * log2(e)
    int32_t n_cols;              // columns written: N - L_obs (SnapKV) or N (H2O)
    float col_mult;              // 1/L_obs (mean) or 1 (sum)
    float *s_out;                // [B][Hq][n_cols]
    float *row_ml;               // workspace [B*Hkv][n_chunks][R][2]
    float *row_lse2;             // workspace [B*Hkv][R rounded up to 128]: each row's log2-sum-exp
                                 // (CUDA-core path: stride R; tensor-core path: negated, stride
                                 // R rounded up to 128, the padding zeroed)
    int32_t n_chunks;
    int32_t chunk;
};
struct ScorePlan {
    int32_t n_chunks, chunk;
    size_t off_ml, off_lse, bytes;
};
ScorePlan score_plan(int B, int Hkv, int G, int N, int L_obs, int n_sm, size_t base_off);
cudaError_t launch_obs_scores(const ScoreParams &p, int dtype, cudaStream_t stream);
// Tensor-core (tcgen05) scoring for bf16 inputs.  Sets *used = false, launching nothing, when
// the shape is not supported (then the CUDA-core kernels are used).
bool obs_scores_tc_supported(const ScoreParams &p);
cudaError_t launch_obs_scores_tc(const ScoreParams &p, int32_t *dev_code, cudaStream_t stream,
                                 bool *used);

// Pool (kernel pool_k, zero padding, divisor pool_k, sum left to right) + max over the G heads.
cudaError_t launch_pool_groupmax(const float *s, int64_t s_row_stride, float *score, int BH,
                                 int G, int n, int pool_k, cudaStream_t stream);

// Exact top-k per row (ties: lower index), ascending emission, then `tail` indices
// n .. n+tail-1 appended.  idx row stride = k + tail.
// SnapKV steps 3-4 fused (pool + group max + top-k) with one thread-block cluster per row; sets
// *used = false, launching nothing, when the row is too long for the cluster's shared memory.
cudaError_t launch_pool_topk(const float *s, int64_t s_row_stride, int rows, int G, int n, int k,
                             int tail, int pool_k, int32_t *idx, int64_t idx_stride,
                             cudaStream_t stream, bool *used);
cudaError_t launch_topk_rows(const float *score, int64_t score_stride, int rows, int n, int k,
                             int tail, int32_t *idx, int64_t idx_stride, cudaStream_t stream);
cudaError_t launch_iota_rows(int32_t *idx, int64_t idx_stride, int rows, int n,
                             cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// DuoAttention append: model KV head kh of the new token goes to retrieval cache index
// index_of[kh] (< n_ret, tail slot len) or streaming ring index index_of[kh] - n_ret.
struct DuoAppendParams {
    void *k, *v;                 // retrieval caches [B][n_ret][cap][D]
    int64_t sb, sh, ss;
    int32_t cap;
    int32_t *len;                // [B*n_ret]
    void *k2, *v2;               // streaming rings [B][n_str][S+W+1][D]
    int64_t sb2, sh2, ss2;
    int32_t S, W;
    const int64_t *t;
    const void *k_new, *v_new;   // [B][Hkv][D]
    int32_t B, Hkv, D, eb, n_ret;
    uint8_t index_of[256];
    int32_t *dev_code;
};
cudaError_t launch_duo_append(const DuoAppendParams &p, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// Block-level eviction over page tables.
struct PagedParams {
    void *k;                     // pool [Hkv][n_pool][bs][D]
    void *v;
    int32_t n_pool, Hkv, bs, D, B, max_blocks;
    int32_t *table;              // [B][max_blocks]
    int32_t *n_blocks;           // [B]
    int32_t *len;                // [B]
    float *score;                // [B][max_blocks]
    int32_t *free_ids;           // [free_cap] stack of free physical blocks
    int32_t *free_top;           // number of ids on the stack
    int32_t free_cap;
    // append
    const void *k_new;           // [B][Hkv][D]
    const void *v_new;
    const int64_t *t;            // nullable
    int32_t *pos;                // nullable [n_pool][bs]
    // accumulate / release
    const float *logits;         // [B*Hq][logits_stride], logical slots
    int64_t logits_stride;
    const float *lse;            // [B*Hq]
    int32_t Hq, budget_blocks, recent_blocks;
    int32_t *released;           // nullable [B]
    int32_t *dev_code;
};
cudaError_t launch_paged_append(const PagedParams &p, int elem_bytes, cudaStream_t stream);

// The prompt's block selection: block scores, the pick, the copy into pool blocks.
struct BlockPromptParams {
    const float *s;              // [B][H][s_stride] per-token scores of the prompt
    int64_t s_stride;
    const void *pk, *pv;         // prompt K/V [B][H][>= N][D] (cache strides, elements)
    int64_t sb, sh, ss;
    void *k, *v;                 // pool [H][n_pool][bs][D]
    int32_t B, H, N, bs, nblk, eb, row_bytes, n_pool, max_blocks;
    int32_t *table, *n_blocks, *len;
    float *score;
    int32_t *free_ids, *free_top;
    int32_t free_cap, budget_blocks, recent_blocks;
    float *ws_score;             // [B][nblk]
    int32_t *ws_src;             // [B][budget_blocks] prompt block of each kept entry
    int32_t *dev_code;
};
cudaError_t launch_block_prompt_select(const BlockPromptParams &p, cudaStream_t stream);
cudaError_t launch_block_accumulate_evict(const PagedParams &p, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// H2O.
struct H2OParams {
    const float *logits;
    int64_t logits_stride;
    const float *lse;
    float *score;
    int32_t *pos;
    int64_t stride;
    int32_t *free_slot;
    int32_t rows, n_slots, L_local, budget;
    int32_t G;                   // query heads per KV row (1: MHA)
    const int64_t *t;
    int32_t *dev_code;
};
cudaError_t launch_h2o_accumulate_evict(const H2OParams &p, cudaStream_t stream);
cudaError_t launch_group_member_copy(const void *q, void *dst, int B, int Hkv, int G, int g, int N,
                                     int row_bytes, cudaStream_t stream);
cudaError_t launch_add_rows(float *acc, const float *x, long long n, cudaStream_t stream);
cudaError_t launch_gather_scores(const float *s_full, int64_t s_stride, const int32_t *idx,
                                 int64_t idx_stride, int rows, int n_keep, float *out,
                                 cudaStream_t stream);

}  // namespace kvc
