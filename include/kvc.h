/*
 * kvc.h -- C ABI of libkvc: KV-cache compression and decode attention over the compressed cache
 * on one NVIDIA GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [KVC]  "Compressão e Poda Dinâmica de KV Cache: StreamingLLM, SnapKV, PyramidKV e
 *          DuoAttention" (produtoramaxvision.com.br blog)
 *   [SINK] "attention sinks" encyclopedia entry (tonho.wtf diário)
 *   [KVCL] "O KV cache", lesson 7.2 of llmdeepdive, section "01 · Conceito"
 *
 * Conventions shared by every entry point
 *   - Plain C types only.  Every tensor argument is a DEVICE pointer owned by the caller unless
 *     the comment says "host".  The library never allocates device memory; operations that
 *     need scratch take a caller-owned workspace whose size is given by a *_workspace_bytes
 *     query.  Workspaces must be 256-byte aligned.
 *   - All work is enqueued on the caller's CUDA stream (`stream`, a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  No entry point synchronises except
 *     kvc_device_status.  Entry points can be captured into a CUDA graph.
 *   - Every entry point validates its arguments on the host before launching anything and
 *     returns a kvc_status; on error nothing is launched and kvc_last_error() describes why.
 *     Values that only exist on the device (lengths, slots, positions) are range-checked by the
 *     kernels: an out-of-range value skips the access and records a code that
 *     kvc_device_status() returns.
 *   - A cache is [batch][n_heads_kv][cap][d_head] with d_head contiguous (see kvc_cache).
 *     d_head is 64, 128 or 256; base pointers are 16-byte aligned and every stride is a
 *     multiple of 16 bytes.  Query head h reads KV head h / (n_heads_q / n_heads_kv)
 *     (grouped-query attention, [KVCL] "01 · Conceito"; [KVC] "O gargalo de memória...").
 *   - Element types: KVC_F32 (fp32 storage and arithmetic) or KVC_BF16 (bf16 storage, fp32
 *     arithmetic).  Queries and new keys/values use the cache's type; outputs are fp32.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVC_OK = 0,
    KVC_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum value               */
    KVC_ERR_SHAPE = 2,         /* unsupported or inconsistent sizes (d_head, head groups)    */
    KVC_ERR_ALIGN = 3,         /* pointer or stride not 16-byte aligned                      */
    KVC_ERR_CAPACITY = 4,      /* a cache or output is too small for the request             */
    KVC_ERR_CUDA = 5,          /* a CUDA runtime call failed (message in kvc_last_error)     */
    KVC_ERR_WORKSPACE = 6,     /* workspace missing, too small or misaligned                 */
    KVC_ERR_DEVICE = 7         /* a kernel's own range check fired (see kvc_device_status)   */
} kvc_status;

typedef enum { KVC_F32 = 0, KVC_BF16 = 1 } kvc_dtype;

/* Device-side range-check codes recorded by kernels (first one wins until read). */
enum {
    KVC_DEV_OK = 0,
    KVC_DEV_TAIL_FULL = 1,      /* append at len >= cap                                       */
    KVC_DEV_BAD_SLOT = 2,       /* free slot outside [0, cap)                                 */
    KVC_DEV_BAD_INDEX = 3,      /* gather index outside [0, src cap)                          */
    KVC_DEV_BAD_POSITION = 4,   /* negative text position                                     */
    KVC_DEV_BAD_LENGTH = 5,     /* len outside [0, cap]                                       */
    KVC_DEV_NO_CANDIDATE = 6,   /* H2O: cache over budget but no historical token to evict    */
    KVC_DEV_TIMEOUT = 7,        /* a bounded wait inside a kernel gave up (results invalid)   */
    KVC_DEV_SCHEDULE = 8,       /* internal schedule bound violated (results invalid)         */
    KVC_DEV_BAD_BLOCK = 9,      /* page-table or free-stack entry outside the block pool      */
    KVC_DEV_POOL_EMPTY = 10,    /* a sequence needed a new block and the free stack was empty */
    KVC_DEV_POOL_OVERFLOW = 11  /* a released block did not fit on the free stack             */
};

/* A KV cache (or a prompt's keys/values) in device memory.
 * Element (b, h, slot, d) of K is at k + b*stride_b + h*stride_h + slot*stride_slot + d
 * (strides in elements).  v follows the same strides; v may be NULL where only keys are read. */
typedef struct {
    void *k;
    void *v;
    int32_t dtype;          /* kvc_dtype */
    int32_t batch;
    int32_t n_heads_kv;
    int32_t cap;            /* slots per (batch, head) */
    int32_t d_head;
    int32_t reserved;
    int64_t stride_b;
    int64_t stride_h;
    int64_t stride_slot;
} kvc_cache;

/* RoPE at in-cache positions for a StreamingLLM cache ([SINK] "como funciona"; [KVC]
 * "Attention Sinks e o StreamingLLM..."): slots 0..n_sink-1 hold the sinks (text positions
 * 0..n_sink-1), slots n_sink..n_sink+window form a ring of window+1 slots in which token
 * a >= n_sink lives at slot n_sink + (a - n_sink) mod (window + 1).  When the token at text
 * position *t is decoded it attends to the sinks and to tokens max(n_sink, t-window) .. t;
 * each attended token's in-cache position is its rank in that set and the query's is
 * min(t, n_sink + window).  Keys are stored before rotation; the query and every key are
 * rotated at those positions on every call (computed through their distance: the rotated dot
 * product depends only on the query position minus the key position).  Pairing: dimension i
 * with i + d_head/2, angle position * theta^(-2i/d_head).  Row p of cos_sin holds the cosines
 * and sines of p times the pair frequencies; since those angles are linear in p, the kernel may
 * also compose a distance from two rows (cos(a+b) = cos a cos b - sin a sin b, and likewise for
 * the sine), which it does for one query head per KV head when n_pos covers one tile of slots
 * (16 KB of keys: 64 rows for bf16 with d_head 128).                                          */
typedef struct {
    int32_t n_sink;         /* S  (4 in the pages' configuration)                            */
    int32_t window;         /* W                                                             */
    const int64_t *t;       /* device scalar: text position of the token being decoded       */
    const float *cos_sin;   /* device [n_pos][2][d_head/2]: cosines then sines (kvc_rope_table) */
    int32_t n_pos;          /* rows of cos_sin; must be >= n_sink + window + 1               */
    int32_t reserved;
} kvc_rope;

/* ALiBi at in-cache positions for a StreamingLLM cache ([SINK] "como funciona": under ALiBi
 * the linear bias runs continuously over the in-cache positions, with no jump where tokens were
 * evicted, so distances never exceed the cache).  Same sink + ring layout, attended set and
 * in-cache positions as kvc_rope; keys are stored and used as given (no rotation).  The logit
 * of query head h against the attended token at in-cache position r is
 *     scale * q.k - slopes[h] * (qpos - r),   qpos = min(t, n_sink + window).
 * The pages print no slope values: the caller passes them (kvc_alibi_slopes gives the usual
 * geometric sequence).                                                                       */
typedef struct {
    int32_t n_sink;         /* S                                                             */
    int32_t window;         /* W                                                             */
    const int64_t *t;       /* device scalar: text position of the token being decoded       */
    const float *slopes;    /* device fp32[n_heads_q]: the bias slope of each query head     */
} kvc_alibi;

/* Paged KV cache for block-level eviction ([KVC] "Implementação prática em vLLM e SGLang": the
 * cache is allocated in blocks of 16 or 32 tokens reached through a page table; blocks leave
 * the page table and return to the free pool without their contents being copied).
 * One pool, one set of page tables and one free stack per layer.
 * Element (blk, h, j, d) of K is at k + ((h*n_blocks + blk)*block_size + j)*d_head + d
 * (v likewise): block blk holds block_size consecutive tokens of every KV head, each head's
 * part in that head's region of the pool (head-major, so the blocks one head reads stay
 * close together whatever ids the page table holds).                                          */
typedef struct {
    void *k;                /* device [n_heads_kv][n_blocks][block_size][d_head]             */
    void *v;
    int32_t dtype;          /* kvc_dtype                                                     */
    int32_t n_blocks;       /* physical blocks in the pool                                   */
    int32_t n_heads_kv;
    int32_t block_size;     /* tokens per block                                              */
    int32_t d_head;
    int32_t reserved;
} kvc_block_pool;

/* Page tables of a batch of sequences.  Sequence b holds len[b] tokens in n_blocks[b] blocks:
 * logical block i is physical block table[b*max_blocks + i]; tokens fill the blocks in table
 * order, so only the last block may be partly filled (n_blocks[b] = ceil(len[b]/block_size)).
 * score[b*max_blocks + i] is logical block i's score (kvc_block_accumulate_evict).           */
typedef struct {
    int32_t *table;         /* device int32[batch][max_blocks]                               */
    int32_t *n_blocks;      /* device int32[batch]                                           */
    int32_t *len;           /* device int32[batch]                                           */
    float *score;           /* device fp32[batch][max_blocks]                                */
    int32_t batch;
    int32_t max_blocks;
} kvc_page_table;

/* The free pool: a stack of free physical block ids, ids[0 .. *top - 1].  Within one call the
 * pops (kvc_paged_append, kvc_block_prompt_select) or the pushes (kvc_block_accumulate_evict)
 * of several sequences take distinct entries through an atomic on *top; calls that use the
 * same free pool must not overlap on the GPU (order them on one stream, or join the streams
 * between them), since a pop racing a push could read an entry before it is written. */
typedef struct {
    int32_t *ids;           /* device int32[capacity]                                        */
    int32_t *top;           /* device int32 scalar: number of free ids                       */
    int32_t capacity;
    int32_t reserved;
} kvc_free_pool;

/* DuoAttention's inference half ([KVC] "Decomposição funcional com o DuoAttention"): the KV
 * heads of a layer are split by a fixed mask gamma (its calibration is training and out of
 * scope).  Retrieval heads (gamma = 1, 20-30 % of the heads on the page) keep the full cache;
 * streaming heads (gamma = 0) keep a constant buffer of n_sink attention sinks and the window
 * tokens before the current one, laid out as the StreamingLLM sink + ring cache of kvc_rope (no
 * positional term: keys are used as stored).  Two caches per layer:
 *   full: [batch][n_retrieval][cap][d_head], tokens at the tail (len per retrieval pair);
 *   ring: [batch][n_streaming][>= n_sink+window+1][d_head].
 * Model KV head h is retrieval index r if retrieval_heads[r] == h, else the next streaming
 * index in ascending head order.                                                             */
typedef struct {
    int32_t n_retrieval;            /* retrieval KV heads (>= 1; the ring holds >= 1 head too) */
    int32_t n_sink;                 /* S (4 on the page)                                        */
    int32_t window;                 /* W (64 on the page)                                       */
    int32_t reserved;
    const int32_t *retrieval_heads; /* HOST int32[n_retrieval]: model KV heads, ascending       */
    const int64_t *t;               /* device scalar: text position of the token being decoded  */
} kvc_duo;

/* ---------------------------------------------------------------------------------------- */
/* Diagnostics                                                                               */

/* Message for the last non-OK status returned on the calling thread ("" if none). */
const char *kvc_last_error(void);

/* Synchronises `stream`, then reads and clears the device range-check code of the current
 * device into *code (KVC_DEV_*).  Returns KVC_ERR_DEVICE if a code was set, else KVC_OK. */
kvc_status kvc_device_status(void *stream, int32_t *code);

/* ---------------------------------------------------------------------------------------- */
/* Host-side sizing                                                                          */

/* Bytes of an uncompressed KV cache: 2 * n_layers * n_heads_kv * d_head * seq_len *
 * bytes_per_elem * batch.  [KVC] "O gargalo de memória do KV Cache em contextos longos",
 * equation Memoria_KV; [KVCL] "01 · Conceito".  Pure host arithmetic. */
uint64_t kvc_kv_bytes(uint64_t n_layers, uint64_t n_heads_kv, uint64_t d_head, uint64_t seq_len,
                      uint64_t bytes_per_elem, uint64_t batch);

/* PyramidKV per-layer budgets, host.  [KVC] "Alocação piramidal com o PyramidKV":
 * B_l = B_base + dB*(N_L-1-l)/(N_L-1) with sum_l B_l = N_L*b_target.  The ramp's steepness is
 * the ratio B_0/B_{N_L-1} = ratio_num/ratio_den (4/1 for a 2x-to-0.5x ramp).  Budgets are
 * floored and the remaining slots go to the largest remainders (lower layer first on ties),
 * so the total is exact.  out: host int64[n_layers]. */
kvc_status kvc_pyramid_budgets(int32_t n_layers, int64_t b_target, int64_t ratio_num,
                               int64_t ratio_den, int64_t *out);

/* RoPE table, host: out[p][0][i] = cos(p*theta^(-2i/d_head)), out[p][1][i] = sin(...) for
 * p < n_pos, i < d_head/2 (each row: d_head/2 cosines, then d_head/2 sines), computed in double
 * and rounded to fp32.  out: host float[n_pos * d_head]; the caller uploads it for
 * kvc_rope.cos_sin. */
kvc_status kvc_rope_table(int32_t n_pos, int32_t d_head, double theta, float *out);

/* ---------------------------------------------------------------------------------------- */
/* SnapKV prefill selection.  [KVC] "SnapKV e a seleção de contexto no prefill", steps 1-4:
 *   1. the last L_obs prompt queries (observation window) attend causally to all seq_len
 *      prompt keys (scale * q.k, softmax per query);
 *   2. s_h[i] = (1/L_obs) * sum over the window of the attention to key i, per query head;
 *   3. average pooling of s_h over the prefix i < seq_len-L_obs, kernel pool_k (odd, <= 15), stride 1,
 *      zero padding, divisor pool_k; then max over the query heads of each KV head;
 *   4. the budget-L_obs prefix positions with the largest pooled score are kept (equal scores
 *      keep the lower index), in ascending order, followed by the window
 *      seq_len-L_obs .. seq_len-1 (always kept).  budget >= seq_len keeps every position.
 * q_obs:  [batch][n_heads_q][L_obs][d_head], prompt->dtype, contiguous.
 * prompt: the prompt keys (prompt->k; prompt->v unused), cap >= seq_len.
 * idx_out: [batch][n_heads_kv][min(budget, seq_len)] int32.
 * scores_out (nullable): [batch][n_heads_q][seq_len-L_obs] fp32, the step-2 column means.
 * bf16 inputs use the tensor cores (fp32 accumulation); fp32 inputs use fp32 FMA.
 * Workspace: kvc_snapkv_select_workspace_bytes(). */
size_t kvc_snapkv_select_workspace_bytes(int32_t batch, int32_t n_heads_q, int32_t n_heads_kv,
                                         int32_t d_head, int32_t seq_len, int32_t L_obs);
kvc_status kvc_snapkv_select(const void *q_obs, const kvc_cache *prompt, int32_t n_heads_q,
                             int32_t seq_len, int32_t L_obs, int32_t pool_k, int32_t budget,
                             float scale, int32_t *idx_out, float *scores_out, void *ws,
                             size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------- */
/* Gather / compaction of retained rows.  [KVC] H2O "Poda e Desalocação" (the discarded
 * tokens' tensors leave physical memory) and "Implementação prática em vLLM e SGLang"
 * (aligned, dense rows).  Out of place: for every (b, h) and j < n_keep,
 *   dst.K[b,h,j] = src.K[b,h,idx[b,h,j]], dst.V[b,h,j] = src.V[b,h,idx[b,h,j]],
 *   pos_dst[b,h,j] = idx[b,h,j] (if pos_dst), len_dst[b*H+h] = n_keep (if len_dst).
 * idx: [batch][n_heads_kv][idx_stride] int32.  Copies are bit exact.  src and dst must not
 * overlap and must agree in dtype, batch, n_heads_kv and d_head; dst->cap >= n_keep. */
kvc_status kvc_compact_gather(const kvc_cache *src, const int32_t *idx, int64_t idx_stride,
                              int32_t n_keep, const kvc_cache *dst, int32_t *pos_dst,
                              int64_t pos_stride, int32_t *len_dst, void *stream);

/* ---------------------------------------------------------------------------------------- */
/* Append one new token's key and value per (batch, KV head).
 * k_new, v_new: [batch][n_heads_kv][d_head], cache dtype, contiguous.  Keys are stored as
 * given (pre-rotation in the StreamingLLM case, [SINK] "como funciona").
 *   KVC_APPEND_TAIL:      slot = len[b*H+h]; then len[b*H+h] += 1 (device int32[batch*H]).
 *                         A full cache (len >= cap) skips the row and records
 *                         KVC_DEV_TAIL_FULL.
 *   KVC_APPEND_RING:      slot of text position *t in the sink + ring layout of kvc_rope
 *                         ([KVC] "Janela Móvel ... buffer circular"); cap >= n_sink+window+1.
 *   KVC_APPEND_FREE_SLOT: slot = free_slot[b*H+h] (set by kvc_h2o_accumulate_evict).
 * t: device int64 scalar, text position of the new token (required for RING, FREE_SLOT and
 * whenever pos is given).  pos (nullable): pos[(b*H+h)*pos_stride + slot] = *t.
 * score (nullable): score[(b*H+h)*score_stride + slot] = 0 (H2O: a new token has s = 0). */
typedef enum {
    KVC_APPEND_TAIL = 0,
    KVC_APPEND_RING = 1,
    KVC_APPEND_FREE_SLOT = 2
} kvc_append_policy;

kvc_status kvc_stream_append(const kvc_cache *cache, int32_t policy, const void *k_new,
                             const void *v_new, const int64_t *t, int32_t *len, int32_t n_sink,
                             int32_t window, const int32_t *free_slot, int32_t *pos,
                             int64_t pos_stride, float *score, int64_t score_stride,
                             void *stream);

/* Adds delta to the device int64 scalar *t (the decode position shared by the calls above),
 * on the stream, so a captured decode step can be replayed. */
kvc_status kvc_position_advance(int64_t *t, int64_t delta, void *stream);

/* ---------------------------------------------------------------------------------------- */
/* Decode attention over the retained slots: for every query head h of every batch row,
 *   out[b,h] = sum_j softmax_j(scale * q[b,h].k_j) v_j
 * over the valid slots j of KV head h/G (the token being decoded is among them once
 * appended).  [KVCL] "01 · Conceito" (the new query attends to the cached keys and mixes the
 * cached values: exact causal attention); [KVC] "O gargalo de memória..." (a GEMV over the
 * whole cache, 1-2 FLOP per byte) and "Implementação prática..." (FlashDecoding parallelises
 * over the time axis: the slots are split across thread blocks and the partial softmax states
 * are merged by log-sum-exp).
 * Valid slots: with rope == NULL, slots 0..len[b*H+h]-1 (or 0..n_valid-1 when len is NULL);
 * with rope, the sink + ring slots of kvc_rope at the decode position *rope->t.
 * q: [batch][n_heads_q][d_head] cache dtype (pre-rotation when rope is given).
 * out: [batch][n_heads_q][d_head] fp32.
 * logits (nullable): logits[(b*n_heads_q+h)*logits_stride + slot] = scale*q.k_slot for valid
 * slots (rotated keys with rope).  lse (nullable): [batch][n_heads_q] log-sum-exp of the
 * logits.  A row with no valid slot gets out = 0 and lse = -inf.
 * Workspace: kvc_decode_attn_workspace_bytes(); it must be zero-filled once before its first
 * use (the kernel leaves it zeroed again), and calls sharing a workspace must not overlap on
 * the GPU. */
size_t kvc_decode_attn_workspace_bytes(int32_t batch, int32_t n_heads_q, int32_t n_heads_kv,
                                       int32_t d_head, int32_t cap);
kvc_status kvc_decode_attn(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                           const int32_t *len, int32_t n_valid, const kvc_rope *rope,
                           float scale, float *out, float *logits, int64_t logits_stride,
                           float *lse, void *ws, size_t ws_bytes, void *stream);

/* kvc_decode_attn with flags (kvc_decode_attn is this call with flags 0).  No counterpart on
 * the pages: it lets the decode kernel overlap the kernel launched before it.
 * KVC_DECODE_KV_SETTLED: the caller guarantees that the cache slots, the lengths (len) and,
 * with rope, the decode position *rope->t that this call reads were last written before an
 * ordering point that this call follows on the stream -- the start of the CUDA graph holding
 * the call, an event the stream waited for, or a kernel launched without programmatic
 * dependent launch (it begins only once all earlier work has finished) -- and that nothing
 * launched between that point and this call writes them.  The kernel may then read them and
 * start loading cache tiles before it waits for the kernel launched just before it, so those
 * loads overlap that kernel's end.  q, out, logits, lse and the workspace are always accessed
 * only after that wait.  The flag is a permission: kernels that cannot use it ignore it.  A
 * call that sets it when the guarantee does not hold may read stale slots or lengths.
 * KVC_DECODE_BALANCE: with len, divide the work among thread blocks by the lengths rather than
 * by the capacity.  By default every (batch, KV head) pair is given cap slots' worth of blocks
 * and the slots past its length are skipped, which costs nothing when the lengths are close to
 * cap; when they differ widely (a ragged batch) the pairs' blocks finish at very different
 * times, and this flag balances them at the price of a scan of the lengths at the start of
 * every block.  Same results either way (the log-sum-exp merge order may differ).
 * KVC_DECODE_TEST_STARVE: a test hook with no counterpart on the pages, for exercising the
 * kernels' bounded waits without a GPU fault.  The kernel issues no cache loads at all, so its
 * first wait for a tile runs out after a short bounded spin; the block then stops (no loads
 * are in flight), every block still finishes, the workspace is left zeroed, and
 * kvc_device_status() reports KVC_DEV_TIMEOUT.  The outputs of such a call are undefined; the
 * next call without the flag is unaffected.  Every wait inside the decode kernels behaves the
 * same way when it gives up for a real reason (a lost arrival): the block stops issuing loads,
 * waits (bounded) for the loads it has in flight, and exits with invalid outputs.
 * Other bits must be 0 (KVC_ERR_INVALID_ARG). */
#define KVC_DECODE_KV_SETTLED 1u
#define KVC_DECODE_BALANCE 2u
#define KVC_DECODE_TEST_STARVE 0x80000000u
kvc_status kvc_decode_attn_ex(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                              const int32_t *len, int32_t n_valid, const kvc_rope *rope,
                              float scale, float *out, float *logits, int64_t logits_stride,
                              float *lse, void *ws, size_t ws_bytes, uint32_t flags,
                              void *stream);

/* Decode attention with ALiBi at in-cache positions over a StreamingLLM sink + ring cache
 * ([SINK] "como funciona", the ALiBi alternative to RoPE; kvc_alibi gives the layout and the
 * logit).  Same q, out, logits (indexed by slot), lse, workspace and flags as
 * kvc_decode_attn_ex with a rope descriptor; the new token is appended with
 * KVC_APPEND_RING first.  cap >= n_sink + window + 1 (else KVC_ERR_CAPACITY); alibi, its t and
 * slopes must not be NULL (KVC_ERR_INVALID_ARG). */
kvc_status kvc_decode_attn_alibi(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                                 const kvc_alibi *alibi, float scale, float *out, float *logits,
                                 int64_t logits_stride, float *lse, void *ws, size_t ws_bytes,
                                 uint32_t flags, void *stream);

/* ALiBi slopes, host: out[h] = 2^(-8 (h+1) / n_heads) for h < n_heads, the geometric sequence
 * of the ALiBi paper (Press et al., "Train Short, Test Long", 2022), defined there for a
 * power-of-two head count; other counts return KVC_ERR_INVALID_ARG (pass your own slopes).
 * out: host float[n_heads]. */
kvc_status kvc_alibi_slopes(int32_t n_heads, float *out);

/* Block-level eviction: append one token per sequence to a paged cache.
 * For every sequence b: if len[b] is a multiple of block_size, a block is popped from the free
 * stack, appended to the page table (n_blocks[b] += 1) with score 0; then the new token's keys
 * and values (every KV head) are written at offset len[b] % block_size of the last block and
 * len[b] += 1.  pos (nullable, with t): device int32[n_blocks][block_size], the text position
 * *t is stored at the token's place in its physical block (it moves with the block).
 * k_new, v_new: [batch][n_heads_kv][d_head], pool dtype, contiguous.
 * When several sequences pop in one call, which free id each receives depends on timing (the
 * page tables stay valid; their logical contents do not depend on it).  An empty free stack
 * records KVC_DEV_POOL_EMPTY and skips that sequence; inconsistent lengths record
 * KVC_DEV_BAD_LENGTH; a table entry outside the pool KVC_DEV_BAD_BLOCK. */
kvc_status kvc_paged_append(const kvc_block_pool *pool, const kvc_page_table *pt,
                            const kvc_free_pool *free_pool, const void *k_new, const void *v_new,
                            const int64_t *t, int32_t *pos, void *stream);

/* Decode attention over a paged cache ("Implementação prática...": FlashDecoding over the
 * blocks the page tables list): for every query head h of sequence b,
 *   out[b,h] = sum_j softmax_j(scale * q[b,h].k_j) v_j
 * over the len[b] tokens of its page table (KV head h / (n_heads_q / n_heads_kv)).
 * q, out, lse, flags and the workspace are those of kvc_decode_attn_ex, with
 * cap = max_blocks * block_size (kvc_decode_attn_workspace_bytes(batch, n_heads_q,
 * n_heads_kv, d_head, cap)); logits (nullable) are indexed by logical slot j = i*block_size +
 * offset, logits_stride >= cap.  KVC_DECODE_KV_SETTLED extends to the page tables. */
kvc_status kvc_decode_attn_paged(const void *q, int32_t n_heads_q, const kvc_block_pool *pool,
                                 const kvc_page_table *pt, float scale, float *out,
                                 float *logits, int64_t logits_stride, float *lse, void *ws,
                                 size_t ws_bytes, uint32_t flags, void *stream);

/* Block-level eviction at the end of the prompt (the one-shot prompt compression of [KVC] H2O,
 * at the block granularity of "Implementação prática em vLLM e SGLang").  For every sequence:
 * prompt block i holds tokens i*block_size .. min(seq_len, (i+1)*block_size) - 1 and scores
 *   Score(i) = sum over the n_heads_kv heads h and its tokens t of s[b][h][t]
 * (s: the prompt's per-token scores, e.g. the column sums kvc_h2o_prefill_select writes to
 * s_full; [batch][n_heads_kv][s_stride] fp32).  The recent_blocks newest blocks are kept with
 * the budget_blocks - recent_blocks highest-scoring older ones (equal scores keep the lower
 * index; a prompt of at most budget_blocks blocks is kept whole).  The kept blocks, in
 * ascending order, take consecutive page-table entries and one contiguous range of ids popped
 * from the free stack; their keys and values are copied from the prompt cache
 * ([batch][n_heads_kv][>= seq_len][d_head]) into the pool; the entries' scores are the block
 * scores; n_blocks and len are set (only the newest block may be partial).
 * The sequences' tables must be empty (n_blocks == 0; else KVC_DEV_BAD_LENGTH); too few free
 * blocks records KVC_DEV_POOL_EMPTY and leaves that sequence empty.
 * 1 <= recent_blocks <= budget_blocks <= max_blocks.  Three kernels: block scores, selection,
 * copy.  Workspace: kvc_block_prompt_select_workspace_bytes(), 256-byte aligned. */
size_t kvc_block_prompt_select_workspace_bytes(int32_t batch, int32_t seq_len,
                                               int32_t block_size, int32_t budget_blocks);
kvc_status kvc_block_prompt_select(const float *s, int64_t s_stride, const kvc_cache *prompt,
                                   int32_t seq_len, const kvc_block_pool *pool,
                                   const kvc_page_table *pt, const kvc_free_pool *free_pool,
                                   int32_t budget_blocks, int32_t recent_blocks, void *ws,
                                   size_t ws_bytes, void *stream);

/* Block-level eviction for one decode step ([KVC] "Implementação prática...": Score(block) =
 * sum over t in the block of s_t; the lowest-scoring blocks leave the page table for the free
 * pool, without copies).  For every sequence b:
 *   score[b,i] += sum over query heads h and tokens j of block i of exp(logits[b,h,j] - lse[b,h])
 *   (s_t is H2O's accumulated attention, summed over the heads: a block holds every head's
 *   keys and values of its tokens);
 *   if n_blocks[b] > budget_blocks: among the logical blocks 0 .. n_blocks[b]-recent_blocks-1
 *   the lowest score is released (equal scores: the newer block); the table and scores after
 *   it move down one entry, n_blocks[b] -= 1, len[b] -= block_size, and its physical id is
 *   pushed onto the free stack.  released (nullable): device int32[batch], the released
 *   logical index or -1.
 * logits: [batch][n_heads_q][logits_stride] from kvc_decode_attn_paged; lse: [batch][n_heads_q].
 * recent_blocks >= 1 (the partly filled block is never released), budget_blocks >= recent_blocks,
 * n_heads_q <= 1024, batch <= 65535.  Two kernels: the score update (one thread block per
 * table entry and sequence), then the release (one warp per sequence). */
kvc_status kvc_block_accumulate_evict(const float *logits, int64_t logits_stride,
                                      const float *lse, int32_t n_heads_q, int32_t block_size,
                                      const kvc_page_table *pt, const kvc_free_pool *free_pool,
                                      int32_t budget_blocks, int32_t recent_blocks,
                                      int32_t *released, void *stream);

/* KV bytes under DuoAttention, host: the memory formula of kvc_kv_bytes with seq_len tokens
 * per retrieval head and min(n_sink + window + 1, seq_len) per streaming head.  With 30 % of
 * the heads retrieving at 128k tokens the saving over kvc_kv_bytes is 70 % ([KVC] DuoAttention:
 * "economizando até 70% de VRAM"). */
uint64_t kvc_duo_kv_bytes(uint64_t n_layers, uint64_t n_retrieval, uint64_t n_streaming,
                          uint64_t d_head, uint64_t seq_len, uint64_t n_sink, uint64_t window,
                          uint64_t bytes_per_elem, uint64_t batch);

/* DuoAttention: append the new token of every KV head to its cache -- a retrieval head's row at
 * the tail of the full cache (slot len[b*n_retrieval+r], then len += 1; a full row records
 * KVC_DEV_TAIL_FULL and is skipped), a streaming head's row at the ring slot of text position
 * *duo->t (slot t for t < n_sink, else n_sink + (t - n_sink) mod (window + 1)).
 * k_new, v_new: [batch][n_heads_kv][d_head] in model head order, cache dtype, contiguous. */
kvc_status kvc_duo_append(const kvc_cache *full, int32_t *len, const kvc_cache *ring,
                          const kvc_duo *duo, const void *k_new, const void *v_new, void *stream);

/* DuoAttention decode ([KVC] DuoAttention with "FlashDecoding esparso"): one launch for both
 * kinds of heads.  Query head h (model order, KV head h / G) attends to all len (or n_valid)
 * slots of its retrieval cache row, or to the min(*t + 1, n_sink + window + 1) valid slots of
 * its ring.  q: [batch][n_heads_q][d_head]; out, lse as kvc_decode_attn; logits (nullable)
 * [batch][n_heads_q][logits_stride] indexed by the slot of the head's own cache,
 * logits_stride >= max(cap, n_sink + window + 1).  Slots of both caches must be dense
 * (stride_slot == d_head).  The work is divided by tiles of each kind, so the streaming heads
 * cost their buffer only.  Flags: KVC_DECODE_KV_SETTLED (as kvc_decode_attn_ex, covering len
 * and *t).  Workspace: kvc_decode_attn_duo_workspace_bytes(); zero-filled once, kept zeroed. */
size_t kvc_decode_attn_duo_workspace_bytes(int32_t batch, int32_t n_heads_q, int32_t n_heads_kv,
                                           int32_t d_head, int32_t cap, int32_t n_retrieval);
kvc_status kvc_decode_attn_duo(const void *q, int32_t n_heads_q, const kvc_cache *full,
                               const int32_t *len, int32_t n_valid, const kvc_cache *ring,
                               const kvc_duo *duo, float scale, float *out, float *logits,
                               int64_t logits_stride, float *lse, void *ws, size_t ws_bytes,
                               uint32_t flags, void *stream);

/* Decode attention without a caller workspace.  No counterpart on the pages: this is a
 * deployment convenience of this library.  Some callers cannot allocate device memory at the
 * point where they decode -- an engine that fixes its whole memory plan at start-up, a plugin
 * running inside another framework's stream capture (an allocation there would invalidate the
 * capture), a process held to an external memory budget -- so they cannot hand
 * kvc_decode_attn a workspace.  This entry point computes exactly what kvc_decode_attn
 * computes (same arguments without ws / ws_bytes) using a scratch array of 8 MiB that the
 * library keeps in its own device module: it allocates and frees nothing.
 * Limits and rules:
 *   - a problem whose workspace (kvc_decode_attn_workspace_bytes) exceeds 8 MiB is rejected
 *     with KVC_ERR_WORKSPACE before anything is launched;
 *   - the scratch is shared by every call in the process on that GPU and keeps the previous
 *     call's contents; each call clears the part that must start at zero on its own stream,
 *     but calls that may overlap on the GPU race on it -- order them on one stream;
 *   - the scratch's device address is looked up once per device by the first call made with
 *     that device current; make that first call before capturing a stream on that device. */
kvc_status kvc_decode_attn_noalloc(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                                   const int32_t *len, int32_t n_valid, const kvc_rope *rope,
                                   float scale, float *out, float *logits,
                                   int64_t logits_stride, float *lse, void *stream);

/* ---------------------------------------------------------------------------------------- */
/* H2O score accumulation and eviction for one decode step.  [KVC] "Heavy-Hitter Oracle (H2O)
 * e a esparsidade de cauda pesada": s_j = sum_t alpha_{t,j}; when the cache is over its
 * budget K, the L_local newest tokens are kept (recent quota) and, among the older tokens,
 * the one with the smallest s is evicted so that only the K_HH largest remain.
 * For every (b, h), h a head of an MHA cache (n_heads_q == n_heads_kv):
 *   score[j] += exp(logits[j] - lse)   for j < n_slots (alpha of this step, from
 *                                      kvc_decode_attn's logits and lse);
 *   if n_slots > budget: among slots with pos[j] <= *t - L_local, the smallest score is
 *   evicted (equal scores: the larger position), free_slot[b*H+h] = that slot.
 * score, pos: [batch][n_heads][stride] (fp32, int32); logits: [batch][n_heads][logits_stride];
 * lse: [batch][n_heads]; free_slot: device int32[batch*n_heads]. */
kvc_status kvc_h2o_accumulate_evict(const float *logits, int64_t logits_stride, const float *lse,
                                    float *score, int32_t *pos, int64_t stride,
                                    int32_t *free_slot, int32_t batch, int32_t n_heads,
                                    int32_t n_slots, const int64_t *t, int32_t L_local,
                                    int32_t budget, void *stream);

/* kvc_h2o_accumulate_evict for a grouped-query cache (n_heads_q = G * n_heads_kv; query head
 * h reads KV head h / G).  A cached row serves the G query heads of its KV head and is evicted
 * for all of them, so its score adds their attention ([KVC] H2O, s_j = sum_t alpha_{t,j}, over
 * the group -- a reading, the pages treat one head):
 *   score[b,kh,j] += sum_g exp(logits[b,kh*G+g,j] - lse[b,kh*G+g])   (g in head order);
 * then the eviction rule of kvc_h2o_accumulate_evict per (b, kh).  score, pos, free_slot are
 * per KV head ([batch][n_heads_kv][stride], device int32[batch*n_heads_kv]); logits and lse per
 * query head ([batch][n_heads_q][logits_stride], [batch][n_heads_q]), as kvc_decode_attn writes
 * them.  n_heads_q == n_heads_kv is kvc_h2o_accumulate_evict (same bits). */
kvc_status kvc_h2o_accumulate_evict_gqa(const float *logits, int64_t logits_stride,
                                        const float *lse, float *score, int32_t *pos,
                                        int64_t stride, int32_t *free_slot, int32_t batch,
                                        int32_t n_heads_q, int32_t n_heads_kv, int32_t n_slots,
                                        const int64_t *t, int32_t L_local, int32_t budget,
                                        void *stream);

/* H2O at the end of the prompt: full causal attention of the prompt (every query row), the
 * column sums s_j = sum_t alpha_{t,j}, then the one-shot compression to the budget: the
 * L_local newest positions plus the K_hh largest s among the older ones (equal scores keep
 * the lower position), ascending.
 * q: [batch][n_heads][seq_len][d_head] (prompt->dtype); prompt: keys (cap >= seq_len), MHA.
 * idx_out: [batch][n_heads][n_keep] int32 and score_out: [batch][n_heads][n_keep] fp32 (the
 * kept tokens' s), n_keep = min(seq_len, K_hh + L_local).  s_full (nullable):
 * [batch][n_heads][seq_len] fp32.  Workspace: kvc_h2o_prefill_workspace_bytes(). */
size_t kvc_h2o_prefill_workspace_bytes(int32_t batch, int32_t n_heads, int32_t d_head,
                                       int32_t seq_len);
kvc_status kvc_h2o_prefill_select(const void *q, const kvc_cache *prompt, int32_t seq_len,
                                  int32_t L_local, int32_t K_hh, float scale, int32_t *idx_out,
                                  float *score_out, float *s_full, void *ws, size_t ws_bytes,
                                  void *stream);

/* kvc_h2o_prefill_select for a grouped-query cache (n_heads_q = G * n_heads_kv; query head h
 * reads KV head h / G).  A cached row is kept or dropped for the whole group, so its score is
 * the sum over the group of each query head's causal column sum ([KVC] H2O, s_j = sum_t
 * alpha_{t,j}, added over the G heads in head order -- a reading, the pages treat one head);
 * then the same compression per (batch, KV head).  q: [batch][n_heads_q][seq_len][d_head]
 * (prompt->dtype, contiguous); idx_out, score_out: [batch][n_heads_kv][n_keep];
 * s_full (nullable): [batch][n_heads_kv][seq_len].  Each group member's heads are copied into
 * the workspace and scored by the one-head kernels.  Workspace:
 * kvc_h2o_prefill_gqa_workspace_bytes() (dtype: kvc_dtype of the prompt), 256-byte aligned. */
size_t kvc_h2o_prefill_gqa_workspace_bytes(int32_t batch, int32_t n_heads_kv, int32_t d_head,
                                           int32_t seq_len, int32_t dtype);
kvc_status kvc_h2o_prefill_select_gqa(const void *q, int32_t n_heads_q, const kvc_cache *prompt,
                                      int32_t seq_len, int32_t L_local, int32_t K_hh,
                                      float scale, int32_t *idx_out, float *score_out,
                                      float *s_full, void *ws, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
