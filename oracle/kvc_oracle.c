/*
 * kvc_oracle.c -- plain, slow CPU oracle for KV-cache compression and decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may load this library.  The product path (the CUDA library) never calls it and
 * shares no code, header, table or constant with it.
 *
 * Everything is computed as written on the source pages, in double precision, from the exact
 * stored input values (bf16 inputs are widened exactly by the caller).  Nothing is blocked,
 * fused or reordered.  Sources, cited by page title and section:
 *   [KVC]  "Compressão e Poda Dinâmica de KV Cache: StreamingLLM, SnapKV, PyramidKV e
 *           DuoAttention" (produtoramaxvision.com.br blog)
 *   [SINK] "attention sinks" encyclopedia entry (tonho.wtf diário)
 *   [KVCL] "O KV cache", lesson 7.2 of llmdeepdive (section "01 · Conceito")
 *
 * Where the pages leave a step open, the reading taken is stated beside the function; every
 * such reading is also listed in the design notes of the repository.
 *
 * Functions whose results no page fixes by example (the attention-quality numbers) are not
 * here: this file only computes what the kernels compute.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

/* Scratch for one call.  The oracle has no error path for a failed allocation: it stops the
 * process with a message rather than compute from a null pointer.                            */
static void *orc_alloc(size_t bytes)
{
    void *p = malloc(bytes > 0 ? bytes : 1);
    if (p == NULL) {
        fprintf(stderr, "kvc oracle: out of host memory (%zu bytes)\n", bytes);
        abort();
    }
    return p;
}

/* ------------------------------------------------------------------------------------------ */
/* KV memory model.  [KVC] "O gargalo de memória do KV Cache em contextos longos", equation
 * Memoria_KV = 2 x n_layers x n_heads_kv x d_head x seq_len x bytes_por_elemento x batch_size;
 * the same model in [KVCL] "01 · Conceito" (factor two for keys plus values).                 */
uint64_t orc_kv_bytes(uint64_t n_layers, uint64_t n_heads_kv, uint64_t d_head, uint64_t seq_len,
                      uint64_t bytes_per_elem, uint64_t batch)
{
    return 2ull * n_layers * n_heads_kv * d_head * seq_len * bytes_per_elem * batch;
}

/* ------------------------------------------------------------------------------------------ */
/* PyramidKV layer budgets.  [KVC] "Alocação piramidal com o PyramidKV":
 *     B_l = B_base + dB * (N_L - 1 - l) / (N_L - 1),    sum_l B_l = N_L * B_target.
 * The pages fix the linear form and the total; the ramp's steepness is given here as the ratio
 * r = B_0 / B_{N_L-1} = ratio_num / ratio_den.  The total then fixes
 *     B_base = 2 * B_target / (1 + r),   dB = (r - 1) * B_base,
 * so B_l = 2*B_target*(num*(N_L-1-l) + den*l) / ((num+den)*(N_L-1)), an exact rational.
 * Reading (the pages do not round): floor every B_l, then give +1 to the layers with the
 * largest remainders (ties: lower layer first) until the total is exactly N_L * B_target.
 * Returns 0, or -1 for invalid arguments.                                                     */
int orc_pyramid_budgets(int n_layers, int64_t b_target, int64_t ratio_num, int64_t ratio_den,
                        int64_t *out)
{
    if (n_layers <= 0 || b_target < 0 || ratio_num <= 0 || ratio_den <= 0) return -1;
    if (n_layers == 1) { out[0] = b_target; return 0; }
    const int64_t nl1 = n_layers - 1;
    /* B_base and dB over the common denominator Q = (num + den) * (N_L - 1). */
    const int64_t Q = (ratio_num + ratio_den) * nl1;
    const int64_t base_num = 2 * b_target * ratio_den * nl1;                 /* B_base * Q    */
    const int64_t delta_num = 2 * b_target * (ratio_num - ratio_den);        /* dB * Q/(N_L-1) */
    int64_t *rem = (int64_t *)orc_alloc(sizeof(int64_t) * (size_t)n_layers);
    int64_t total = 0;
    for (int l = 0; l < n_layers; ++l) {
        const int64_t num = base_num + delta_num * (nl1 - l);               /* B_l * Q      */
        out[l] = num / Q;
        rem[l] = num % Q;
        total += out[l];
    }
    int64_t deficit = (int64_t)n_layers * b_target - total;
    while (deficit > 0) {
        int best = -1;
        for (int l = 0; l < n_layers; ++l)
            if (rem[l] >= 0 && (best < 0 || rem[l] > rem[best])) best = l;
        out[best] += 1;
        rem[best] = -1;     /* each layer rounds up at most once */
        --deficit;
    }
    free(rem);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Rotary position embedding.  [SINK] "como funciona": keys are stored before rotation and the
 * positional rotation is applied at every decode step at the in-cache position.  The pages give
 * no RoPE formula; the reading taken is the usual half-split pairing: dimension i pairs with
 * i + D/2 and the pair is rotated by the angle pos * theta^(-2i/D).                          */
void orc_rope(int D, double theta, int64_t pos, const double *x, double *y)
{
    const int h = D / 2;
    for (int i = 0; i < h; ++i) {
        const double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)D);
        const double c = cos(ang), s = sin(ang);
        const double a = x[i], b = x[i + h];
        y[i] = a * c - b * s;
        y[i + h] = a * s + b * c;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Decode attention of one query over n cached keys.  [KVCL] "01 · Conceito": the new token's
 * query attends to the cached keys and mixes the cached values; this is exact causal attention.
 * [KVC] "O gargalo de memória...": each emitted token reads the whole cache (a GEMV).
 * Reading: scaled dot product with the caller's scale (1/sqrt(D)), max-subtracted softmax.
 *   logits (nullable): l_j = scale * q.k_j          lse (nullable): log sum_j exp(l_j)
 * n == 0 gives out = 0 and lse = -inf.                                                        */
void orc_attend(int n, int D, double scale, const double *q, const double *K, const double *V,
                double *out, double *logits, double *lse)
{
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n <= 0) {
        if (lse) *lse = -INFINITY;
        return;
    }
    double *l = (double *)orc_alloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * K[(size_t)j * D + d];
        l[j] = scale * acc;
        if (l[j] > m) m = l[j];
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) z += exp(l[j] - m);
    for (int j = 0; j < n; ++j) {
        const double p = exp(l[j] - m) / z;
        for (int d = 0; d < D; ++d) out[d] += p * V[(size_t)j * D + d];
    }
    if (logits) for (int j = 0; j < n; ++j) logits[j] = l[j];
    if (lse) *lse = m + log(z);
    free(l);
}

/* ------------------------------------------------------------------------------------------ */
/* StreamingLLM.  [KVC] "Attention Sinks e o StreamingLLM para fluxos contínuos": the cache is
 * the first S tokens (attention sinks, fixed) plus a rolling window of the W most recent tokens
 * in a circular buffer.  [SINK] "como funciona": positions are assigned inside the cache, not in
 * the text: a cache holding [0,1,2,3,6,7,8] while decoding the next token uses positions 0..7.
 *
 * Reading: when the token at text position t is decoded, it attends to the sinks that exist
 * (text positions < min(S, t+1)) and to the W tokens before it plus itself (text positions
 * max(S, t-W) .. t).  The in-cache position of each attended token is its rank in that set,
 * sorted by text position; the query's position is the rank of t (the last one).
 * Returns the count n and fills tok[n] (text positions) and cpos[n] (in-cache positions).     */
int orc_stream_window(int64_t t, int S, int W, int64_t *tok, int64_t *cpos, int64_t *qpos)
{
    int n = 0;
    const int64_t sink_end = t + 1 < S ? t + 1 : S;          /* sinks that exist so far   */
    for (int64_t a = 0; a < sink_end; ++a) { tok[n] = a; cpos[n] = n; ++n; }
    const int64_t recent_begin = t - W > S ? t - W : S;      /* window, token t included  */
    for (int64_t a = recent_begin; a <= t; ++a) { tok[n] = a; cpos[n] = n; ++n; }
    *qpos = cpos[n - 1];
    return n;
}

/* Physical slot of token a in a cache laid out as S sink slots followed by a ring of W+1
 * slots.  Reading: the ring holds the W window tokens plus the token being decoded, so the
 * slot written for token t is the one that held token t-W-1, which has just left the window. */
int64_t orc_stream_slot(int64_t a, int S, int W)
{
    if (a < S) return a;
    return S + (a - S) % (int64_t)(W + 1);
}

/* Decode of the token at text position t under StreamingLLM with RoPE at in-cache positions.
 * hist_k / hist_v hold the pre-rotation keys and the values of text positions 0..t (the token
 * itself included), q_pre the pre-rotation query.  Every attended key is rotated from its
 * stored value at its in-cache position, the query at its own in-cache position.             */
void orc_stream_decode(int64_t t, int S, int W, int D, double theta, double scale,
                       const double *q_pre, const double *hist_k, const double *hist_v,
                       double *out)
{
    const size_t cap = (size_t)(S + W + 1);
    int64_t *tok = (int64_t *)orc_alloc(sizeof(int64_t) * cap);
    int64_t *cpos = (int64_t *)orc_alloc(sizeof(int64_t) * cap);
    int64_t qpos;
    const int n = orc_stream_window(t, S, W, tok, cpos, &qpos);
    double *Kr = (double *)orc_alloc(sizeof(double) * (size_t)n * D);
    double *Vs = (double *)orc_alloc(sizeof(double) * (size_t)n * D);
    double *qr = (double *)orc_alloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < n; ++j) {
        orc_rope(D, theta, cpos[j], hist_k + (size_t)tok[j] * D, Kr + (size_t)j * D);
        memcpy(Vs + (size_t)j * D, hist_v + (size_t)tok[j] * D, sizeof(double) * (size_t)D);
    }
    orc_rope(D, theta, qpos, q_pre, qr);
    orc_attend(n, D, scale, qr, Kr, Vs, out, NULL, NULL);
    free(tok); free(cpos); free(Kr); free(Vs); free(qr);
}

/* StreamingLLM with ALiBi.  [SINK] "como funciona": under ALiBi the linear bias is applied
 * continuously at the in-cache positions (no jump over the evicted tokens), so distances never
 * exceed the cache length.  The pages print no ALiBi formula; the reading taken is the usual
 * one: the logit of the query at in-cache position p_q against a key at in-cache position p_k
 * is scale * q.k - slope * (p_q - p_k), with `slope` the head's constant (given by the caller).
 * Keys are used as stored (no rotation).  The attended set and the positions are those of
 * orc_stream_window.  logits (nullable): per attended token in rank order; lse (nullable).    */
void orc_stream_decode_alibi(int64_t t, int S, int W, int D, double slope, double scale,
                             const double *q, const double *hist_k, const double *hist_v,
                             double *out, double *logits, double *lse)
{
    const size_t cap = (size_t)(S + W + 1);
    int64_t *tok = (int64_t *)orc_alloc(sizeof(int64_t) * cap);
    int64_t *cpos = (int64_t *)orc_alloc(sizeof(int64_t) * cap);
    int64_t qpos;
    const int n = orc_stream_window(t, S, W, tok, cpos, &qpos);
    double *l = (double *)orc_alloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * hist_k[(size_t)tok[j] * D + d];
        l[j] = scale * acc - slope * (double)(qpos - cpos[j]);
        if (l[j] > m) m = l[j];
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) z += exp(l[j] - m);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int j = 0; j < n; ++j) {
        const double p = exp(l[j] - m) / z;
        for (int d = 0; d < D; ++d) out[d] += p * hist_v[(size_t)tok[j] * D + d];
    }
    if (logits) for (int j = 0; j < n; ++j) logits[j] = l[j];
    if (lse) *lse = m + log(z);
    free(tok); free(cpos); free(l);
}

/* ------------------------------------------------------------------------------------------ */
/* Top-k with the tie rule used throughout: keep the k largest scores, equal scores keep the
 * lower index; the kept indices are returned in ascending order (original order preserved).
 * A library sort serves as the step.                                                          */
typedef struct { double v; int32_t i; } orc_scored;

static int orc_cmp_desc(const void *pa, const void *pb)
{
    const orc_scored *a = (const orc_scored *)pa, *b = (const orc_scored *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

static int orc_cmp_int(const void *pa, const void *pb)
{
    const int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

void orc_topk_ascending(int n, int k, const double *score, int32_t *idx)
{
    if (k > n) k = n;
    if (k <= 0) return;
    orc_scored *e = (orc_scored *)orc_alloc(sizeof(orc_scored) * (size_t)n);
    for (int i = 0; i < n; ++i) { e[i].v = score[i]; e[i].i = i; }
    qsort(e, (size_t)n, sizeof(orc_scored), orc_cmp_desc);
    for (int j = 0; j < k; ++j) idx[j] = e[j].i;
    qsort(idx, (size_t)k, sizeof(int32_t), orc_cmp_int);
    free(e);
}

/* ------------------------------------------------------------------------------------------ */
/* SnapKV.  [KVC] "SnapKV e a seleção de contexto no prefill", steps 1-4:
 *   1. observation window: the last L_obs prompt queries attend to the prompt (A_{h,L_obs,N});
 *   2. mean over the window: s_i = (1/L_obs) sum_t A_{h,t,i};
 *   3. 1-D pooling with kernel 5 smooths the scores;
 *   4. per-head top-k keeps the positions with the largest values.
 *
 * Steps 1-2 for one query head.  Qobs holds the L_obs window queries (text positions
 * N-L_obs .. N-1), K the N prompt keys.  Reading: causal attention inside the window (query t
 * sees keys at text positions <= its own), scaled by `scale`; the mean divides every column by
 * L_obs.  s receives all N columns (the window's own columns included; they sum with the
 * prefix to 1 per query head).                                                                */
void orc_snapkv_obs_scores(int L_obs, int N, int D, double scale, const double *Qobs,
                           const double *K, double *s)
{
    double *row = (double *)orc_alloc(sizeof(double) * (size_t)N);
    for (int i = 0; i < N; ++i) s[i] = 0.0;
    for (int t = 0; t < L_obs; ++t) {
        const int p = N - L_obs + t;            /* text position of this query */
        double m = -INFINITY;
        for (int i = 0; i <= p; ++i) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += Qobs[(size_t)t * D + d] * K[(size_t)i * D + d];
            row[i] = scale * acc;
            if (row[i] > m) m = row[i];
        }
        double z = 0.0;
        for (int i = 0; i <= p; ++i) z += exp(row[i] - m);
        for (int i = 0; i <= p; ++i) s[i] += exp(row[i] - m) / z;   /* A_{h,t,i} */
    }
    for (int i = 0; i < N; ++i) s[i] /= (double)L_obs;
    free(row);
}

/* Step 3.  Reading: average pooling, odd kernel k, stride 1, zero padding (k-1)/2 on each side,
 * divisor always k ("Conv1D" with a box kernel), over the n prefix scores only.              */
void orc_pool1d(int n, int k, const double *s, double *p)
{
    const int r = (k - 1) / 2;
    for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int j = i - r; j <= i + r; ++j)
            if (j >= 0 && j < n) acc += s[j];
        p[i] = acc / (double)k;
    }
}

/* Whole selection for one KV head whose query group has G heads.  Reading: the G pooled score
 * rows are reduced by max (one top-k per KV head); the budget counts the observation window,
 * which is always kept; k = budget - L_obs prefix positions are chosen; the kept prefix
 * indices (ascending) are followed by the window N-L_obs .. N-1.  budget >= N keeps all.
 * Qobs: [G][L_obs][D].  s_out (nullable): [G][N] column means; score_out (nullable): [N-L_obs].
 * Returns the number of kept indices, or -1 for invalid arguments.                          */
int orc_snapkv_select(int G, int L_obs, int N, int D, int pool_k, int budget, double scale,
                      const double *Qobs, const double *K, int32_t *idx, double *s_out,
                      double *score_out)
{
    if (G <= 0 || L_obs <= 0 || L_obs > N || pool_k <= 0 || (pool_k % 2) == 0 ||
        budget < L_obs)
        return -1;
    const int n = N - L_obs;
    double *s = (double *)orc_alloc(sizeof(double) * (size_t)G * N);
    double *p = (double *)orc_alloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *score = (double *)orc_alloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int g = 0; g < G; ++g)
        orc_snapkv_obs_scores(L_obs, N, D, scale, Qobs + (size_t)g * L_obs * D, K,
                              s + (size_t)g * N);
    for (int i = 0; i < n; ++i) score[i] = -INFINITY;
    for (int g = 0; g < G; ++g) {
        orc_pool1d(n, pool_k, s + (size_t)g * N, p);
        for (int i = 0; i < n; ++i)
            if (p[i] > score[i]) score[i] = p[i];
    }
    int kept;
    if (budget >= N) {
        for (int i = 0; i < N; ++i) idx[i] = i;
        kept = N;
    } else {
        const int k = budget - L_obs;
        orc_topk_ascending(n, k, score, idx);
        for (int t = 0; t < L_obs; ++t) idx[k + t] = n + t;
        kept = budget;
    }
    if (s_out) memcpy(s_out, s, sizeof(double) * (size_t)G * N);
    if (score_out) memcpy(score_out, score, sizeof(double) * (size_t)n);
    free(s); free(p); free(score);
    return kept;
}

/* Steps 3-4 replayed in single precision from given fp32 column means (the GPU's own), with the
 * arithmetic order fixed: the pooled sum adds s[i-r] .. s[i+r] left to right in fp32 (terms
 * outside the prefix are skipped), then divides by k in fp32; max over the group; top-k as
 * above on the fp32 values.  s: [G][n_prefix] (row stride n_prefix).  This is the reference for
 * the bit-exact index contract; it takes the same decisions as the kernels given their own
 * scores, since both sides decide in fp32.                                                    */
int orc_snapkv_stage_f32(int G, int n_prefix, int pool_k, int L_obs, int budget,
                         const float *s, int32_t *idx)
{
    const int N = n_prefix + L_obs;
    if (budget < L_obs || pool_k <= 0 || (pool_k % 2) == 0) return -1;
    if (budget >= N) {
        for (int i = 0; i < N; ++i) idx[i] = i;
        return N;
    }
    const int r = (pool_k - 1) / 2;
    double *score = (double *)orc_alloc(sizeof(double) * (size_t)(n_prefix > 0 ? n_prefix : 1));
    for (int i = 0; i < n_prefix; ++i) {
        float best = -INFINITY;
        for (int g = 0; g < G; ++g) {
            const float *sg = s + (size_t)g * n_prefix;
            float acc = 0.0f;
            for (int j = i - r; j <= i + r; ++j)
                if (j >= 0 && j < n_prefix) acc = acc + sg[j];
            const float pooled = acc / (float)pool_k;
            if (pooled > best) best = pooled;
        }
        score[i] = (double)best;   /* exact widening: order is unchanged */
    }
    const int k = budget - L_obs;
    orc_topk_ascending(n_prefix, k, score, idx);
    for (int t = 0; t < L_obs; ++t) idx[k + t] = n_prefix + t;
    free(score);
    return budget;
}

/* ------------------------------------------------------------------------------------------ */
/* H2O.  [KVC] "Heavy-Hitter Oracle (H2O) e a esparsidade de cauda pesada":
 *   s_j = sum_t alpha_{t,j}  (attention received by token j, accumulated over steps t);
 *   when the cache reaches its budget K: a guaranteed quota for the L_local newest tokens, the
 *   historical tokens ordered by s_j keep only the K_HH largest, the rest are freed.
 *
 * Prompt scores.  Reading: the prompt is processed by full causal attention; s_j sums the
 * attention column j over all N prompt queries.  Q, K: [N][D]; s: [N].                       */
void orc_h2o_prompt_scores(int N, int D, double scale, const double *Q, const double *K,
                           double *s)
{
    double *row = (double *)orc_alloc(sizeof(double) * (size_t)N);
    for (int j = 0; j < N; ++j) s[j] = 0.0;
    for (int t = 0; t < N; ++t) {
        double m = -INFINITY;
        for (int j = 0; j <= t; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += Q[(size_t)t * D + d] * K[(size_t)j * D + d];
            row[j] = scale * acc;
            if (row[j] > m) m = row[j];
        }
        double z = 0.0;
        for (int j = 0; j <= t; ++j) z += exp(row[j] - m);
        for (int j = 0; j <= t; ++j) s[j] += exp(row[j] - m) / z;   /* alpha_{t,j} */
    }
    free(row);
}

/* Prompt scores of a grouped-query KV head.  Reading (as for the decode steps of a grouped
 * cache): a cached row serves the G query heads of its KV head and is kept or dropped for all
 * of them, so its score is the sum over the group of each query head's column sum.
 * Q: [G][N][D] (the group's query heads); K: [N][D]; s: [N].                                 */
void orc_h2o_prompt_scores_group(int G, int N, int D, double scale, const double *Q,
                                 const double *K, double *s)
{
    double *sg = (double *)orc_alloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int j = 0; j < N; ++j) s[j] = 0.0;
    for (int g = 0; g < G; ++g) {
        orc_h2o_prompt_scores(N, D, scale, Q + (size_t)g * N * D, K, sg);
        for (int j = 0; j < N; ++j) s[j] += sg[j];
    }
    free(sg);
}

/* One-shot compression at the end of the prompt.  Reading: the L_local newest prompt positions
 * are kept (recent quota), the K_HH largest s among the older positions are kept (ties: lower
 * position), the kept positions are returned ascending.  If N <= L_local + K_HH everything is
 * kept.  Returns the count.                                                                   */
int orc_h2o_prompt_select(int N, int L_local, int K_hh, const double *s, int32_t *idx)
{
    if (N <= L_local + K_hh) {
        for (int j = 0; j < N; ++j) idx[j] = j;
        return N;
    }
    const int n_old = N - L_local;
    orc_topk_ascending(n_old, K_hh, s, idx);
    for (int j = 0; j < L_local; ++j) idx[K_hh + j] = n_old + j;
    return K_hh + L_local;
}

/* One decode step over the current cache.  The slots hold the retained tokens and the token
 * being decoded (already appended with pos = t and s = 0).  Reading of the step order: attend
 * over every slot (self included), add each slot's attention to its score, then, if the cache
 * holds more than `budget` tokens, evict one token among the historical ones (pos <= t-L_local,
 * i.e. outside the recent quota): the lowest score, equal scores evict the larger position.
 * Returns the evicted slot or -1.  alpha (nullable): the step's attention weights per slot.   */
int orc_h2o_step(int n_slots, int D, double scale, const double *q, const double *K,
                 const double *V, const int64_t *pos, double *s, int64_t t, int L_local,
                 int budget, double *out, double *alpha)
{
    double *l = (double *)orc_alloc(sizeof(double) * (size_t)(n_slots > 0 ? n_slots : 1));
    double lse;
    orc_attend(n_slots, D, scale, q, K, V, out, l, &lse);
    for (int j = 0; j < n_slots; ++j) {
        const double a = exp(l[j] - lse);
        s[j] += a;
        if (alpha) alpha[j] = a;
    }
    free(l);
    if (n_slots <= budget) return -1;
    int ev = -1;
    for (int j = 0; j < n_slots; ++j) {
        if (pos[j] > t - L_local) continue;
        if (ev < 0 || s[j] < s[ev] || (s[j] == s[ev] && pos[j] > pos[ev])) ev = j;
    }
    return ev;
}

/* H2O on a grouped-query cache.  [KVC] H2O fixes s_j = sum over steps of alpha_j for one
 * head; with grouped-query attention ([KVCL] "01 · Conceito": several query heads share one
 * KV head) a cached row serves G query heads and can only be evicted for all of them.
 * Reading: the row's score is the sum over the group of its query heads' attention,
 * s_j += sum_g alpha_{g,j}; the eviction rule is that of orc_h2o_step.  q: [G][D];
 * out: [G][D].  Returns the evicted slot or -1.                                              */
int orc_h2o_step_group(int G, int n_slots, int D, double scale, const double *q,
                       const double *K, const double *V, const int64_t *pos, double *s,
                       int64_t t, int L_local, int budget, double *out)
{
    double *l = (double *)orc_alloc(sizeof(double) * (size_t)(n_slots > 0 ? n_slots : 1));
    for (int g = 0; g < G; ++g) {
        double lse;
        orc_attend(n_slots, D, scale, q + (size_t)g * D, K, V, out + (size_t)g * D, l, &lse);
        for (int j = 0; j < n_slots; ++j) s[j] += exp(l[j] - lse);
    }
    free(l);
    if (n_slots <= budget) return -1;
    int ev = -1;
    for (int j = 0; j < n_slots; ++j) {
        if (pos[j] > t - L_local) continue;
        if (ev < 0 || s[j] < s[ev] || (s[j] == s[ev] && pos[j] > pos[ev])) ev = j;
    }
    return ev;
}

/* The eviction decision alone, in fp32, on given fp32 scores (the GPU's own). */
int orc_h2o_evict_f32(int n_slots, const float *s, const int64_t *pos, int64_t t, int L_local)
{
    int ev = -1;
    for (int j = 0; j < n_slots; ++j) {
        if (pos[j] > t - L_local) continue;
        if (ev < 0 || s[j] < s[ev] || (s[j] == s[ev] && pos[j] > pos[ev])) ev = j;
    }
    return ev;
}

/* ------------------------------------------------------------------------------------------ */
/* Block-level eviction.  [KVC] "Implementação prática em vLLM e SGLang": the cache lives in
 * physical blocks of 16 or 32 tokens reached through a page table; the engine rates a whole
 * block by the sum of its tokens' importance, Score(block) = sum over t in the block of s_t,
 * and when memory runs out the scheduler releases the lowest-scoring blocks from the page
 * table; they return to the free pool without copying any data.
 * Readings (the pages leave these open):
 *   - s_t is H2O's accumulated attention of token t ([KVC] H2O: s_j = sum over steps of
 *     alpha), summed over the query heads: a block holds every head's keys and values of its
 *     tokens, so only a per-token total can rank it;
 *   - step order as for H2O: the new token is appended (opening a new block when the last one
 *     is full), every head attends over all cached tokens (itself included), each block's score
 *     grows by its share of this step's attention, and then, if the sequence holds more than
 *     budget_blocks blocks, one block is released;
 *   - the recent_blocks newest blocks (the partly filled one included) are never released,
 *     the counterpart of H2O's recent quota; among the others the lowest score goes, equal
 *     scores releasing the newer block (the larger index; the older one is kept, as in H2O).
 *
 * One decode step of one sequence, computed as written.  The cache holds n_tok tokens in
 * page-table order; block i holds tokens i*bs .. min(n_tok, (i+1)*bs) - 1.  Query head h
 * (h < Hq) reads KV head h / (Hq / Hkv).  q: [Hq][D]; K, V: [Hkv][n_tok][D] (tokens gathered
 * in table order); score: [nb] block scores, updated in place.  out: [Hq][D].
 * Returns the index of the released block, or -1.                                             */
int orc_block_step(int Hq, int Hkv, int D, int n_tok, int bs, double scale, const double *q,
                   const double *K, const double *V, double *score, int budget_blocks,
                   int recent_blocks, double *out)
{
    const int G = Hq / Hkv;
    const int nb = (n_tok + bs - 1) / bs;
    double *l = (double *)orc_alloc(sizeof(double) * (size_t)(n_tok > 0 ? n_tok : 1));
    for (int h = 0; h < Hq; ++h) {
        const int kh = h / G;
        double lse;
        orc_attend(n_tok, D, scale, q + (size_t)h * D, K + (size_t)kh * n_tok * D,
                   V + (size_t)kh * n_tok * D, out + (size_t)h * D, l, &lse);
        for (int j = 0; j < n_tok; ++j) score[j / bs] += exp(l[j] - lse);
    }
    free(l);
    if (nb <= budget_blocks) return -1;
    int ev = -1;
    for (int i = 0; i < nb - recent_blocks; ++i)
        if (ev < 0 || score[i] <= score[ev]) ev = i;     /* <=: equal scores take the newer */
    return ev;
}

/* The release decision alone, in fp32, on given fp32 block scores (the GPU's own). */
int orc_block_evict_f32(int nb, const float *score, int budget_blocks, int recent_blocks)
{
    if (nb <= budget_blocks) return -1;
    int ev = -1;
    for (int i = 0; i < nb - recent_blocks; ++i)
        if (ev < 0 || score[i] <= score[ev]) ev = i;
    return ev;
}

/* ------------------------------------------------------------------------------------------ */
/* DuoAttention, inference half.  [KVC] "Decomposição funcional com o DuoAttention": retrieval
 * heads (gamma = 1, 20-30 % of the heads) keep the full KV cache; streaming heads (gamma = 0)
 * keep a constant buffer of 64 local tokens and 4 attention sinks.  The mask gamma comes from a
 * calibration (training), out of scope here: it is an input.
 * Readings: a streaming head attends to the set StreamingLLM attends to (orc_stream_window: the
 * n_sink first tokens, the `window` tokens before t and t itself); no positional term is added
 * (keys as stored, already position-encoded); a retrieval head attends to tokens 0..t.
 * hist_k, hist_v: [t+1][D], the head's keys and values of text positions 0..t.              */
void orc_duo_decode(int retrieval, int64_t t, int S, int W, int D, double scale,
                    const double *q, const double *hist_k, const double *hist_v, double *out)
{
    if (retrieval) {
        orc_attend((int)(t + 1), D, scale, q, hist_k, hist_v, out, NULL, NULL);
        return;
    }
    const size_t cap = (size_t)(S + W + 1);
    int64_t *tok = (int64_t *)orc_alloc(sizeof(int64_t) * cap);
    int64_t *cpos = (int64_t *)orc_alloc(sizeof(int64_t) * cap);
    int64_t qpos;
    const int n = orc_stream_window(t, S, W, tok, cpos, &qpos);
    double *K = (double *)orc_alloc(sizeof(double) * (size_t)n * D);
    double *V = (double *)orc_alloc(sizeof(double) * (size_t)n * D);
    for (int j = 0; j < n; ++j) {
        memcpy(K + (size_t)j * D, hist_k + (size_t)tok[j] * D, sizeof(double) * (size_t)D);
        memcpy(V + (size_t)j * D, hist_v + (size_t)tok[j] * D, sizeof(double) * (size_t)D);
    }
    orc_attend(n, D, scale, q, K, V, out, NULL, NULL);
    free(tok); free(cpos); free(K); free(V);
}

/* KV bytes under DuoAttention: the memory formula of [KVC] "O gargalo de memória..." with the
 * sequence length replaced per head: seq_len tokens for a retrieval head, at most
 * n_sink + window + 1 for a streaming head (its buffer, the token being decoded included).   */
uint64_t orc_duo_kv_bytes(uint64_t n_layers, uint64_t n_retrieval, uint64_t n_streaming,
                          uint64_t d_head, uint64_t seq_len, uint64_t n_sink, uint64_t window,
                          uint64_t bytes_per_elem, uint64_t batch)
{
    uint64_t buf = n_sink + window + 1;
    if (buf > seq_len) buf = seq_len;
    return 2ull * n_layers * d_head * bytes_per_elem * batch *
           (n_retrieval * seq_len + n_streaming * buf);
}

/* Block-level eviction at the end of the prompt: the prompt's tokens are grouped into blocks
 * of bs (block i holds tokens i*bs .. min(N, (i+1)*bs) - 1), each block is rated by
 * Score(block) = sum over its tokens t and the H heads of s[h][t] (the prompt's accumulated
 * attention, [KVC] H2O column sums), and the cache keeps the recent_blocks newest blocks plus
 * the budget_blocks - recent_blocks highest-scoring older ones (equal scores keep the lower
 * index, as for tokens), in ascending order.  Reading: the one-shot prompt compression of H2O
 * ([KVC] H2O), taken at block granularity as "Implementação prática em vLLM e SGLang" rates
 * blocks.  s: [H][N]; score_blk (nullable): [nblk] block scores; keep: [nblk] ascending kept
 * block indices.  Returns the number kept.                                                   */
int orc_block_prompt_select(int H, int N, int bs, const double *s, int budget_blocks,
                            int recent_blocks, double *score_blk, int32_t *keep)
{
    const int nblk = (N + bs - 1) / bs;
    double *sc = (double *)orc_alloc(sizeof(double) * (size_t)(nblk > 0 ? nblk : 1));
    for (int i = 0; i < nblk; ++i) sc[i] = 0.0;
    for (int h = 0; h < H; ++h)
        for (int t = 0; t < N; ++t) sc[t / bs] += s[(size_t)h * N + t];
    if (score_blk) for (int i = 0; i < nblk; ++i) score_blk[i] = sc[i];
    int n_keep;
    if (nblk <= budget_blocks) {
        for (int i = 0; i < nblk; ++i) keep[i] = i;
        n_keep = nblk;
    } else {
        const int recent = recent_blocks < nblk ? recent_blocks : nblk;
        const int n_old = nblk - recent;
        const int k_old = budget_blocks - recent;
        orc_topk_ascending(n_old, k_old, sc, keep);
        for (int j = 0; j < recent; ++j) keep[k_old + j] = n_old + j;
        n_keep = k_old + recent;
    }
    free(sc);
    return n_keep;
}
