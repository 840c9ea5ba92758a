// api.cu -- the C ABI of libkvc (include/kvc.h): argument validation, planning, dispatch.
//
// Every entry point validates on the host and returns a kvc_status before launching anything;
// nothing here allocates device memory or synchronises (except kvc_device_status).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/kvc.h"
#include "internal.h"

namespace {

thread_local std::string g_last_error;

// Device-side range-check code (KVC_DEV_*); kernels receive its address.
__device__ int32_t g_dev_code;

constexpr int kMaxDevices = 64;
// polls before a wait gives up under KVC_DECODE_TEST_STARVE (a short, bounded stall)
constexpr uint32_t kTestSpinLimit = 1024;
std::mutex g_mutex;
int32_t *g_code_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

kvc_status fail(kvc_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
kvc_status fail(kvc_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

kvc_status ok()
{
    g_last_error.clear();
    return KVC_OK;
}

kvc_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(KVC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Per-device facts, looked up once per device.
kvc_status device_info(int32_t **code_ptr, int *n_sm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(KVC_ERR_CUDA, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_code_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dev_code);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device code)");
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_code_ptr[dev] = static_cast<int32_t *>(p);
        g_sm_count[dev] = sms;
    }
    if (code_ptr) *code_ptr = g_code_ptr[dev];
    if (n_sm) *n_sm = g_sm_count[dev];
    return KVC_OK;
}

// SM count for workspace sizing; 152 (GB300) when no device is usable from this thread.
int sm_count_or_default()
{
    int n_sm = 0;
    if (device_info(nullptr, &n_sm) != KVC_OK || n_sm <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n_sm;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

int elem_bytes(int dtype) { return dtype == KVC_BF16 ? 2 : 4; }

kvc_status check_cache(const kvc_cache *c, const char *name, bool need_v)
{
    if (c == nullptr) return fail(KVC_ERR_INVALID_ARG, "%s: null cache descriptor", name);
    if (c->k == nullptr || (need_v && c->v == nullptr))
        return fail(KVC_ERR_INVALID_ARG, "%s: null k/v pointer", name);
    if (c->dtype != KVC_F32 && c->dtype != KVC_BF16)
        return fail(KVC_ERR_INVALID_ARG, "%s: dtype %d", name, c->dtype);
    if (c->batch <= 0 || c->n_heads_kv <= 0 || c->cap < 0)
        return fail(KVC_ERR_SHAPE, "%s: batch %d heads %d cap %d", name, c->batch,
                    c->n_heads_kv, c->cap);
    if (c->d_head != 64 && c->d_head != 128 && c->d_head != 256)
        return fail(KVC_ERR_SHAPE, "%s: d_head %d (supported: 64, 128, 256)", name, c->d_head);
    if (c->stride_slot < c->d_head || c->stride_b < 0 || c->stride_h < 0)
        return fail(KVC_ERR_SHAPE, "%s: strides", name);
    const int64_t eb = elem_bytes(c->dtype);
    if (!aligned16(c->k) || (need_v && !aligned16(c->v)) || (c->stride_slot * eb) % 16 ||
        (c->stride_h * eb) % 16 || (c->stride_b * eb) % 16)
        return fail(KVC_ERR_ALIGN, "%s: pointers and strides must be 16-byte aligned", name);
    return KVC_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

namespace kvc {

void set_last_error(const char *msg) { g_last_error = msg; }

DecodePlan decode_plan(int B, int Hq, int Hkv, int D, int cap, int n_sm, int seg_pairs)
{
    // The decode kernel divides the P = B*Hkv pairs' slot tiles evenly over at most C = 2*n_sm
    // persistent blocks (two per SM).  A pair's tiles then meet at most floor(C / P) + 2
    // blocks, which bounds the partial states kept per pair; the bound does not depend on the
    // tile size (so not on the element type either).
    (void)cap;
    DecodePlan pl{};
    const long long pairs = (long long)B * Hkv;
    const long long ctas = 2LL * (n_sm > 0 ? n_sm : 152);
    const long long alike = seg_pairs > 0 && seg_pairs < pairs ? seg_pairs : pairs;
    long long max_seg = ctas / alike + 2;
    if (max_seg > ctas) max_seg = ctas;
    pl.max_seg = (int)max_seg;
    const size_t G = (size_t)(Hq / Hkv);
    pl.off_o = 0;
    pl.off_ml = align256(pl.off_o + (size_t)pairs * max_seg * G * D * sizeof(float));
    pl.off_cnt = align256(pl.off_ml + (size_t)pairs * max_seg * G * 2 * sizeof(float));
    pl.bytes = align256(pl.off_cnt + (size_t)pairs * sizeof(int32_t));
    return pl;
}

}  // namespace kvc

// ==========================================================================================
extern "C" {

const char *kvc_last_error(void) { return g_last_error.c_str(); }

kvc_status kvc_device_status(void *stream, int32_t *code)
{
    if (code == nullptr) return fail(KVC_ERR_INVALID_ARG, "kvc_device_status: null code");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    kvc_status st = device_info(nullptr, nullptr);
    if (st != KVC_OK) return st;
    int32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, g_dev_code, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
    const int32_t zero = 0;
    e = cudaMemcpyToSymbol(g_dev_code, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    *code = v;
    if (v != 0) return fail(KVC_ERR_DEVICE, "device range check fired: code %d", v);
    return ok();
}

uint64_t kvc_kv_bytes(uint64_t n_layers, uint64_t n_heads_kv, uint64_t d_head, uint64_t seq_len,
                      uint64_t bytes_per_elem, uint64_t batch)
{
    // Keys and values (factor 2) for every layer, KV head, head dimension, position, batch row.
    return 2ull * n_layers * n_heads_kv * d_head * seq_len * bytes_per_elem * batch;
}

kvc_status kvc_pyramid_budgets(int32_t n_layers, int64_t b_target, int64_t ratio_num,
                               int64_t ratio_den, int64_t *out)
{
    if (out == nullptr || n_layers <= 0 || b_target < 0 || ratio_num <= 0 || ratio_den <= 0)
        return fail(KVC_ERR_INVALID_ARG, "kvc_pyramid_budgets: invalid arguments");
    if (n_layers == 1) {
        out[0] = b_target;
        return ok();
    }
    // B_l * (num+den)*(N_L-1) = 2*b_target*(num*(N_L-1-l) + den*l), exact in integers.
    const int64_t last = n_layers - 1;
    const int64_t denom = (ratio_num + ratio_den) * last;
    std::vector<std::pair<int64_t, int32_t>> frac(n_layers);
    int64_t assigned = 0;
    for (int32_t l = 0; l < n_layers; ++l) {
        const int64_t numer = 2 * b_target * (ratio_num * (last - l) + ratio_den * l);
        out[l] = numer / denom;
        frac[l] = {numer % denom, l};
        assigned += out[l];
    }
    std::sort(frac.begin(), frac.end(), [](const auto &a, const auto &b) {
        return a.first != b.first ? a.first > b.first : a.second < b.second;
    });
    const int64_t missing = (int64_t)n_layers * b_target - assigned;
    for (int64_t i = 0; i < missing; ++i) out[frac[(size_t)i].second] += 1;
    return ok();
}

kvc_status kvc_rope_table(int32_t n_pos, int32_t d_head, double theta, float *out)
{
    if (out == nullptr || n_pos < 0 || d_head <= 0 || (d_head % 2) || !(theta > 0))
        return fail(KVC_ERR_INVALID_ARG, "kvc_rope_table: invalid arguments");
    const int half = d_head / 2;
    std::vector<double> inv_freq(half);
    for (int i = 0; i < half; ++i) inv_freq[i] = std::pow(theta, -2.0 * i / d_head);
    for (int32_t p = 0; p < n_pos; ++p)
        for (int i = 0; i < half; ++i) {
            const double a = (double)p * inv_freq[i];
            out[(size_t)p * d_head + i] = (float)std::cos(a);
            out[(size_t)p * d_head + half + i] = (float)std::sin(a);
        }
    return ok();
}

// ------------------------------------------------------------------------------------------
size_t kvc_decode_attn_workspace_bytes(int32_t batch, int32_t n_heads_q, int32_t n_heads_kv,
                                       int32_t d_head, int32_t cap)
{
    if (batch <= 0 || n_heads_q <= 0 || n_heads_kv <= 0 || d_head <= 0 || cap < 0) return 0;
    return kvc::decode_plan(batch, n_heads_q, n_heads_kv, d_head, cap, sm_count_or_default())
        .bytes;
}

kvc_status kvc_decode_attn(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                           const int32_t *len, int32_t n_valid, const kvc_rope *rope,
                           float scale, float *out, float *logits, int64_t logits_stride,
                           float *lse, void *ws, size_t ws_bytes, void *stream)
{
    return kvc_decode_attn_ex(q, n_heads_q, cache, len, n_valid, rope, scale, out, logits,
                              logits_stride, lse, ws, ws_bytes, 0u, stream);
}

// Paged decode: the page tables of a paged cache (pool described by the kvc_cache view).
struct PagedView {
    const int32_t *table;
    const int32_t *len;
    int32_t max_blocks, bs, n_pool;
};

// Shared body of the decode entry points: at most one of rope / alibi / paged is given.
static kvc_status decode_impl(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                              const int32_t *len, int32_t n_valid, const kvc_rope *rope,
                              const kvc_alibi *alibi, const PagedView *paged, float scale,
                              float *out, float *logits, int64_t logits_stride, float *lse,
                              void *ws, size_t ws_bytes, uint32_t flags, void *stream)
{
    if (flags & ~(uint32_t)(KVC_DECODE_KV_SETTLED | KVC_DECODE_BALANCE | KVC_DECODE_TEST_STARVE))
        return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn: unknown flags 0x%x", flags);
    kvc_status st = check_cache(cache, "kvc_decode_attn", true);
    if (st != KVC_OK) return st;
    if (q == nullptr || out == nullptr) return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn: null q/out");
    if (!aligned16(q)) return fail(KVC_ERR_ALIGN, "kvc_decode_attn: q must be 16-byte aligned");
    if (n_heads_q <= 0 || n_heads_q % cache->n_heads_kv)
        return fail(KVC_ERR_SHAPE, "kvc_decode_attn: n_heads_q %d not a multiple of n_heads_kv %d",
                    n_heads_q, cache->n_heads_kv);
    const int G = n_heads_q / cache->n_heads_kv;
    if (G != 1 && G != 2 && G != 4 && G != 6 && G != 8)
        return fail(KVC_ERR_SHAPE, "kvc_decode_attn: group size %d (supported: 1,2,4,6,8)", G);
    if (!std::isfinite(scale)) return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn: scale");
    int slots_max = cache->cap;
    if (rope != nullptr) {
        if (rope->t == nullptr || rope->cos_sin == nullptr || rope->n_sink < 0 || rope->window < 0)
            return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn: rope descriptor");
        const long long ring = (long long)rope->n_sink + rope->window + 1;
        if (ring > cache->cap)
            return fail(KVC_ERR_CAPACITY, "kvc_decode_attn: cap %d < n_sink + window + 1 = %lld",
                        cache->cap, ring);
        if (rope->n_pos < ring)
            return fail(KVC_ERR_CAPACITY, "kvc_decode_attn: rope table has %d rows, needs %lld",
                        rope->n_pos, ring);
        if (!aligned16(rope->cos_sin))
            return fail(KVC_ERR_ALIGN, "kvc_decode_attn: cos_sin must be 16-byte aligned");
        slots_max = (int)ring;
    } else if (alibi != nullptr) {
        if (alibi->t == nullptr || alibi->slopes == nullptr || alibi->n_sink < 0 ||
            alibi->window < 0)
            return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn_alibi: alibi descriptor");
        const long long ring = (long long)alibi->n_sink + alibi->window + 1;
        if (ring > cache->cap)
            return fail(KVC_ERR_CAPACITY,
                        "kvc_decode_attn_alibi: cap %d < n_sink + window + 1 = %lld", cache->cap,
                        ring);
        slots_max = (int)ring;
    } else if (paged != nullptr) {
        slots_max = cache->cap;
    } else if (len == nullptr && (n_valid < 0 || n_valid > cache->cap)) {
        return fail(KVC_ERR_CAPACITY, "kvc_decode_attn: n_valid %d outside [0, cap %d]", n_valid,
                    cache->cap);
    }
    if (logits != nullptr && logits_stride < slots_max)
        return fail(KVC_ERR_CAPACITY, "kvc_decode_attn: logits_stride %lld < %d slots",
                    (long long)logits_stride, slots_max);
    int32_t *code = nullptr;
    int n_sm = 0;
    st = device_info(&code, &n_sm);
    if (st != KVC_OK) return st;
    const kvc::DecodePlan pl = kvc::decode_plan(cache->batch, n_heads_q, cache->n_heads_kv,
                                                cache->d_head, cache->cap, n_sm);
    if (ws == nullptr || ws_bytes < pl.bytes)
        return fail(KVC_ERR_WORKSPACE, "kvc_decode_attn: workspace needs %zu bytes, got %zu",
                    pl.bytes, ws_bytes);
    if (!aligned256(ws)) return fail(KVC_ERR_WORKSPACE, "kvc_decode_attn: workspace alignment");
    kvc::DecodeParams p{};
    p.q = q;
    p.k = cache->k;
    p.v = cache->v;
    p.sb = cache->stride_b; p.sh = cache->stride_h; p.ss = cache->stride_slot;
    p.B = cache->batch; p.Hq = n_heads_q; p.Hkv = cache->n_heads_kv; p.cap = cache->cap;
    p.len = len;
    p.n_valid = n_valid;
    if (rope != nullptr) {
        p.rope = 1; p.S = rope->n_sink; p.W = rope->window; p.t = rope->t;
        p.cos_sin = rope->cos_sin;
        p.n_pos = rope->n_pos;
    } else if (alibi != nullptr) {
        p.S = alibi->n_sink; p.W = alibi->window; p.t = alibi->t;
        p.alibi = alibi->slopes;
    } else if (paged != nullptr) {
        p.len = paged->len;
        p.table = paged->table;
        p.max_blocks = paged->max_blocks;
        p.bs = paged->bs;
        p.n_pool = paged->n_pool;
    }
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out; p.logits = logits; p.logits_stride = logits_stride; p.lse = lse;
    char *wsb = static_cast<char *>(ws);
    p.ws_o = reinterpret_cast<float *>(wsb + pl.off_o);
    p.ws_ml = reinterpret_cast<float *>(wsb + pl.off_ml);
    p.ws_cnt = reinterpret_cast<int32_t *>(wsb + pl.off_cnt);
    p.P = cache->batch * cache->n_heads_kv;
    p.max_seg = pl.max_seg;
    p.n_sm = n_sm > 0 ? n_sm : 152;
    p.kv_settled = (flags & KVC_DECODE_KV_SETTLED) ? 1 : 0;
    p.balance = (flags & KVC_DECODE_BALANCE) ? 1 : 0;
    if (flags & KVC_DECODE_TEST_STARVE) {
        p.starve = 1;
        p.spin_limit = kTestSpinLimit;
    }
    p.dev_code = code;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    bool used = false;
    if (p.table != nullptr) {
        e = cache->dtype == KVC_BF16 ? kvc::launch_decode_attn_bf16_paged(p, cache->d_head, G, s)
                                     : kvc::launch_decode_attn_f32_paged(p, cache->d_head, G, s);
        if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
        return ok();
    }
    if (p.alibi != nullptr) {
        e = cache->dtype == KVC_BF16 ? kvc::launch_decode_attn_bf16_alibi(p, cache->d_head, G, s)
                                     : kvc::launch_decode_attn_f32_alibi(p, cache->d_head, G, s);
        if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
        return ok();
    }
    if (cache->dtype == KVC_BF16 && !p.rope && G > 1) {
        // query groups: the two matrix products of the group run on the tensor cores
        e = kvc::launch_decode_attn_mma(p, cache->d_head, G, s, &used);
        if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
        if (used) return ok();
    }
    if (cache->dtype == KVC_BF16)
        e = p.rope ? kvc::launch_decode_attn_bf16_rope(p, cache->d_head, G, s)
                   : kvc::launch_decode_attn_bf16(p, cache->d_head, G, s);
    else
        e = p.rope ? kvc::launch_decode_attn_f32_rope(p, cache->d_head, G, s)
                   : kvc::launch_decode_attn_f32(p, cache->d_head, G, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
    return ok();
}

kvc_status kvc_decode_attn_ex(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                              const int32_t *len, int32_t n_valid, const kvc_rope *rope,
                              float scale, float *out, float *logits, int64_t logits_stride,
                              float *lse, void *ws, size_t ws_bytes, uint32_t flags, void *stream)
{
    return decode_impl(q, n_heads_q, cache, len, n_valid, rope, nullptr, nullptr, scale, out,
                       logits, logits_stride, lse, ws, ws_bytes, flags, stream);
}

kvc_status kvc_decode_attn_alibi(const void *q, int32_t n_heads_q, const kvc_cache *cache,
                                 const kvc_alibi *alibi, float scale, float *out, float *logits,
                                 int64_t logits_stride, float *lse, void *ws, size_t ws_bytes,
                                 uint32_t flags, void *stream)
{
    if (alibi == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn_alibi: null alibi descriptor");
    return decode_impl(q, n_heads_q, cache, nullptr, 0, nullptr, alibi, nullptr, scale, out,
                       logits, logits_stride, lse, ws, ws_bytes, flags, stream);
}

// ------------------------------------------------------------------------------------------
// DuoAttention.
namespace {

struct DuoMap {
    int n_ret = 0, n_str = 0, Hkv = 0;
    uint8_t head_of[256] = {};    // retrieval heads in the given order, then the others ascending
    uint8_t index_of[256] = {};   // inverse of head_of
};

kvc_status duo_check(const kvc_cache *full, const kvc_cache *ring, const kvc_duo *duo,
                     const char *name, DuoMap *m)
{
    if (duo == nullptr || duo->t == nullptr || duo->n_retrieval < 0 || duo->n_sink < 0 ||
        duo->window < 0 || (duo->n_retrieval > 0 && duo->retrieval_heads == nullptr))
        return fail(KVC_ERR_INVALID_ARG, "%s: duo descriptor", name);
    if (full == nullptr || ring == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "%s: null cache descriptor", name);
    kvc_status st = check_cache(full, name, true);
    if (st != KVC_OK) return st;
    st = check_cache(ring, name, true);
    if (st != KVC_OK) return st;
    if (full->dtype != ring->dtype || full->d_head != ring->d_head || full->batch != ring->batch)
        return fail(KVC_ERR_SHAPE, "%s: the two caches differ in dtype, d_head or batch", name);
    if (full->stride_slot != full->d_head || ring->stride_slot != ring->d_head)
        return fail(KVC_ERR_SHAPE, "%s: cache slots must be dense (stride_slot == d_head)", name);
    if (full->n_heads_kv != duo->n_retrieval)
        return fail(KVC_ERR_SHAPE, "%s: full cache has %d heads, n_retrieval is %d", name,
                    full->n_heads_kv, duo->n_retrieval);
    const long long ring_cap = (long long)duo->n_sink + duo->window + 1;
    if (ring->cap < ring_cap)
        return fail(KVC_ERR_CAPACITY, "%s: ring cap %d < n_sink + window + 1 = %lld", name,
                    ring->cap, ring_cap);
    m->n_ret = duo->n_retrieval;
    m->n_str = ring->n_heads_kv;
    m->Hkv = m->n_ret + m->n_str;
    if (m->Hkv > 256) return fail(KVC_ERR_SHAPE, "%s: more than 256 KV heads", name);
    bool used[256] = {};
    for (int r = 0; r < m->n_ret; ++r) {
        const int h = duo->retrieval_heads[r];
        if (h < 0 || h >= m->Hkv || used[h] || (r > 0 && h <= duo->retrieval_heads[r - 1]))
            return fail(KVC_ERR_INVALID_ARG, "%s: retrieval_heads must be ascending, distinct "
                        "KV heads below %d", name, m->Hkv);
        used[h] = true;
        m->head_of[r] = (uint8_t)h;
        m->index_of[h] = (uint8_t)r;
    }
    int i = m->n_ret;
    for (int h = 0; h < m->Hkv; ++h)
        if (!used[h]) {
            m->head_of[i] = (uint8_t)h;
            m->index_of[h] = (uint8_t)i;
            ++i;
        }
    return KVC_OK;
}

}  // namespace

uint64_t kvc_duo_kv_bytes(uint64_t n_layers, uint64_t n_retrieval, uint64_t n_streaming,
                          uint64_t d_head, uint64_t seq_len, uint64_t n_sink, uint64_t window,
                          uint64_t bytes_per_elem, uint64_t batch)
{
    // per head: seq_len tokens (retrieval) or the constant buffer, never more than seq_len
    const uint64_t buffer = std::min<uint64_t>(n_sink + window + 1, seq_len);
    return 2ull * n_layers * d_head * bytes_per_elem * batch *
           (n_retrieval * seq_len + n_streaming * buffer);
}

kvc_status kvc_duo_append(const kvc_cache *full, int32_t *len, const kvc_cache *ring,
                          const kvc_duo *duo, const void *k_new, const void *v_new, void *stream)
{
    DuoMap m;
    kvc_status st = duo_check(full, ring, duo, "kvc_duo_append", &m);
    if (st != KVC_OK) return st;
    if (k_new == nullptr || v_new == nullptr || (m.n_ret > 0 && len == nullptr))
        return fail(KVC_ERR_INVALID_ARG, "kvc_duo_append: null k_new/v_new/len");
    if (!aligned16(k_new) || !aligned16(v_new))
        return fail(KVC_ERR_ALIGN, "kvc_duo_append: k_new/v_new must be 16-byte aligned");
    int32_t *code = nullptr;
    st = device_info(&code, nullptr);
    if (st != KVC_OK) return st;
    kvc::DuoAppendParams p{};
    p.k = full->k; p.v = full->v;
    p.sb = full->stride_b; p.sh = full->stride_h; p.ss = full->stride_slot; p.cap = full->cap;
    p.len = len;
    p.k2 = ring->k; p.v2 = ring->v;
    p.sb2 = ring->stride_b; p.sh2 = ring->stride_h; p.ss2 = ring->stride_slot;
    p.S = duo->n_sink; p.W = duo->window; p.t = duo->t;
    p.k_new = k_new; p.v_new = v_new;
    p.B = full->batch; p.Hkv = m.Hkv; p.D = full->d_head; p.eb = elem_bytes(full->dtype);
    p.n_ret = m.n_ret;
    std::memcpy(p.index_of, m.index_of, sizeof(p.index_of));
    p.dev_code = code;
    cudaError_t e = kvc::launch_duo_append(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "duo append launch");
    return ok();
}

size_t kvc_decode_attn_duo_workspace_bytes(int32_t batch, int32_t n_heads_q, int32_t n_heads_kv,
                                           int32_t d_head, int32_t cap, int32_t n_retrieval)
{
    if (batch <= 0 || n_heads_q <= 0 || n_heads_kv <= 0 || d_head <= 0 || cap < 0 ||
        n_retrieval < 0 || n_retrieval > n_heads_kv)
        return 0;
    return kvc::decode_plan(batch, n_heads_q, n_heads_kv, d_head, cap, sm_count_or_default(),
                            batch * (n_retrieval > 0 ? n_retrieval : 1))
        .bytes;
}

kvc_status kvc_decode_attn_duo(const void *q, int32_t n_heads_q, const kvc_cache *full,
                               const int32_t *len, int32_t n_valid, const kvc_cache *ring,
                               const kvc_duo *duo, float scale, float *out, float *logits,
                               int64_t logits_stride, float *lse, void *ws, size_t ws_bytes,
                               uint32_t flags, void *stream)
{
    if (flags & ~(uint32_t)KVC_DECODE_KV_SETTLED)
        return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn_duo: unknown flags 0x%x", flags);
    DuoMap m;
    kvc_status st = duo_check(full, ring, duo, "kvc_decode_attn_duo", &m);
    if (st != KVC_OK) return st;
    if (q == nullptr || out == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn_duo: null q/out");
    if (!aligned16(q)) return fail(KVC_ERR_ALIGN, "kvc_decode_attn_duo: q must be 16-byte aligned");
    if (n_heads_q <= 0 || n_heads_q % m.Hkv)
        return fail(KVC_ERR_SHAPE, "kvc_decode_attn_duo: n_heads_q %d not a multiple of %d KV "
                    "heads", n_heads_q, m.Hkv);
    const int G = n_heads_q / m.Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 6 && G != 8)
        return fail(KVC_ERR_SHAPE, "kvc_decode_attn_duo: group size %d (supported: 1,2,4,6,8)", G);
    if (!std::isfinite(scale)) return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attn_duo: scale");
    if (len == nullptr && (n_valid < 0 || n_valid > full->cap))
        return fail(KVC_ERR_CAPACITY, "kvc_decode_attn_duo: n_valid %d outside [0, cap %d]",
                    n_valid, full->cap);
    const int ring_cap = duo->n_sink + duo->window + 1;
    if (logits != nullptr && logits_stride < std::max(full->cap, ring_cap))
        return fail(KVC_ERR_CAPACITY, "kvc_decode_attn_duo: logits_stride %lld too small",
                    (long long)logits_stride);
    int32_t *code = nullptr;
    int n_sm = 0;
    st = device_info(&code, &n_sm);
    if (st != KVC_OK) return st;
    const int B = full->batch;
    const kvc::DecodePlan pl = kvc::decode_plan(B, n_heads_q, m.Hkv, full->d_head, full->cap,
                                                n_sm, B * (m.n_ret > 0 ? m.n_ret : 1));
    if (ws == nullptr || ws_bytes < pl.bytes)
        return fail(KVC_ERR_WORKSPACE, "kvc_decode_attn_duo: workspace needs %zu bytes, got %zu",
                    pl.bytes, ws_bytes);
    if (!aligned256(ws)) return fail(KVC_ERR_WORKSPACE, "kvc_decode_attn_duo: workspace alignment");
    kvc::DecodeParams p{};
    p.q = q;
    p.k = full->k; p.v = full->v;
    p.sb = full->stride_b; p.sh = full->stride_h; p.ss = full->stride_slot;
    p.B = B; p.Hq = n_heads_q; p.Hkv = m.Hkv; p.cap = full->cap;
    p.len = len; p.n_valid = n_valid;
    p.t = duo->t;
    p.n_ret = m.n_ret; p.n_str = m.n_str; p.ring_cap = ring_cap;
    p.k2 = ring->k; p.v2 = ring->v; p.sb2 = ring->stride_b; p.sh2 = ring->stride_h;
    std::memcpy(p.head_of, m.head_of, sizeof(p.head_of));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out; p.logits = logits; p.logits_stride = logits_stride; p.lse = lse;
    char *wsb = static_cast<char *>(ws);
    p.ws_o = reinterpret_cast<float *>(wsb + pl.off_o);
    p.ws_ml = reinterpret_cast<float *>(wsb + pl.off_ml);
    p.ws_cnt = reinterpret_cast<int32_t *>(wsb + pl.off_cnt);
    p.P = B * m.Hkv;
    p.max_seg = pl.max_seg;
    p.n_sm = n_sm > 0 ? n_sm : 152;
    p.kv_settled = (flags & KVC_DECODE_KV_SETTLED) ? 1 : 0;
    p.dev_code = code;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = full->dtype == KVC_BF16
                        ? kvc::launch_decode_attn_bf16_duo(p, full->d_head, G, s)
                        : kvc::launch_decode_attn_f32_duo(p, full->d_head, G, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
    return ok();
}

// ------------------------------------------------------------------------------------------
// Block-level eviction over page tables.
static kvc_status check_paged(const kvc_block_pool *pool, const kvc_page_table *pt,
                              const char *name, kvc_cache *view)
{
    if (pool == nullptr || pt == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "%s: null pool or page-table descriptor", name);
    if (pt->table == nullptr || pt->n_blocks == nullptr || pt->len == nullptr ||
        pt->score == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "%s: null page-table array", name);
    if (pool->n_blocks <= 0 || pool->block_size <= 0 || pt->batch <= 0 || pt->max_blocks <= 0)
        return fail(KVC_ERR_SHAPE, "%s: n_blocks %d block_size %d batch %d max_blocks %d", name,
                    pool->n_blocks, pool->block_size, pt->batch, pt->max_blocks);
    if ((long long)pt->max_blocks * pool->block_size > (1LL << 30))
        return fail(KVC_ERR_SHAPE, "%s: max_blocks * block_size too large", name);
    kvc_cache c{};
    c.k = pool->k;
    c.v = pool->v;
    c.dtype = pool->dtype;
    c.batch = pt->batch;
    c.n_heads_kv = pool->n_heads_kv;
    c.cap = pt->max_blocks * pool->block_size;
    c.d_head = pool->d_head;
    c.stride_b = 0;
    c.stride_h = (int64_t)pool->n_blocks * pool->block_size * pool->d_head;   // head-major
    c.stride_slot = pool->d_head;
    *view = c;
    return check_cache(&c, name, true);
}

static kvc_status check_free_pool(const kvc_free_pool *fp, const char *name)
{
    if (fp == nullptr || fp->ids == nullptr || fp->top == nullptr || fp->capacity <= 0)
        return fail(KVC_ERR_INVALID_ARG, "%s: free pool descriptor", name);
    return KVC_OK;
}

kvc_status kvc_paged_append(const kvc_block_pool *pool, const kvc_page_table *pt,
                            const kvc_free_pool *free_pool, const void *k_new, const void *v_new,
                            const int64_t *t, int32_t *pos, void *stream)
{
    kvc_cache view;
    kvc_status st = check_paged(pool, pt, "kvc_paged_append", &view);
    if (st != KVC_OK) return st;
    st = check_free_pool(free_pool, "kvc_paged_append");
    if (st != KVC_OK) return st;
    if (k_new == nullptr || v_new == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_paged_append: null k_new/v_new");
    if (!aligned16(k_new) || !aligned16(v_new))
        return fail(KVC_ERR_ALIGN, "kvc_paged_append: k_new/v_new must be 16-byte aligned");
    int32_t *code = nullptr;
    st = device_info(&code, nullptr);
    if (st != KVC_OK) return st;
    kvc::PagedParams p{};
    p.k = pool->k; p.v = pool->v;
    p.n_pool = pool->n_blocks; p.Hkv = pool->n_heads_kv; p.bs = pool->block_size;
    p.D = pool->d_head; p.B = pt->batch; p.max_blocks = pt->max_blocks;
    p.table = pt->table; p.n_blocks = pt->n_blocks; p.len = pt->len; p.score = pt->score;
    p.free_ids = free_pool->ids; p.free_top = free_pool->top; p.free_cap = free_pool->capacity;
    p.k_new = k_new; p.v_new = v_new; p.t = t; p.pos = pos;
    p.dev_code = code;
    cudaError_t e = kvc::launch_paged_append(p, elem_bytes(pool->dtype),
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged append launch");
    return ok();
}

kvc_status kvc_decode_attn_paged(const void *q, int32_t n_heads_q, const kvc_block_pool *pool,
                                 const kvc_page_table *pt, float scale, float *out,
                                 float *logits, int64_t logits_stride, float *lse, void *ws,
                                 size_t ws_bytes, uint32_t flags, void *stream)
{
    kvc_cache view;
    kvc_status st = check_paged(pool, pt, "kvc_decode_attn_paged", &view);
    if (st != KVC_OK) return st;
    PagedView pv{pt->table, pt->len, pt->max_blocks, pool->block_size, pool->n_blocks};
    return decode_impl(q, n_heads_q, &view, nullptr, 0, nullptr, nullptr, &pv, scale, out,
                       logits, logits_stride, lse, ws, ws_bytes, flags, stream);
}

size_t kvc_block_prompt_select_workspace_bytes(int32_t batch, int32_t seq_len,
                                               int32_t block_size, int32_t budget_blocks)
{
    if (batch <= 0 || seq_len <= 0 || block_size <= 0 || budget_blocks <= 0) return 0;
    const size_t nblk = ((size_t)seq_len + block_size - 1) / block_size;
    return align256((size_t)batch * nblk * sizeof(float)) +
           align256((size_t)batch * budget_blocks * sizeof(int32_t));
}

kvc_status kvc_block_prompt_select(const float *s, int64_t s_stride, const kvc_cache *prompt,
                                   int32_t seq_len, const kvc_block_pool *pool,
                                   const kvc_page_table *pt, const kvc_free_pool *free_pool,
                                   int32_t budget_blocks, int32_t recent_blocks, void *ws,
                                   size_t ws_bytes, void *stream)
{
    kvc_cache view;
    kvc_status st = check_paged(pool, pt, "kvc_block_prompt_select", &view);
    if (st != KVC_OK) return st;
    st = check_free_pool(free_pool, "kvc_block_prompt_select");
    if (st != KVC_OK) return st;
    st = check_cache(prompt, "kvc_block_prompt_select", true);
    if (st != KVC_OK) return st;
    if (s == nullptr) return fail(KVC_ERR_INVALID_ARG, "kvc_block_prompt_select: null scores");
    if (prompt->dtype != pool->dtype || prompt->n_heads_kv != pool->n_heads_kv ||
        prompt->d_head != pool->d_head || prompt->batch != pt->batch)
        return fail(KVC_ERR_SHAPE, "kvc_block_prompt_select: prompt and pool differ in dtype, "
                    "heads, d_head or batch");
    if (seq_len <= 0 || seq_len > prompt->cap || s_stride < seq_len)
        return fail(KVC_ERR_CAPACITY, "kvc_block_prompt_select: seq_len %d (prompt cap %d, "
                    "score stride %lld)", seq_len, prompt->cap, (long long)s_stride);
    if (recent_blocks < 1 || budget_blocks < recent_blocks || budget_blocks > pt->max_blocks)
        return fail(KVC_ERR_INVALID_ARG, "kvc_block_prompt_select: need 1 <= recent_blocks <= "
                    "budget_blocks <= max_blocks (%d, %d, %d)", recent_blocks, budget_blocks,
                    pt->max_blocks);
    if (pt->batch > 65535 || pool->n_heads_kv > 65535)
        return fail(KVC_ERR_SHAPE, "kvc_block_prompt_select: batch %d, heads %d", pt->batch,
                    pool->n_heads_kv);
    const size_t need = kvc_block_prompt_select_workspace_bytes(pt->batch, seq_len,
                                                                pool->block_size, budget_blocks);
    if (ws == nullptr || ws_bytes < need || !aligned256(ws))
        return fail(KVC_ERR_WORKSPACE, "kvc_block_prompt_select: workspace needs %zu bytes "
                    "(256-byte aligned), got %zu", need, ws_bytes);
    int32_t *code = nullptr;
    st = device_info(&code, nullptr);
    if (st != KVC_OK) return st;
    kvc::BlockPromptParams p{};
    p.s = s; p.s_stride = s_stride;
    p.pk = prompt->k; p.pv = prompt->v;
    p.sb = prompt->stride_b; p.sh = prompt->stride_h; p.ss = prompt->stride_slot;
    p.k = pool->k; p.v = pool->v;
    p.B = pt->batch; p.H = pool->n_heads_kv; p.N = seq_len; p.bs = pool->block_size;
    p.nblk = (seq_len + pool->block_size - 1) / pool->block_size;
    p.eb = elem_bytes(pool->dtype); p.row_bytes = pool->d_head * p.eb;
    p.n_pool = pool->n_blocks; p.max_blocks = pt->max_blocks;
    p.table = pt->table; p.n_blocks = pt->n_blocks; p.len = pt->len; p.score = pt->score;
    p.free_ids = free_pool->ids; p.free_top = free_pool->top; p.free_cap = free_pool->capacity;
    p.budget_blocks = budget_blocks; p.recent_blocks = recent_blocks;
    char *wsb = static_cast<char *>(ws);
    p.ws_score = reinterpret_cast<float *>(wsb);
    p.ws_src = reinterpret_cast<int32_t *>(wsb + align256((size_t)p.B * p.nblk * sizeof(float)));
    p.dev_code = code;
    cudaError_t e = kvc::launch_block_prompt_select(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "block prompt selection launch");
    return ok();
}

kvc_status kvc_block_accumulate_evict(const float *logits, int64_t logits_stride,
                                      const float *lse, int32_t n_heads_q, int32_t block_size,
                                      const kvc_page_table *pt, const kvc_free_pool *free_pool,
                                      int32_t budget_blocks, int32_t recent_blocks,
                                      int32_t *released, void *stream)
{
    if (pt == nullptr || pt->table == nullptr || pt->n_blocks == nullptr || pt->len == nullptr ||
        pt->score == nullptr || logits == nullptr || lse == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_block_accumulate_evict: null argument");
    kvc_status st = check_free_pool(free_pool, "kvc_block_accumulate_evict");
    if (st != KVC_OK) return st;
    if (pt->batch <= 0 || pt->batch > 65535 || pt->max_blocks <= 0 || block_size <= 0 ||
        n_heads_q <= 0 || n_heads_q > 1024)
        return fail(KVC_ERR_SHAPE, "kvc_block_accumulate_evict: batch %d max_blocks %d "
                    "block_size %d n_heads_q %d", pt->batch, pt->max_blocks, block_size,
                    n_heads_q);
    if (recent_blocks < 1 || budget_blocks < recent_blocks)
        return fail(KVC_ERR_INVALID_ARG, "kvc_block_accumulate_evict: recent_blocks %d must be "
                    ">= 1 and <= budget_blocks %d", recent_blocks, budget_blocks);
    if (logits_stride < (int64_t)pt->max_blocks * block_size)
        return fail(KVC_ERR_CAPACITY, "kvc_block_accumulate_evict: logits_stride %lld < %lld",
                    (long long)logits_stride, (long long)pt->max_blocks * block_size);
    int32_t *code = nullptr;
    st = device_info(&code, nullptr);
    if (st != KVC_OK) return st;
    kvc::PagedParams p{};
    p.bs = block_size; p.B = pt->batch; p.max_blocks = pt->max_blocks;
    p.table = pt->table; p.n_blocks = pt->n_blocks; p.len = pt->len; p.score = pt->score;
    p.free_ids = free_pool->ids; p.free_top = free_pool->top; p.free_cap = free_pool->capacity;
    p.logits = logits; p.logits_stride = logits_stride; p.lse = lse; p.Hq = n_heads_q;
    p.budget_blocks = budget_blocks; p.recent_blocks = recent_blocks; p.released = released;
    p.n_pool = 0x7fffffff;
    p.dev_code = code;
    cudaError_t e = kvc::launch_block_accumulate_evict(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "block accumulate/evict launch");
    return ok();
}

kvc_status kvc_alibi_slopes(int32_t n_heads, float *out)
{
    // Geometric sequence starting at and stepping by 2^(-8/n): head h gets 2^(-8(h+1)/n).
    if (out == nullptr || n_heads <= 0 || (n_heads & (n_heads - 1)) != 0)
        return fail(KVC_ERR_INVALID_ARG,
                    "kvc_alibi_slopes: n_heads %d must be a positive power of two", n_heads);
    for (int32_t h = 0; h < n_heads; ++h)
        out[h] = (float)std::exp2(-8.0 * (double)(h + 1) / (double)n_heads);
    return ok();
}

// ------------------------------------------------------------------------------------------
kvc_status kvc_stream_append(const kvc_cache *cache, int32_t policy, const void *k_new,
                             const void *v_new, const int64_t *t, int32_t *len, int32_t n_sink,
                             int32_t window, const int32_t *free_slot, int32_t *pos,
                             int64_t pos_stride, float *score, int64_t score_stride,
                             void *stream)
{
    kvc_status st = check_cache(cache, "kvc_stream_append", true);
    if (st != KVC_OK) return st;
    if (k_new == nullptr || v_new == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_stream_append: null k_new/v_new");
    if (!aligned16(k_new) || !aligned16(v_new))
        return fail(KVC_ERR_ALIGN, "kvc_stream_append: k_new/v_new must be 16-byte aligned");
    if (policy == KVC_APPEND_TAIL) {
        if (len == nullptr) return fail(KVC_ERR_INVALID_ARG, "kvc_stream_append: TAIL needs len");
    } else if (policy == KVC_APPEND_RING) {
        if (t == nullptr || n_sink < 0 || window < 0)
            return fail(KVC_ERR_INVALID_ARG, "kvc_stream_append: RING needs t, n_sink, window");
        if ((long long)n_sink + window + 1 > cache->cap)
            return fail(KVC_ERR_CAPACITY, "kvc_stream_append: cap %d < n_sink + window + 1",
                        cache->cap);
    } else if (policy == KVC_APPEND_FREE_SLOT) {
        if (t == nullptr || free_slot == nullptr)
            return fail(KVC_ERR_INVALID_ARG, "kvc_stream_append: FREE_SLOT needs t and free_slot");
    } else {
        return fail(KVC_ERR_INVALID_ARG, "kvc_stream_append: policy %d", policy);
    }
    if ((pos != nullptr && (t == nullptr || pos_stride < cache->cap)) ||
        (score != nullptr && score_stride < cache->cap))
        return fail(KVC_ERR_INVALID_ARG, "kvc_stream_append: pos needs t; strides >= cap");
    int32_t *code = nullptr;
    st = device_info(&code, nullptr);
    if (st != KVC_OK) return st;
    kvc::AppendParams p{};
    p.k = cache->k; p.v = cache->v;
    p.sb = cache->stride_b; p.sh = cache->stride_h; p.ss = cache->stride_slot;
    p.B = cache->batch; p.H = cache->n_heads_kv; p.cap = cache->cap; p.D = cache->d_head;
    p.policy = policy;
    p.k_new = k_new; p.v_new = v_new; p.t = t; p.len = len;
    p.S = n_sink; p.W = window; p.free_slot = free_slot;
    p.pos = pos; p.pos_stride = pos_stride; p.score = score; p.score_stride = score_stride;
    p.dev_code = code;
    cudaError_t e = kvc::launch_append(p, elem_bytes(cache->dtype), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return ok();
}

kvc_status kvc_position_advance(int64_t *t, int64_t delta, void *stream)
{
    if (t == nullptr) return fail(KVC_ERR_INVALID_ARG, "kvc_position_advance: null t");
    cudaError_t e = kvc::launch_position_advance(t, delta, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "position advance launch");
    return ok();
}

// ------------------------------------------------------------------------------------------
kvc_status kvc_compact_gather(const kvc_cache *src, const int32_t *idx, int64_t idx_stride,
                              int32_t n_keep, const kvc_cache *dst, int32_t *pos_dst,
                              int64_t pos_stride, int32_t *len_dst, void *stream)
{
    kvc_status st = check_cache(src, "kvc_compact_gather(src)", true);
    if (st != KVC_OK) return st;
    st = check_cache(dst, "kvc_compact_gather(dst)", true);
    if (st != KVC_OK) return st;
    if (idx == nullptr || n_keep < 0 || idx_stride < n_keep)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact_gather: idx / n_keep / idx_stride");
    if (src->dtype != dst->dtype || src->batch != dst->batch ||
        src->n_heads_kv != dst->n_heads_kv || src->d_head != dst->d_head)
        return fail(KVC_ERR_SHAPE, "kvc_compact_gather: src and dst disagree in shape or dtype");
    if (dst->cap < n_keep)
        return fail(KVC_ERR_CAPACITY, "kvc_compact_gather: dst cap %d < n_keep %d", dst->cap, n_keep);
    if (src->k == dst->k || src->v == dst->v || src->k == dst->v || src->v == dst->k)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact_gather: out of place only");
    if (pos_dst != nullptr && pos_stride < n_keep)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact_gather: pos_stride < n_keep");
    int32_t *code = nullptr;
    st = device_info(&code, nullptr);
    if (st != KVC_OK) return st;
    kvc::GatherParams p{};
    p.sk = src->k; p.sv = src->v;
    p.s_sb = src->stride_b; p.s_sh = src->stride_h; p.s_ss = src->stride_slot; p.s_cap = src->cap;
    p.dk = dst->k; p.dv = dst->v;
    p.d_sb = dst->stride_b; p.d_sh = dst->stride_h; p.d_ss = dst->stride_slot;
    p.B = src->batch; p.H = src->n_heads_kv; p.D = src->d_head;
    p.idx = idx; p.idx_stride = idx_stride; p.n_keep = n_keep;
    p.pos_dst = pos_dst; p.pos_stride = pos_stride; p.len_dst = len_dst;
    p.dev_code = code;
    cudaError_t e = kvc::launch_gather(p, elem_bytes(src->dtype), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    return ok();
}

// ------------------------------------------------------------------------------------------
// Observation-window scores: bf16 inputs of supported shapes run on the tensor cores, the rest
// (fp32, short windows with several heads) on the CUDA-core kernels.
static cudaError_t run_scores(const kvc::ScoreParams &sp, int dtype, float scale, int32_t *code,
                              cudaStream_t s)
{
    if (dtype == KVC_BF16 && scale > 0.f) {
        bool used = false;
        cudaError_t e = kvc::launch_obs_scores_tc(sp, code, s, &used);
        if (e != cudaSuccess || used) return e;
    }
    return kvc::launch_obs_scores(sp, dtype, s);
}

// SnapKV workspace: [s (G heads, prefix columns)] [pooled score] [row states] [row lse].
static void snapkv_layout(int B, int Hq, int Hkv, int N, int L_obs, int n_sm, size_t *off_s,
                          size_t *off_score, kvc::ScorePlan *pl)
{
    const size_t n = (size_t)(N - L_obs);
    *off_s = 0;
    *off_score = align256((size_t)B * Hq * n * sizeof(float));
    const size_t base = align256(*off_score + (size_t)B * Hkv * n * sizeof(float));
    *pl = kvc::score_plan(B, Hkv, Hq / Hkv, N, L_obs, n_sm, base);
}

size_t kvc_snapkv_select_workspace_bytes(int32_t batch, int32_t n_heads_q, int32_t n_heads_kv,
                                         int32_t d_head, int32_t seq_len, int32_t L_obs)
{
    (void)d_head;
    if (batch <= 0 || n_heads_kv <= 0 || n_heads_q <= 0 || n_heads_q % n_heads_kv ||
        L_obs <= 0 || seq_len < L_obs)
        return 0;
    size_t off_s, off_score;
    kvc::ScorePlan pl;
    snapkv_layout(batch, n_heads_q, n_heads_kv, seq_len, L_obs, sm_count_or_default(), &off_s,
                  &off_score, &pl);
    return pl.bytes;
}

kvc_status kvc_snapkv_select(const void *q_obs, const kvc_cache *prompt, int32_t n_heads_q,
                             int32_t seq_len, int32_t L_obs, int32_t pool_k, int32_t budget,
                             float scale, int32_t *idx_out, float *scores_out, void *ws,
                             size_t ws_bytes, void *stream)
{
    kvc_status st = check_cache(prompt, "kvc_snapkv_select", false);
    if (st != KVC_OK) return st;
    if (q_obs == nullptr || idx_out == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_snapkv_select: null q_obs/idx_out");
    if (n_heads_q <= 0 || n_heads_q % prompt->n_heads_kv)
        return fail(KVC_ERR_SHAPE, "kvc_snapkv_select: n_heads_q %d vs n_heads_kv %d", n_heads_q,
                    prompt->n_heads_kv);
    if (L_obs <= 0 || seq_len < L_obs || seq_len > prompt->cap)
        return fail(KVC_ERR_SHAPE, "kvc_snapkv_select: need 0 < L_obs <= seq_len <= cap");
    if (pool_k <= 0 || pool_k % 2 == 0 || pool_k > 15)
        return fail(KVC_ERR_INVALID_ARG, "kvc_snapkv_select: pool_k %d must be odd, 1..15",
                    pool_k);
    if (budget < L_obs)
        return fail(KVC_ERR_CAPACITY, "kvc_snapkv_select: budget %d < L_obs %d", budget, L_obs);
    if (!std::isfinite(scale)) return fail(KVC_ERR_INVALID_ARG, "kvc_snapkv_select: scale");
    int32_t *code = nullptr;
    int n_sm = 0;
    st = device_info(&code, &n_sm);
    if (st != KVC_OK) return st;
    const int B = prompt->batch, Hkv = prompt->n_heads_kv, G = n_heads_q / Hkv;
    size_t off_s, off_score;
    kvc::ScorePlan pl;
    snapkv_layout(B, n_heads_q, Hkv, seq_len, L_obs, n_sm, &off_s, &off_score, &pl);
    if (ws == nullptr || ws_bytes < pl.bytes || !aligned256(ws))
        return fail(KVC_ERR_WORKSPACE, "kvc_snapkv_select: workspace needs %zu aligned bytes",
                    pl.bytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n = seq_len - L_obs;
    const int n_keep = std::min(budget, seq_len);
    if (budget >= seq_len && scores_out == nullptr) {
        cudaError_t e = kvc::launch_iota_rows(idx_out, n_keep, B * Hkv, n_keep, s);
        if (e != cudaSuccess) return cuda_fail(e, "iota launch");
        return ok();
    }
    char *wsb = static_cast<char *>(ws);
    float *s_cols = scores_out ? scores_out : reinterpret_cast<float *>(wsb + off_s);
    float *pooled = reinterpret_cast<float *>(wsb + off_score);
    kvc::ScoreParams sp{};
    sp.q = q_obs; sp.k = prompt->k;
    sp.sb = prompt->stride_b; sp.sh = prompt->stride_h; sp.ss = prompt->stride_slot;
    sp.B = B; sp.Hq = n_heads_q; sp.Hkv = Hkv; sp.G = G; sp.D = prompt->d_head; sp.N = seq_len;
    sp.L_obs = L_obs;
    sp.scale_log2 = scale * 1.4426950408889634f;
    sp.n_cols = n;
    sp.col_mult = 1.0f / (float)L_obs;
    sp.s_out = s_cols;
    sp.row_ml = reinterpret_cast<float *>(wsb + pl.off_ml);
    sp.row_lse2 = reinterpret_cast<float *>(wsb + pl.off_lse);
    sp.n_chunks = pl.n_chunks;
    sp.chunk = pl.chunk;
    cudaError_t e = run_scores(sp, prompt->dtype, scale, code, s);
    if (e != cudaSuccess) return cuda_fail(e, "observation scores launch");
    if (budget >= seq_len) {
        e = kvc::launch_iota_rows(idx_out, n_keep, B * Hkv, n_keep, s);
        if (e != cudaSuccess) return cuda_fail(e, "iota launch");
        return ok();
    }
    bool fused = false;
    e = kvc::launch_pool_topk(s_cols, n, B * Hkv, G, n, budget - L_obs, L_obs, pool_k, idx_out,
                              budget, s, &fused);
    if (e != cudaSuccess) return cuda_fail(e, "pool + top-k launch");
    if (fused) return ok();
    e = kvc::launch_pool_groupmax(s_cols, n, pooled, B * Hkv, G, n, pool_k, s);
    if (e != cudaSuccess) return cuda_fail(e, "pool launch");
    e = kvc::launch_topk_rows(pooled, n, B * Hkv, n, budget - L_obs, L_obs, idx_out, budget, s);
    if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
    return ok();
}

// ------------------------------------------------------------------------------------------
kvc_status kvc_h2o_accumulate_evict(const float *logits, int64_t logits_stride, const float *lse,
                                    float *score, int32_t *pos, int64_t stride,
                                    int32_t *free_slot, int32_t batch, int32_t n_heads,
                                    int32_t n_slots, const int64_t *t, int32_t L_local,
                                    int32_t budget, void *stream)
{
    return kvc_h2o_accumulate_evict_gqa(logits, logits_stride, lse, score, pos, stride, free_slot,
                                        batch, n_heads, n_heads, n_slots, t, L_local, budget,
                                        stream);
}

kvc_status kvc_h2o_accumulate_evict_gqa(const float *logits, int64_t logits_stride,
                                        const float *lse, float *score, int32_t *pos,
                                        int64_t stride, int32_t *free_slot, int32_t batch,
                                        int32_t n_heads_q, int32_t n_heads_kv, int32_t n_slots,
                                        const int64_t *t, int32_t L_local, int32_t budget,
                                        void *stream)
{
    if (logits == nullptr || lse == nullptr || score == nullptr || pos == nullptr ||
        free_slot == nullptr || t == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_h2o_accumulate_evict: null pointer");
    if (batch <= 0 || n_heads_kv <= 0 || n_heads_q < n_heads_kv || n_heads_q % n_heads_kv ||
        n_slots < 0 || L_local < 0 || budget < 0 || logits_stride < n_slots || stride < n_slots)
        return fail(KVC_ERR_SHAPE, "kvc_h2o_accumulate_evict: sizes");
    const int n_heads = n_heads_kv;
    int32_t *code = nullptr;
    kvc_status st = device_info(&code, nullptr);
    if (st != KVC_OK) return st;
    kvc::H2OParams p{};
    p.logits = logits; p.logits_stride = logits_stride; p.lse = lse;
    p.score = score; p.pos = pos; p.stride = stride; p.free_slot = free_slot;
    p.rows = batch * n_heads; p.n_slots = n_slots; p.L_local = L_local; p.budget = budget;
    p.G = n_heads_q / n_heads_kv;
    p.t = t; p.dev_code = code;
    cudaError_t e = kvc::launch_h2o_accumulate_evict(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "H2O launch");
    return ok();
}

// H2O prefill workspace: [s_full] [row states] [row lse].
static void h2o_layout(int B, int H, int N, int n_sm, size_t *off_s, kvc::ScorePlan *pl)
{
    *off_s = 0;
    const size_t base = align256((size_t)B * H * N * sizeof(float));
    *pl = kvc::score_plan(B, H, 1, N, N, n_sm, base);
}

size_t kvc_h2o_prefill_workspace_bytes(int32_t batch, int32_t n_heads, int32_t d_head,
                                       int32_t seq_len)
{
    (void)d_head;
    if (batch <= 0 || n_heads <= 0 || seq_len <= 0) return 0;
    size_t off_s;
    kvc::ScorePlan pl;
    h2o_layout(batch, n_heads, seq_len, sm_count_or_default(), &off_s, &pl);
    return pl.bytes;
}

kvc_status kvc_h2o_prefill_select(const void *q, const kvc_cache *prompt, int32_t seq_len,
                                  int32_t L_local, int32_t K_hh, float scale, int32_t *idx_out,
                                  float *score_out, float *s_full, void *ws, size_t ws_bytes,
                                  void *stream)
{
    kvc_status st = check_cache(prompt, "kvc_h2o_prefill_select", false);
    if (st != KVC_OK) return st;
    if (q == nullptr || idx_out == nullptr || score_out == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_h2o_prefill_select: null pointer");
    if (seq_len <= 0 || seq_len > prompt->cap || L_local < 0 || K_hh < 0)
        return fail(KVC_ERR_SHAPE, "kvc_h2o_prefill_select: sizes");
    if (!std::isfinite(scale)) return fail(KVC_ERR_INVALID_ARG, "kvc_h2o_prefill_select: scale");
    int32_t *code = nullptr;
    int n_sm = 0;
    st = device_info(&code, &n_sm);
    if (st != KVC_OK) return st;
    const int B = prompt->batch, H = prompt->n_heads_kv, N = seq_len;
    size_t off_s;
    kvc::ScorePlan pl;
    h2o_layout(B, H, N, n_sm, &off_s, &pl);
    if (ws == nullptr || ws_bytes < pl.bytes || !aligned256(ws))
        return fail(KVC_ERR_WORKSPACE, "kvc_h2o_prefill_select: workspace needs %zu aligned bytes",
                    pl.bytes);
    char *wsb = static_cast<char *>(ws);
    float *sf = s_full ? s_full : reinterpret_cast<float *>(wsb + off_s);
    kvc::ScoreParams sp{};
    sp.q = q; sp.k = prompt->k;
    sp.sb = prompt->stride_b; sp.sh = prompt->stride_h; sp.ss = prompt->stride_slot;
    sp.B = B; sp.Hq = H; sp.Hkv = H; sp.G = 1; sp.D = prompt->d_head; sp.N = N; sp.L_obs = N;
    sp.scale_log2 = scale * 1.4426950408889634f;
    sp.n_cols = N;
    sp.col_mult = 1.0f;
    sp.s_out = sf;
    sp.row_ml = reinterpret_cast<float *>(wsb + pl.off_ml);
    sp.row_lse2 = reinterpret_cast<float *>(wsb + pl.off_lse);
    sp.n_chunks = pl.n_chunks;
    sp.chunk = pl.chunk;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = run_scores(sp, prompt->dtype, scale, code, s);
    if (e != cudaSuccess) return cuda_fail(e, "prompt scores launch");
    const long long keep_ll = (long long)K_hh + L_local;
    const int n_keep = (int)std::min<long long>(N, keep_ll);
    if (N <= keep_ll) {
        e = kvc::launch_iota_rows(idx_out, n_keep, B * H, n_keep, s);
    } else {
        e = kvc::launch_topk_rows(sf, N, B * H, N - L_local, K_hh, L_local, idx_out, n_keep, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "H2O selection launch");
    e = kvc::launch_gather_scores(sf, N, idx_out, n_keep, B * H, n_keep, score_out, s);
    if (e != cudaSuccess) return cuda_fail(e, "score gather launch");
    return ok();
}

// Grouped-query prompt selection: [s_acc][s_g][q of one group member][scoring plan].
static size_t h2o_gqa_layout(int B, int Hkv, int N, int D, int eb, int n_sm, size_t *off_g,
                             size_t *off_q, kvc::ScorePlan *pl)
{
    const size_t s_bytes = align256((size_t)B * Hkv * N * sizeof(float));
    *off_g = s_bytes;
    *off_q = 2 * s_bytes;
    const size_t base = *off_q + align256((size_t)B * Hkv * N * D * eb);
    *pl = kvc::score_plan(B, Hkv, 1, N, N, n_sm, base);
    return pl->bytes;
}

size_t kvc_h2o_prefill_gqa_workspace_bytes(int32_t batch, int32_t n_heads_kv, int32_t d_head,
                                           int32_t seq_len, int32_t dtype)
{
    if (batch <= 0 || n_heads_kv <= 0 || seq_len <= 0 || d_head <= 0 ||
        (dtype != KVC_F32 && dtype != KVC_BF16))
        return 0;
    size_t og, oq;
    kvc::ScorePlan pl;
    return h2o_gqa_layout(batch, n_heads_kv, seq_len, d_head, elem_bytes(dtype),
                          sm_count_or_default(), &og, &oq, &pl);
}

kvc_status kvc_h2o_prefill_select_gqa(const void *q, int32_t n_heads_q, const kvc_cache *prompt,
                                      int32_t seq_len, int32_t L_local, int32_t K_hh,
                                      float scale, int32_t *idx_out, float *score_out,
                                      float *s_full, void *ws, size_t ws_bytes, void *stream)
{
    kvc_status st = check_cache(prompt, "kvc_h2o_prefill_select_gqa", false);
    if (st != KVC_OK) return st;
    if (q == nullptr || idx_out == nullptr || score_out == nullptr)
        return fail(KVC_ERR_INVALID_ARG, "kvc_h2o_prefill_select_gqa: null pointer");
    if (!aligned16(q)) return fail(KVC_ERR_ALIGN, "kvc_h2o_prefill_select_gqa: q alignment");
    const int Hkv = prompt->n_heads_kv;
    if (n_heads_q <= 0 || n_heads_q % Hkv)
        return fail(KVC_ERR_SHAPE, "kvc_h2o_prefill_select_gqa: n_heads_q %d not a multiple of "
                    "%d KV heads", n_heads_q, Hkv);
    if (seq_len <= 0 || seq_len > prompt->cap || L_local < 0 || K_hh < 0)
        return fail(KVC_ERR_SHAPE, "kvc_h2o_prefill_select_gqa: sizes");
    if (!std::isfinite(scale))
        return fail(KVC_ERR_INVALID_ARG, "kvc_h2o_prefill_select_gqa: scale");
    int32_t *code = nullptr;
    int n_sm = 0;
    st = device_info(&code, &n_sm);
    if (st != KVC_OK) return st;
    const int B = prompt->batch, N = seq_len, D = prompt->d_head, G = n_heads_q / Hkv;
    const int eb = elem_bytes(prompt->dtype);
    size_t off_g, off_q;
    kvc::ScorePlan pl;
    const size_t need = h2o_gqa_layout(B, Hkv, N, D, eb, n_sm, &off_g, &off_q, &pl);
    if (ws == nullptr || ws_bytes < need || !aligned256(ws))
        return fail(KVC_ERR_WORKSPACE, "kvc_h2o_prefill_select_gqa: workspace needs %zu aligned "
                    "bytes", need);
    char *wsb = static_cast<char *>(ws);
    float *acc = s_full ? s_full : reinterpret_cast<float *>(wsb);
    float *sg = reinterpret_cast<float *>(wsb + off_g);
    void *qg = wsb + off_q;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kvc::ScoreParams sp{};
    sp.q = qg; sp.k = prompt->k;
    sp.sb = prompt->stride_b; sp.sh = prompt->stride_h; sp.ss = prompt->stride_slot;
    sp.B = B; sp.Hq = Hkv; sp.Hkv = Hkv; sp.G = 1; sp.D = D; sp.N = N; sp.L_obs = N;
    sp.scale_log2 = scale * 1.4426950408889634f;
    sp.n_cols = N;
    sp.col_mult = 1.0f;
    sp.row_ml = reinterpret_cast<float *>(wsb + pl.off_ml);
    sp.row_lse2 = reinterpret_cast<float *>(wsb + pl.off_lse);
    sp.n_chunks = pl.n_chunks;
    sp.chunk = pl.chunk;
    cudaError_t e;
    for (int g = 0; g < G; ++g) {
        // member g of every group, then its causal column sums, added in head order
        e = kvc::launch_group_member_copy(q, qg, B, Hkv, G, g, N, D * eb, s);
        if (e != cudaSuccess) return cuda_fail(e, "group member copy launch");
        sp.s_out = g == 0 ? acc : sg;
        e = run_scores(sp, prompt->dtype, scale, code, s);
        if (e != cudaSuccess) return cuda_fail(e, "prompt scores launch");
        if (g > 0) {
            e = kvc::launch_add_rows(acc, sg, (long long)B * Hkv * N, s);
            if (e != cudaSuccess) return cuda_fail(e, "group sum launch");
        }
    }
    const long long keep_ll = (long long)K_hh + L_local;
    const int n_keep = (int)std::min<long long>(N, keep_ll);
    if (N <= keep_ll)
        e = kvc::launch_iota_rows(idx_out, n_keep, B * Hkv, n_keep, s);
    else
        e = kvc::launch_topk_rows(acc, N, B * Hkv, N - L_local, K_hh, L_local, idx_out, n_keep, s);
    if (e != cudaSuccess) return cuda_fail(e, "H2O selection launch");
    e = kvc::launch_gather_scores(acc, N, idx_out, n_keep, B * Hkv, n_keep, score_out, s);
    if (e != cudaSuccess) return cuda_fail(e, "score gather launch");
    return ok();
}

}  // extern "C"
