// obs_scores_tc.cu -- observation-window attention scores on the 5th-generation tensor cores.
//
// SnapKV steps 1-2 ("Compressão e Poda Dinâmica de KV Cache", "SnapKV e a seleção de contexto
// no prefill") and H2O's prompt column sums (section "Heavy-Hitter Oracle (H2O)..."), for bf16
// inputs.  The product of the window queries with the prompt keys is a genuine dense
// contraction (rows x keys x d_head), so it runs on tcgen05.mma (bf16 operands, fp32
// accumulators in tensor memory); softmax and the reductions run in the epilogue warps.
//
// Same two passes as the CUDA-core kernels (obs_scores.cu):
//   pass 1 (ROWSTATS): A = a 128-row tile of window queries, B = 128-key tiles streamed along
//     the prompt; the accumulator has one row per TMEM lane, so each epilogue thread folds its
//     own row's logits into a running (max, sum of exp2) with no cross-thread reduction;
//   pass 2 (COLSUM): the transposed product, A = 128-key tiles, B = 128-row blocks of the
//     window queries; the accumulator has one key per TMEM lane, so each epilogue thread sums
//     its key's probabilities exp2(l - lse) over the rows of each query head, again without
//     cross-thread reduction, and writes each column sum once (deterministic).  When every head
//     lies inside one 128-row block (SnapKV windows of 32, 64 or 128 queries), a block keeps one
//     row block resident and streams a chunk of key tiles; otherwise (H2O's whole-prompt
//     window, one head of many row blocks) a block keeps one key tile and streams the row
//     blocks that can see it.
//
// Block roles (320 threads): warp 0 issues TMA loads (cp.async.bulk.tensor, 128-byte swizzle,
// K-major tiles of 128 rows x 64 elements), warp 1 owns the tensor-memory allocation and one
// of its threads issues the MMAs (M = N = 128, K = 16 per instruction) and the commits, warps
// 2-9 are the epilogue in two sets of four (each warp reads its 32 TMEM lanes with tcgen05.ld).
// The epilogue (exp2 and sums of 16K logits per tile) is the long stage, so the two sets take
// alternate tiles: with four accumulators in tensor memory the MMAs run up to four tiles ahead
// and two epilogue warps share each scheduler.  Operand stages and accumulators are handed over
// with mbarriers; every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int TC_ROWS = 128;         // MMA M and N
constexpr int TC_THREADS = 320;      // TMA warp, MMA warp, two epilogue sets of four warps
constexpr int TC_SUB_BYTES = TC_ROWS * 128;   // one 128-row x 64-element bf16 sub-tile
constexpr int TC_NACC = 4;                    // fp32 accumulators of 128 columns
constexpr uint32_t TC_TMEM_COLS = 128 * TC_NACC;

// ---- tcgen05 / TMA helpers ---------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
// The same load with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap *map, int c0,
                                                 int c1, int c2, int c3, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
        "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;               // leading-dimension offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;     // stride between 8-row groups
    d |= (uint64_t)1 << 46;               // descriptor version
    d |= (uint64_t)2 << 61;               // 128-byte swizzle
    return d;
}
// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major, M = N = 128.
constexpr uint32_t kIdescBf16M128N128 =
    (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdescBf16M128N128), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                     "r"(bar)
                 : "memory");
}
// All 128 columns of a tile (four 32-column loads, one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[4][32])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t *r = reinterpret_cast<uint32_t *>(v[c]);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
            "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
              "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
              "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
              "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
              "=r"(r[31])
            : "r"(taddr + c * 32));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 columns, issued without waiting (tmem_wait_ld before the registers are read).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, float (&v)[32])
{
    uint32_t *r = reinterpret_cast<uint32_t *>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 64 columns (two 32-column loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[2][32])
{
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t *r = reinterpret_cast<uint32_t *>(v[c]);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
            "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
              "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
              "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
              "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
              "=r"(r[31])
            : "r"(taddr + c * 32));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// sum_j exp2(v[j] * scale + off[j]) over 32 values with packed fp32x2 FMA and adds (two
// independent chains); `off` is one value for all (off_u) or per element (off_v, 16-byte aligned).
__device__ __forceinline__ float exp2_sum32(const float *v, float scale, float off_u,
                                            const float *off_v)
{
    const float2 s2 = make_float2(scale, scale);
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 o = off_v ? *reinterpret_cast<const float4 *>(off_v + j)
                               : make_float4(off_u, off_u, off_u, off_u);
        const float2 o0 = make_float2(o.x, o.y), o1 = make_float2(o.z, o.w);
        float2 x = __ffma2_rn(make_float2(v[j], v[j + 1]), s2, o0);
        float2 y = __ffma2_rn(make_float2(v[j + 2], v[j + 3]), s2, o1);
        x.x = ex2(x.x);
        x.y = ex2(x.y);
        y.x = ex2(y.x);
        y.y = ex2(y.y);
        a0 = __fadd2_rn(a0, x);
        a1 = __fadd2_rn(a1, y);
    }
    const float2 a = __fadd2_rn(a0, a1);
    return a.x + a.y;
}
__device__ __forceinline__ float max32(const float *x)
{
    float a0 = x[0], a1 = x[1], a2 = x[2], a3 = x[3];
#pragma unroll
    for (int j = 4; j < 32; j += 4) {
        a0 = fmaxf(a0, x[j]);
        a1 = fmaxf(a1, x[j + 1]);
        a2 = fmaxf(a2, x[j + 2]);
        a3 = fmaxf(a3, x[j + 3]);
    }
    return fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
}

// After a wait ran out (the device code is set), a block's producer waits (bounded) for the last
// phase of each of the n ring barriers it armed (`used` loads in all, load j on barrier j % n),
// so that no copy is still writing into shared memory when the block exits.  In normal
// operation nothing is waited for: the drain is skipped.
__device__ __forceinline__ bool timeout_recorded(const int32_t *code)
{
    return code != nullptr && *reinterpret_cast<const volatile int32_t *>(code) != 0;
}
__device__ __forceinline__ void drain_loads(uint32_t bars, int n, long long used, int32_t *code)
{
    for (long long j = used > n ? used - n : 0; j < used; ++j)
        if (!mbar_wait_ok(bars + 8 * (uint32_t)(j % n), (uint32_t)((j / n) & 1), kMbarSpinLimit))
            record_code(code, kDevCodeTimeout);
}

// Named barriers: 1 over every epilogue warp that takes part (128 threads per set), 2 + set
// over the four warps of one set.
__device__ __forceinline__ void epilogue_sync(int nsets)
{
    asm volatile("bar.sync 1, %0;" ::"r"(128 * nsets) : "memory");
}
__device__ __forceinline__ void set_sync(int set)
{
    asm volatile("bar.sync %0, 128;" ::"r"(2 + set) : "memory");
}

// Column sums over one block of rows r0 .. r0 + rows_blk - 1 (tensor-memory columns from tcol,
// 64 per read, or 32 with LD32: half the registers) for this thread's key.  (g_cur, acc_g) carry the sum of the head in progress; a
// finished head's sum (times col_mult) goes to out[head * out_stride + out_idx] when out_ok.
// nlse: the rows' negated log2-sum-exp.  The head g_a and row-in-head rem of each 32-row chunk
// advance incrementally (heads have at least 32 rows, or there is one head).
template <bool LD32 = false>
__device__ __forceinline__ void colsum_rows(const ScoreParams &p, int first_pos, uint32_t tcol,
                                            int r0, int rows_blk, int key, bool mask_tile,
                                            const float *nlse, float *out, int out_stride,
                                            int out_idx, bool out_ok, int &g_cur, float &acc_g)
{
    int g_a = r0 / p.L_obs;
    int rem = r0 - g_a * p.L_obs;
    float vt[2][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c * 32 >= rows_blk) break;
        // LD32: 32 columns per tensor-memory read; otherwise 64 (one wait for two chunks)
        if (LD32) {
            tmem_ld32_async(tcol + c * 32, vt[0]);
            tmem_wait_ld();
        } else if ((c & 1) == 0) tmem_ld64(tcol + c * 32, vt);
        const float *v = vt[LD32 ? 0 : (c & 1)];
        const int rows_here = min(32, rows_blk - c * 32);
        const int split = min(rows_here, p.L_obs - rem);      // rows in head g_a
        if (g_a != g_cur) {                                   // flush the finished head
            if (out_ok) out[(size_t)g_cur * out_stride + out_idx] = acc_g * p.col_mult;
            acc_g = 0.f;
            g_cur = g_a;
        }
        // rows see keys up to their positions; the smallest in the chunk is its first row, or
        // the next head's first window row past a head boundary
        const bool mask_c = mask_tile && key > first_pos + (split < rows_here ? 0 : rem);
        if (split == 32 && !mask_c) {
            acc_g += exp2_sum32(v, p.scale_log2, 0.f, nlse + c * 32);
        } else {
            float s_a = 0.f, s_b = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float pr = ex2(fmaf(v[j], p.scale_log2, nlse[c * 32 + j]));
                if (mask_c) {
                    const int w = j < split ? rem + j : j - split;   // row inside its head
                    if (key > first_pos + w) pr = 0.f;
                }
                if (j < split) s_a += pr;
                else if (j < rows_here) s_b += pr;
            }
            acc_g += s_a;
            if (split < rows_here) {                          // into head g_a + 1
                if (out_ok) out[(size_t)g_cur * out_stride + out_idx] = acc_g * p.col_mult;
                g_cur = g_a + 1;
                acc_g = s_b;
            }
        }
        rem += 32;
        if (rem >= p.L_obs) {
            rem -= p.L_obs;
            ++g_a;
        }
    }
}

// Row statistics of one 128-key tile for this thread's row (accumulator lanes = rows): the
// logits past the row's position (or past the prompt) are masked, then the running (max, sum
// of exp2) in log2 units is updated.
__device__ __forceinline__ void rowstats_tile(uint32_t taddr, int k0, int pos, int N,
                                              float scale_log2, float &m_run, float &z_run)
{
    // this row sees keys up to its own position: mask only where the tile reaches past it (or
    // past the prompt)
    const bool need_mask = k0 + TC_ROWS - 1 > pos || k0 + TC_ROWS > N;
    float v[4][32];
    tmem_ld128(taddr, v);
    if (need_mask) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int key = k0 + c * 32 + j;
                if (key > pos || key >= N) v[c][j] = -INFINITY;
            }
    }
    const float mx = fmaxf(fmaxf(max32(v[0]), max32(v[1])), fmaxf(max32(v[2]), max32(v[3])));
    const float m_new = fmaxf(m_run, mx * scale_log2);
    const float z = (exp2_sum32(v[0], scale_log2, -m_new, nullptr) +
                     exp2_sum32(v[1], scale_log2, -m_new, nullptr)) +
                    (exp2_sum32(v[2], scale_log2, -m_new, nullptr) +
                     exp2_sum32(v[3], scale_log2, -m_new, nullptr));
    z_run = z_run * ex2(m_run - m_new) + z;
    m_run = m_new;
}

// The same update for 64 keys k0 .. k0 + 63 (one tensor-memory read), with a lazy running max:
// the exp2 values are summed relative to the running max as it stands, without finding the
// keys' max first; only when that sum comes out above 2^32 (a logit more than 32 above the
// running max, and always on a row's first visible keys, whose running max is still kNegBig)
// is their max taken and the sum rescaled to it.  z_run is then a sum relative to m_run that
// may exceed 1, which every (m, z) merge downstream handles as it stands.
__device__ __forceinline__ void rowstats_half_lazy(uint32_t taddr, int k0, int pos, int N,
                                                   float scale_log2, float &m_run, float &z_run)
{
    const bool need_mask = k0 + 63 > pos || k0 + 64 > N;
    float v[2][32];
    tmem_ld64(taddr, v);
    if (need_mask) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int key = k0 + c * 32 + j;
                if (key > pos || key >= N) v[c][j] = -INFINITY;
            }
    }
    const float z = exp2_sum32(v[0], scale_log2, -m_run, nullptr) +
                    exp2_sum32(v[1], scale_log2, -m_run, nullptr);
    if (z <= 4294967296.f) {
        z_run += z;
        return;
    }
    const float m_new = fmaxf(m_run, fmaxf(max32(v[0]), max32(v[1])) * scale_log2);
    const float zn = exp2_sum32(v[0], scale_log2, -m_new, nullptr) +
                     exp2_sum32(v[1], scale_log2, -m_new, nullptr);
    z_run = z_run * ex2(m_run - m_new) + zn;
    m_run = m_new;
}

struct TcParams {
    ScoreParams sp;       // shapes, scale, outputs, workspace (see internal.h)
    int32_t n_mtiles;     // row tiles of 128 per (batch, KV head)    (pass 1)
    int32_t chunk_tiles;  // key tiles of 128 per pass-1 block
    int32_t n_col_tiles;  // key tiles of 128 covering the n_cols written columns (pass 2)
    int32_t col_chunks;   // pass 2 with a resident row block: key-tile chunks per row block
    int32_t col_chunk_tiles;
    int32_t n_work;       // work items of the launch (blocks take them round-robin)
    int32_t n_fp;         // resident tile pairs per (pair, chunk) (tile-pair kernel)
    int32_t n_sup;        // units per (pair, chunk): resident pairs i and n_fp - 1 - i together
    int32_t *dev_code;
};

// Window row r of the group -> (head g, text position) with rows ordered g*L_obs + w.
__device__ __forceinline__ int row_pos(const ScoreParams &p, int r)
{
    return p.N - p.L_obs + (r % p.L_obs);
}

// One work item: a resident ("fixed") operand tile and a run of streamed tiles.
//   MODE 0: fixed = a 128-row tile of window queries, streamed = key tiles of one chunk;
//   MODE 1: fixed = one key tile, streamed = the row blocks that can see it;
//   MODE 2: fixed = a 128-row block holding whole heads, streamed = key tiles of one chunk.
struct TcItem {
    int pair, fixed_row0, t_begin, n_tiles, chunk, ktile;
};

template <int MODE>
__device__ __forceinline__ TcItem tc_item(const TcParams &tp, int u)
{
    const ScoreParams &p = tp.sp;
    const int R = p.G * p.L_obs;
    const int first_pos = p.N - p.L_obs;
    TcItem it{};
    if (MODE == 0) {
        const int per_pair = tp.n_mtiles * p.n_chunks;
        it.pair = u / per_pair;
        const int mtile = (u % per_pair) / p.n_chunks;
        it.chunk = u % p.n_chunks;
        // keys a row tile can see: up to the largest position among its rows
        const int r_lo = mtile * TC_ROWS;
        const int r_hi = min(r_lo + TC_ROWS, R) - 1;
        const int w_hi = (r_lo / p.L_obs != r_hi / p.L_obs) ? p.L_obs - 1 : r_hi % p.L_obs;
        const int kt_needed = (first_pos + w_hi) / TC_ROWS + 1;
        it.t_begin = it.chunk * tp.chunk_tiles;
        it.n_tiles = max(0, min(it.t_begin + tp.chunk_tiles, kt_needed) - it.t_begin);
        it.fixed_row0 = r_lo;
    } else if (MODE == 2) {
        const int n_rb = (R + TC_ROWS - 1) / TC_ROWS;
        const int per_pair = n_rb * tp.col_chunks;
        it.pair = u / per_pair;
        const int mtile = (u % per_pair) / tp.col_chunks;      // resident row block
        it.chunk = u % tp.col_chunks;
        it.t_begin = it.chunk * tp.col_chunk_tiles;              // first key tile
        it.n_tiles = max(0, min(it.t_begin + tp.col_chunk_tiles, tp.n_col_tiles) - it.t_begin);
        it.fixed_row0 = mtile * TC_ROWS;
    } else {
        it.pair = u / tp.n_col_tiles;
        it.ktile = u % tp.n_col_tiles;
        // row blocks whose rows can see this key tile: positions >= its first key
        const int k0 = it.ktile * TC_ROWS;
        int rb0 = 0;
        if (k0 > first_pos) rb0 = (k0 - first_pos) / TC_ROWS;   // rows sorted by position when G = 1
        if (p.G > 1) rb0 = 0;
        it.t_begin = rb0;
        it.n_tiles = max(0, (R + TC_ROWS - 1) / TC_ROWS - rb0);
    }
    return it;
}

// CONTIG: blocks take contiguous item ranges whose items mostly share the resident tile (the key
// chunks of one pair), which is then reloaded only when it changes, from one buffer; the room
// goes to more streamed stages.  Otherwise items are taken round-robin and every item reloads
// (double-buffered where it fits).
template <int D, bool CONTIG>
struct TcPlan {
    static constexpr int SUBS = D / 64;                       // 64-element sub-tiles per tile
    static constexpr int TILE_BYTES = SUBS * TC_SUB_BYTES;
    static constexpr int NFIX = (CONTIG || D >= 256) ? 1 : 2;  // resident tile buffers
    static constexpr int NS_RAW = (200 * 1024 - NFIX * TILE_BYTES) / TILE_BYTES;
    static constexpr int NS_CAP = CONTIG ? 8 : 4;
    static constexpr int NS = NS_RAW > NS_CAP ? NS_CAP : NS_RAW;   // streamed tiles in flight
    static_assert(NS >= 2, "tensor-core scoring needs two operand stages");
    static constexpr int BAR_BYTES = 8 * (2 * NFIX + 2 * NS + 2 * TC_NACC + 2) + 16;
    static constexpr int SMEM_USED = 1024 + (NFIX + NS) * TILE_BYTES + BAR_BYTES +
                                     4 * TC_ROWS * 4 + 2 * TC_ROWS * 2 * 4 + 64;
    // every block allocates all of tensor memory: one block per SM, so at least half the SM's
    // shared memory is requested
    static constexpr int SMEM = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
};

// Persistent blocks: block c takes a contiguous range of work items (CONTIG) or the items
// c, c + gridDim.x, ...  The roles walk the same item sequence; stage, accumulator and
// epilogue-set indices follow block-global tile counters; the resident tile is loaded into the
// next of NFIX buffers whenever an item's resident tile differs from the previous item's, and the
// MMA thread releases a buffer after the last item that uses it.
// MODE 0: row statistics; 1: column sums, key tile resident; 2: column sums, row block resident
template <int D, int MODE, bool CONTIG>
__global__ void __launch_bounds__(TC_THREADS, 1)
tc_scores_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 const TcParams tp)
{
    using PL = TcPlan<D, CONTIG>;
    constexpr int SUBS = PL::SUBS, TILE_BYTES = PL::TILE_BYTES, NFIX = PL::NFIX, NS = PL::NS;
    constexpr int KSTEPS = D / 16;
    const ScoreParams &p = tp.sp;
    // epilogue sets: with a resident key tile the column sums carry across row blocks; two sets
    // (alternate row blocks, partial sums merged per item) when every row is one head, one set
    // when a key's column crosses heads
    const int NSETS = (MODE == 1 && p.G > 1) ? 1 : 2;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned operand area (the swizzle pattern is anchored to 1024-byte lines)
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t fixed0 = base;                         // NFIX resident tiles
    const uint32_t stage0 = base + NFIX * TILE_BYTES;     // NS streamed tiles
    const uint32_t bars = stage0 + NS * TILE_BYTES;       // mbarriers
    const uint32_t bar_fix_full = bars;                   // NFIX
    const uint32_t bar_fix_empty = bar_fix_full + 8 * NFIX;   // NFIX
    const uint32_t bar_full = bar_fix_empty + 8 * NFIX;   // NS
    const uint32_t bar_empty = bar_full + 8 * NS;         // NS
    const uint32_t bar_acc_full = bar_empty + 8 * NS;     // TC_NACC
    const uint32_t bar_acc_empty = bar_acc_full + 8 * TC_NACC;   // TC_NACC
    const uint32_t bar_done = bar_acc_empty + 8 * TC_NACC;       // the MMA thread's last commit
    const uint32_t tmem_slot = bar_done + 16;                    // u32 written by tcgen05.alloc
    float *sm_lse = reinterpret_cast<float *>(smem_raw + (tmem_slot + 16 - raw));   // [4][128]
    float *sm_mz = sm_lse + 4 * TC_ROWS;                  // [2][128][2] second set's states

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int R = p.G * p.L_obs;
    const int first_pos = p.N - p.L_obs;
    const int C = gridDim.x;
    // this block's item sequence
    const int u_first = CONTIG ? (int)((long long)blockIdx.x * tp.n_work / C) : (int)blockIdx.x;
    const int u_end = CONTIG ? (int)((long long)(blockIdx.x + 1) * tp.n_work / C) : tp.n_work;
    const int u_step = CONTIG ? 1 : C;
    // identity of an item's resident tile
    auto fixed_id = [&](const TcItem &it) -> long long {
        return (long long)it.pair * (1LL << 32) + (MODE == 1 ? it.ktile : it.fixed_row0);
    };

    if (threadIdx.x == 0) {
        for (int f = 0; f < NFIX; ++f) {
            mbar_init(bar_fix_full + 8 * f, 1);
            mbar_init(bar_fix_empty + 8 * f, 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int a = 0; a < TC_NACC; ++a) {
            mbar_init(bar_acc_full + 8 * a, 1);
            mbar_init(bar_acc_empty + 8 * a, 4);   // the four warps of the set owning it
        }
        mbar_init(bar_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         tmem_slot),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t tmem_base;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem_base) : "r"(tmem_slot));

    long long loads_streamed = 0;               // the producer's counts (for the drain)
    int loads_fixed = 0;
    if (warp == 0 && lane == 0) {
        // ================================ TMA producer ============================================
        long long g = 0;                            // streamed tiles so far
        int nrl = 0;                                // resident-tile loads so far
        long long prev_id = -1;
        // keys streamed once per pass (one row tile per pair) are marked evict-first, so that
        // what the pass writes (and the next kernel reads) is not pushed out of L2 by them
        const bool once = MODE != 1 && tp.n_mtiles == 1;
        const uint64_t pol = l2_evict_first_policy();
        for (int u = u_first; u < u_end; u += u_step) {
            const TcItem it = tc_item<MODE>(tp, u);
            if (it.n_tiles == 0) continue;
            const int b = it.pair / p.Hkv, kh = it.pair % p.Hkv;
            const int qrow_group = (b * p.Hq + kh * p.G) * p.L_obs;
            const long long id = fixed_id(it);
            if (id != prev_id) {
                prev_id = id;
                const int f = nrl % NFIX;
                if (nrl >= NFIX)
                    mbar_wait(bar_fix_empty + 8 * f, ((nrl / NFIX) - 1) & 1, tp.dev_code);
                const uint32_t fx = fixed0 + f * TILE_BYTES;
                mbar_arrive_expect_tx(bar_fix_full + 8 * f, TILE_BYTES);
                for (int a = 0; a < SUBS; ++a) {
                    if (MODE != 1)
                        tma_load_2d(fx + a * TC_SUB_BYTES, &qmap, a * 64,
                                    qrow_group + it.fixed_row0, bar_fix_full + 8 * f);
                    else
                        tma_load_4d(fx + a * TC_SUB_BYTES, &kmap, a * 64, it.ktile * TC_ROWS, kh,
                                    b, bar_fix_full + 8 * f);
                }
                ++nrl;
            }
            for (int i = 0; i < it.n_tiles; ++i, ++g) {
                const int s = (int)(g % NS);
                if (g >= NS) mbar_wait(bar_empty + 8 * s, (int)((g / NS) - 1) & 1, tp.dev_code);
                const uint32_t dst = stage0 + s * TILE_BYTES;
                mbar_arrive_expect_tx(bar_full + 8 * s, TILE_BYTES);
                for (int a = 0; a < SUBS; ++a) {
                    if (MODE != 1 && once)
                        tma_load_4d_hint(dst + a * TC_SUB_BYTES, &kmap, a * 64,
                                         (it.t_begin + i) * TC_ROWS, kh, b, bar_full + 8 * s, pol);
                    else if (MODE != 1)
                        tma_load_4d(dst + a * TC_SUB_BYTES, &kmap, a * 64,
                                    (it.t_begin + i) * TC_ROWS, kh, b, bar_full + 8 * s);
                    else
                        tma_load_2d(dst + a * TC_SUB_BYTES, &qmap, a * 64,
                                    qrow_group + (it.t_begin + i) * TC_ROWS, bar_full + 8 * s);
                }
            }
        }
        loads_streamed = g;
        loads_fixed = nrl;
    } else if (warp == 1 && lane == 0) {
        // ================================ MMA issuer ==============================================
        long long g = 0;
        int nrl = 0, f = 0;
        long long prev_id = -1;
        for (int u = u_first; u < u_end; u += u_step) {
            const TcItem it = tc_item<MODE>(tp, u);
            if (it.n_tiles == 0) continue;
            const long long id = fixed_id(it);
            if (id != prev_id) {
                prev_id = id;
                f = nrl % NFIX;
                mbar_wait(bar_fix_full + 8 * f, (nrl / NFIX) & 1, tp.dev_code);
                ++nrl;
            }
            const uint32_t fx = fixed0 + f * TILE_BYTES;
            for (int i = 0; i < it.n_tiles; ++i, ++g) {
                const int s = (int)(g % NS), ab = (int)(g % TC_NACC);
                mbar_wait(bar_full + 8 * s, (int)(g / NS) & 1, tp.dev_code);
                if (g >= TC_NACC)
                    mbar_wait(bar_acc_empty + 8 * ab, (int)((g / TC_NACC) - 1) & 1, tp.dev_code);
                tc_fence_after();
                // MODE 0/1: A = resident tile, B = streamed tile; MODE 2: A = streamed keys,
                // B = resident rows (the accumulator then has one key per lane)
                const uint32_t a_base = MODE == 2 ? stage0 + s * TILE_BYTES : fx;
                const uint32_t b_base = MODE == 2 ? fx : stage0 + s * TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const uint32_t off = (kk >> 2) * TC_SUB_BYTES + (kk & 3) * 32;
                    umma_bf16(tmem_base + ab * 128, sw128_desc(a_base + off),
                              sw128_desc(b_base + off), kk > 0 ? 1u : 0u);
                }
                umma_commit(bar_empty + 8 * s);       // operand stage free once the MMAs finish
                umma_commit(bar_acc_full + 8 * ab);   // accumulator ready for the epilogue
            }
            // release the resident buffer after its last item: the next item with tiles loads
            // a different resident tile (or there is none)
            long long next_id = -1;
            for (int v = u + u_step; v < u_end; v += u_step) {
                const TcItem nx = tc_item<MODE>(tp, v);
                if (nx.n_tiles > 0) {
                    next_id = fixed_id(nx);
                    break;
                }
            }
            if (next_id != -1 && next_id != id) umma_commit(bar_fix_empty + 8 * f);
        }
    } else if (warp >= 2 && (warp - 2) / 4 < NSETS) {
        // ================================ epilogue ================================================
        const int set = (warp - 2) / 4;           // global tiles g with g % NSETS == set
        const int q4 = warp & 3;                  // TMEM lanes 32*q4 .. 32*q4+31
        const int et = q4 * 32 + lane;            // this thread's lane (row or key)
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        long long g = 0;
        int k = 0;
        // MODE 2: this thread's resident row, its negated log2-sum-exp, and whose it is
        long long nlse_id = -1;
        float my_nlse = 0.f;
        for (int u = u_first; u < u_end; u += u_step) {
            const TcItem it = tc_item<MODE>(tp, u);
            const int b = it.pair / p.Hkv, kh = it.pair % p.Hkv;
            if (MODE == 0) {
                const int r = it.fixed_row0 + et;     // window row of the group
                const bool row_ok = r < R;
                float *dst = p.row_ml + (((size_t)it.pair * p.n_chunks + it.chunk) * R + r) * 2;
                if (it.n_tiles == 0) {
                    // no key tile reaches these rows: an empty state for every row
                    if (set == 0 && row_ok) {
                        dst[0] = kNegBig;
                        dst[1] = 0.f;
                    }
                    continue;
                }
                const int pos = row_ok ? row_pos(p, r) : -1;
                float m_run = kNegBig, z_run = 0.f;
                for (int i = 0; i < it.n_tiles; ++i) {
                    const long long gg = g + i;
                    if ((int)(gg % NSETS) != set) continue;
                    const int ab = (int)(gg % TC_NACC);
                    mbar_wait(bar_acc_full + 8 * ab, (int)(gg / TC_NACC) & 1, tp.dev_code);
                    tc_fence_after();
                    rowstats_tile(tmem_base + ab * 128 + lane_off, (it.t_begin + i) * TC_ROWS, pos,
                                  p.N, p.scale_log2, m_run, z_run);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acc_empty + 8 * ab);
                }
                // the second set hands its row states to the first, which merges and writes
                float *mz = sm_mz + (k & 1) * 2 * TC_ROWS;
                if (set == 1) {
                    mz[2 * et] = m_run;
                    mz[2 * et + 1] = z_run;
                }
                epilogue_sync(NSETS);
                if (set == 0 && row_ok) {
                    const float m1 = mz[2 * et], z1 = mz[2 * et + 1];
                    const float M = fmaxf(m_run, m1);
                    dst[0] = M;
                    dst[1] = z_run * ex2(m_run - M) + z1 * ex2(m1 - M);
                }
            } else if (MODE == 2) {
                if (it.n_tiles == 0) continue;
                // resident rows fixed_row0 .. +127 hold whole heads: per key tile, each thread
                // sums its key's column over each head and writes it (lse_buf holds -lse)
                float *lse_buf = sm_lse + (k & 1) * TC_ROWS;
                if (set == 0) {
                    // the row's log2-sum-exp from pass 1's per-chunk (max, sum) states, when
                    // the resident row block changes (same arithmetic as rowlse_tc_kernel)
                    const long long id = fixed_id(it);
                    if (id != nlse_id) {
                        nlse_id = id;
                        const int r = it.fixed_row0 + et;
                        my_nlse = 0.f;
                        if (r < R) {
                            const float *st = p.row_ml + ((size_t)it.pair * p.n_chunks * R + r) * 2;
                            const size_t cstep = (size_t)R * 2;
                            float M = kNegBig;
                            for (int c = 0; c < p.n_chunks; ++c) M = fmaxf(M, st[c * cstep]);
                            float Z = 0.f;
                            for (int c = 0; c < p.n_chunks; ++c)
                                Z += st[c * cstep + 1] * exp2f(st[c * cstep] - M);
                            my_nlse = -(M + log2f(Z));
                        }
                    }
                    lse_buf[et] = my_nlse;
                }
                epilogue_sync(NSETS);
                float *s_base = p.s_out + (size_t)(b * p.Hq + kh * p.G) * p.n_cols;
                const int rows_blk = min(TC_ROWS, R - it.fixed_row0);
                for (int i = 0; i < it.n_tiles; ++i) {
                    const long long gg = g + i;
                    if ((int)(gg % NSETS) != set) continue;
                    const int ab = (int)(gg % TC_NACC);
                    const int key = (it.t_begin + i) * TC_ROWS + et;
                    const bool mask_tile = (it.t_begin + i) * TC_ROWS + TC_ROWS - 1 > first_pos;
                    mbar_wait(bar_acc_full + 8 * ab, (int)(gg / TC_NACC) & 1, tp.dev_code);
                    tc_fence_after();
                    int g_cur = it.fixed_row0 / p.L_obs;
                    float acc_g = 0.f;
                    colsum_rows(p, first_pos, tmem_base + ab * 128 + lane_off, it.fixed_row0,
                                rows_blk, key, mask_tile, lse_buf, s_base, p.n_cols, key,
                                key < p.n_cols, g_cur, acc_g);
                    if (key < p.n_cols) s_base[(size_t)g_cur * p.n_cols + key] = acc_g * p.col_mult;
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acc_empty + 8 * ab);
                }
            } else {
                if (it.n_tiles == 0) continue;
                const int key = it.ktile * TC_ROWS + et;
                const float *lse_g = p.row_lse2 + (size_t)it.pair * tp.n_mtiles * TC_ROWS;
                const bool mask_tile = it.ktile * TC_ROWS + TC_ROWS - 1 > first_pos;
                float *s_base = p.s_out + (size_t)(b * p.Hq + kh * p.G) * p.n_cols;
                int g_cur = it.t_begin * TC_ROWS / p.L_obs;   // head of the first row handled
                float acc_g = 0.f;
                int n_mine = 0;                               // this set's row blocks so far
                // this thread's row of the set's next row block, loaded one block ahead
                auto lse_of = [&](int i) -> float {
                    const int r = (it.t_begin + i) * TC_ROWS + et;
                    return (i < it.n_tiles && r < R) ? lse_g[r] : 0.f;
                };
                const int i_first = (int)(((set - g) % NSETS + NSETS) % NSETS);
                float lse_next = lse_of(i_first);
                for (int i = 0; i < it.n_tiles; ++i) {
                    const long long gg = g + i;
                    if ((int)(gg % NSETS) != set) continue;
                    const int ab = (int)(gg % TC_NACC);
                    const int r0 = (it.t_begin + i) * TC_ROWS;   // first row of this block
                    // stage the block's negated row log2-sum-exp values (per set, double
                    // buffered)
                    float *lse_buf = sm_lse + (set * 2 + ((int)(gg / NSETS) & 1)) * TC_ROWS;
                    lse_buf[et] = lse_next;
                    lse_next = lse_of(i + NSETS);
                    set_sync(set);
                    mbar_wait(bar_acc_full + 8 * ab, (int)(gg / TC_NACC) & 1, tp.dev_code);
                    tc_fence_after();
                    ++n_mine;
                    colsum_rows(p, first_pos, tmem_base + ab * 128 + lane_off, r0,
                                min(TC_ROWS, R - r0), key, mask_tile, lse_buf, s_base, p.n_cols,
                                key, key < p.n_cols, g_cur, acc_g);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acc_empty + 8 * ab);
                }
                (void)n_mine;
                if (NSETS == 1) {
                    if (key < p.n_cols) s_base[(size_t)g_cur * p.n_cols + key] = acc_g * p.col_mult;
                } else {
                    // one head (G == 1): the second set hands its partial sum to the first
                    float *part = sm_mz + (k & 1) * 2 * TC_ROWS;
                    if (set == 1) part[et] = acc_g;
                    epilogue_sync(NSETS);
                    if (set == 0 && key < p.n_cols)
                        s_base[key] = (acc_g + part[et]) * p.col_mult;
                }
            }
            g += it.n_tiles;
            if (it.n_tiles > 0) ++k;
        }
    }

    tc_fence_before();
    __syncthreads();
    // after a wait ran out: the last loads have landed and every product issued has completed
    // before the block frees tensor memory and exits
    if ((threadIdx.x == 0 || threadIdx.x == 32) && timeout_recorded(tp.dev_code)) {
        if (threadIdx.x == 0) {
            drain_loads(bar_full, NS, loads_streamed, tp.dev_code);
            drain_loads(bar_fix_full, NFIX, loads_fixed, tp.dev_code);
        } else {
            umma_commit(bar_done);
            mbar_wait(bar_done, 0, tp.dev_code);
        }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TC_TMEM_COLS)
                     : "memory");
}

// ---- resident tile pairs ------------------------------------------------------------------------
// For windows of many 128-row tiles (H2O's whole-prompt window) a work item keeps TWO resident
// tiles, a pair of window-row tiles for the row statistics (MODE 0) or a pair of key tiles for
// the column sums (MODE 1), and streams the other operand once for both: each streamed tile
// feeds two products (A = resident tile e, B = streamed tile, so the accumulator lanes are rows
// in MODE 0 and keys in MODE 1), which doubles the product time per streamed byte.  Each tile
// has two accumulators in tensor memory (its products alternate between them).  The epilogue
// has four sets of four warps (four warps per SM sub-partition: the exp2 sums of a product need
// that many to keep the special-function unit busy, one or two warps leave it mostly idle on
// latency); sets (e, 0) and (e, 1) take every product of resident tile e, one 64-column half
// each (keys in MODE 0, window rows in MODE 1), and at the end of an item they merge their
// partial row states or column sums through shared memory.  In a causal window the item
// lengths grow with the tile index, so a block takes the resident pairs i and n - 1 - i of one
// (pair, chunk) as one unit and every unit costs about the same.  MODE 1 streams window-row
// blocks with their negated row log-sum-exp values (a 512-byte bulk copy per block into a ring
// of its own, released by the epilogue warps once read).
constexpr int TP_LSE_SLOTS = 8;
constexpr int TP_THREADS = 576;     // TMA warp, MMA warp, four epilogue sets of four warps
constexpr int TP_MAX_G = 8;         // MODE 1: query heads per KV head (shared-memory partials)

template <int D>
struct TpPlan {
    static constexpr int SUBS = D / 64;
    static constexpr int TILE_BYTES = SUBS * TC_SUB_BYTES;
    static constexpr int NS_RAW = (196 * 1024 - 2 * TILE_BYTES) / TILE_BYTES;
    static constexpr int NS = NS_RAW > 8 ? 8 : NS_RAW;       // streamed tiles in flight
    static_assert(NS >= 3, "resident tile pairs need three streamed stages");
    static constexpr int LSE_BYTES = TP_LSE_SLOTS * TC_ROWS * 4;
    // MODE 0: [2 tiles][128 rows][2] (m, z); MODE 1: [4 sets][G][128 keys] partial sums
    static constexpr int PART_BYTES = 4 * TP_MAX_G * TC_ROWS * 4;
    static constexpr int BAR_BYTES = 8 * (2 + 2 * NS + 2 * TC_NACC + 2 * TP_LSE_SLOTS + 2) + 16;
    static constexpr int SMEM_USED =
        1024 + (2 + NS) * TILE_BYTES + LSE_BYTES + PART_BYTES + BAR_BYTES;
    static constexpr int SMEM = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
    static_assert(SMEM <= 227 * 1024, "tile-pair plan exceeds shared memory");
};

struct TpItem {
    int pair, chunk, fp;      // (batch, KV head) pair, key chunk (MODE 0), resident tile pair
    int n_fix;                // resident tiles: 1 or 2
    int s_begin, n_str;       // first streamed tile, streamed tiles
    int lo0, hi0, lo1, hi1;   // set s takes the streamed tiles lo_s <= i < hi_s
    __device__ __forceinline__ int lo(int s) const { return s ? lo1 : lo0; }
    __device__ __forceinline__ int hi(int s) const { return s ? hi1 : hi0; }
};

// Units: (pair, chunk, su) for MODE 0, (pair, su) for MODE 1; unit su covers the resident pairs
// su and n_fp - 1 - su (one of them when they coincide).
__device__ __forceinline__ int tp_subitems(const TcParams &tp, int u)
{
    const int su = u % tp.n_sup;
    return tp.n_fp - 1 - su != su ? 2 : 1;
}

template <int MODE>
__device__ __forceinline__ TpItem tp_item(const TcParams &tp, int u, int sub)
{
    const ScoreParams &p = tp.sp;
    const int R = p.G * p.L_obs;
    const int first_pos = p.N - p.L_obs;
    const int su = u % tp.n_sup;
    TpItem it{};
    it.fp = sub == 0 ? su : tp.n_fp - 1 - su;
    if (MODE == 0) {
        it.pair = u / (tp.n_sup * p.n_chunks);
        it.chunk = (u / tp.n_sup) % p.n_chunks;
        it.s_begin = it.chunk * tp.chunk_tiles;
        it.n_fix = (2 * it.fp + 1) * TC_ROWS < R ? 2 : 1;
        // keys the rows of tile s can see: up to the largest position among them
        auto need = [&](int s) {
            const int r_lo = (2 * it.fp + s) * TC_ROWS;
            const int r_hi = min(r_lo + TC_ROWS, R) - 1;
            const int w_hi = (r_lo / p.L_obs != r_hi / p.L_obs) ? p.L_obs - 1 : r_hi % p.L_obs;
            const int kt_needed = (first_pos + w_hi) / TC_ROWS + 1;
            return max(0, min(it.s_begin + tp.chunk_tiles, kt_needed) - it.s_begin);
        };
        it.lo0 = it.lo1 = 0;
        it.hi0 = need(0);
        it.hi1 = it.n_fix == 2 ? need(1) : 0;
        it.n_str = max(it.hi0, it.hi1);
    } else {
        it.pair = u / tp.n_sup;
        it.n_fix = 2 * it.fp + 1 < tp.n_col_tiles ? 2 : 1;
        const int n_rb = (R + TC_ROWS - 1) / TC_ROWS;
        // row blocks whose rows can see key tile s: positions >= its first key (rows are sorted
        // by position when G = 1)
        auto first_rb = [&](int s) {
            const int k0 = (2 * it.fp + s) * TC_ROWS;
            return (p.G == 1 && k0 > first_pos) ? (k0 - first_pos) / TC_ROWS : 0;
        };
        it.s_begin = first_rb(0);
        it.n_str = n_rb - it.s_begin;
        it.lo0 = 0;
        it.hi0 = it.n_str;
        it.lo1 = it.n_fix == 2 ? first_rb(1) - it.s_begin : 0;
        it.hi1 = it.n_fix == 2 ? it.n_str : 0;
    }
    return it;
}

__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t cnt)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(cnt) : "memory");
}

__device__ __forceinline__ void pair_sync(int id)
{
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// Persistent blocks take units u = blockIdx.x, blockIdx.x + gridDim.x, ...; the three roles walk
// the same item sequence.  The resident pair has one buffer, reloaded per item once the item's
// last products are done (the epilogue still drains its last products meanwhile).
template <int D, int MODE>
__global__ void __launch_bounds__(TP_THREADS, 1)
tc_pair_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const TcParams tp)
{
    using PL = TpPlan<D>;
    constexpr int SUBS = PL::SUBS, TILE_BYTES = PL::TILE_BYTES, NS = PL::NS;
    constexpr int KSTEPS = D / 16;
    constexpr int LS = TP_LSE_SLOTS;
    const ScoreParams &p = tp.sp;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t fixed0 = base;                          // two resident tiles
    const uint32_t stage0 = base + 2 * TILE_BYTES;         // NS streamed tiles
    const uint32_t lse0 = stage0 + NS * TILE_BYTES;        // LS x 128 floats (MODE 1)
    const uint32_t part0 = lse0 + PL::LSE_BYTES;           // the sets' partial states
    const uint32_t bars = part0 + PL::PART_BYTES;
    const uint32_t bar_fix_full = bars;
    const uint32_t bar_fix_empty = bar_fix_full + 8;
    const uint32_t bar_full = bar_fix_empty + 8;           // NS
    const uint32_t bar_empty = bar_full + 8 * NS;          // NS
    const uint32_t bar_acc_full = bar_empty + 8 * NS;      // TC_NACC
    const uint32_t bar_acc_empty = bar_acc_full + 8 * TC_NACC;   // TC_NACC
    const uint32_t bar_lse_full = bar_acc_empty + 8 * TC_NACC;   // LS
    const uint32_t bar_lse_empty = bar_lse_full + 8 * LS;        // LS
    const uint32_t bar_done = bar_lse_empty + 8 * LS;      // the MMA thread's last commit
    const uint32_t tmem_slot = bar_done + 16;
    const float *sm_lse = reinterpret_cast<const float *>(smem_raw + (lse0 - raw));
    float *sm_part = reinterpret_cast<float *>(smem_raw + (part0 - raw));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int R = p.G * p.L_obs;
    const int first_pos = p.N - p.L_obs;
    const int C = gridDim.x;
    const int lse_stride = tp.n_mtiles * TC_ROWS;

    if (threadIdx.x == 0) {
        mbar_init(bar_fix_full, 1);
        mbar_init(bar_fix_empty, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int a = 0; a < TC_NACC; ++a) {
            mbar_init(bar_acc_full + 8 * a, 1);
            mbar_init(bar_acc_empty + 8 * a, 8);   // the eight warps of the tile's two sets
        }
        for (int l = 0; l < LS; ++l) {
            mbar_init(bar_lse_full + 8 * l, 1);
            mbar_init(bar_lse_empty + 8 * l, 16);  // the warps of the (two or four) sets reading it
        }
        mbar_init(bar_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         tmem_slot),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t tmem_base;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem_base) : "r"(tmem_slot));

    long long loads_streamed = 0;               // the producer's counts (for the drain)
    int loads_fixed = 0;
    if (warp == 0 && lane == 0) {
        // ================================ TMA producer ============================================
        long long g = 0;
        int nrl = 0;
        for (int u = blockIdx.x; u < tp.n_work; u += C) {
            const int nsub = tp_subitems(tp, u);
            for (int sub = 0; sub < nsub; ++sub) {
                const TpItem it = tp_item<MODE>(tp, u, sub);
                if (it.n_str == 0) continue;
                const int b = it.pair / p.Hkv, kh = it.pair % p.Hkv;
                const int qrow_group = (b * p.Hq + kh * p.G) * p.L_obs;
                if (nrl > 0) mbar_wait(bar_fix_empty, (nrl - 1) & 1, tp.dev_code);
                mbar_arrive_expect_tx(bar_fix_full, it.n_fix * TILE_BYTES);
                for (int f = 0; f < it.n_fix; ++f)
                    for (int a = 0; a < SUBS; ++a) {
                        const uint32_t dst = fixed0 + f * TILE_BYTES + a * TC_SUB_BYTES;
                        if (MODE == 0)
                            tma_load_2d(dst, &qmap, a * 64,
                                        qrow_group + (2 * it.fp + f) * TC_ROWS, bar_fix_full);
                        else
                            tma_load_4d(dst, &kmap, a * 64, (2 * it.fp + f) * TC_ROWS, kh, b,
                                        bar_fix_full);
                    }
                ++nrl;
                for (int i = 0; i < it.n_str; ++i, ++g) {
                    const int s = (int)(g % NS);
                    if (g >= NS) mbar_wait(bar_empty + 8 * s, (int)((g / NS) - 1) & 1, tp.dev_code);
                    const uint32_t dst = stage0 + s * TILE_BYTES;
                    mbar_arrive_expect_tx(bar_full + 8 * s, TILE_BYTES);
                    for (int a = 0; a < SUBS; ++a) {
                        if (MODE == 0)
                            tma_load_4d(dst + a * TC_SUB_BYTES, &kmap, a * 64,
                                        (it.s_begin + i) * TC_ROWS, kh, b, bar_full + 8 * s);
                        else
                            tma_load_2d(dst + a * TC_SUB_BYTES, &qmap, a * 64,
                                        qrow_group + (it.s_begin + i) * TC_ROWS, bar_full + 8 * s);
                    }
                    if (MODE == 1) {
                        // the row block's negated log2-sum-exp values (padded rows are zero)
                        const int l = (int)(g % LS);
                        if (g >= LS)
                            mbar_wait(bar_lse_empty + 8 * l, (int)((g / LS) - 1) & 1, tp.dev_code);
                        mbar_arrive_expect_tx(bar_lse_full + 8 * l, TC_ROWS * 4);
                        bulk_g2s(lse0 + l * TC_ROWS * 4,
                                 p.row_lse2 + (size_t)it.pair * lse_stride +
                                     (size_t)(it.s_begin + i) * TC_ROWS,
                                 TC_ROWS * 4, bar_lse_full + 8 * l);
                    }
                }
            }
        }
        loads_streamed = g;
        loads_fixed = nrl;
    } else if (warp == 1 && lane == 0) {
        // ================================ MMA issuer ==============================================
        long long g = 0;
        int nrl = 0;
        int uses0 = 0, uses1 = 0;             // accumulator uses per set
        for (int u = blockIdx.x; u < tp.n_work; u += C) {
            const int nsub = tp_subitems(tp, u);
            for (int sub = 0; sub < nsub; ++sub) {
                const TpItem it = tp_item<MODE>(tp, u, sub);
                if (it.n_str == 0) continue;
                mbar_wait(bar_fix_full, nrl & 1, tp.dev_code);
                ++nrl;
                for (int i = 0; i < it.n_str; ++i, ++g) {
                    const int s = (int)(g % NS);
                    mbar_wait(bar_full + 8 * s, (int)(g / NS) & 1, tp.dev_code);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (i < it.lo(e) || i >= it.hi(e)) continue;
                        const int k = e ? uses1++ : uses0++;
                        const int acc = 2 * (k & 1) + e;
                        if (k >= 2)
                            mbar_wait(bar_acc_empty + 8 * acc, ((k >> 1) - 1) & 1, tp.dev_code);
                        tc_fence_after();
                        const uint32_t a_base = fixed0 + e * TILE_BYTES;
                        const uint32_t b_base = stage0 + s * TILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < KSTEPS; ++kk) {
                            const uint32_t off = (kk >> 2) * TC_SUB_BYTES + (kk & 3) * 32;
                            umma_bf16(tmem_base + acc * 128, sw128_desc(a_base + off),
                                      sw128_desc(b_base + off), kk > 0 ? 1u : 0u);
                        }
                        umma_commit(bar_acc_full + 8 * acc);
                    }
                    umma_commit(bar_empty + 8 * s);   // streamed stage free once both products end
                }
                umma_commit(bar_fix_empty);           // resident pair free after the item
            }
        }
    } else if (warp >= 2) {
        // ================================ epilogue ================================================
        const int sg = (warp - 2) / 4;            // set
        const int e = sg & 1;                     // resident tile e of every item ...
        const int h = sg >> 1;                    // ... columns 64 h .. 64 h + 63 of its products
        const int q4 = warp & 3;                  // TMEM lanes 32*q4 .. 32*q4+31
        const int et = q4 * 32 + lane;            // this thread's lane (row or key)
        const uint32_t tcol = tmem_base + e * 128 + h * 64 + ((uint32_t)(q4 * 32) << 16);
        const int bar_id = 1 + e * 4 + q4;        // the two sets of tile e, this lane quarter
        long long g = 0;
        int k = 0;                                // products of tile e so far
        for (int u = blockIdx.x; u < tp.n_work; u += C) {
            const int nsub = tp_subitems(tp, u);
            for (int sub = 0; sub < nsub; ++sub) {
                const TpItem it = tp_item<MODE>(tp, u, sub);
                if (e >= it.n_fix) {
                    g += it.n_str;
                    continue;
                }
                const int b = it.pair / p.Hkv, kh = it.pair % p.Hkv;
                if (MODE == 0) {
                    const int r = (2 * it.fp + e) * TC_ROWS + et;   // window row of the group
                    const bool row_ok = r < R;
                    const int pos = row_ok ? row_pos(p, r) : -1;
                    float m_run = kNegBig, z_run = 0.f;
                    for (int i = it.lo(e); i < it.hi(e); ++i, ++k) {
                        const int acc = 2 * (k & 1) + e;
                        mbar_wait(bar_acc_full + 8 * acc, (k >> 1) & 1, tp.dev_code);
                        tc_fence_after();
                        rowstats_half_lazy(tcol + (k & 1) * 256, (it.s_begin + i) * TC_ROWS + h * 64,
                                           pos, p.N, p.scale_log2, m_run, z_run);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_acc_empty + 8 * acc);
                    }
                    // the second set hands its rows' states to the first, which merges and
                    // writes them (an empty state where no key tile of the chunk reaches a row)
                    float *mz = sm_part + (e * TC_ROWS + et) * 2;
                    if (h == 1) {
                        mz[0] = m_run;
                        mz[1] = z_run;
                    }
                    pair_sync(bar_id);
                    if (h == 0 && row_ok) {
                        const float m1 = mz[0], z1 = mz[1];
                        const float M = fmaxf(m_run, m1);
                        float *dst =
                            p.row_ml + (((size_t)it.pair * p.n_chunks + it.chunk) * R + r) * 2;
                        dst[0] = M;
                        dst[1] = z_run * ex2(m_run - M) + z1 * ex2(m1 - M);
                    }
                    pair_sync(bar_id);
                } else {
                    const bool other = it.n_fix == 2;     // does tile 1 take part?
                    const int kt = 2 * it.fp + e;
                    const int key = kt * TC_ROWS + et;
                    const bool mask_tile = kt * TC_ROWS + TC_ROWS - 1 > first_pos;
                    // this set's per-head partial sums of its key: [G][128]
                    float *part = sm_part + (size_t)sg * TP_MAX_G * TC_ROWS;
                    for (int gq = 0; gq < p.G; ++gq) part[gq * TC_ROWS + et] = 0.f;
                    int g_cur = -1;
                    float acc_g = 0.f;
                    for (int i = it.lo(e); i < it.hi(e); ++i, ++k) {
                        const long long gg = g + i;
                        const int l = (int)(gg % LS);
                        const int acc = 2 * (k & 1) + e;
                        const int r0 = (it.s_begin + i) * TC_ROWS + h * 64;   // this half's rows
                        const int rows = min(64, R - r0);
                        mbar_wait(bar_lse_full + 8 * l, (int)(gg / LS) & 1, tp.dev_code);
                        mbar_wait(bar_acc_full + 8 * acc, (k >> 1) & 1, tp.dev_code);
                        tc_fence_after();
                        // (warp-uniform: the tensor-memory loads below are .sync.aligned)
                        if (p.G == 1 && rows == 64 &&
                            __all_sync(0xffffffffu, key <= first_pos + r0)) {
                            // one head, and every row of this half sees every key of the warp:
                            // the 64 rows' probabilities summed with no head or mask bookkeeping
                            float v[2][32];
                            tmem_ld64(tcol + (k & 1) * 256, v);
                            const float *nl = sm_lse + l * TC_ROWS + h * 64;
                            acc_g += exp2_sum32(v[0], p.scale_log2, 0.f, nl) +
                                     exp2_sum32(v[1], p.scale_log2, 0.f, nl + 32);
                            g_cur = 0;
                        } else if (rows > 0) {
                            if (g_cur < 0) g_cur = r0 / p.L_obs;
                            colsum_rows<true>(p, first_pos, tcol + (k & 1) * 256, r0, rows, key,
                                        mask_tile, sm_lse + l * TC_ROWS + h * 64, part, TC_ROWS,
                                        et, true, g_cur, acc_g);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(bar_acc_empty + 8 * acc);
                            // tile 0 takes every row block: its set also releases the slot for
                            // tile 1 where tile 1 does not take this block
                            const bool alone = e == 0 && !(other && i >= it.lo1);
                            mbar_arrive_cnt(bar_lse_empty + 8 * l, alone ? 2u : 1u);
                        }
                    }
                    if (g_cur >= 0) part[g_cur * TC_ROWS + et] = acc_g * p.col_mult;
                    pair_sync(bar_id);
                    if (h == 0 && key < p.n_cols) {
                        const float *part1 = sm_part + (size_t)(sg + 2) * TP_MAX_G * TC_ROWS;
                        float *s_base = p.s_out + (size_t)(b * p.Hq + kh * p.G) * p.n_cols + key;
                        for (int gq = 0; gq < p.G; ++gq)
                            s_base[(size_t)gq * p.n_cols] =
                                part[gq * TC_ROWS + et] + part1[gq * TC_ROWS + et];
                    }
                    pair_sync(bar_id);
                }
                g += it.n_str;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // after a wait ran out: the last loads have landed and every product issued has completed
    // before the block frees tensor memory and exits
    if ((threadIdx.x == 0 || threadIdx.x == 32) && timeout_recorded(tp.dev_code)) {
        if (threadIdx.x == 0) {
            drain_loads(bar_full, NS, loads_streamed, tp.dev_code);
            drain_loads(bar_fix_full, 1, loads_fixed, tp.dev_code);
            if (MODE == 1) drain_loads(bar_lse_full, LS, loads_streamed, tp.dev_code);
        } else {
            umma_commit(bar_done);
            mbar_wait(bar_done, 0, tp.dev_code);
        }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TC_TMEM_COLS)
                     : "memory");
}

template <int D>
constexpr int tc_smem_bytes()
{
    return TcPlan<D, false>::SMEM > TcPlan<D, true>::SMEM ? TcPlan<D, false>::SMEM
                                                          : TcPlan<D, true>::SMEM;
}

// ---- host: tensor maps through the driver entry point ------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode != nullptr;
}

bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t row_bytes)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, TC_ROWS};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_4d(CUtensorMap *m, const void *ptr, uint64_t d, uint64_t n, uint64_t h, uint64_t bsz,
               uint64_t s_slot, uint64_t s_h, uint64_t s_b)
{
    cuuint64_t dims[4] = {d, n, h, bsz};
    cuuint64_t strides[3] = {s_slot, s_h, s_b};
    cuuint32_t box[4] = {64, TC_ROWS, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Each row's negated log2-sum-exp from pass 1's per-chunk (max, sum) states, stored with the row
// count rounded up to 128 per pair (whole row blocks for the bulk copies; the padding is zero).
__global__ void rowlse_tc_kernel(const ScoreParams p)
{
    const int R = p.G * p.L_obs;
    const int Rp = (R + TC_ROWS - 1) / TC_ROWS * TC_ROWS;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)p.B * p.Hkv * Rp) return;
    const long long bkh = i / Rp;
    const int r = (int)(i % Rp);
    if (r >= R) {
        p.row_lse2[i] = 0.f;
        return;
    }
    float M = kNegBig;
    for (int c = 0; c < p.n_chunks; ++c)
        M = fmaxf(M, p.row_ml[((bkh * p.n_chunks + c) * R + r) * 2]);
    float Z = 0.f;
    for (int c = 0; c < p.n_chunks; ++c) {
        const float *s = p.row_ml + ((bkh * p.n_chunks + c) * R + r) * 2;
        Z += s[1] * exp2f(s[0] - M);
    }
    p.row_lse2[i] = -(M + log2f(Z));
}

template <int D>
cudaError_t launch_tc_typed(const ScoreParams &sp, const CUtensorMap &qm, const CUtensorMap &km,
                            int32_t *dev_code, cudaStream_t stream)
{
    constexpr int SMEM = tc_smem_bytes<D>();
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        void (*kerns[5])(const CUtensorMap, const CUtensorMap, const TcParams) = {
            tc_scores_kernel<D, 0, false>, tc_scores_kernel<D, 0, true>,
            tc_scores_kernel<D, 1, false>, tc_scores_kernel<D, 2, false>,
            tc_scores_kernel<D, 2, true>};
        for (auto kf : kerns) {
            cudaError_t e =
                cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
            if (e != cudaSuccess) return e;
        }
        if constexpr (D <= 128) {
            for (auto kf : {tc_pair_kernel<D, 0>, tc_pair_kernel<D, 1>}) {
                cudaError_t e = cudaFuncSetAttribute(
                    kf, cudaFuncAttributeMaxDynamicSharedMemorySize, TpPlan<D>::SMEM);
                if (e != cudaSuccess) return e;
            }
        }
        configured[dev] = true;
    }
    int n_sm = 152;
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (n_sm <= 0) n_sm = 152;
    const int R = sp.G * sp.L_obs;
    TcParams tp;
    tp.sp = sp;
    tp.n_mtiles = (R + TC_ROWS - 1) / TC_ROWS;
    tp.chunk_tiles = sp.chunk / TC_ROWS;
    tp.n_col_tiles = (sp.n_cols + TC_ROWS - 1) / TC_ROWS;
    tp.col_chunks = 1;
    tp.col_chunk_tiles = tp.n_col_tiles;
    tp.n_fp = 0;
    tp.n_sup = 0;
    tp.dev_code = dev_code;
    // one persistent block per SM (at most one per work item); round-robin items with a single
    // resident buffer would stall the pipeline at every item, so each gets its own block there
    auto grid = [&](long long work, bool contig) {
        return (unsigned)((!contig && TcPlan<D, false>::NFIX == 1) || work < n_sm ? work : n_sm);
    };
    const long long pairs = (long long)sp.B * sp.Hkv;
    const long long work0 = pairs * tp.n_mtiles * sp.n_chunks;
    if (work0 > 0x7fffffffLL) return cudaErrorInvalidValue;
    tp.n_work = (int)work0;
    // several key chunks per row tile: contiguous items share the resident tile (where that buys
    // streamed stages: with d_head 256 two stages is all that fits either way)
    constexpr bool kContigPays = TcPlan<D, true>::NS > TcPlan<D, false>::NS;
    // windows of several row tiles (up to d_head 128, where two resident tiles and three
    // streamed stages fit): resident row-tile pairs
    constexpr bool kPairs = D <= 128;
    if (kPairs && tp.n_mtiles >= 2) {
        if constexpr (kPairs) {
            tp.n_fp = (tp.n_mtiles + 1) / 2;
            tp.n_sup = (tp.n_fp + 1) / 2;
            const long long work = pairs * sp.n_chunks * tp.n_sup;
            if (work > 0x7fffffffLL) return cudaErrorInvalidValue;
            tp.n_work = (int)work;
            tc_pair_kernel<D, 0><<<(unsigned)(work < n_sm ? work : n_sm), TP_THREADS,
                                   TpPlan<D>::SMEM, stream>>>(qm, km, tp);
        }
    } else if (kContigPays && sp.n_chunks >= 2)
        tc_scores_kernel<D, 0, true><<<grid(work0, true), TC_THREADS, SMEM, stream>>>(qm, km, tp);
    else
        tc_scores_kernel<D, 0, false><<<grid(work0, false), TC_THREADS, SMEM, stream>>>(qm, km, tp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int n_rb = (R + TC_ROWS - 1) / TC_ROWS;
    const bool rows_resident = R <= TC_ROWS || (sp.G > 1 && TC_ROWS % sp.L_obs == 0);
    // the column pass with resident rows folds each row's chunk states itself; with streamed
    // rows (or no column pass) the row log-sum-exp values are written first
    if (!rows_resident || tp.n_col_tiles == 0) {
        const long long rows = pairs * n_rb * TC_ROWS;
        rowlse_tc_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, stream>>>(sp);
        e = cudaGetLastError();
        if (e != cudaSuccess || tp.n_col_tiles == 0) return e;
    }
    if (rows_resident) {
        // every head inside one row block: keep the row block, stream the key tiles
        const long long base = pairs * n_rb;
        long long chunks = (4LL * n_sm + base - 1) / base;
        if (chunks > tp.n_col_tiles) chunks = tp.n_col_tiles;
        tp.col_chunk_tiles = (int)((tp.n_col_tiles + chunks - 1) / chunks);
        tp.col_chunks = (tp.n_col_tiles + tp.col_chunk_tiles - 1) / tp.col_chunk_tiles;
        const long long work2 = base * tp.col_chunks;
        if (work2 > 0x7fffffffLL) return cudaErrorInvalidValue;
        tp.n_work = (int)work2;
        if (kContigPays && tp.col_chunks >= 2)
            tc_scores_kernel<D, 2, true><<<grid(work2, true), TC_THREADS, SMEM, stream>>>(qm, km,
                                                                                         tp);
        else
            tc_scores_kernel<D, 2, false><<<grid(work2, false), TC_THREADS, SMEM, stream>>>(qm, km,
                                                                                           tp);
    } else if (kPairs && sp.G <= TP_MAX_G) {
        // stream the row blocks past resident key-tile pairs
        tp.n_fp = (tp.n_col_tiles + 1) / 2;
        tp.n_sup = (tp.n_fp + 1) / 2;
        const long long work = pairs * tp.n_sup;
        if (work > 0x7fffffffLL) return cudaErrorInvalidValue;
        tp.n_work = (int)work;
        if constexpr (kPairs)
            tc_pair_kernel<D, 1><<<(unsigned)(work < n_sm ? work : n_sm), TP_THREADS,
                                   TpPlan<D>::SMEM, stream>>>(qm, km, tp);
    } else {
        const long long work1 = pairs * tp.n_col_tiles;
        if (work1 > 0x7fffffffLL) return cudaErrorInvalidValue;
        tp.n_work = (int)work1;
        tc_scores_kernel<D, 1, false><<<grid(work1, false), TC_THREADS, SMEM, stream>>>(qm, km,
                                                                                       tp);
    }
    return cudaGetLastError();
}

}  // namespace

bool obs_scores_tc_supported(const ScoreParams &p)
{
    return (p.D == 64 || p.D == 128 || p.D == 256) && (p.L_obs >= 32 || p.G == 1) &&
           p.chunk % TC_ROWS == 0;
}

cudaError_t launch_obs_scores_tc(const ScoreParams &p, int32_t *dev_code, cudaStream_t stream,
                                 bool *used)
{
    *used = false;
    if (!obs_scores_tc_supported(p) || !get_encoder()) return cudaSuccess;
    CUtensorMap qm, km;
    const uint64_t eb = 2;
    if (!encode_2d(&qm, p.q, (uint64_t)p.D, (uint64_t)p.B * p.Hq * p.L_obs, (uint64_t)p.D * eb))
        return cudaSuccess;
    if (!encode_4d(&km, p.k, (uint64_t)p.D, (uint64_t)p.N, (uint64_t)p.Hkv, (uint64_t)p.B,
                   (uint64_t)p.ss * eb, (uint64_t)p.sh * eb, (uint64_t)p.sb * eb))
        return cudaSuccess;
    *used = true;
    switch (p.D) {
    case 64: return launch_tc_typed<64>(p, qm, km, dev_code, stream);
    case 128: return launch_tc_typed<128>(p, qm, km, dev_code, stream);
    default: return launch_tc_typed<256>(p, qm, km, dev_code, stream);
    }
}

}  // namespace kvc
