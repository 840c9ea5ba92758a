// decode_mma.cu -- grouped-query decode attention on the tensor cores (bf16 caches, no RoPE).
//
// Same result and same schedule as decode_attn.cuh (persistent blocks over the flattened
// (pair, tile) space, a shared-memory ring, last-block log-sum-exp merge), but the arithmetic of
// a query group runs as matrix products.  With G query heads sharing every K/V row, the logits
// of a tile are the [G x D] x [D x keys] product and the output update the [G x keys] x
// [keys x D] product -- a dense contraction of G rows.  On CUDA cores the bf16 widening, the
// FMAs and the cross-lane reductions per key exceed what the SMs can issue while HBM delivers
// the cache at full rate once G >= 4, so these two products use mma.sync (m16n8k16, bf16 in,
// fp32 accumulate) with the G heads as rows 0..G-1 of the 16-row tile.
//
// Data movement.  K and V tiles (TK slots x D) arrive by TMA (cp.async.bulk.tensor, 4-D tensor
// map over [batch][head][slot][dim], 128-byte swizzle) into an NS-stage ring; ldmatrix reads
// the swizzled tiles without bank conflicts (.trans for V, whose rows are keys).
//
// Warp layout.  Each warp owns 16 keys of the tile: it computes their logits for all heads,
// updates its online-softmax state (lazy running max, base-2 exponentials), converts the
// probabilities in place into the A operand of the P.V product (the accumulator layout of
// m16n8 is the operand layout of m16k16) and accumulates o.  For D = 256 two warps share the
// same 16 keys and split the head dimension of o.  The probabilities P enter the P.V product as
// two bf16 terms, P = hi + lo with hi = bf16(P) and lo = bf16(P - hi), each multiplied by V on
// the tensor cores into the same fp32 accumulator: P is carried to 16 significant bits (a
// relative error below 2^-17, against 2^-9 for P rounded once), so the arithmetic stays fp32
// class while the inputs are bf16.  The sums l are kept in fp32.
//
// Bounded waits (p.spin_limit polls): one that gives up records KVC_DEV_TIMEOUT and raises the
// block's abort flag -- no more loads, the other waits give up at once, the tiles and merge
// tickets are still walked so that every block finishes -- and the issuing thread waits
// (bounded) for its last loads before the block exits.  The outputs of such a call are invalid.
// The flag is read only after a first poll has failed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int MW = 8;                        // warps per block
constexpr int M_THREADS = MW * 32;
constexpr float kSlack = 8.0f;               // lazy running max, log2 units

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D(16x8 fp32) += A(16x16 bf16, rows 8..15 zero) * B(16x8 bf16)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Byte offset of (row, 8-element chunk) inside a tile stored as D/64 sub-tiles of rows x 128 B
// with the 128-byte swizzle (16-byte chunk c of row r at c ^ (r mod 8)).
__device__ __forceinline__ uint32_t sw_off(int row, int chunk, int rows_per_sub)
{
    const int sub = chunk >> 3, c = chunk & 7;
    return (uint32_t)(sub * rows_per_sub * 128 + row * 128 + ((c ^ (row & 7)) << 4));
}
__device__ __forceinline__ int cta_of(long long t, long long T, int C)
{
    return (int)(((t + 1) * (long long)C - 1) / T);
}

constexpr int kPrefMax = 1024;               // pairs whose tile offsets a block scans into smem

template <int D, int G>
struct MmaPlan {
    static constexpr int TK = D == 256 ? 64 : 128;             // slots per tile
    static constexpr int PAIRS = D == 256 ? 2 : 1;             // warps sharing 16 keys
    static constexpr int KGROUPS = MW / PAIRS;                  // 16-key groups per tile
    static_assert(KGROUPS * 16 == TK, "tile = 16 keys per key group");
    static constexpr int DW = D / PAIRS;                        // output dims per warp
    static constexpr int TILE_BYTES = TK * D * 2;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int MERGE_BYTES = KGROUPS * G * (D + 2) * 4 + 16;
    static constexpr int BAR_BYTES = 128;
    static constexpr int PREF_BYTES = ((kPrefMax + 1) * 4 + 15) / 16 * 16;
    static constexpr int SMEM_MAX = 227 * 1024;                 // dynamic shared memory per block
    static constexpr int NS_fit =
        (SMEM_MAX - 1024 - MERGE_BYTES - BAR_BYTES - PREF_BYTES) / STAGE_BYTES;
    static constexpr int NS = NS_fit > 4 ? 4 : NS_fit;
    static_assert(NS >= 2, "two stages at least");
    static constexpr int SMEM = 1024 + NS * STAGE_BYTES + BAR_BYTES + MERGE_BYTES + PREF_BYTES;
};


// Bulk copy global -> shared memory, completion counted in bytes on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Log-sum-exp merge of the nseg partial states of one pair, segment s held in workspace slot
// slot_of(s).  Every load of a batch of segments is issued before any is used: the merge costs
// one L2 round trip per eight segments.
template <int G, int D>
__device__ __forceinline__ void merge_segments(const float *ws_o, const float *ws_ml, int slot0,
                                               int c_lo, int nseg, float *out, float *lse,
                                               int rows0)
{
    constexpr int NCH = G * D / 4;                         // 16-byte chunks of the G output rows
    constexpr int CPT = (NCH + M_THREADS - 1) / M_THREADS; // chunks per thread
    constexpr int UNR = 8;                                 // segments per batch of loads
    float M[CPT], L[CPT];
    float4 O[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        M[k] = kNegBig;
        L[k] = 0.f;
        O[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int s0 = 0; s0 < nseg; s0 += UNR) {
        float4 o[CPT][UNR];
        float m[CPT][UNR], l[CPT][UNR];
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int ch = threadIdx.x + k * M_THREADS;
            const int g = ch * 4 / D, d = ch * 4 % D;
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int s = s0 + u;
                if (ch < NCH && s < nseg) {
                    const size_t st = (size_t)(s == 0 ? slot0 : 2 * (c_lo + s)) * G + g;
                    o[k][u] = __ldcg(reinterpret_cast<const float4 *>(ws_o + st * D + d));
                    m[k][u] = __ldcg(ws_ml + st * 2);
                    l[k][u] = __ldcg(ws_ml + st * 2 + 1);
                } else {
                    o[k][u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    m[k][u] = kNegBig;
                    l[k][u] = 0.f;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            float mb = M[k];
#pragma unroll
            for (int u = 0; u < UNR; ++u) mb = fmaxf(mb, m[k][u]);
            const float cm = ex2(M[k] - mb);
            L[k] *= cm;
            O[k].x *= cm; O[k].y *= cm; O[k].z *= cm; O[k].w *= cm;
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const float c = ex2(m[k][u] - mb);
                L[k] += l[k][u] * c;
                O[k].x += o[k][u].x * c; O[k].y += o[k][u].y * c;
                O[k].z += o[k][u].z * c; O[k].w += o[k][u].w * c;
            }
            M[k] = mb;
        }
    }
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        const int ch = threadIdx.x + k * M_THREADS;
        if (ch >= NCH) continue;
        const int g = ch * 4 / D, d = ch * 4 % D;
        const bool any = L[k] > 0.f;
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        if (any) r = make_float4(O[k].x / L[k], O[k].y / L[k], O[k].z / L[k], O[k].w / L[k]);
        *reinterpret_cast<float4 *>(out + (size_t)(rows0 + g) * D + d) = r;
        if (d == 0 && lse != nullptr)
            lse[rows0 + g] = any ? (M[k] + log2f(L[k])) * kLn2 : -INFINITY;
    }
}

// Schedule.  The tiles of all pairs form one sequence (pair by pair, TK slots per tile) that
// the blocks split into equal contiguous ranges.  Pair q holds tiles [pref(q), pref(q + 1)):
//   len == nullptr:         ceil(n_valid / TK) tiles for every pair;
//   balance, P <= kPrefMax: ceil(len[q] / TK) tiles, offsets from a block-wide scan of the
//                           lengths (every tile holds slots, so the ranges balance the bytes
//                           read however the lengths differ; the scan delays each block's first
//                           load by a read of the lengths and two block barriers);
//   otherwise:              ceil(cap / TK) tiles; tiles past the length are skipped.
// A pair split over several blocks leaves one partial state per block: block c keeps the state
// of the first pair of its range in workspace slot 2c and that of its last pair in slot 2c + 1
// (a block's other pairs are complete inside its range).  The block that takes a pair's last
// ticket merges them.
template <int D, int G>
__global__ void __launch_bounds__(M_THREADS, 1)
decode_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p)
{
    using PL = MmaPlan<D, G>;
    constexpr int TK = PL::TK, NS = PL::NS, DW = PL::DW;
    constexpr int KSTEPS = D / 16;
    constexpr int NB = DW / 8;                 // 8-dim output blocks per warp
    static_assert(G <= 8, "group fits rows 0..7 of the 16-row tile");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t stage0 = base;
    const uint32_t bars = stage0 + NS * PL::STAGE_BYTES;
    const uint32_t bar_full = bars, bar_empty = bars + 8 * NS, bar_merge = bars + 16 * NS;
    float *sm_m = reinterpret_cast<float *>(smem_raw + (bars + PL::BAR_BYTES - raw));
    float *sm_l = sm_m + PL::KGROUPS * G;
    float *sm_o = sm_l + PL::KGROUPS * G;      // [KGROUPS][G][D]
    int *sm_flag = reinterpret_cast<int *>(sm_o + PL::KGROUPS * G * D);
    volatile int *sm_abort = sm_flag + 1;      // set once a bounded wait has given up
    int *sm_pref = reinterpret_cast<int *>(reinterpret_cast<unsigned char *>(sm_m) + PL::MERGE_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kg = warp / PL::PAIRS;           // key group (16 keys of the tile)
    const int half = warp % PL::PAIRS;         // output-dim half (D = 256)
    const int gr = lane >> 2, tq = lane & 3;   // mma fragment row / column pair
    const int C = gridDim.x, cta = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, MW);
        }
        mbar_init(bar_merge, 1);
        *sm_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Lengths and cache slots written before the previous kernel began may be read before
    // waiting for it; everything else (q, outputs, workspace) only after.
    if (!p.kv_settled) {
        pdl_trigger();
        pdl_wait();                            // inputs may come from the previous kernel
    }

    auto pair_slots = [&](int q) -> int {
        if (p.len != nullptr) {
            const int n = p.len[q];
            return n < 0 ? 0 : (n > p.cap ? p.cap : n);
        }
        return p.n_valid < 0 ? 0 : (p.n_valid > p.cap ? p.cap : p.n_valid);
    };
    const int mode = p.len == nullptr ? 0 : (p.balance && p.P <= kPrefMax ? 1 : 2);
    const int ntq = mode == 0 ? (pair_slots(0) + TK - 1) / TK : p.NT;
    if (mode == 1) {
        // exclusive scan of the pairs' tile counts into sm_pref[0..P]
        constexpr int PER = (kPrefMax + M_THREADS - 1) / M_THREADS;
        int cnt[PER], sum = 0;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int q = threadIdx.x * PER + k;
            cnt[k] = q < p.P ? (pair_slots(q) + TK - 1) / TK : 0;
            sum += cnt[k];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int *wsum = reinterpret_cast<int *>(sm_m);   // MW warp totals (merge area, free now)
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int run = incl - sum;
        for (int w = 0; w < warp; ++w) run += wsum[w];
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int q = threadIdx.x * PER + k;
            if (q < p.P) sm_pref[q] = run;
            run += cnt[k];
        }
        if (threadIdx.x == M_THREADS - 1) sm_pref[p.P] = run;
        __syncthreads();
    }
    auto pref = [&](int q) -> long long {
        return mode == 1 ? (long long)sm_pref[q] : (long long)q * ntq;
    };
    const long long T = pref(p.P);
    // the first Ce blocks split the tiles, each at least one (a pair's segments are then the
    // blocks c_lo..c_hi, every one of which takes a ticket)
    const int Ce = T < C ? (int)T : C;
    const long long t_begin = cta < Ce ? (long long)cta * T / Ce : 0;
    const long long t_end = cta < Ce ? (long long)(cta + 1) * T / Ce : 0;
    const int n_tiles = (int)(t_end - t_begin);
    // pair holding tile t < T: the last q with pref(q) <= t
    auto pair_of = [&](long long t) -> int {
        if (mode != 1) return (int)(t / ntq);
        int lo = 0, hi = p.P - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm_pref[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    };
    // tile cursors (pair q covers tiles [q_lo, q_hi)), advanced monotonically
    struct Cursor {
        int q;
        long long lo, hi;
    };
    auto cursor_at = [&](long long t) -> Cursor {
        Cursor c;
        c.q = pair_of(t);
        c.lo = pref(c.q);
        c.hi = pref(c.q + 1);
        return c;
    };
    auto advance = [&](Cursor &c, long long t) {
        while (t >= c.hi) {
            ++c.q;
            c.lo = c.hi;
            c.hi = pref(c.q + 1);
        }
    };

    // The issuing thread keeps the slot count of the pair it is loading: one global read per
    // pair, not one per tile on the critical path of every copy.
    Cursor ic{};
    int iss_q = -1, iss_slots = 0;
    int last_issued = -1;                      // the issuing thread's last tile (abort drain)
    auto issue_tile = [&](int i) {
        if (p.starve) return;                  // test hook: no loads, no arrivals
        last_issued = i;
        const long long t = t_begin + i;
        const int s = i % NS;
        advance(ic, t);
        const int q = ic.q;
        const int j0 = (int)(t - ic.lo) * TK;
        const uint32_t full = bar_full + 8 * s;
        if (q != iss_q) {
            iss_q = q;
            iss_slots = pair_slots(q);
        }
        if (j0 >= iss_slots) {
            mbar_arrive(full);
            return;
        }
        const int b = q / p.Hkv, kh = q % p.Hkv;
        const uint32_t kdst = stage0 + s * PL::STAGE_BYTES, vdst = kdst + PL::TILE_BYTES;
        mbar_arrive_expect_tx(full, (uint32_t)PL::STAGE_BYTES);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub) {
            tma_load_4d(kdst + sub * TK * 128, &kmap, sub * 64, j0, kh, b, full);
            tma_load_4d(vdst + sub * TK * 128, &vmap, sub * 64, j0, kh, b, full);
        }
    };
    if (threadIdx.x == 0 && n_tiles > 0) {
        ic = cursor_at(t_begin);
        for (int i = 0; i < NS && i < n_tiles; ++i) issue_tile(i);
    }
    if (p.kv_settled) {
        pdl_trigger();
        pdl_wait();                            // q, outputs and workspace follow the previous kernel
    }

    // pairs without a tile (no valid slot) still get their rows: out = 0, lse = -inf
    if (mode != 2) {
        for (int q = cta; q < p.P; q += C) {
            if (pref(q + 1) != pref(q)) continue;
            const int rows0 = (q / p.Hkv) * p.Hq + (q % p.Hkv) * G;
            for (int i = threadIdx.x; i < G * D; i += M_THREADS) {
                p.out[(size_t)rows0 * D + i] = 0.f;
                if (i % D == 0 && p.lse != nullptr) p.lse[rows0 + i / D] = -INFINITY;
            }
        }
    }

    // ---- per-pair state ---------------------------------------------------------------------
    uint32_t qa0[KSTEPS], qa2[KSTEPS];         // q rows as A fragments (rows >= G are zero)
    float o[NB][4];
    float m_row = kNegBig, l_part = 0.f;       // row gr (head gr); l summed over the 4 lanes later
    int cur_slots = 0;
    float *lg_row = nullptr;

    auto start_pair = [&](int q) {
        cur_slots = pair_slots(q);
        const int b = q / p.Hkv, kh = q % p.Hkv;
        const __nv_bfloat16 *qb =
            static_cast<const __nv_bfloat16 *>(p.q) + ((size_t)b * p.Hq + (size_t)kh * G) * D;
#pragma unroll
        for (int s = 0; s < KSTEPS; ++s) {
            if (gr < G) {
                qa0[s] = *reinterpret_cast<const uint32_t *>(qb + (size_t)gr * D + 16 * s + 2 * tq);
                qa2[s] = *reinterpret_cast<const uint32_t *>(qb + (size_t)gr * D + 16 * s + 2 * tq + 8);
            } else {
                qa0[s] = 0u;
                qa2[s] = 0u;
            }
        }
#pragma unroll
        for (int n = 0; n < NB; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m_row = kNegBig;
        l_part = 0.f;
        lg_row = (p.logits != nullptr && gr < G)
                     ? p.logits + (size_t)((q / p.Hkv) * p.Hq + (q % p.Hkv) * G + gr) * p.logits_stride
                     : nullptr;
    };

    // Merge of the pair this block finishes last, its ring of stages idle by then: every partial
    // state comes into shared memory by bulk copies issued at once (one round trip to L2 for up
    // to GS segments), then each thread combines its 16-byte chunks of the G output rows.
    auto merge_staged = [&](int slot0, int c_lo, int nseg, int rows0) {
        constexpr int O_BYTES = G * D * 4, ML_BYTES = G * 8;
        constexpr int GS = NS * PL::STAGE_BYTES / (O_BYTES + ML_BYTES);
        static_assert(GS >= 1, "one partial state fits the ring");
        constexpr int NCH = G * D / 4;
        constexpr int CPT = (NCH + M_THREADS - 1) / M_THREADS;
        const float *so = reinterpret_cast<const float *>(smem_raw + (stage0 - raw));
        const float *sml = reinterpret_cast<const float *>(smem_raw + (stage0 - raw) + GS * O_BYTES);
        float M[CPT], L[CPT];
        float4 O[CPT];
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            M[k] = kNegBig;
            L[k] = 0.f;
            O[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        uint32_t phase = 0;
        for (int s0 = 0; s0 < nseg; s0 += GS) {
            const int ng = min(GS, nseg - s0);
            if (warp == 0) {
                // the partial states were written by other blocks through the generic proxy
                // (made visible by the acquire); the ring was last read by this block's warps
                asm volatile("fence.proxy.async.global;" ::: "memory");
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (lane == 0)
                    mbar_arrive_expect_tx(bar_merge, (uint32_t)(ng * (O_BYTES + ML_BYTES)));
                __syncwarp();
                for (int u = lane; u < ng; u += 32) {       // the copies issued by 32 lanes
                    const int s = s0 + u;
                    const size_t slot = (size_t)(s == 0 ? slot0 : 2 * (c_lo + s));
                    bulk_g2s(stage0 + u * O_BYTES, p.ws_o + slot * G * D, O_BYTES, bar_merge);
                    bulk_g2s(stage0 + GS * O_BYTES + u * ML_BYTES, p.ws_ml + slot * G * 2,
                             ML_BYTES, bar_merge);
                }
            }
            const bool got = mbar_wait_abortable(bar_merge, phase & 1u, p.spin_limit, sm_abort);
            ++phase;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int ch = threadIdx.x + k * M_THREADS;
                if (ch >= NCH) continue;
                const int g = ch * 4 / D, d = ch * 4 % D;
                float mb = M[k];
                for (int u = 0; u < ng; ++u) mb = fmaxf(mb, sml[u * 2 * G + 2 * g]);
                const float cm = ex2(M[k] - mb);
                L[k] *= cm;
                O[k].x *= cm; O[k].y *= cm; O[k].z *= cm; O[k].w *= cm;
                for (int u = 0; u < ng; ++u) {
                    const float c = ex2(sml[u * 2 * G + 2 * g] - mb);
                    const float4 v = *reinterpret_cast<const float4 *>(so + u * G * D + g * D + d);
                    L[k] += sml[u * 2 * G + 2 * g + 1] * c;
                    O[k].x += v.x * c; O[k].y += v.y * c; O[k].z += v.z * c; O[k].w += v.w * c;
                }
                M[k] = mb;
            }
            // the next group's copies reuse the ring; a wait that gave up ends the merge after
            // a bounded wait for this group's copies
            if (__syncthreads_or(!got)) {
                if (threadIdx.x == 0) {
                    record_code(p.dev_code, kDevCodeTimeout);
                    *sm_abort = 1;
                    mbar_wait_ok(bar_merge, (phase - 1) & 1u, p.spin_limit);
                }
                __syncthreads();
                break;
            }
        }
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int ch = threadIdx.x + k * M_THREADS;
            if (ch >= NCH) continue;
            const int g = ch * 4 / D, d = ch * 4 % D;
            const bool any = L[k] > 0.f;
            float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
            if (any) r = make_float4(O[k].x / L[k], O[k].y / L[k], O[k].z / L[k], O[k].w / L[k]);
            *reinterpret_cast<float4 *>(p.out + (size_t)(rows0 + g) * D + d) = r;
            if (d == 0 && p.lse != nullptr)
                p.lse[rows0 + g] = any ? (M[k] + log2f(L[k])) * kLn2 : -INFINITY;
        }
    };

    auto finish_pair = [&](int q, long long q_lo, long long q_hi, bool ring_idle) {
        float l_row = l_part;
        l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
        l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
        if (gr < G) {
#pragma unroll
            for (int n = 0; n < NB; ++n) {
                const int d = half * DW + 8 * n + 2 * tq;
                sm_o[(kg * G + gr) * D + d] = o[n][0];
                sm_o[(kg * G + gr) * D + d + 1] = o[n][1];
            }
            if (tq == 0 && half == 0) {
                sm_m[kg * G + gr] = m_row;
                sm_l[kg * G + gr] = l_row;
            }
        }
        __syncthreads();
        const int c_lo = cta_of(q_lo, T, Ce);
        const int c_hi = cta_of(q_hi - 1, T, Ce);
        const int nseg = c_hi - c_lo + 1;
        const int slot = 2 * cta + (t_begin < q_lo ? 1 : 0);
        const int rows0 = (q / p.Hkv) * p.Hq + (q % p.Hkv) * G;
        for (int i = threadIdx.x; i < G * D; i += M_THREADS) {
            const int g = i / D, d = i % D;
            float M = sm_m[g];
#pragma unroll
            for (int w = 1; w < PL::KGROUPS; ++w) M = fmaxf(M, sm_m[w * G + g]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < PL::KGROUPS; ++w) {
                const float c = ex2(sm_m[w * G + g] - M);
                L += sm_l[w * G + g] * c;
                O += sm_o[(w * G + g) * D + d] * c;
            }
            if (nseg == 1) {
                p.out[(size_t)(rows0 + g) * D + d] = L > 0.f ? O / L : 0.f;
                if (d == 0 && p.lse != nullptr)
                    p.lse[rows0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
            } else {
                const size_t st = (size_t)slot * G + g;
                p.ws_o[st * D + d] = O;
                if (d == 0) {
                    p.ws_ml[st * 2] = M;
                    p.ws_ml[st * 2 + 1] = L;
                }
            }
        }
        __syncthreads();
        if (nseg > 1) {
            if (threadIdx.x == 0) *sm_flag = (ticket_acq_rel(&p.ws_cnt[q]) == nseg - 1);
            __syncthreads();
            if (*sm_flag) {
                const long long tb_lo = (long long)c_lo * T / Ce;  // first tile of block c_lo
                const int slot0 = 2 * c_lo + (tb_lo < q_lo ? 1 : 0);
                // (an aborting block's ring may still receive tile loads: not used then)
                if (ring_idle && nseg > 8 && *sm_abort == 0)   // one batch of registers <= 8
                    merge_staged(slot0, c_lo, nseg, rows0);
                else
                    merge_segments<G, D>(p.ws_o, p.ws_ml, slot0, c_lo, nseg, p.out, p.lse, rows0);
                if (threadIdx.x == 0) p.ws_cnt[q] = 0;
            }
            __syncthreads();
        }
    };

    Cursor mc{};
    if (n_tiles > 0) mc = cursor_at(t_begin);
    int cur = -1;
    long long cur_lo = 0, cur_hi = 0;
    for (int i = 0; i < n_tiles; ++i) {
        const long long t = t_begin + i;
        const int s = i % NS;
        advance(mc, t);
        if (mc.q != cur) {
            if (cur >= 0) finish_pair(cur, cur_lo, cur_hi, false);
            cur = mc.q;
            cur_lo = mc.lo;
            cur_hi = mc.hi;
            start_pair(cur);
        }
        if (!mbar_wait_abortable(bar_full + 8 * s, (i / NS) & 1, p.spin_limit, sm_abort)) {
            record_code(p.dev_code, kDevCodeTimeout);
            *sm_abort = 1;
        }
        const int j0 = (int)(t - cur_lo) * TK;
        const int key0 = kg * 16;                          // this warp's 16 keys in the tile
        if (j0 + key0 < cur_slots) {
            const uint32_t kst = stage0 + s * PL::STAGE_BYTES, vst = kst + PL::TILE_BYTES;
            // ---- logits: S[16 x 16 keys] = Q . K^T over D -------------------------------------
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const int mrow = lane & 7, mi = lane >> 3;    // ldmatrix: matrix mi, row mrow
#pragma unroll
            for (int sp = 0; sp < KSTEPS / 2; ++sp) {
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kst + sw_off(key0 + 8 * nb + mrow, 4 * sp + mi, TK), b0, b1, b2, b3);
                    mma16816(sc[nb], qa0[2 * sp], qa2[2 * sp], b0, b1);
                    mma16816(sc[nb], qa0[2 * sp + 1], qa2[2 * sp + 1], b2, b3);
                }
            }
            // ---- online softmax on row gr (keys key0 + 8nb + 2tq + e) ---------------------------
            float lg[2][2];
            float mx = -INFINITY;
#pragma unroll
            for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = j0 + key0 + 8 * nb + 2 * tq + e;
                    const float v = sc[nb][e] * p.scale_log2;
                    lg[nb][e] = j < cur_slots ? v : -INFINITY;
                    mx = fmaxf(mx, lg[nb][e]);
                    if (lg_row != nullptr && j < cur_slots) lg_row[j] = v * kLn2;
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            if (mx > m_row + kSlack) {
                const float corr = ex2(m_row - mx);
                l_part *= corr;
#pragma unroll
                for (int n = 0; n < NB; ++n) {
                    o[n][0] *= corr;
                    o[n][1] *= corr;
                }
                m_row = mx;
            }
            float pr[2][2];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    pr[nb][e] = ex2(lg[nb][e] - m_row);
                    l_part += pr[nb][e];
                }
            const uint32_t pa0 = pack_bf16(pr[0][0], pr[0][1]);   // keys 2tq, 2tq+1
            const uint32_t pa2 = pack_bf16(pr[1][0], pr[1][1]);   // keys 8+2tq, 9+2tq
            // the rounding residuals (exact in fp32), themselves rounded to bf16
            const uint32_t pb0 = pack_bf16(pr[0][0] - bf16_lo(pa0), pr[0][1] - bf16_hi(pa0));
            const uint32_t pb2 = pack_bf16(pr[1][0] - bf16_lo(pa2), pr[1][1] - bf16_hi(pa2));
            // ---- o[16 x DW] += P[16 x 16 keys] . V[16 keys x DW] --------------------------------
            // Slots past the pair's length are still in the tile (the cache may hold any bytes
            // there); their probabilities are 0, but 0 * NaN would poison the product, so the
            // warp zeroes those rows of its dim range first.
            const int valid_here = cur_slots - (j0 + key0);
            if (valid_here < 16) {
                constexpr int CH = DW / 8;                 // 16-byte chunks per row in my range
                for (int x = lane; x < (16 - valid_here) * CH; x += 32) {
                    const int rr = key0 + valid_here + x / CH;
                    const int chunk = (half * DW) / 8 + x % CH;
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                                     vst + sw_off(rr, chunk, TK)),
                                 "r"(0u)
                                 : "memory");
                }
                __syncwarp();
                // order these generic-proxy writes before the next TMA write into the stage
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            const int vrow = key0 + (mi & 1) * 8 + mrow;
#pragma unroll
            for (int n = 0; n < NB; n += 2) {
                uint32_t b0, b1, b2, b3;
                const int chunk = (half * DW) / 8 + n + (mi >> 1);
                ldsm_x4_t(vst + sw_off(vrow, chunk, TK), b0, b1, b2, b3);
                mma16816(o[n], pa0, pa2, b0, b1);
                mma16816(o[n + 1], pa0, pa2, b2, b3);
                mma16816(o[n], pb0, pb2, b0, b1);
                mma16816(o[n + 1], pb0, pb2, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        if (threadIdx.x == 0 && i + NS < n_tiles && *sm_abort == 0) {
            // a warp that gave up on this stage set the abort flag before releasing it
            if (!mbar_wait_abortable(bar_empty + 8 * s, (i / NS) & 1, p.spin_limit, sm_abort)) {
                record_code(p.dev_code, kDevCodeTimeout);
                *sm_abort = 1;
            } else if (*sm_abort == 0) {
                issue_tile(i + NS);
            }
        }
    }
    if (cur >= 0) finish_pair(cur, cur_lo, cur_hi, true);
    // after an abort the last NS tiles issued (one per stage) may still be landing
    if (threadIdx.x == 0 && *sm_abort != 0)
        for (int i = max(0, last_issued - NS + 1); i <= last_issued; ++i)
            mbar_wait_ok(bar_full + 8 * (i % NS), (i / NS) & 1, p.spin_limit);
}

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;

bool encoder()
{
    std::call_once(g_enc_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_enc != nullptr;
}

bool encode_cache(CUtensorMap *m, const void *ptr, const DecodeParams &p, int D, int TK)
{
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.cap, (cuuint64_t)p.Hkv, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {(cuuint64_t)p.ss * 2, (cuuint64_t)p.sh * 2, (cuuint64_t)p.sb * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)TK, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_typed(const DecodeParams &p, cudaStream_t stream, bool *used)
{
    using PL = MmaPlan<D, G>;
    CUtensorMap km, vm;
    if (!encode_cache(&km, p.k, p, D, PL::TK) || !encode_cache(&vm, p.v, p, D, PL::TK))
        return cudaSuccess;   // not encodable (unusual strides): the caller falls back
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, PL::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    DecodeParams q = p;
    if (q.spin_limit == 0) q.spin_limit = kMbarSpinLimit;
    q.NT = p.cap > 0 ? (p.cap + PL::TK - 1) / PL::TK : 1;
    const long long T_all = (long long)q.P * q.NT;
    long long C = T_all < p.n_sm ? T_all : p.n_sm;
    // two partial-state slots per block in the workspace
    const long long slots = (long long)q.P * q.max_seg;
    if (2 * C > slots) C = slots / 2;
    if (C < 1) C = 1;
    *used = true;
    return launch_pdl(decode_mma_kernel<D, G>, dim3((unsigned)C), dim3(M_THREADS), (size_t)PL::SMEM,
                      stream, km, vm, q);
}

}  // namespace

cudaError_t launch_decode_attn_mma(const DecodeParams &p, int D, int G, cudaStream_t stream,
                                   bool *used)
{
    *used = false;
    if (p.rope || !encoder()) return cudaSuccess;
#define KVC_MMA_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_typed<DD, GG>(p, stream, used);
    KVC_MMA_CASE(64, 2) KVC_MMA_CASE(64, 4) KVC_MMA_CASE(64, 6) KVC_MMA_CASE(64, 8)
    KVC_MMA_CASE(128, 2) KVC_MMA_CASE(128, 4) KVC_MMA_CASE(128, 6) KVC_MMA_CASE(128, 8)
    KVC_MMA_CASE(256, 2) KVC_MMA_CASE(256, 4) KVC_MMA_CASE(256, 6) KVC_MMA_CASE(256, 8)
#undef KVC_MMA_CASE
    return cudaSuccess;
}

}  // namespace kvc
