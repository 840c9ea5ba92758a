// decode_attn.cuh -- decode attention over the retained slots of a KV cache (sm_103a).
//
// What it computes ("O KV cache", llmdeepdive 7.2, "01 · Conceito"): the new token's query
// attends to every valid cached key of its KV head and mixes the cached values -- exact causal
// attention.  Where the time goes ("Compressão e Poda Dinâmica de KV Cache", "O gargalo de
// memória do KV Cache..."): every emitted token reads the whole retained cache from HBM in a
// GEMV at 1-2 FLOP per byte, so this kernel is an HBM stream.  How the work is split
// ("Implementação prática em vLLM e SGLang": FlashDecoding parallelises along the time axis):
// the slots of every (batch, KV head) pair are cut into tiles, and the flattened sequence of
// (pair, tile) work items is divided evenly among persistent thread blocks, so a pair's slots
// may be shared by several blocks; each block keeps an online-softmax state (max m, sum l,
// weighted values o) per query head of the group, and when a pair spans several blocks the last
// block to finish it (atomic ticket, no waiting) merges the states by log-sum-exp.
//
// Data movement.  K and V tiles (TK slots x d_head; 16 KB of keys per tile) stream from HBM into
// an NS-stage shared-memory ring with cp.async.bulk, completion tracked by mbarriers
// (transaction bytes); the block's eight warps compute from shared memory and release each stage
// through a second mbarrier, after which warp 0 refills it NS tiles ahead, the tile's copies
// dealt out over its lanes.  Bytes in flight per SM come from the ring depth and the blocks per
// SM, not registers.
//
// Arithmetic.  fp32 throughout, with Blackwell's packed fp32x2 FMA (two lanes of a float2 per
// instruction) for the q.k dot products and the p*v accumulation.  A key row is read by
// LPK = D/(2*VW) lanes; lane lk holds the VW elements at lk*VW of the first half of the row and
// the VW elements at the same offset of the second half, so both members of every RoPE pair
// (i, i + D/2) sit in one lane.  q is pre-scaled by scale*log2(e) so the softmax is base 2; the
// running max only moves when a logit exceeds it by more than 2^8 (the weights stay below 256,
// far from fp32 overflow), which spares most rescales of o.
//
// RoPE at in-cache positions ("attention sinks", "como funciona"): the logit of query position
// p_q against key position p_k depends only on the distance p_q - p_k, since rotations compose:
// (R(p_q) q).(R(p_k) k) = q.R(p_k - p_q) k.  So q is never rotated; every key is combined with q
// through the rotation by its distance, whose cos and sin come from the distance-indexed table
// (planar rows: d_head/2 cosines then d_head/2 sines).  The attended keys are visited in rank
// order -- the sinks, then the ring from its oldest token to the newest -- which is their
// in-cache position r, so the distance of key r is simply qpos - r.  A tile of TK ranks maps to
// at most three contiguous runs of physical slots (sinks; ring up to its last slot; ring from its
// first slot), copied separately into consecutive rows of the stage.
//
// Factored rotation (one query head per KV head, table of at least TK rows).  Reading a table
// row per key puts an L2 round trip in front of every logit.  Instead, each lane always holds
// the same key offsets kk of a tile, and within the tile starting at rank r0
//     dist = base + (TK - 1 - kk),   base = qpos - r0 - (TK - 1).
// With pair i of the head dimension written as a complex number, the logit term is
// Re(conj(q_i) k_i e^{-i dist th_i}) = Re([conj(q_i) e^{-i (TK-1-kk) th_i}] e^{-i base th_i} k_i).
// The bracket is a per-lane constant formed once per pair from table row TK-1-kk; the issuing
// thread copies row |base| into the stage with the keys, so the per-key work reads only shared
// memory.  A negative base (the newest tile) uses row |base| with the sine negated.
//
// ALiBi at in-cache positions ("attention sinks", "como funciona": the linear bias is applied
// continuously over the cache, never with a jump where tokens were evicted).  The same rank-order
// walk gives every key its distance qpos - r directly, and the logit becomes
// scale * q.k - slope_h * (qpos - r), with the query head's slope from the caller; keys are not
// rotated.
//
// Paged cache ("Implementação prática em vLLM e SGLang": blocks of 16 or 32 tokens behind a page
// table).  The slots of a sequence are its page table's blocks in order; a tile of TK logical
// slots is copied run by run, one bulk copy per block it touches, from the pool's
// [head][block][slot][d] rows, so the compute loop is unchanged.  The pool is head-major: all
// of one head's blocks lie in one region (n_blocks * block_size rows), so the blocks a (sequence,
// head) pair reads stay within a few large pages wherever the page table puts them.  A table entry outside the pool
// records KVC_DEV_BAD_BLOCK and reads block 0 instead (the copy sizes stay as announced).
//
// DuoAttention ("Decomposição funcional com o DuoAttention": retrieval heads keep the full
// cache, streaming heads a constant buffer of sinks and recent tokens).  One launch covers both
// kinds.  The tiles of the retrieval pairs (B x n_ret, full caches, NT tiles each) are split
// evenly over the blocks as usual; each streaming pair (B x n_str, ring caches, NT2 tiles) goes
// whole to one block, round-robin, ahead of that block's retrieval range -- a streaming pair is
// almost all fixed cost (its q, its output), so spreading them keeps any block from collecting
// many.  head_of maps each pair back to the model's KV head for q, the outputs and the logits.
//
// Waits on mbarriers are bounded (p.spin_limit polls).  A wait that gives up records
// KVC_DEV_TIMEOUT and raises the block's abort flag: the issuing thread loads nothing more,
// the other waits of the block give up at once, and the block still walks its tiles (computing
// on whatever the stages hold) and takes part in the merge tickets, so every block finishes
// and the tickets are left zeroed.  Before exiting, the issuing thread waits (again bounded)
// for the loads it issued last, so no copy is still landing in the block's shared memory when
// it exits.  The outputs of such a call are invalid.  The flag is read only once a first poll
// has failed, so the waits that succeed at once cost what they did without it.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace kvc {

constexpr int kDecodeWarps = 8;
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kDecodeTileKeyBytes = 16384;   // bytes of keys per tile
constexpr int kDevCodeSchedule = 8;          // KVC_DEV_SCHEDULE
constexpr float kLazyMaxSlack = 8.0f;        // log2 units

// VW elements of T at a shared address, widened to VW/2 float2 (consecutive elements paired).
template <typename T, int VW>
__device__ __forceinline__ void lds_pairs(uint32_t addr, float2 *f)
{
    if constexpr (sizeof(T) == 4) {
        static_assert(VW == 4, "fp32 lane vector");
        float4 x;
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                     : "r"(addr));
        f[0] = make_float2(x.x, x.y);
        f[1] = make_float2(x.z, x.w);
    } else if constexpr (VW == 8) {
        uint32_t a, b, c, d;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                     : "r"(addr));
        f[0] = make_float2(bf16_lo(a), bf16_hi(a));
        f[1] = make_float2(bf16_lo(b), bf16_hi(b));
        f[2] = make_float2(bf16_lo(c), bf16_hi(c));
        f[3] = make_float2(bf16_lo(d), bf16_hi(d));
    } else {
        static_assert(VW == 4, "bf16 lane vector");
        uint32_t a, b;
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
        f[0] = make_float2(bf16_lo(a), bf16_hi(a));
        f[1] = make_float2(bf16_lo(b), bf16_hi(b));
    }
}

// Persistent schedule: tile t (pair-major) belongs to block floor(((t+1)*C - 1) / T).
__device__ __forceinline__ int cta_of_tile(long long t, long long T, int C)
{
    return (int)(((t + 1) * (long long)C - 1) / T);
}

// Shared-memory plan of one instantiation (host and device agree): two blocks per SM with a
// three-stage ring where they fit (and the group is small enough for 128 registers a thread),
// else one block with a deeper ring.
template <typename T, int D, int G, int RM = 0>
struct DecodeSmem {
    static constexpr int TK = kDecodeTileKeyBytes / (D * (int)sizeof(T));
    static constexpr int kTileBytes = TK * D * (int)sizeof(T);
    static constexpr int kRotBytes = RM == 2 ? D * 4 : 0;   // staged base row (factored RoPE)
    static constexpr int kStageBytes = 2 * kTileBytes + kRotBytes;
    static constexpr int kMergeBytes = kDecodeWarps * G * (D + 2) * 4 + 16;
    static constexpr int kBarBytes = 256;
    static constexpr int kTwoBlockBytes = kBarBytes + 3 * kStageBytes + kMergeBytes;
    static constexpr int CPS = (G <= 4 && 2 * (kTwoBlockBytes + 1024) <= 233472) ? 2 : 1;
    static constexpr int NS_one = (220 * 1024 - kMergeBytes - kBarBytes) / kStageBytes;
    static constexpr int NS = CPS == 2 ? 3 : (NS_one > 6 ? 6 : NS_one);
    static_assert(NS >= 2, "decode pipeline needs at least two stages");
    static constexpr int kBytes = kBarBytes + NS * kStageBytes + kMergeBytes;
};

// RM: 0 no RoPE, 1 RoPE with one table row per key, 2 factored RoPE (G == 1, n_pos >= TK),
// 3 ALiBi, 4 paged (no positional term), 5 DuoAttention (no positional term).  Modes 1-3 read
// the StreamingLLM sink + ring layout in rank order.
template <typename T, int D, int G, int VW, int UNR, int RM, int CPS>
__global__ void __launch_bounds__(kDecodeThreads, CPS)
decode_attn_kernel(const DecodeParams p)
{
    using SM = DecodeSmem<T, D, G, RM>;
    constexpr bool RANKED = RM >= 1 && RM <= 3;   // sink + ring layout, visited in rank order
    constexpr bool PAGED = RM == 4;
    constexpr bool DUO = RM == 5;
    constexpr bool ROPE = RM == 1 || RM == 2;
    constexpr bool FACT = RM == 2;
    constexpr bool ALIBI = RM == 3;
    constexpr int TK = SM::TK;
    constexpr int NS = SM::NS;
    constexpr int NW = kDecodeWarps;
    constexpr int HALF = D / 2;
    constexpr int LPK = HALF / VW;
    static_assert(LPK >= 1 && LPK <= 32 && (32 % LPK) == 0, "lane layout");
    static_assert(VW % 2 == 0, "pairs of elements");
    constexpr int KPW = 32 / LPK;
    constexpr int P2 = VW / 2;          // float2 per half-row per lane
    constexpr int KEYS_PER_STEP = NW * KPW * UNR;
    static_assert(TK % KEYS_PER_STEP == 0, "tile must be a whole number of steps");
    constexpr int STEPS = TK / KEYS_PER_STEP;
    constexpr int EB = (int)sizeof(T);
    static_assert(!FACT || (G == 1 && STEPS == 1), "factored RoPE: fixed key offsets per lane");

    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar_full = sbase;                 // NS x 8 bytes
    const uint32_t bar_empty = sbase + 8 * NS;       // NS x 8 bytes
    const uint32_t stage0 = sbase + SM::kBarBytes;
    // bytes 128..255 of the barrier area: the issuing thread's cache of page-table entries
    static_assert(16 * NS <= 128, "barriers fit below the table cache");
    constexpr int kTabCache = 32;
    float *sm_m = reinterpret_cast<float *>(smem + SM::kBarBytes + NS * SM::kStageBytes);
    float *sm_l = sm_m + NW * G;
    float *sm_o = sm_l + NW * G;                     // [NW][G][D]
    int *sm_flag = reinterpret_cast<int *>(sm_o + NW * G * D);
    volatile int *sm_abort = sm_flag + 1;            // set once a bounded wait has given up

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int C = gridDim.x;
    const int cta = blockIdx.x;
    // DuoAttention: the even split covers the T_ret retrieval tiles only; streaming pairs
    // cta, cta + C, ... (n_own of them) come first in this block's list
    const long long T_ret = DUO ? (long long)p.B * p.n_ret * p.NT : 0;
    const int P_ret = DUO ? p.B * p.n_ret : 0;
    const int P_str = DUO ? p.B * p.n_str : 0;
    const int n_own = DUO ? (cta < P_str ? (P_str - 1 - cta) / C + 1 : 0) : 0;
    const long long T_all = DUO ? T_ret : (long long)p.P * p.NT;
    const long long t_begin = (long long)cta * T_all / C;
    const long long t_end = (long long)(cta + 1) * T_all / C;
    const int n_tiles = (int)(t_end - t_begin) + n_own * (DUO ? p.NT2 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, NW);
        }
        *sm_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // With a settled cache the position, the lengths and the first tiles are read before
    // waiting for the previous kernel; q, the outputs and the workspace always after.
    if (!p.kv_settled) {
        pdl_trigger();
        pdl_wait();                                  // inputs may come from the previous kernel
    }

    // ---- decode position (StreamingLLM layout) --------------------------------------------
    // With RoPE or ALiBi the tiles run over ranks: rank r < S is sink slot r; rank r >= S is ring token
    // a_old + (r - S), at slot S + (ring_off + r - S) mod (W + 1), a_old = max(S, t - W) being the
    // oldest ring token still attended.  n_att = min(t + 1, S + W + 1) ranks are attended.
    int qpos = 0, n_att = 0, ring_off = 0;
    int n_ring = 0;            // DuoAttention: valid slots of a streaming head's ring
    if (DUO) {
        int64_t tpos = *p.t;
        if (tpos < 0) {
            if (threadIdx.x == 0) record_code(p.dev_code, 4 /* KVC_DEV_BAD_POSITION */);
            tpos = 0;
        }
        n_ring = (int)(tpos + 1 < (int64_t)p.ring_cap ? tpos + 1 : (int64_t)p.ring_cap);
    }
    if (RANKED) {
        int64_t tpos = *p.t;
        if (tpos < 0) {
            if (threadIdx.x == 0) record_code(p.dev_code, 4 /* KVC_DEV_BAD_POSITION */);
            tpos = 0;
        }
        const int64_t sw = (int64_t)p.S + p.W;
        qpos = (int)(tpos < sw ? tpos : sw);
        n_att = qpos + 1;
        const int64_t a_old = tpos - p.W > (int64_t)p.S ? tpos - p.W : (int64_t)p.S;
        ring_off = (int)((a_old - p.S) % (int64_t)(p.W + 1));
    }
    auto rank_slot = [&](int r) -> int {
        if (r < p.S) return r;
        int x = ring_off + (r - p.S);
        if (x > p.W) x -= p.W + 1;
        return p.S + x;
    };
    // ---- pairs and tiles -------------------------------------------------------------------
    // this block's tile i -> its pair q and first slot j0
    auto locate = [&](int i, int &q, int &j0) {
        if constexpr (DUO) {
            const int own = n_own * p.NT2;
            if (i < own) {
                q = P_ret + cta + (i / p.NT2) * C;
                j0 = (i % p.NT2) * TK;
            } else {
                const long long t = t_begin + (i - own);
                q = (int)(t / p.NT);
                j0 = (int)(t % p.NT) * TK;
            }
        } else {
            const long long t = t_begin + i;
            q = (int)(t / p.NT);
            j0 = (int)(t % p.NT) * TK;
        }
    };
    // Walking this block's tiles in order: one division at the start, then the pair and first
    // slot advance by one tile at a time.  DuoAttention's streaming pairs come first in its list,
    // so it keeps locate(); so does the per-key rotation, whose registers are all taken.
    constexpr bool CURSOR = !DUO && RM != 1;
    struct TileCursor {
        int i, q, j0;
    };
    auto cursor_start = [&]() -> TileCursor {
        TileCursor c{0, 0, 0};
        if constexpr (CURSOR) {
            c.q = (int)(t_begin / p.NT);
            c.j0 = (int)(t_begin % p.NT) * TK;
        }
        return c;
    };
    auto cursor_get = [&](const TileCursor &c, int &q, int &j0) {
        if constexpr (!CURSOR) {
            locate(c.i, q, j0);
        } else {
            q = c.q;
            j0 = c.j0;
        }
    };
    auto cursor_next = [&](TileCursor &c) {
        ++c.i;
        if constexpr (CURSOR) {
            c.j0 += TK;
            if (c.j0 >= p.NT * TK) {
                c.j0 = 0;
                ++c.q;
            }
        }
    };
    // first tile and tile count of pair q in the even split (DuoAttention: retrieval pairs;
    // a streaming pair is one block's alone)
    auto pair_first = [&](int q) -> long long { return (long long)q * p.NT; };
    auto pair_tiles = [&](int q) -> int { return p.NT; };
    // batch row and model KV head of pair q
    auto pair_bk = [&](int q, int &b, int &kh) {
        if constexpr (DUO) {
            if (q < P_ret) {
                b = q / p.n_ret;
                kh = p.head_of[q % p.n_ret];
            } else {
                b = (q - P_ret) / p.n_str;
                kh = p.head_of[p.n_ret + (q - P_ret) % p.n_str];
            }
        } else {
            b = q / p.Hkv;
            kh = q % p.Hkv;
        }
    };
    // number of work items (slots without RoPE, ranks with it) of pair q
    auto pair_slots = [&](int q) -> int {
        if (RANKED) return n_att;
        if (DUO && q >= P_ret) return n_ring;
        if (PAGED) {
            const int n = p.len[q / p.Hkv];
            return n < 0 ? 0 : (n > p.cap ? p.cap : n);
        }
        if (p.len != nullptr) {
            const int n = p.len[q];
            return n < 0 ? 0 : (n > p.cap ? p.cap : n);
        }
        return p.n_valid;
    };

    // ---- tile loader: warp 0 issues the bulk copies of tile i into stage i % NS ------------
    // Every lane of warp 0 walks the same tiles; a tile's copies (its K and V runs, the RoPE base
    // row, or the page blocks it touches) are dealt out over the lanes, so issuing them costs
    // one copy's issue time rather than the sum (each bulk copy takes a few hundred cycles to
    // issue: 360 ns per tile for two copies, 790 ns for a paged tile's four, against ~500 ns of
    // the issuing warp's own arithmetic), and lane 0 arrives on the stage's barrier with the byte
    // count.  DuoAttention (two contiguous copies per tile) keeps one issuing thread, which
    // leaves warp 0's other lanes free to start the next tile while it refills (97 % against
    // 92.5 % of the HBM peak issued by the warp).
    constexpr bool WARP_ISSUE = !DUO;
    const bool LOADER = WARP_ISSUE ? warp == 0 : threadIdx.x == 0;
    const bool dense = (p.ss == D);
    // The loader keeps the slot count of the pair it is loading: one global read per pair, not
    // one per tile on the critical path of every copy.
    int iss_q = -1, iss_slots = 0;
    // Paged: it also keeps a window of kTabCache page-table entries of the sequence it is
    // loading in shared memory, fetched together with cp.async, one entry per lane (one round
    // trip per window, not one per block on the critical path of every copy).
    int tab_b = -1, tab_lo = 0, tab_cnt = 0;
    auto table_entry = [&](int b, int lb) -> int {
        if (b != tab_b || lb < tab_lo || lb >= tab_lo + tab_cnt) {
            // aligned windows: every head of a sequence restarts at block 0, and a sequence of
            // at most kTabCache blocks is fetched once
            tab_b = b;
            tab_lo = lb - lb % kTabCache;
            tab_cnt = min(kTabCache, p.max_blocks - tab_lo);
            const int32_t *src = p.table + (size_t)b * p.max_blocks + tab_lo;
            static_assert(kTabCache <= 32, "one table entry per lane");
            if (lane < tab_cnt)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                             :: "r"(sbase + 128 + 4 * lane), "l"(src + lane) : "memory");
            asm volatile("cp.async.wait_all;" ::: "memory");
            __syncwarp();
        }
        return reinterpret_cast<const int32_t *>(smem + 128)[lb - tab_lo];
    };
    int last_issued = -1;      // the loader's last tile (the drain after an abort)
    TileCursor iss_cur = cursor_start();
    auto issue_tile = [&](int i) {
        if (p.starve) return;  // test hook: no loads, no arrivals (the waits run out)
        last_issued = i;
        const int s = i % NS;
        int q, j0;
        cursor_get(iss_cur, q, j0);
        cursor_next(iss_cur);
        if (q != iss_q) {
            // paged: the pairs of a sequence share its length
            if (!PAGED || iss_q < 0 || q / p.Hkv != iss_q / p.Hkv) iss_slots = pair_slots(q);
            iss_q = q;
        }
        const int rows = max(0, min(TK, iss_slots - j0));
        const uint32_t full = bar_full + 8 * s;
        const uint32_t kdst = stage0 + s * SM::kStageBytes;
        const uint32_t vdst = kdst + SM::kTileBytes;
        const int b = q / p.Hkv, kh = q % p.Hkv;
        const T *kb, *vb;
        if constexpr (DUO) {
            // the pair's own cache: a retrieval head's full cache or a streaming head's ring
            if (q < P_ret) {
                const size_t base = (size_t)(q / p.n_ret) * p.sb + (size_t)(q % p.n_ret) * p.sh;
                kb = static_cast<const T *>(p.k) + base;
                vb = static_cast<const T *>(p.v) + base;
            } else {
                const int qs = q - P_ret;
                const size_t base = (size_t)(qs / p.n_str) * p.sb2 + (size_t)(qs % p.n_str) * p.sh2;
                kb = static_cast<const T *>(p.k2) + base;
                vb = static_cast<const T *>(p.v2) + base;
            }
        } else {
            const size_t base = (size_t)b * p.sb + (size_t)kh * p.sh;
            kb = static_cast<const T *>(p.k) + base;
            vb = static_cast<const T *>(p.v) + base;
        }
        if (rows == 0) {
            if (lane == 0) mbar_arrive(full);
            return;
        }
        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(2 * rows * D * EB + SM::kRotBytes));
        // the tile's copies, dealt out over the lanes in order
        int job = 0;
        auto copy = [&](uint32_t dst, const void *src, uint32_t bytes) {
            if (((WARP_ISSUE ? job : 0) & 31) == lane) bulk_g2s(dst, src, bytes, full);
            ++job;
        };
        if constexpr (FACT) {
            // |base| <= max(TK - 1, qpos) < n_pos (checked on the host)
            const int row = min(abs(qpos - j0 - (TK - 1)), p.n_pos - 1);
            copy(vdst + SM::kTileBytes, p.cos_sin + (size_t)row * D, D * 4);
        }
        // copy rows [r_a, r_b) of the tile's work items, physically contiguous from slot j_a
        auto copy_run = [&](int r_a, int r_b, int j_a) {
            if (r_b <= r_a) return;
            const uint32_t off = (uint32_t)((r_a - j0) * D * EB);
            if (dense) {
                copy(kdst + off, kb + (size_t)j_a * D, (r_b - r_a) * D * EB);
                copy(vdst + off, vb + (size_t)j_a * D, (r_b - r_a) * D * EB);
            } else {
                for (int r = 0; r < r_b - r_a; ++r) {
                    copy(kdst + off + r * D * EB, kb + (size_t)(j_a + r) * p.ss, D * EB);
                    copy(vdst + off + r * D * EB, vb + (size_t)(j_a + r) * p.ss, D * EB);
                }
            }
        };
        const int j1 = j0 + rows;
        if constexpr (PAGED) {
            // one run per block of the page table the tile touches; one division per tile
            const T *kh_k = static_cast<const T *>(p.k) + (size_t)kh * p.n_pool * p.bs * D;
            const T *kh_v = static_cast<const T *>(p.v) + (size_t)kh * p.n_pool * p.bs * D;
            int lb = j0 / p.bs;
            int off = j0 - lb * p.bs;
            uint32_t doff = 0;
            for (int r = j0; r < j1; ++lb) {
                const int n = min(j1 - r, p.bs - off);
                int phys = table_entry(b, lb);
                if (phys < 0 || phys >= p.n_pool) {
                    if (lane == 0) record_code(p.dev_code, 9 /* KVC_DEV_BAD_BLOCK */);
                    phys = 0;
                }
                const size_t src = (size_t)phys * p.bs * D + (size_t)off * D;
                const uint32_t bytes = (uint32_t)n * (uint32_t)(D * EB);
                copy(kdst + doff, kh_k + src, bytes);
                copy(vdst + doff, kh_v + src, bytes);
                doff += bytes;
                r += n;
                off = 0;
            }
        } else if (!RANKED) {
            copy_run(j0, j1, j0);
        } else {
            copy_run(j0, min(j1, p.S), j0);                          // sinks
            const int ra = max(j0, p.S);
            if (ra < j1) {
                const int sa = rank_slot(ra);                        // ring, up to its last slot
                const int rb = min(j1, ra + (p.S + p.W + 1 - sa));
                copy_run(ra, rb, sa);
                copy_run(rb, j1, p.S);                               // ring, from its first slot
            }
        }
    };
    if (LOADER)
        for (int i = 0; i < NS && i < n_tiles; ++i) issue_tile(i);
    if (p.kv_settled) {
        pdl_trigger();
        pdl_wait();
    }

    // ================================= compute ===================================================
    const int lk = lane % LPK;
    const int ks = lane / LPK;
    const int d0 = lk * VW;

    float2 q1[G][P2], q2[G][P2], q2n[G][P2];   // q halves (pre-scaled); q2n = -q2 (RoPE form)
    float2 pr[UNR][P2], pi[UNR][P2];            // factored RoPE: conj(q) e^{-i (TK-1-kk) th}
    float2 o1[G][P2], o2[G][P2];
    float m[G], l[G];
    float slope2[G];           // ALiBi: the query heads' slopes times log2(e)
    int cur = -1;              // pair in progress
    int cur_slots = 0;
    int cur_li = -1;           // whose length cur_slots holds (paged: the pairs of a sequence share it)

    // The loads a pair starts with -- its query rows and, with the factored rotation, the table
    // rows of the lane's key offsets -- are issued before the previous pair's merge, whose
    // barriers and ticket then hide their latency (the old pair's q and rotation registers are
    // free by then).
    constexpr int QW = VW * (int)sizeof(T) / 4;       // 32-bit words of a lane's half-row
    constexpr int FU = FACT ? UNR : 1;
    constexpr int FR = FACT ? P2 / 2 : 1;
    struct PairFetch {
        uint32_t qa[G][QW], qc[G][QW];                // q: first and second half, raw words
        float4 rc[FU][FR], rs[FU][FR];                // factored rotation: cosines, sines
    };
    auto load_words = [](const T *src, uint32_t (&w)[QW]) {
        if constexpr (QW == 4) {
            const uint4 x = *reinterpret_cast<const uint4 *>(src);
            w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        } else {
            static_assert(QW == 2, "lane vector of 8 or 16 bytes");
            const uint2 x = *reinterpret_cast<const uint2 *>(src);
            w[0] = x.x; w[1] = x.y;
        }
    };
    auto words_to_floats = [](const uint32_t (&w)[QW], float *f) {
#pragma unroll
        for (int i = 0; i < QW; ++i) {
            if constexpr (sizeof(T) == 4) {
                f[i] = __uint_as_float(w[i]);
            } else {
                f[2 * i] = bf16_lo(w[i]);
                f[2 * i + 1] = bf16_hi(w[i]);
            }
        }
    };
    auto fetch_pair = [&](int q) -> PairFetch {
        PairFetch f;
        int b, kh;
        pair_bk(q, b, kh);
        const T *qb = static_cast<const T *>(p.q) + ((size_t)b * p.Hq + (size_t)kh * G) * D;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            load_words(qb + (size_t)g * D + d0, f.qa[g]);
            load_words(qb + (size_t)g * D + HALF + d0, f.qc[g]);
        }
        if constexpr (FACT) {
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int rk = TK - 1 - (warp * KPW * UNR + ks + u * KPW);
                const float *row = p.cos_sin + (size_t)rk * D;
#pragma unroll
                for (int i2 = 0; i2 < P2; i2 += 2) {
                    f.rc[u][i2 / 2] = __ldg(reinterpret_cast<const float4 *>(row + d0 + 2 * i2));
                    f.rs[u][i2 / 2] =
                        __ldg(reinterpret_cast<const float4 *>(row + HALF + d0 + 2 * i2));
                }
            }
        }
        return f;
    };
    auto start_pair = [&](int q, const PairFetch &f) {
        cur = q;
        const int li = PAGED ? q / p.Hkv : q;
        if (li != cur_li) {
            cur_li = li;
            cur_slots = pair_slots(q);
        }
        int b, kh;
        pair_bk(q, b, kh);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float a[VW], c[VW];
            words_to_floats(f.qa[g], a);
            words_to_floats(f.qc[g], c);
#pragma unroll
            for (int i = 0; i < P2; ++i) {
                q1[g][i] = make_float2(a[2 * i] * p.scale_log2, a[2 * i + 1] * p.scale_log2);
                q2[g][i] = make_float2(c[2 * i] * p.scale_log2, c[2 * i + 1] * p.scale_log2);
                q2n[g][i] = make_float2(-q2[g][i].x, -q2[g][i].y);
                o1[g][i] = make_float2(0.f, 0.f);
                o2[g][i] = make_float2(0.f, 0.f);
            }
            m[g] = kNegBig;
            l[g] = 0.f;
            slope2[g] = ALIBI ? __ldg(p.alibi + kh * G + g) * kLog2e : 0.f;
        }
        if constexpr (FACT) {
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
#pragma unroll
                for (int i2 = 0; i2 < P2; i2 += 2) {
                    const float4 c4 = f.rc[u][i2 / 2], s4 = f.rs[u][i2 / 2];
                    const float2 cc[2] = {make_float2(c4.x, c4.y), make_float2(c4.z, c4.w)};
                    const float2 ss[2] = {make_float2(s4.x, s4.y), make_float2(s4.z, s4.w)};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // (q1 - i q2)(c - i s) = (q1 c - q2 s) - i (q1 s + q2 c)
                        const float2 a = q1[0][i2 + h], b = q2[0][i2 + h];
                        pr[u][i2 + h] = __ffma2_rn(q2n[0][i2 + h], ss[h], __fmul2_rn(a, cc[h]));
                        const float2 t = __ffma2_rn(a, ss[h], __fmul2_rn(b, cc[h]));
                        pi[u][i2 + h] = make_float2(-t.x, -t.y);
                    }
                }
            }
        }
    };

    // Merge this block's state for pair `q` and write the output or a partial state; the last
    // block of a shared pair merges every partial.
    auto finish_pair = [&](int q) {
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float m_o = __shfl_xor_sync(0xffffffffu, m[g], off);
                const float l_o = __shfl_xor_sync(0xffffffffu, l[g], off);
                const float m_n = fmaxf(m[g], m_o);
                const float c1 = ex2(m[g] - m_n), c2 = ex2(m_o - m_n);
                l[g] = l[g] * c1 + l_o * c2;
#pragma unroll
                for (int i = 0; i < P2; ++i) {
                    const float2 x = o1[g][i], y = o2[g][i];
                    o1[g][i].x = x.x * c1 + __shfl_xor_sync(0xffffffffu, x.x, off) * c2;
                    o1[g][i].y = x.y * c1 + __shfl_xor_sync(0xffffffffu, x.y, off) * c2;
                    o2[g][i].x = y.x * c1 + __shfl_xor_sync(0xffffffffu, y.x, off) * c2;
                    o2[g][i].y = y.y * c1 + __shfl_xor_sync(0xffffffffu, y.y, off) * c2;
                }
                m[g] = m_n;
            }
        }
        if (ks == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float *row = sm_o + (warp * G + g) * D;
#pragma unroll
                for (int i = 0; i < P2; ++i) {
                    row[d0 + 2 * i] = o1[g][i].x;
                    row[d0 + 2 * i + 1] = o1[g][i].y;
                    row[HALF + d0 + 2 * i] = o2[g][i].x;
                    row[HALF + d0 + 2 * i + 1] = o2[g][i].y;
                }
                if (lk == 0) {
                    sm_m[warp * G + g] = m[g];
                    sm_l[warp * G + g] = l[g];
                }
            }
        }
        __syncthreads();
        const long long t_first = pair_first(q);
        const bool whole = DUO && q >= P_ret;        // a streaming pair: this block alone
        const int c_lo = whole ? cta : cta_of_tile(t_first, T_all, C);
        const int c_hi = whole ? cta : cta_of_tile(t_first + pair_tiles(q) - 1, T_all, C);
        const int nseg = c_hi - c_lo + 1;
        const int seg = cta - c_lo;
        const bool seg_ok = nseg <= p.max_seg;   // guaranteed by the host plan; checked anyway
        if (!seg_ok && threadIdx.x == 0) record_code(p.dev_code, kDevCodeSchedule);
        int pb, pkh;
        pair_bk(q, pb, pkh);
        const int rows0 = pb * p.Hq + pkh * G;
        for (int i = threadIdx.x; i < G * D; i += kDecodeThreads) {
            const int g = i / D, d = i % D;
            float M = sm_m[g];
#pragma unroll
            for (int w = 1; w < NW; ++w) M = fmaxf(M, sm_m[w * G + g]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float c = ex2(sm_m[w * G + g] - M);
                L += sm_l[w * G + g] * c;
                O += sm_o[(w * G + g) * D + d] * c;
            }
            if (nseg == 1) {
                p.out[(size_t)(rows0 + g) * D + d] = L > 0.f ? O / L : 0.f;
                if (d == 0 && p.lse != nullptr)
                    p.lse[rows0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
            } else if (seg_ok) {
                const size_t slot = ((size_t)q * p.max_seg + seg) * G + g;
                p.ws_o[slot * D + d] = O;
                if (d == 0) {
                    p.ws_ml[slot * 2] = M;
                    p.ws_ml[slot * 2 + 1] = L;
                }
            }
        }
        if (nseg > 1 && seg_ok) {
            // the block barrier orders every thread's partial-state writes before thread 0's
            // release; its acquire (and the barrier after it) orders the last block's reads of
            // the other blocks' states after their writes
            __syncthreads();
            if (threadIdx.x == 0) *sm_flag = (ticket_acq_rel(&p.ws_cnt[q]) == nseg - 1);
            __syncthreads();
            if (*sm_flag) {
                merge_pair_partials<G, D, kDecodeThreads>(p.ws_o, p.ws_ml, p.max_seg, q, nseg, p.out,
                                                    p.lse, rows0, sm_o, NW * G * D);
                if (threadIdx.x == 0) p.ws_cnt[q] = 0;   // leave the ticket zeroed
            }
        }
        __syncthreads();   // the merge area is reused by the next pair
    };

    TileCursor cmp_cur = cursor_start();
    for (int i = 0; i < n_tiles; ++i) {
        const int s = i % NS;
        int q, j0;
        cursor_get(cmp_cur, q, j0);
        cursor_next(cmp_cur);
        if (q != cur) {
            const PairFetch pf = fetch_pair(q);
            if (cur >= 0) finish_pair(cur);
            start_pair(q, pf);
        }
        if (!mbar_wait_abortable(bar_full + 8 * s, (i / NS) & 1, p.spin_limit, sm_abort)) {
            record_code(p.dev_code, kDevCodeTimeout);
            *sm_abort = 1;
        }
        const uint32_t kst = stage0 + s * SM::kStageBytes;
        const uint32_t vst = kst + SM::kTileBytes;
        int lb_, lkh_;
        pair_bk(q, lb_, lkh_);
        float *lg_out =
            p.logits ? p.logits + (size_t)(lb_ * p.Hq + lkh_ * G) * p.logits_stride : nullptr;
        // factored RoPE: the tile's base row e^{-i base th} (cosines, sines signed by base)
        float2 cb[P2], ncb[P2], sb[P2];
        if constexpr (FACT) {
            const float *row =
                reinterpret_cast<const float *>(smem + (vst - sbase) + SM::kTileBytes);
            const float sg = (qpos - j0 - (TK - 1)) < 0 ? -1.f : 1.f;
#pragma unroll
            for (int x = 0; x < VW; x += 4) {
                const float4 c4 = *reinterpret_cast<const float4 *>(row + d0 + x);
                const float4 s4 = *reinterpret_cast<const float4 *>(row + HALF + d0 + x);
                cb[x / 2] = make_float2(c4.x, c4.y);
                cb[x / 2 + 1] = make_float2(c4.z, c4.w);
                sb[x / 2] = make_float2(sg * s4.x, sg * s4.y);
                sb[x / 2 + 1] = make_float2(sg * s4.z, sg * s4.w);
            }
#pragma unroll
            for (int i2 = 0; i2 < P2; ++i2) ncb[i2] = make_float2(-cb[i2].x, -cb[i2].y);
        }
#pragma unroll 1
        for (int st = 0; st < STEPS; ++st) {
            const int kbase = st * KEYS_PER_STEP + warp * KPW * UNR + ks;
            float lg[UNR][G];
            bool valid[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int kk = kbase + u * KPW;
                const int j = j0 + kk;
                const bool ok = j < cur_slots;
                valid[u] = ok;
                float2 k1[P2], k2[P2];
                const uint32_t row = kst + (uint32_t)(kk * D * EB);
                lds_pairs<T, VW>(row + d0 * EB, k1);
                lds_pairs<T, VW>(row + (HALF + d0) * EB, k2);
                if constexpr (FACT) {
                    // q' = (pr + i pi) e^{-i base th};  logit = Re(q' (k1 + i k2))
                    //    = k1 (pr c + pi s) + k2 (pr s - pi c)
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i2 = 0; i2 < P2; ++i2) {
                        const float2 re = __ffma2_rn(pi[u][i2], sb[i2], __fmul2_rn(pr[u][i2], cb[i2]));
                        const float2 w2 = __ffma2_rn(pr[u][i2], sb[i2], __fmul2_rn(pi[u][i2], ncb[i2]));
                        acc = __ffma2_rn(k1[i2], re, acc);
                        acc = __ffma2_rn(k2[i2], w2, acc);
                    }
                    lg[u][0] = acc.x + acc.y;
                } else if constexpr (ROPE) {
                    // rotate q by the key's distance (rank j: qpos - j) and dot with the key
                    const float *cs = p.cos_sin + (size_t)(ok ? qpos - j : 0) * D;
                    float2 cd[P2], sd[P2];
#pragma unroll
                    for (int i2 = 0; i2 < P2; i2 += 2) {
                        const float4 c4 = __ldg(reinterpret_cast<const float4 *>(cs + d0 + 2 * i2));
                        const float4 s4 =
                            __ldg(reinterpret_cast<const float4 *>(cs + HALF + d0 + 2 * i2));
                        cd[i2] = make_float2(c4.x, c4.y);
                        sd[i2] = make_float2(s4.x, s4.y);
                        cd[i2 + 1] = make_float2(c4.z, c4.w);
                        sd[i2 + 1] = make_float2(s4.z, s4.w);
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i2 = 0; i2 < P2; ++i2) {
                            // u = q1 c - q2 s, w = q2 c + q1 s; logit += k1 u + k2 w
                            const float2 uu =
                                __ffma2_rn(q2n[g][i2], sd[i2], __fmul2_rn(q1[g][i2], cd[i2]));
                            const float2 ww =
                                __ffma2_rn(q1[g][i2], sd[i2], __fmul2_rn(q2[g][i2], cd[i2]));
                            acc = __ffma2_rn(k1[i2], uu, acc);
                            acc = __ffma2_rn(k2[i2], ww, acc);
                        }
                        lg[u][g] = acc.x + acc.y;
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i2 = 0; i2 < P2; ++i2) {
                            acc = __ffma2_rn(k1[i2], q1[g][i2], acc);
                            acc = __ffma2_rn(k2[i2], q2[g][i2], acc);
                        }
                        lg[u][g] = acc.x + acc.y;
                    }
                }
            }
#pragma unroll
            for (int off = LPK / 2; off > 0; off >>= 1)
#pragma unroll
                for (int u = 0; u < UNR; ++u)
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        lg[u][g] += __shfl_xor_sync(0xffffffffu, lg[u][g], off);
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                if constexpr (ALIBI) {
                    // the key of rank j sits qpos - j positions before the query
                    const float dist = (float)(qpos - (j0 + kbase + u * KPW));
#pragma unroll
                    for (int g = 0; g < G; ++g) lg[u][g] = fmaf(-slope2[g], dist, lg[u][g]);
                }
                if (!valid[u]) {
#pragma unroll
                    for (int g = 0; g < G; ++g) lg[u][g] = -INFINITY;
                } else if (lg_out != nullptr && lk == 0) {
                    const int j = RANKED ? rank_slot(j0 + kbase + u * KPW) : j0 + kbase + u * KPW;
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        lg_out[(size_t)g * p.logits_stride + j] = lg[u][g] * kLn2;
                }
            }
            // lazy running max: move it only when a logit exceeds it by more than the slack
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = lg[0][g];
#pragma unroll
                for (int u = 1; u < UNR; ++u) mx = fmaxf(mx, lg[u][g]);
                if (mx > m[g] + kLazyMaxSlack) {
                    const float corr = ex2(m[g] - mx);
                    l[g] *= corr;
                    const float2 c2 = make_float2(corr, corr);
#pragma unroll
                    for (int i2 = 0; i2 < P2; ++i2) {
                        o1[g][i2] = __fmul2_rn(o1[g][i2], c2);
                        o2[g][i2] = __fmul2_rn(o2[g][i2], c2);
                    }
                    m[g] = mx;
                }
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                // masked keys are skipped outright: their shared-memory rows may hold stale
                // bytes, and 0 * (NaN or Inf) would poison the sum
                if (!valid[u]) continue;
                const int kk = kbase + u * KPW;
                float2 v1[P2], v2[P2];
                const uint32_t row = vst + (uint32_t)(kk * D * EB);
                lds_pairs<T, VW>(row + d0 * EB, v1);
                lds_pairs<T, VW>(row + (HALF + d0) * EB, v2);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float pu = ex2(lg[u][g] - m[g]);
                    l[g] += pu;
                    const float2 p2 = make_float2(pu, pu);
#pragma unroll
                    for (int i2 = 0; i2 < P2; ++i2) {
                        o1[g][i2] = __ffma2_rn(p2, v1[i2], o1[g][i2]);
                        o2[g][i2] = __ffma2_rn(p2, v2[i2], o2[g][i2]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        if (LOADER && i + NS < n_tiles) {
            // every warp has released stage s: refill it with tile i + NS (a warp that gave up
            // on this stage set the abort flag before it released it, so the refill never lands
            // on a load still in flight); lane 0 waits, the loader issues
            int go = 0;
            if (lane == 0 && *sm_abort == 0) {
                if (!mbar_wait_abortable(bar_empty + 8 * s, (i / NS) & 1, p.spin_limit,
                                         sm_abort)) {
                    record_code(p.dev_code, kDevCodeTimeout);
                    *sm_abort = 1;
                } else {
                    go = *sm_abort == 0;
                }
            }
            if (WARP_ISSUE) go = __shfl_sync(0xffffffffu, go, 0);
            if (go) issue_tile(i + NS);
        }
    }
    if (cur >= 0) finish_pair(cur);
    // after an abort the last NS tiles issued (one per stage) may still be landing: wait for
    // them, bounded, before the block's shared memory is released
    if (threadIdx.x == 0 && *sm_abort != 0)
        for (int i = max(0, last_issued - NS + 1); i <= last_issued; ++i)
            mbar_wait_ok(bar_full + 8 * (i % NS), (i / NS) & 1, p.spin_limit);
}

// Elements per lane-half by (type, group size): keeps q and o (4*G*VW floats) in registers.
template <typename T, int G>
constexpr int decode_vw()
{
    if constexpr (sizeof(T) == 4) return 4;
    else return G <= 2 ? 8 : 4;
}
constexpr int kDecodeUnroll = 2;

template <typename T, int D, int G, int RM>
cudaError_t launch_decode_rm(const DecodeParams &p, cudaStream_t stream)
{
    constexpr int VW = decode_vw<T, G>();
    using SM = DecodeSmem<T, D, G, RM>;
    auto kern = decode_attn_kernel<T, D, G, VW, kDecodeUnroll, RM, SM::CPS>;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SM::kBytes);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    DecodeParams q = p;
    if (q.spin_limit == 0) q.spin_limit = kMbarSpinLimit;
    q.NT = p.cap > 0 ? (p.cap + SM::TK - 1) / SM::TK : 1;
    if (q.NT < 1) q.NT = 1;
    long long T_all = (long long)q.P * q.NT;
    if constexpr (RM == 5) {
        // retrieval tiles split evenly; at least as many blocks as streaming pairs would use
        q.NT2 = p.ring_cap > 0 ? (p.ring_cap + SM::TK - 1) / SM::TK : 1;
        const long long t_ret = (long long)p.B * p.n_ret * q.NT;
        const long long p_str = (long long)p.B * p.n_str;
        T_all = t_ret > p_str ? t_ret : p_str;
    }
    const long long max_ctas = (long long)p.n_sm * SM::CPS;
    const int C = (int)(T_all < max_ctas ? T_all : max_ctas);
    return launch_pdl(kern, dim3((unsigned)C), dim3(kDecodeThreads), (size_t)SM::kBytes, stream, q);
}

// Position handling of an instantiation unit.
constexpr int kDecodePlain = 0;   // valid slots 0 .. len-1, no positional term
constexpr int kDecodeRope = 1;    // StreamingLLM layout, RoPE at in-cache positions
constexpr int kDecodeAlibi = 2;   // StreamingLLM layout, ALiBi at in-cache positions
constexpr int kDecodePaged = 3;   // page-table cache, no positional term
constexpr int kDecodeDuo = 4;     // DuoAttention: full and ring caches in one launch

// RoPE with one query head per KV head takes the factored rotation when the table covers the
// per-lane offsets 0 .. TK-1; otherwise each key reads its table row.
template <typename T, int D, int G, int MODE>
cudaError_t launch_decode_typed(const DecodeParams &p, cudaStream_t stream)
{
    if constexpr (MODE == kDecodePlain) {
        return launch_decode_rm<T, D, G, 0>(p, stream);
    } else if constexpr (MODE == kDecodeAlibi) {
        return launch_decode_rm<T, D, G, 3>(p, stream);
    } else if constexpr (MODE == kDecodePaged) {
        return launch_decode_rm<T, D, G, 4>(p, stream);
    } else if constexpr (MODE == kDecodeDuo) {
        return launch_decode_rm<T, D, G, 5>(p, stream);
    } else if constexpr (G == 1) {
        if (p.n_pos >= DecodeSmem<T, D, G, 2>::TK) return launch_decode_rm<T, D, G, 2>(p, stream);
        return launch_decode_rm<T, D, G, 1>(p, stream);
    } else {
        return launch_decode_rm<T, D, G, 1>(p, stream);
    }
}

template <typename T, int MODE>
cudaError_t launch_decode_variant(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
#define KVC_DECODE_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_decode_typed<T, DD, GG, MODE>(p, stream);
#define KVC_DECODE_D(DD) \
    KVC_DECODE_CASE(DD, 1) KVC_DECODE_CASE(DD, 2) KVC_DECODE_CASE(DD, 4) \
    KVC_DECODE_CASE(DD, 6) KVC_DECODE_CASE(DD, 8)
    KVC_DECODE_D(64)
    KVC_DECODE_D(128)
    KVC_DECODE_D(256)
#undef KVC_DECODE_D
#undef KVC_DECODE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvc
