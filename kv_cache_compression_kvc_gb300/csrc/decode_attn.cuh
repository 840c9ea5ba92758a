// decode_attn.cuh -- decode attention over the retained slots of a KV cache.
//
// What it computes ("O KV cache", llmdeepdive 7.2, "01 · Conceito"): the new token's query
// attends to every cached key of its KV head and mixes the cached values -- exact causal
// attention.  Where the time goes ("Compressão e Poda Dinâmica de KV Cache", "O gargalo de
// memória do KV Cache..."): every emitted token reads the whole cache from HBM in a GEMV at
// 1-2 FLOP per byte, so this kernel is an HBM stream.  How it is parallelised ("Implementação
// prática em vLLM e SGLang": FlashDecoding splits the work along the time axis): the slots of
// each (batch, KV head) are cut into n_splits contiguous chunks, one thread block each; each
// block keeps an online softmax state (max m, sum l, weighted values o) for all G query heads
// of the group, and the last block to finish a KV head (atomic ticket, nobody waits) merges
// the chunk states by log-sum-exp.
//
// Lane layout.  A key row of D elements is read by LPK = D/(2*VW) lanes; lane lk holds the VW
// elements starting at lk*VW in the first half of the row and the VW elements at the same
// offset in the second half, so the two members of every RoPE pair (i, i + D/2) sit in one
// lane and rotating keys needs no shuffle.  32/LPK keys are in flight per warp step, UNR steps
// are loaded before any arithmetic (K and V together) to keep enough bytes in flight.
// Arithmetic is fp32; q is pre-scaled by scale*log2(e) so the softmax uses exp2.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace kvc {

template <typename T, int D, int G, int VW, int NW, int UNR>
__global__ void __launch_bounds__(NW * 32)
decode_attn_kernel(const DecodeParams p)
{
    constexpr int HALF = D / 2;
    constexpr int LPK = HALF / VW;
    static_assert(LPK >= 1 && LPK <= 32 && (32 % LPK) == 0, "lane layout");
    constexpr int KPW = 32 / LPK;
    constexpr int E = 2 * VW;

    const int split = blockIdx.x;
    const int kh = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int lk = lane % LPK;
    const int ks = lane / LPK;
    const int d0 = lk * VW;
    const int bkh = b * p.Hkv + kh;

    // ---- valid slots ----------------------------------------------------------------------
    int n_slots;
    int64_t t = 0;
    int qpos = 0, ring_base = 0;
    if (p.rope) {
        t = *p.t;
        if (t < 0) {
            record_code(p.dev_code, 4 /* KVC_DEV_BAD_POSITION */);
            t = 0;
        }
        n_slots = p.S + p.W + 1;
        const int64_t sw = (int64_t)p.S + p.W;
        qpos = (int)(t < sw ? t : sw);
        if (t >= p.S) ring_base = (int)((t - p.S) % (int64_t)(p.W + 1));
    } else if (p.len != nullptr) {
        n_slots = p.len[bkh];
        if (n_slots < 0 || n_slots > p.cap) {
            if (split == 0 && threadIdx.x == 0) record_code(p.dev_code, 5 /* BAD_LENGTH */);
            n_slots = n_slots < 0 ? 0 : p.cap;
        }
    } else {
        n_slots = p.n_valid;
    }
    const int s_begin = split * p.chunk;
    const int s_end = min(s_begin + p.chunk, n_slots);

    // ---- query: G heads, this lane's 2*VW dims, rotated and pre-scaled --------------------
    float qf[G][E];
    {
        const T *qb = static_cast<const T *>(p.q) + ((size_t)b * p.Hq + (size_t)kh * G) * D;
        float cs[2 * VW];
        if (p.rope) {
            const float *row = p.cos_sin + ((size_t)qpos * HALF + d0) * 2;
#pragma unroll
            for (int i = 0; i < 2 * VW; ++i) cs[i] = row[i];
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            load_cached<T, VW>(qb + (size_t)g * D + d0, &qf[g][0]);
            load_cached<T, VW>(qb + (size_t)g * D + HALF + d0, &qf[g][VW]);
            if (p.rope) {
#pragma unroll
                for (int i = 0; i < VW; ++i) {
                    const float x1 = qf[g][i], x2 = qf[g][VW + i];
                    const float c = cs[2 * i], s = cs[2 * i + 1];
                    qf[g][i] = x1 * c - x2 * s;
                    qf[g][VW + i] = x1 * s + x2 * c;
                }
            }
#pragma unroll
            for (int e = 0; e < E; ++e) qf[g][e] *= p.scale_log2;
        }
    }

    float m[G], l[G], o[G][E];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = kNegBig;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[g][e] = 0.f;
    }

    const T *kb = static_cast<const T *>(p.k) + (size_t)b * p.sb + (size_t)kh * p.sh;
    const T *vb = static_cast<const T *>(p.v) + (size_t)b * p.sb + (size_t)kh * p.sh;
    float *lg_out = p.logits ? p.logits + (size_t)(b * p.Hq + kh * G) * p.logits_stride : nullptr;

    constexpr int STEP = KPW * UNR;
    for (int blk = s_begin + warp * STEP; blk < s_end; blk += NW * STEP) {
        RawVec<T, VW> kr[UNR][2], vr[UNR][2];
        bool valid[UNR];
        int kpos[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int j = blk + u * KPW + ks;
            bool ok = j < s_end;
            int pj = j;
            if (p.rope && ok) {
                if (j < p.S) {
                    ok = j <= t;
                } else {
                    int dd = ring_base - (j - p.S);
                    if (dd < 0) dd += p.W + 1;
                    ok = (t >= p.S) && ((int64_t)dd <= t - p.S);
                    pj = qpos - dd;
                }
            }
            valid[u] = ok;
            kpos[u] = pj;
            if (ok) {
                const size_t row = (size_t)j * p.ss;
                kr[u][0].load(kb + row + d0);
                kr[u][1].load(kb + row + HALF + d0);
                vr[u][0].load(vb + row + d0);
                vr[u][1].load(vb + row + HALF + d0);
            } else {
                kr[u][0].zero(); kr[u][1].zero();
                vr[u][0].zero(); vr[u][1].zero();
            }
        }

        float lg[UNR][G];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            float kf[E];
            kr[u][0].to_float(&kf[0]);
            kr[u][1].to_float(&kf[VW]);
            if (p.rope && valid[u]) {
                const float *row = p.cos_sin + ((size_t)kpos[u] * HALF + d0) * 2;
#pragma unroll
                for (int i = 0; i < VW; i += 2) {
                    const float4 cs = *reinterpret_cast<const float4 *>(row + 2 * i);
                    const float a0 = kf[i], b0 = kf[VW + i];
                    const float a1 = kf[i + 1], b1 = kf[VW + i + 1];
                    kf[i] = a0 * cs.x - b0 * cs.y;
                    kf[VW + i] = a0 * cs.y + b0 * cs.x;
                    kf[i + 1] = a1 * cs.z - b1 * cs.w;
                    kf[VW + i + 1] = a1 * cs.w + b1 * cs.z;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) acc = fmaf(qf[g][e], kf[e], acc);
                lg[u][g] = acc;
            }
        }
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) {
#pragma unroll
            for (int u = 0; u < UNR; ++u)
#pragma unroll
                for (int g = 0; g < G; ++g)
                    lg[u][g] += __shfl_xor_sync(0xffffffffu, lg[u][g], off);
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            if (!valid[u]) {
#pragma unroll
                for (int g = 0; g < G; ++g) lg[u][g] = -INFINITY;
            } else if (lg_out != nullptr && lk == 0) {
                const int j = blk + u * KPW + ks;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    lg_out[(size_t)g * p.logits_stride + j] = lg[u][g] * kLn2;
            }
        }

#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = lg[0][g];
#pragma unroll
            for (int u = 1; u < UNR; ++u) mx = fmaxf(mx, lg[u][g]);
            const float m_new = fmaxf(m[g], mx);
            const float corr = exp2f(m[g] - m_new);
            l[g] *= corr;
#pragma unroll
            for (int e = 0; e < E; ++e) o[g][e] *= corr;
            m[g] = m_new;
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            float vf[E];
            vr[u][0].to_float(&vf[0]);
            vr[u][1].to_float(&vf[VW]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pu = exp2f(lg[u][g] - m[g]);
                l[g] += pu;
#pragma unroll
                for (int e = 0; e < E; ++e) o[g][e] = fmaf(pu, vf[e], o[g][e]);
            }
        }
    }

    // ---- merge the KPW lane groups of the warp --------------------------------------------
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float m_o = __shfl_xor_sync(0xffffffffu, m[g], off);
            const float l_o = __shfl_xor_sync(0xffffffffu, l[g], off);
            const float m_n = fmaxf(m[g], m_o);
            const float c1 = exp2f(m[g] - m_n), c2 = exp2f(m_o - m_n);
            l[g] = l[g] * c1 + l_o * c2;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o_o = __shfl_xor_sync(0xffffffffu, o[g][e], off);
                o[g][e] = o[g][e] * c1 + o_o * c2;
            }
            m[g] = m_n;
        }
    }

    // ---- merge the warps of the block ------------------------------------------------------
    __shared__ float sm_m[NW][G], sm_l[NW][G];
    __shared__ float sm_o[NW][G][D];
    __shared__ int sm_last;
    if (ks == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int i = 0; i < VW; ++i) {
                sm_o[warp][g][d0 + i] = o[g][i];
                sm_o[warp][g][HALF + d0 + i] = o[g][VW + i];
            }
            if (lk == 0) {
                sm_m[warp][g] = m[g];
                sm_l[warp][g] = l[g];
            }
        }
    }
    __syncthreads();

    const int rows0 = b * p.Hq + kh * G;   // first query row of this KV head
    for (int i = threadIdx.x; i < G * D; i += NW * 32) {
        const int g = i / D, d = i % D;
        float M = sm_m[0][g];
#pragma unroll
        for (int w = 1; w < NW; ++w) M = fmaxf(M, sm_m[w][g]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float c = exp2f(sm_m[w][g] - M);
            L += sm_l[w][g] * c;
            O += sm_o[w][g][d] * c;
        }
        if (p.n_splits == 1) {
            p.out[(size_t)(rows0 + g) * D + d] = L > 0.f ? O / L : 0.f;
            if (d == 0 && p.lse != nullptr)
                p.lse[rows0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        } else {
            const size_t slot = (size_t)(rows0 + g) * p.n_splits + split;
            p.ws_o[slot * D + d] = O;
            if (d == 0) {
                p.ws_ml[slot * 2] = M;
                p.ws_ml[slot * 2 + 1] = L;
            }
        }
    }
    if (p.n_splits == 1) return;

    // ---- last block of this KV head merges the n_splits partial states ---------------------
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) sm_last = (atomicAdd(&p.ws_cnt[bkh], 1) == p.n_splits - 1);
    __syncthreads();
    if (!sm_last) return;
    __threadfence();

    for (int i = threadIdx.x; i < G * D; i += NW * 32) {
        const int g = i / D, d = i % D;
        const size_t base = (size_t)(rows0 + g) * p.n_splits;
        float M = kNegBig;
        for (int s = 0; s < p.n_splits; ++s) M = fmaxf(M, __ldcg(&p.ws_ml[(base + s) * 2]));
        float L = 0.f, O = 0.f;
        for (int s = 0; s < p.n_splits; ++s) {
            const float c = exp2f(__ldcg(&p.ws_ml[(base + s) * 2]) - M);
            L += __ldcg(&p.ws_ml[(base + s) * 2 + 1]) * c;
            O += __ldcg(&p.ws_o[(base + s) * D + d]) * c;
        }
        p.out[(size_t)(rows0 + g) * D + d] = L > 0.f ? O / L : 0.f;
        if (d == 0 && p.lse != nullptr)
            p.lse[rows0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    if (threadIdx.x == 0) p.ws_cnt[bkh] = 0;   // leave the ticket zeroed for the next call
}

// Elements per lane-half by (type, group size): keeps q and o (2*G*2*VW floats) in registers.
template <typename T, int G>
constexpr int decode_vw()
{
    if constexpr (sizeof(T) == 4) return 4;
    else return G <= 2 ? 8 : 4;
}

constexpr int kDecodeWarps = 4;
constexpr int kDecodeUnroll = 4;

template <typename T, int D, int G>
cudaError_t launch_decode_typed(const DecodeParams &p, cudaStream_t stream)
{
    constexpr int VW = decode_vw<T, G>();
    dim3 grid(p.n_splits, p.Hkv, p.B);
    decode_attn_kernel<T, D, G, VW, kDecodeWarps, kDecodeUnroll>
        <<<grid, kDecodeWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode_dtype(const DecodeParams &p, int D, int G, cudaStream_t stream)
{
#define KVC_DECODE_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_decode_typed<T, DD, GG>(p, stream);
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
