// append_gather.cu -- row movers: append one token per (batch, KV head), gather retained rows
// into a compacted cache, advance the device decode position.
//
// Both movers are HBM copies with 16-byte vectors.  A row (d_head elements) is handled by one
// group of lanes inside a single warp, so per-row bookkeeping (reading a length, then bumping
// it) is ordered by __syncwarp alone.
#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

// Row of `vpr` 16-byte vectors copied by `lpr` lanes (vpr / lpr vectors each).
struct RowMap {
    int lpr;   // lanes per row
    int rpw;   // rows per warp
    int vpl;   // vectors per lane
};

__host__ __device__ inline RowMap row_map(int row_bytes)
{
    const int vpr = row_bytes / 16;
    RowMap m;
    m.lpr = vpr < 32 ? vpr : 32;
    m.rpw = 32 / m.lpr;
    m.vpl = vpr / m.lpr;
    return m;
}

// ---------------------------------------------------------------------------------------------
// Append.  Slot by policy: TAIL = len (then len + 1), RING = sink + ring layout of the text
// position t ("Attention Sinks e o StreamingLLM...": 4 fixed sinks plus a circular window),
// FREE_SLOT = the slot H2O freed at the previous step.
__global__ void append_kernel(const AppendParams p, int row_bytes)
{
    const RowMap rm = row_map(row_bytes);
    const int warp_g = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int row = warp_g * rm.rpw + lane / rm.lpr;
    const int li = lane % rm.lpr;
    const bool active = row < p.B * p.H;
    const int b = active ? row / p.H : 0, h = active ? row % p.H : 0;
    pdl_trigger();
    pdl_wait();                                 // lengths, slots and t may come from the previous kernel

    int64_t t = p.t != nullptr ? *p.t : 0;
    int slot = -1;
    if (active) {
        if (p.policy == 0) {
            const int len = p.len[row];
            if (len < 0 || len >= p.cap) {
                if (li == 0) record_code(p.dev_code, len < 0 ? 5 : 1);
            } else {
                slot = len;
            }
        } else if (p.policy == 1) {
            if (t < 0) {
                if (li == 0) record_code(p.dev_code, 4);
            } else {
                slot = t < p.S ? (int)t : p.S + (int)((t - p.S) % (int64_t)(p.W + 1));
            }
        } else {
            const int fs = p.free_slot[row];
            if (fs < 0 || fs >= p.cap) {
                if (li == 0) record_code(p.dev_code, 2);
            } else {
                slot = fs;
            }
        }
    }
    __syncwarp();   // every lane has read len / free_slot before any lane writes
    if (slot < 0) return;

    const size_t dst = ((size_t)b * p.sb + (size_t)h * p.sh + (size_t)slot * p.ss) *
                       (size_t)(row_bytes / p.D);
    const size_t src = (size_t)row * row_bytes;
    const char *kn = static_cast<const char *>(p.k_new) + src;
    const char *vn = static_cast<const char *>(p.v_new) + src;
    char *kd = static_cast<char *>(p.k) + dst;
    char *vd = static_cast<char *>(p.v) + dst;
    for (int i = 0; i < rm.vpl; ++i) {
        const int off = (i * rm.lpr + li) * 16;
        *reinterpret_cast<uint4 *>(kd + off) = *reinterpret_cast<const uint4 *>(kn + off);
        *reinterpret_cast<uint4 *>(vd + off) = *reinterpret_cast<const uint4 *>(vn + off);
    }
    if (li == 0) {
        if (p.pos != nullptr) p.pos[(size_t)row * p.pos_stride + slot] = (int32_t)t;
        if (p.score != nullptr) p.score[(size_t)row * p.score_stride + slot] = 0.f;
        if (p.policy == 0) p.len[row] = slot + 1;
    }
}

// ---------------------------------------------------------------------------------------------
// Gather: dst row j of (b, h) <- src row idx[b, h, j]; bit-exact copies.
__global__ void gather_kernel(const GatherParams p, int row_bytes)
{
    const RowMap rm = row_map(row_bytes);
    const int warp_g = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long row = (long long)warp_g * rm.rpw + lane / rm.lpr;   // (b*H + h)*n_keep + j
    const int li = lane % rm.lpr;
    const long long rows = (long long)p.B * p.H * p.n_keep;
    if (row >= rows) return;
    const int bh = (int)(row / p.n_keep);
    const int j = (int)(row % p.n_keep);
    const int b = bh / p.H, h = bh % p.H;
    const int src_slot = p.idx[(size_t)bh * p.idx_stride + j];
    if (src_slot < 0 || src_slot >= p.s_cap) {
        if (li == 0) record_code(p.dev_code, 3);
        return;
    }
    const int eb = row_bytes / p.D;
    const size_t s_off = ((size_t)b * p.s_sb + (size_t)h * p.s_sh + (size_t)src_slot * p.s_ss) * eb;
    const size_t d_off = ((size_t)b * p.d_sb + (size_t)h * p.d_sh + (size_t)j * p.d_ss) * eb;
    const char *sk = static_cast<const char *>(p.sk) + s_off;
    const char *sv = static_cast<const char *>(p.sv) + s_off;
    char *dk = static_cast<char *>(p.dk) + d_off;
    char *dv = static_cast<char *>(p.dv) + d_off;
    for (int i = 0; i < rm.vpl; ++i) {
        const int off = (i * rm.lpr + li) * 16;
        const uint4 kx = ld_stream_16(sk + off);
        const uint4 vx = ld_stream_16(sv + off);
        *reinterpret_cast<uint4 *>(dk + off) = kx;
        *reinterpret_cast<uint4 *>(dv + off) = vx;
    }
    if (li == 0) {
        if (p.pos_dst != nullptr) p.pos_dst[(size_t)bh * p.pos_stride + j] = src_slot;
        if (p.len_dst != nullptr && j == 0) p.len_dst[bh] = p.n_keep;
    }
}

__global__ void position_advance_kernel(int64_t *t, int64_t delta)
{
    pdl_trigger();
    pdl_wait();
    *t += delta;
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, int elem_bytes, cudaStream_t stream)
{
    const int row_bytes = p.D * elem_bytes;
    const RowMap rm = row_map(row_bytes);
    const int rows = p.B * p.H;
    const int warps = (rows + rm.rpw - 1) / rm.rpw;
    const int threads = 256;
    const int blocks = (warps * 32 + threads - 1) / threads;
    return launch_pdl(append_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, p, row_bytes);
}

cudaError_t launch_gather(const GatherParams &p, int elem_bytes, cudaStream_t stream)
{
    const int row_bytes = p.D * elem_bytes;
    const RowMap rm = row_map(row_bytes);
    const long long rows = (long long)p.B * p.H * p.n_keep;
    if (rows == 0) return cudaSuccess;
    const long long warps = (rows + rm.rpw - 1) / rm.rpw;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    gather_kernel<<<(unsigned)blocks, threads, 0, stream>>>(p, row_bytes);
    return cudaGetLastError();
}

cudaError_t launch_position_advance(int64_t *t, int64_t delta, cudaStream_t stream)
{
    return launch_pdl(position_advance_kernel, dim3(1), dim3(1), 0, stream, t, delta);
}

}  // namespace kvc
