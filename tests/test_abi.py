"""The C ABI library builds, loads and exports every symbol include/kvc.h declares; its host-only
entry points agree with the oracle; argument validation rejects bad calls before any launch.
No GPU needed: nothing here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_kvc_gb300 import build, kvc as k
    build.build()
    k.load()
    return k


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for n in ("kvc_snapkv_select", "kvc_compact_gather", "kvc_stream_append",
              "kvc_h2o_accumulate_evict", "kvc_decode_attn"):
        assert n in names


def test_library_exports_every_declared_symbol(kvc):
    lib = ctypes.CDLL(kvc.library_path())
    missing = [n for n in _declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
    # the binding declares a signature for each of them, no more, no less
    assert sorted(kvc.SIGNATURES) == _declared_symbols()


def test_kv_bytes_matches_oracle(kvc):
    for args in [(64, 4, 256, 262144, 2, 1), (16, 4, 256, 262144, 2, 1), (32, 32, 128, 2049, 2, 16),
                 (1, 1, 64, 1, 4, 1)]:
        assert kvc.kvc_kv_bytes(*args) == oracle.kv_bytes(*args)


@pytest.mark.parametrize("n_layers,target,num,den", [(16, 8192, 4, 1), (32, 5243, 4, 1),
                                                     (3, 1, 3, 1), (7, 1001, 1, 4), (1, 9, 4, 1),
                                                     (40, 123457, 7, 3)])
def test_pyramid_budgets_match_oracle(kvc, n_layers, target, num, den):
    assert kvc.kvc_pyramid_budgets(n_layers, target, num, den) == \
        [int(x) for x in oracle.pyramid_budgets(n_layers, target, num, den)]


def test_rope_table_matches_oracle_rotation(kvc):
    D, n = 128, 300
    tab = kvc.kvc_rope_table(n, D, 10000.0).numpy().astype(np.float64)
    rng = np.random.default_rng(3)
    x = rng.standard_normal(D)
    for p in (0, 1, 17, 299):
        c, s = tab[p, 0], tab[p, 1]
        y = np.concatenate([x[:D // 2] * c - x[D // 2:] * s, x[:D // 2] * s + x[D // 2:] * c])
        assert np.max(np.abs(y - oracle.rope(x, p))) < 1e-5   # fp32 table entries


def test_validation_rejects_bad_calls_before_launch(kvc):
    lib = kvc.load()
    c = kvc.kvc_cache()
    c.k = c.v = 4096
    c.dtype, c.batch, c.n_heads_kv, c.cap, c.d_head = kvc.KVC_BF16, 1, 1, 16, 96
    c.stride_b, c.stride_h, c.stride_slot = 16 * 96, 16 * 96, 96
    st = lib.kvc_decode_attn(4096, 1, ctypes.byref(c), None, 4, None, 1.0, 4096, None, 0, None,
                             None, 0, None)
    assert st == 2 and "d_head" in kvc.kvc_last_error()           # KVC_ERR_SHAPE
    c.d_head, c.stride_slot = 128, 128
    st = lib.kvc_decode_attn(4096, 3, ctypes.byref(c), None, 4, None, 1.0, 4096, None, 0, None,
                             None, 0, None)
    assert st == 2                                                 # group size 3 unsupported
    c.k = 4100
    st = lib.kvc_decode_attn(4096, 1, ctypes.byref(c), None, 4, None, 1.0, 4096, None, 0, None,
                             None, 0, None)
    assert st == 3                                                 # KVC_ERR_ALIGN
    c.k = 4096
    st = lib.kvc_decode_attn(4096, 1, ctypes.byref(c), None, 17, None, 1.0, 4096, None, 0, None,
                             None, 0, None)
    assert st == 4                                                 # n_valid > cap
    st = lib.kvc_decode_attn_ex(4096, 1, ctypes.byref(c), None, 4, None, 1.0, 4096, None, 0,
                                None, None, 0, 4, None)
    assert st == 1 and "flags" in kvc.kvc_last_error()            # unknown flag bit
    st = lib.kvc_stream_append(ctypes.byref(c), 7, 4096, 4096, None, None, 0, 0, None, None, 0,
                               None, 0, None)
    assert st == 1                                                 # bad policy
    st = lib.kvc_stream_append(ctypes.byref(c), kvc.KVC_APPEND_RING, 4096, 4096, 4096, None, 4,
                               20, None, None, 0, None, 0, None)
    assert st == 4                                                 # ring does not fit cap 16
    st = lib.kvc_snapkv_select(4096, ctypes.byref(c), 1, 16, 8, 4, 20, 1.0, 4096, None, None, 0,
                               None)
    assert st == 1                                                 # even pool kernel
    st = lib.kvc_snapkv_select(4096, ctypes.byref(c), 1, 16, 8, 5, 7, 1.0, 4096, None, None, 0,
                               None)
    assert st == 4                                                 # budget < L_obs
    d = kvc.kvc_cache.from_buffer_copy(c)
    st = lib.kvc_compact_gather(ctypes.byref(c), 4096, 8, 8, ctypes.byref(d), None, 0, None, None)
    assert st == 1                                                 # in place is refused
    assert lib.kvc_pyramid_budgets(0, 10, 4, 1, None) == 1
    assert kvc.kvc_last_error() != ""


def test_alibi_slopes_geometric_sequence(kvc):
    """Eight heads: 1/2, 1/4, ..., 1/256 (the ALiBi paper's example); sixteen heads interleave
    the square roots; a head count that is not a power of two is refused."""
    assert kvc.kvc_alibi_slopes(8).tolist() == [2.0 ** -(h + 1) for h in range(8)]
    s16 = kvc.kvc_alibi_slopes(16).double().numpy()
    assert np.allclose(s16, [2.0 ** (-(h + 1) / 2) for h in range(16)], rtol=1e-7, atol=0)
    assert np.allclose(s16[1::2], [2.0 ** -(h + 1) for h in range(8)], rtol=0, atol=0)
    with pytest.raises(kvc.KvcError):
        kvc.kvc_alibi_slopes(6)


def test_alibi_validation_before_launch(kvc):
    lib = kvc.load()
    c = kvc.kvc_cache()
    c.k = c.v = 4096
    c.dtype, c.batch, c.n_heads_kv, c.cap, c.d_head = kvc.KVC_BF16, 1, 1, 16, 128
    c.stride_b, c.stride_h, c.stride_slot = 16 * 128, 16 * 128, 128
    st = lib.kvc_decode_attn_alibi(4096, 1, ctypes.byref(c), None, 1.0, 4096, None, 0, None,
                                   None, 0, 0, None)
    assert st == 1 and "alibi" in kvc.kvc_last_error()            # no descriptor
    a = kvc.kvc_alibi()
    a.n_sink, a.window, a.t, a.slopes = 4, 20, 4096, 4096
    st = lib.kvc_decode_attn_alibi(4096, 1, ctypes.byref(c), ctypes.byref(a), 1.0, 4096, None,
                                   0, None, None, 0, 0, None)
    assert st == 4                                                 # ring does not fit cap 16
    a.window, a.slopes = 3, None
    st = lib.kvc_decode_attn_alibi(4096, 1, ctypes.byref(c), ctypes.byref(a), 1.0, 4096, None,
                                   0, None, None, 0, 0, None)
    assert st == 1                                                 # no slopes


def test_paged_validation_before_launch(kvc):
    lib = kvc.load()
    pool = kvc.kvc_block_pool()
    pool.k = pool.v = 4096
    pool.dtype, pool.n_blocks, pool.n_heads_kv, pool.block_size, pool.d_head = \
        kvc.KVC_BF16, 8, 2, 16, 96
    pt = kvc.kvc_page_table()
    pt.table = pt.n_blocks = pt.len = pt.score = 4096
    pt.batch, pt.max_blocks = 2, 4
    fp = kvc.kvc_free_pool()
    fp.ids, fp.top, fp.capacity = 4096, 4096, 8
    B = ctypes.byref
    st = lib.kvc_decode_attn_paged(4096, 2, B(pool), B(pt), 1.0, 4096, None, 0, None, None, 0,
                                   0, None)
    assert st == 2 and "d_head" in kvc.kvc_last_error()           # KVC_ERR_SHAPE
    pool.d_head = 128
    pt.table = None
    st = lib.kvc_paged_append(B(pool), B(pt), B(fp), 4096, 4096, None, None, None)
    assert st == 1                                                 # null page-table array
    pt.table = 4096
    fp.capacity = 0
    st = lib.kvc_paged_append(B(pool), B(pt), B(fp), 4096, 4096, None, None, None)
    assert st == 1                                                 # empty free-pool descriptor
    fp.capacity = 8
    st = lib.kvc_block_accumulate_evict(4096, 64, 4096, 4, 16, B(pt), B(fp), 3, 0, None, None)
    assert st == 1 and "recent_blocks" in kvc.kvc_last_error()    # recent quota of 0 blocks
    st = lib.kvc_block_accumulate_evict(4096, 63, 4096, 4, 16, B(pt), B(fp), 3, 1, None, None)
    assert st == 4                                                 # logits_stride < 4 * 16
    st = lib.kvc_decode_attn_paged(4096, 2, B(pool), B(pt), 1.0, 4096, 4096, 32, None, None, 0,
                                   0, None)
    assert st == 4                                                 # logits_stride < cap 64


def test_duo_kv_bytes_matches_oracle(kvc):
    for args in [(32, 3, 7, 128, 131072, 4, 64, 2, 1), (1, 1, 1, 64, 10, 4, 64, 4, 2),
                 (16, 8, 24, 256, 4096, 4, 64, 2, 8)]:
        assert kvc.kvc_duo_kv_bytes(*args) == oracle.duo_kv_bytes(*args)


def test_duo_validation_before_launch(kvc):
    lib = kvc.load()
    full, ring = kvc.kvc_cache(), kvc.kvc_cache()
    for c, h, cap in ((full, 2, 64), (ring, 6, 69)):
        c.k = c.v = 4096
        c.dtype, c.batch, c.n_heads_kv, c.cap, c.d_head = kvc.KVC_BF16, 1, h, cap, 128
        c.stride_b, c.stride_h, c.stride_slot = h * cap * 128, cap * 128, 128
    duo = kvc.Duo([1, 5], 4, 64, torch.zeros(1, dtype=torch.int64))
    B = ctypes.byref
    st = lib.kvc_decode_attn_duo(4096, 6, B(full), None, 10, B(ring), B(duo.desc), 1.0, 4096,
                                 None, 0, None, None, 0, 0, None)
    assert st == 2                                                 # 6 query heads over 8 KV heads
    bad = kvc.Duo([5, 1], 4, 64, torch.zeros(1, dtype=torch.int64))
    st = lib.kvc_decode_attn_duo(4096, 8, B(full), None, 10, B(ring), B(bad.desc), 1.0, 4096,
                                 None, 0, None, None, 0, 0, None)
    assert st == 1 and "ascending" in kvc.kvc_last_error()
    three = kvc.Duo([0, 1, 2], 4, 64, torch.zeros(1, dtype=torch.int64))
    st = lib.kvc_duo_append(B(full), 4096, B(ring), B(three.desc), 4096, 4096, None)
    assert st == 2                                                 # full cache holds 2 heads
    ring.cap = 68
    st = lib.kvc_duo_append(B(full), 4096, B(ring), B(duo.desc), 4096, 4096, None)
    assert st == 4                                                 # ring < 4 + 64 + 1 slots


def test_block_prompt_select_validation_before_launch(kvc):
    lib = kvc.load()
    B = ctypes.byref
    pool = kvc.kvc_block_pool()
    pool.k = pool.v = 4096
    pool.dtype, pool.n_blocks, pool.n_heads_kv, pool.block_size, pool.d_head = \
        kvc.KVC_BF16, 32, 2, 16, 128
    pt = kvc.kvc_page_table()
    pt.table = pt.n_blocks = pt.len = pt.score = 4096
    pt.batch, pt.max_blocks = 1, 8
    fp = kvc.kvc_free_pool()
    fp.ids, fp.top, fp.capacity = 4096, 4096, 32
    pr = kvc.kvc_cache()
    pr.k = pr.v = 4096
    pr.dtype, pr.batch, pr.n_heads_kv, pr.cap, pr.d_head = kvc.KVC_BF16, 1, 2, 100, 128
    pr.stride_b, pr.stride_h, pr.stride_slot = 2 * 100 * 128, 100 * 128, 128
    st = lib.kvc_block_prompt_select(4096, 100, B(pr), 100, B(pool), B(pt), B(fp), 4, 0, 4096,
                                     1 << 20, None)
    assert st == 1 and "recent_blocks" in kvc.kvc_last_error()    # recent quota of 0 blocks
    st = lib.kvc_block_prompt_select(4096, 100, B(pr), 100, B(pool), B(pt), B(fp), 9, 1, 4096,
                                     1 << 20, None)
    assert st == 1                                                 # budget beyond max_blocks
    st = lib.kvc_block_prompt_select(4096, 100, B(pr), 101, B(pool), B(pt), B(fp), 4, 1, 4096,
                                     1 << 20, None)
    assert st == 4                                                 # seq_len beyond the prompt
    st = lib.kvc_block_prompt_select(4096, 50, B(pr), 100, B(pool), B(pt), B(fp), 4, 1, 4096,
                                     1 << 20, None)
    assert st == 4                                                 # score rows too short
    pr.n_heads_kv, pr.stride_b = 3, 3 * 100 * 128
    st = lib.kvc_block_prompt_select(4096, 100, B(pr), 100, B(pool), B(pt), B(fp), 4, 1, 4096,
                                     1 << 20, None)
    assert st == 2                                                 # prompt heads != pool heads
    assert lib.kvc_block_prompt_select_workspace_bytes(1, 100, 16, 4) == 256 + 256


def test_workspace_queries_of_the_added_entry_points(kvc):
    """Host sizing: the DuoAttention decode allows more blocks per retrieval pair than the
    plain decode of the same shape; the grouped H2O prompt selection holds one group member's
    queries and two score arrays beside the one-head scoring state; bad arguments give 0."""
    plain = kvc.kvc_decode_attn_workspace_bytes(1, 32, 32, 128, 131080)
    duo = kvc.kvc_decode_attn_duo_workspace_bytes(1, 32, 32, 128, 131080, 8)
    assert duo > plain > 0
    B, Hkv, D, N = 16, 8, 128, 4096
    gqa = kvc.kvc_h2o_prefill_gqa_workspace_bytes(B, Hkv, D, N, kvc.KVC_BF16)
    assert gqa >= B * Hkv * N * D * 2 + 2 * B * Hkv * N * 4
    assert kvc.kvc_h2o_prefill_gqa_workspace_bytes(B, Hkv, D, N, kvc.KVC_F32) > gqa
    assert kvc.kvc_h2o_prefill_gqa_workspace_bytes(B, Hkv, D, N, 7) == 0
    assert kvc.kvc_decode_attn_duo_workspace_bytes(1, 32, 32, 128, 100, 33) == 0


@pytest.mark.parametrize("B,H,N", [(16, 32, 4096), (2, 3, 333), (1, 1, 129), (1, 2, 128)])
def test_scoring_workspace_holds_whole_row_blocks(kvc, B, H, N):
    """Host sizing of the prompt scoring: besides the column sums and at least one (max, sum)
    state per window row, the workspace holds every row's log-sum-exp padded to whole 128-row
    blocks (the column pass streams those values one 512-byte block at a time)."""
    rows_padded = (N + 127) // 128 * 128
    need = B * H * (N + 2 * N + rows_padded) * 4
    assert kvc.kvc_h2o_prefill_workspace_bytes(B, H, 128, N) >= need
    G, L_obs = 4, 64
    if N > L_obs:
        R = G * L_obs
        need_s = B * H * ((N - L_obs) * (G + 1) + 2 * R + (R + 127) // 128 * 128) * 4
        assert kvc.kvc_snapkv_select_workspace_bytes(B, H * G, H, 128, N, L_obs) >= need_s
