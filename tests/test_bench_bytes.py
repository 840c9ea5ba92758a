"""Host logic of the bench (no GPU): the algorithmic bytes the roofline figures divide by, for
the block-eviction and DuoAttention workloads, against counts written out here from the
workloads' shapes, and the token counts the block workload attends step by step."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _paged():
    import bench
    from kv_cache_compression_kvc_gb300 import inputs as I
    R = object.__new__(bench.PagedBlocks)
    R.w = I.WORKLOADS["paged"]
    R.bs, R.nb, R.recent = bench.PagedBlocks.block_shape(R.w)
    return R


def test_block_shape_rounds_budget_and_quota_up_to_blocks():
    R = _paged()
    assert (R.bs, R.nb, R.recent) == (32, 26, 13)            # 819 -> 832 tokens, 410 -> 416


def test_block_workload_tokens_per_step():
    """Full tables of 26 blocks: a step that opens a block attends 833 tokens then releases one
    (801 left); the last block then refills one token per step up to 832."""
    R = _paged()
    seq = [R.tokens_at(s) for s in range(70)]
    assert seq[0] == 833 and seq[1] == 802 and seq[31] == 832 and seq[32] == 833
    assert min(seq) == 802 and max(seq) == 833
    assert sum(seq[:32]) / 32 == 817.5


def test_block_workload_decode_bytes():
    R = _paged()
    w = R.w
    n = 833
    kv = 2 * w.batch * w.n_heads_kv * n * w.d_head * 2           # K and V, bf16
    qo = w.batch * w.n_heads_q * w.d_head * (2 + 4)               # q bf16, out fp32
    logits = w.batch * w.n_heads_q * (n + 1) * 4
    assert R.decode_bytes(0, 1) == kv + qo + logits


def test_duo_workload_decode_bytes():
    import bench
    from kv_cache_compression_kvc_gb300 import inputs as I
    R = object.__new__(bench.DuoAttention)
    R.w = w = I.WORKLOADS["duo"]
    R.n_ret, R.n_str, R.ring_cap = 8, 24, w.n_sink + w.window + 1
    step = 5
    full = w.prompt + step + 1                                    # the appended token included
    kv = 2 * w.batch * w.d_head * 2 * (8 * full + 24 * 69)
    qo = w.batch * w.n_heads_q * w.d_head * (2 + 4)
    assert R.decode_bytes(step, 1) == kv + qo
    assert R.ring_cap == 69
