"""kvc_decode_attn_noalloc: decode attention for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace (an engine whose device-memory plan is fixed
at start-up, a plugin running inside someone else's stream capture, a process held to an
external memory budget).  This entry point uses the library's own fixed 8 MiB device scratch
instead.  Its result must equal kvc_decode_attn's (same kernel, same schedule) on consecutive
calls that reuse the shared scratch, and a problem too large for the scratch must be refused
before anything is launched.  This file is collected last on purpose.
"""
import math

import pytest
import torch

from gpu_helpers import TOL, assert_close, cuda_or_skip, lib
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu

LIMIT = 8 << 20


def _compare_twice(kvc, q, K, V, dtype, **kw):
    B, Hq, D = q.shape
    lse_ref = torch.empty((B, Hq), device=q.device)
    ref = kvc.kvc_decode_attn(q, K, V, lse=lse_ref, **kw).clone()
    for call in range(2):
        lse = torch.full((B, Hq), float("nan"), device=q.device)
        out = torch.full((B, Hq, D), float("nan"), device=q.device)
        kvc.kvc_decode_attn_noalloc(q, K, V, out=out, lse=lse, **kw)
        assert kvc.kvc_device_status() == 0
        assert_close(out.cpu(), ref.cpu(), TOL[dtype], f"no-alloc call {call}")
        assert_close(lse.cpu(), lse_ref.cpu(), 1e-4, f"no-alloc lse call {call}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_workspace_entry_point(dtype):
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, G, D, cap = 2, 2, 4, 128, 3000
    assert 0 < kvc.kvc_decode_attn_workspace_bytes(B, Hkv * G, Hkv, D, cap) <= LIMIT
    K = I.randn((B, Hkv, cap, D), 501, dev, dtype)
    V = I.randn((B, Hkv, cap, D), 502, dev, dtype)
    q = I.randn((B, Hkv * G, D), 503, dev, dtype)
    lens = torch.tensor([2999, 17, 1500, 3000], dtype=torch.int32, device=dev)
    _compare_twice(kvc, q, K, V, dtype, scale=1 / math.sqrt(D), len=lens)


def test_noalloc_streaming_rope():
    dev = cuda_or_skip()
    kvc = lib()
    S, W, D, B, H = 4, 300, 128, 1, 2
    K = I.randn((B, H, S + W + 1, D), 511, dev, torch.bfloat16)
    V = I.randn((B, H, S + W + 1, D), 512, dev, torch.bfloat16)
    q = I.randn((B, H, D), 513, dev, torch.bfloat16)
    table = kvc.kvc_rope_table(S + W + 1, D).to(dev)
    t = torch.tensor([1234], dtype=torch.int64, device=dev)
    _compare_twice(kvc, q, K, V, torch.bfloat16, scale=1 / math.sqrt(D),
                   rope=kvc.make_rope(S, W, t, table))


def test_noalloc_refuses_problems_beyond_its_scratch():
    dev = cuda_or_skip()
    kvc = lib()
    candidates = [(1, 1, 8, 256, 100000), (64, 64, 8, 256, 64), (16, 16, 8, 256, 4096)]
    shape = next((c for c in candidates
                  if kvc.kvc_decode_attn_workspace_bytes(c[0], c[1] * c[2], c[1], c[3], c[4])
                  > LIMIT), None)
    assert shape is not None, "no candidate exceeds the fixed scratch"
    B, Hkv, G, D, cap = shape
    K = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=dev)
    V = torch.zeros_like(K)
    q = torch.zeros((B, Hkv * G, D), dtype=torch.bfloat16, device=dev)
    out = torch.full((B, Hkv * G, D), 7.0, device=dev)
    with pytest.raises(kvc.KvcError) as err:
        kvc.kvc_decode_attn_noalloc(q, K, V, scale=0.1, n_valid=cap, out=out)
    assert err.value.status == 6 and "scratch" in str(err.value)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)          # nothing was launched
