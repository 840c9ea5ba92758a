"""GPU: the decode kernels' bounded waits, made to run out without any fault.

KVC_DECODE_TEST_STARVE makes the tile issuer load nothing, so the first wait of every block
gives up after a short bounded spin.  The call must finish, report KVC_DEV_TIMEOUT through
kvc_device_status, leave the workspace's merge tickets zeroed, and the next ordinary call on the
same workspace must give the same bits as before.  No copy is ever issued in this mode, so
nothing can still be landing in shared memory when a block exits.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, assert_close, cuda_or_skip, f64, lib
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu

KVC_DEV_TIMEOUT = 7


# (dtype, G, D, B, Hkv, cap): one head per KV head (CUDA-core kernel), query groups on the
# tensor cores, pairs spread over many blocks (merge tickets in use) and many small pairs
@pytest.mark.parametrize("dtype,G,D,B,Hkv,cap", [
    (torch.float32, 1, 64, 1, 2, 20000),
    (torch.bfloat16, 1, 128, 3, 4, 3000),
    (torch.bfloat16, 4, 128, 1, 1, 30000),
    (torch.bfloat16, 6, 256, 2, 4, 9000),
])
def test_decode_wait_runs_out_and_next_call_is_exact(dtype, G, D, B, Hkv, cap):
    dev = cuda_or_skip()
    kvc = lib()
    Hq = Hkv * G
    K = I.randn((B, Hkv, cap, D), 500 + D + G, dev, dtype)
    V = I.randn((B, Hkv, cap, D), 501 + D + G, dev, dtype)
    q = I.randn((B, Hq, D), 502 + D + G, dev, dtype)
    lens = torch.full((B * Hkv,), cap, dtype=torch.int32, device=dev)
    lens[0] = cap - 77
    scale = 1 / math.sqrt(D)
    ws = kvc.decode_workspace(B, Hq, Hkv, D, cap, dev)
    lse0 = torch.empty((B, Hq), device=dev)
    out0 = kvc.kvc_decode_attn_ex(q, K, V, scale=scale, len=lens, lse=lse0, ws=ws).clone()
    assert kvc.kvc_device_status() == 0
    # the starved call: every block gives up on its first tile and still finishes
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvc.kvc_decode_attn_ex(q, K, V, scale=scale, len=lens, ws=ws,
                           flags=kvc.KVC_DECODE_TEST_STARVE)
    assert kvc.kvc_device_status() == KVC_DEV_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    # a starved block still takes part in the merge tickets, so they come back zeroed: the
    # next call on the same workspace merges every pair exactly as the first one did
    lse1 = torch.empty((B, Hq), device=dev)
    out1 = kvc.kvc_decode_attn_ex(q, K, V, scale=scale, len=lens, lse=lse1, ws=ws)
    assert kvc.kvc_device_status() == 0
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    # and it is the attention the oracle computes
    for b, h in [(0, 0), (B - 1, Hq - 1)]:
        n = int(lens[b * Hkv + h // G])
        ref, _, _ = oracle.attend(f64(q[b, h]), f64(K[b, h // G, :n]), f64(V[b, h // G, :n]),
                                  scale)
        assert_close(out1[b, h].cpu().numpy(), ref, TOL[dtype], f"out ({b},{h})")


def test_decode_unknown_flag_refused_and_starved_call_then_normal_call():
    """The test flag is a bit of its own: unknown bits are still refused on the host."""
    dev = cuda_or_skip()
    kvc = lib()
    K = torch.zeros((1, 1, 64, 64), device=dev)
    q = torch.zeros((1, 1, 64), device=dev)
    with pytest.raises(kvc.KvcError):
        kvc.kvc_decode_attn_ex(q, K, K, scale=0.125, n_valid=4, flags=0x40000000)
    out = kvc.kvc_decode_attn_ex(q, K, K, scale=0.125, n_valid=4,
                                 flags=kvc.KVC_DECODE_TEST_STARVE)
    assert kvc.kvc_device_status() == KVC_DEV_TIMEOUT
    out = kvc.kvc_decode_attn_ex(q, K, K, scale=0.125, n_valid=4)
    assert kvc.kvc_device_status() == 0 and torch.all(out == 0)
    assert np.isfinite(out.cpu().numpy()).all()
