"""GPU parity: DuoAttention's inference half (retrieval heads over full caches, streaming heads
over sink + ring buffers, one decode launch), through the C ABI, against the oracle."""
import math

import pytest
import torch

import oracle
from gpu_helpers import TOL, assert_close, cuda_or_skip, f64, lib
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _caches(B, n_ret, n_str, cap, ring_cap, D, dtype, dev):
    full_k = torch.zeros((B, n_ret, cap, D), device=dev, dtype=dtype)
    full_v = torch.zeros_like(full_k)
    ring_k = torch.zeros((B, n_str, ring_cap, D), device=dev, dtype=dtype)
    ring_v = torch.zeros_like(ring_k)
    return full_k, full_v, ring_k, ring_v


@pytest.mark.parametrize("dtype,D,G,ret_heads,Hkv,S,W", [
    (torch.float32, 64, 1, [1, 3], 4, 4, 20),
    (torch.bfloat16, 128, 1, [0], 3, 4, 9),
    (torch.bfloat16, 128, 4, [2, 3], 5, 4, 64),
    (torch.float32, 256, 2, [0, 1, 4], 6, 0, 30),
])
def test_duo_decode_every_step_from_empty(dtype, D, G, ret_heads, Hkv, S, W):
    """Token by token: the append sends each KV head's row to its own cache, then one decode
    launch; every query head against the oracle's DuoAttention decode from the full history."""
    dev = cuda_or_skip()
    kvc = lib()
    B = 2
    Hq = Hkv * G
    n_ret, n_str = len(ret_heads), Hkv - len(ret_heads)
    T = S + 2 * (W + 1) + 7
    cap = T + 3
    fk, fv, rk, rv = _caches(B, n_ret, n_str, cap, S + W + 1, D, dtype, dev)
    full, ring = kvc.cache_view(fk, fv), kvc.cache_view(rk, rv)
    ln = torch.zeros(B * n_ret, dtype=torch.int32, device=dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    duo = kvc.Duo(ret_heads, S, W, t_dev)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, T, 90 + D + G, dev, dtype)
    hk, hv = f64(ks), f64(vs)
    scale = 1 / math.sqrt(D)
    lse = torch.empty((B, Hq), device=dev)
    for t in range(T):
        t_dev.fill_(t)
        kvc.kvc_duo_append(full, ln, ring, duo, ks[t], vs[t])
        out = kvc.kvc_decode_attn_duo(qs[t], full, ring, duo, scale=scale, len=ln, lse=lse)
        t_dev.add_(0)        # a plain kernel: an ordering point after the append (kvc.h)
        out_s = kvc.kvc_decode_attn_duo(qs[t], full, ring, duo, scale=scale, len=ln,
                                        flags=kvc.KVC_DECODE_KV_SETTLED)
        assert torch.equal(out, out_s), "settled-cache load order changed the result"
        o = out.cpu().numpy()
        for b in range(B):
            for h in range(Hq):
                kh = h // G
                ref = oracle.duo_decode(kh in ret_heads, t, S, W, f64(qs[t, b, h]),
                                        hk[:t + 1, b, kh], hv[:t + 1, b, kh], scale)
                assert_close(o[b, h], ref, TOL[dtype], f"t={t} b={b} h={h}")
    assert kvc.kvc_device_status() == 0
    assert ln.cpu().tolist() == [T] * (B * n_ret)


def test_duo_long_retrieval_heads_many_blocks():
    """Retrieval heads of 6000 tokens (many tiles, a pair split over many blocks and merged)
    beside streaming heads of 4 + 64 + 1 slots, the page's buffer; one decode step at t = 6000,
    every head against the oracle; the logits at each head's own slots."""
    dev = cuda_or_skip()
    kvc = lib()
    dtype, D, G, B, Hkv, S, W, N = torch.bfloat16, 128, 1, 2, 8, 4, 64, 6000
    ret_heads = [2, 5]
    Hq = Hkv * G
    n_ret, n_str = len(ret_heads), Hkv - len(ret_heads)
    hist_k = I.randn((N + 1, B, Hkv, D), 501, dev, dtype)
    hist_v = I.randn((N + 1, B, Hkv, D), 502, dev, dtype)
    q = I.randn((B, Hq, D), 503, dev, dtype)
    fk, fv, rk, rv = _caches(B, n_ret, n_str, N + 8, S + W + 1, D, dtype, dev)
    str_heads = [h for h in range(Hkv) if h not in ret_heads]
    for r, h in enumerate(ret_heads):                       # prompt tokens 0 .. N-1
        fk[:, r, :N] = hist_k[:N, :, h].permute(1, 0, 2)
        fv[:, r, :N] = hist_v[:N, :, h].permute(1, 0, 2)
    for s_, h in enumerate(str_heads):                      # their ring slots
        for a in list(range(S)) + list(range(N - W, N)):
            slot = oracle.stream_slot(a, S, W)
            rk[:, s_, slot] = hist_k[a, :, h]
            rv[:, s_, slot] = hist_v[a, :, h]
    full, ring = kvc.cache_view(fk, fv), kvc.cache_view(rk, rv)
    ln = torch.full((B * n_ret,), N, dtype=torch.int32, device=dev)
    t_dev = torch.tensor([N], dtype=torch.int64, device=dev)
    duo = kvc.Duo(ret_heads, S, W, t_dev)
    kvc.kvc_duo_append(full, ln, ring, duo, hist_k[N].contiguous(), hist_v[N].contiguous())
    logits = torch.full((B, Hq, N + 8), float("nan"), device=dev)
    out = kvc.kvc_decode_attn_duo(q, full, ring, duo, scale=1 / math.sqrt(D), len=ln,
                                  logits=logits)
    assert kvc.kvc_device_status() == 0
    o, lg = out.cpu().numpy(), logits.cpu().numpy()
    hk, hv = f64(hist_k), f64(hist_v)
    scale = 1 / math.sqrt(D)
    tok, _, _ = oracle.stream_window(N, S, W)
    for b in range(B):
        for h in range(Hq):
            kh = h // G
            ret = kh in ret_heads
            ref = oracle.duo_decode(ret, N, S, W, f64(q[b, h]), hk[:, b, kh], hv[:, b, kh], scale)
            assert_close(o[b, h], ref, TOL[dtype], f"b={b} h={h}")
            if ret:
                _, ref_lg, _ = oracle.attend(f64(q[b, h]), hk[:, b, kh], hv[:, b, kh], scale)
                assert_close(lg[b, h, :N + 1], ref_lg, 1e-3, f"logits b={b} h={h}")
            else:
                slots = [oracle.stream_slot(int(a), S, W) for a in tok]
                want = scale * (hk[tok, b, kh] @ f64(q[b, h]))
                assert_close(lg[b, h, slots], want, 1e-3, f"ring logits b={b} h={h}")


def test_duo_empty_retrieval_caches():
    """Retrieval heads with no token yet (len 0) give out = 0 and lse = -inf; the streaming
    heads at t = 0 attend their one slot."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, G, D, S, W = 2, 3, 2, 64, 4, 8
    Hq = Hkv * G
    fk, fv, rk, rv = _caches(B, 1, Hkv - 1, 16, S + W + 1, D, torch.float32, dev)
    rk[:, :, 0] = I.randn((B, Hkv - 1, D), 601, dev)
    rv[:, :, 0] = I.randn((B, Hkv - 1, D), 602, dev)
    full, ring = kvc.cache_view(fk, fv), kvc.cache_view(rk, rv)
    ln = torch.zeros(B, dtype=torch.int32, device=dev)
    t = torch.zeros(1, dtype=torch.int64, device=dev)
    duo = kvc.Duo([1], S, W, t)
    q = I.randn((B, Hq, D), 603, dev)
    lse = torch.empty((B, Hq), device=dev)
    out = kvc.kvc_decode_attn_duo(q, full, ring, duo, scale=0.125, len=ln, lse=lse)
    assert kvc.kvc_device_status() == 0
    o, ls = out.cpu(), lse.cpu()
    for h in range(Hq):
        if h // G == 1:                                     # the retrieval head
            assert torch.all(o[:, h] == 0) and torch.all(torch.isneginf(ls[:, h]))
        else:                                               # one slot: its value
            s_idx = 0 if h // G == 0 else 1
            assert torch.allclose(o[:, h], rv[:, s_idx, 0].cpu(), atol=1e-6)
            assert torch.allclose(ls[:, h], 0.125 * (q[:, h] * rk[:, s_idx, 0]).sum(-1).cpu(),
                                  atol=1e-4)
