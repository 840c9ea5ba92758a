"""GPU parity: decode attention, append and the StreamingLLM ring, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, TOL_SPLIT_P, assert_close, assert_rel, cuda_or_skip, f64, lib
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _oracle_decode(q, K, V, lens, scale, G):
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    logits = {}
    lse = np.zeros((B, Hq))
    for b in range(B):
        for h in range(Hq):
            n = int(lens[b, h // G])
            o, lg, ls = oracle.attend(f64(q[b, h]), f64(K[b, h // G, :n]), f64(V[b, h // G, :n]),
                                      scale)
            out[b, h], lse[b, h], logits[(b, h)] = o, ls, lg
    return out, logits, lse


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D,G", [(64, 4), (128, 1), (128, 2), (256, 6), (128, 8), (64, 1)])
def test_decode_matches_oracle_ragged(dtype, D, G):
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, cap = 2, 2, 1040
    Hq = Hkv * G
    K = I.randn((B, Hkv, cap, D), 11 + D + G, dev, dtype)
    V = I.randn((B, Hkv, cap, D), 12 + D + G, dev, dtype)
    q = I.randn((B, Hq, D), 13 + D + G, dev, dtype)
    lens = torch.tensor([[1037, 1], [300, 64]], dtype=torch.int32, device=dev)
    scale = 1 / math.sqrt(D)
    logits = torch.full((B, Hq, cap), float("nan"), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    out = kvc.kvc_decode_attn(q, K, V, scale=scale, len=lens.flatten(), logits=logits, lse=lse)
    assert kvc.kvc_device_status() == 0
    # the settled-cache load order gives the same bits
    lg2, lse2 = torch.full_like(logits, float("nan")), torch.empty_like(lse)
    out2 = kvc.kvc_decode_attn_ex(q, K, V, scale=scale, flags=kvc.KVC_DECODE_KV_SETTLED,
                                  len=lens.flatten(), logits=lg2, lse=lse2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert torch.equal(torch.nan_to_num(logits, 7.0), torch.nan_to_num(lg2, 7.0))
    ref, ref_lg, ref_lse = _oracle_decode(q, K, V, lens.cpu().numpy(), scale, G)
    # grouped bf16 heads run on the tensor cores (split-P product): the recorded bound there
    err = assert_close(out.cpu(), ref, TOL_SPLIT_P if dtype == torch.bfloat16 and G >= 2
                       else TOL[dtype], "decode out")
    print(f"decode {dtype} D={D} G={G}: max abs error {err:.2e}")
    assert_close(lse.cpu(), ref_lse, 1e-4, "lse")
    lg = logits.cpu().numpy()
    for (b, h), r in ref_lg.items():
        assert_close(lg[b, h, :len(r)], r, 1e-4, f"logits {b},{h}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_host_n_valid_and_empty(dtype):
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, G, D, cap = 3, 1, 2, 128, 700
    K = I.randn((B, Hkv, cap, D), 21, dev, dtype)
    V = I.randn((B, Hkv, cap, D), 22, dev, dtype)
    q = I.randn((B, Hkv * G, D), 23, dev, dtype)
    scale = 1 / math.sqrt(D)
    for n in (0, 1, 129, 700):
        lse = torch.empty((B, Hkv * G), device=dev)
        out = kvc.kvc_decode_attn(q, K, V, scale=scale, n_valid=n, lse=lse)
        ref, _, ref_lse = _oracle_decode(q, K, V, np.full((B, Hkv), n), scale, G)
        assert_close(out.cpu(), ref, TOL[dtype], f"n_valid={n}")
        if n == 0:
            assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("D,G", [(128, 4), (256, 6), (64, 8)])
@pytest.mark.parametrize("case", ["ragged", "one_pair", "many_pairs"])
def test_gqa_decode_schedules(D, G, case):
    """Tensor-core group decode under both schedules -- blocks split by capacity (default) and
    by the lengths (KVC_DECODE_BALANCE; capacity again past 1024 pairs) -- on ragged pairs with
    empty and full ones, one pair split over every block, and many pairs.  Both orderings of
    the first loads (KVC_DECODE_KV_SETTLED or not) give the same bits."""
    dev = cuda_or_skip()
    kvc = lib()
    dtype = torch.bfloat16
    if case == "ragged":
        B, Hkv, cap = 5, 4, 2000
    elif case == "one_pair":
        B, Hkv, cap = 1, 1, 20000
    else:
        B, Hkv, cap = 65, 16, 200
    Hq = Hkv * G
    seed = 100 + D + G + len(case)
    K = I.randn((B, Hkv, cap, D), seed, dev, dtype)
    V = I.randn((B, Hkv, cap, D), seed + 1, dev, dtype)
    q = I.randn((B, Hq, D), seed + 2, dev, dtype)
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, cap + 1, size=(B, Hkv))
    if case == "ragged":
        lens.flat[:4] = [0, cap, 1, 129]
    elif case == "one_pair":
        lens[:] = cap
    else:
        lens.flat[:3] = [0, cap, 1]
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev).flatten()
    scale = 1 / math.sqrt(D)
    S, BAL = kvc.KVC_DECODE_KV_SETTLED, kvc.KVC_DECODE_BALANCE
    outs = {}
    for flags in (0, S, BAL, S | BAL):
        lse = torch.empty((B, Hq), device=dev)
        out = kvc.kvc_decode_attn_ex(q, K, V, scale=scale, flags=flags, len=lens_t, lse=lse)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        outs[flags] = (out.cpu(), lse.cpu())
    for a, b in ((0, S), (BAL, S | BAL)):
        assert torch.equal(outs[a][0], outs[b][0]) and torch.equal(outs[a][1], outs[b][1])
    if case == "many_pairs":                 # a sample of the heads
        heads = [(b, h) for b in range(B) for h in range(Hq)]
        pick = rng.choice(len(heads), size=300, replace=False)
        heads = [heads[i] for i in pick] + [(0, g) for g in range(G)]
    else:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    Kc, Vc, qh = K.cpu(), V.cpu(), f64(q)
    for b, h in heads:
        n = int(lens[b, h // G])
        o, _, ls = oracle.attend(qh[b, h], f64(Kc[b, h // G, :n]), f64(Vc[b, h // G, :n]), scale)
        for flags in (0, BAL):
            out, lse = outs[flags]
            assert_close(out[b, h].numpy(), o, TOL[dtype], f"out ({b},{h}) n={n} flags={flags}")
            if n == 0:
                assert torch.all(out[b, h] == 0) and math.isinf(float(lse[b, h]))
            else:
                assert abs(float(lse[b, h]) - ls) <= 1e-3, (b, h, flags, float(lse[b, h]), ls)


def test_decode_strided_cache_view():
    """A cache that is a slice of a larger buffer (slot stride > d_head, capacity padding)."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, G, D = 2, 3, 2, 64
    big_k = I.randn((B, Hkv, 900, 2 * D), 31, dev, torch.bfloat16)
    big_v = I.randn((B, Hkv, 900, 2 * D), 32, dev, torch.bfloat16)
    K, V = big_k[:, :, 100:800, D:], big_v[:, :, 100:800, D:]
    q = I.randn((B, Hkv * G, D), 33, dev, torch.bfloat16)
    out = kvc.kvc_decode_attn(q, K, V, scale=0.125, n_valid=650)
    ref, _, _ = _oracle_decode(q, K, V, np.full((B, Hkv), 650), 0.125, G)
    assert_close(out.cpu(), ref, TOL[torch.bfloat16], "strided")


def test_append_tail_and_free_slot_layout():
    dev = cuda_or_skip()
    kvc = lib()
    B, H, cap, D = 2, 3, 10, 64
    K = torch.zeros((B, H, cap, D), device=dev, dtype=torch.bfloat16)
    V = torch.zeros_like(K)
    lens = torch.tensor([0, 3, 9, 5, 2, 0], dtype=torch.int32, device=dev)
    kn = I.randn((B, H, D), 41, dev, torch.bfloat16)
    vn = I.randn((B, H, D), 42, dev, torch.bfloat16)
    t = torch.tensor([77], dtype=torch.int64, device=dev)
    pos = torch.full((B, H, cap), -1, dtype=torch.int32, device=dev)
    kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_TAIL, kn, vn, t=t, len=lens, pos=pos)
    assert kvc.kvc_device_status() == 0
    before = [0, 3, 9, 5, 2, 0]
    assert lens.cpu().tolist() == [x + 1 for x in before]
    for r, s in enumerate(before):
        b, h = divmod(r, H)
        assert torch.equal(K[b, h, s], kn[b, h]) and torch.equal(V[b, h, s], vn[b, h])
        assert int(pos[b, h, s]) == 77
    # a full row records KVC_DEV_TAIL_FULL and is left untouched
    lens2 = torch.tensor([cap, 0, 0, 0, 0, 0], dtype=torch.int32, device=dev)
    snapshot = K.clone()
    kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_TAIL, kn, vn, len=lens2)
    assert kvc.kvc_device_status() == 1
    assert torch.equal(K[0, 0], snapshot[0, 0]) and int(lens2[0]) == cap
    # FREE_SLOT writes at the given slot, sets pos = t and score = 0
    free = torch.tensor([4, 0, 9, 1, 1, 7], dtype=torch.int32, device=dev)
    score = torch.ones((B, H, cap), device=dev)
    kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_FREE_SLOT, kn, vn, t=t, free_slot=free, pos=pos,
                          score=score)
    assert kvc.kvc_device_status() == 0
    for r, s in enumerate(free.cpu().tolist()):
        b, h = divmod(r, H)
        assert torch.equal(K[b, h, s], kn[b, h]) and float(score[b, h, s]) == 0.0
        assert int(pos[b, h, s]) == 77


# (dtype, D, G, S, W, extra table rows, wraps of the ring).  With one query head per KV head and
# a table of at least one tile of rows, the kernel factors the rotation into a per-lane constant
# and per-tile base rows; the cases with extra rows exercise that form: rings spanning several
# tiles (wrap point inside a tile), sinks spanning two tiles, no sinks, a partial last tile.
@pytest.mark.parametrize("dtype,D,G,S,W,extra,wraps", [
    (torch.float32, 64, 1, 4, 20, 0, 3),
    (torch.bfloat16, 128, 2, 4, 37, 0, 3),
    (torch.bfloat16, 64, 1, 0, 9, 0, 3),
    (torch.float32, 256, 4, 2, 130, 0, 3),
    (torch.bfloat16, 128, 1, 4, 150, 64, 2),
    (torch.bfloat16, 64, 1, 0, 200, 0, 2),
    (torch.float32, 64, 1, 70, 20, 0, 2),
    (torch.bfloat16, 256, 1, 3, 40, 30, 3),
    (torch.float32, 128, 1, 1, 45, 5, 3),
])
def test_streaming_ring_rope_matches_oracle_every_step(dtype, D, G, S, W, extra, wraps):
    """Token by token from an empty cache: ring append then decode with RoPE at in-cache
    positions; every step against the oracle's StreamingLLM decode from the full history."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv = 2, 2
    Hq = Hkv * G
    T = S + wraps * (W + 1) + 5
    cap = S + W + 1 + 3                        # extra slots past the ring are never used
    K = torch.zeros((B, Hkv, cap, D), device=dev, dtype=dtype)
    V = torch.zeros_like(K)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, T, 50 + D + W, dev, dtype)
    table = kvc.kvc_rope_table(S + W + 1 + extra, D, 10000.0).to(dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    rope = kvc.make_rope(S, W, t_dev, table)
    scale = 1 / math.sqrt(D)
    hk, hv = f64(ks), f64(vs)
    for t in range(T):
        t_dev.fill_(t)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, ks[t], vs[t], t=t_dev, n_sink=S,
                              window=W)
        out_t = kvc.kvc_decode_attn(qs[t], K, V, scale=scale, rope=rope)
        t_dev.add_(0)        # a plain kernel: an ordering point after the append (kvc.h)
        out_s = kvc.kvc_decode_attn_ex(qs[t], K, V, scale=scale, rope=rope,
                                       flags=kvc.KVC_DECODE_KV_SETTLED)
        assert torch.equal(out_t, out_s), "settled-cache load order changed the result"
        out = out_t.cpu().numpy()
        for b in range(B):
            for h in range(Hq):
                ref = oracle.stream_decode(t, S, W, f64(qs[t, b, h]), hk[:t + 1, b, h // G],
                                           hv[:t + 1, b, h // G], scale)
                assert_close(out[b, h], ref, TOL[dtype], f"t={t} b={b} h={h}")
    assert kvc.kvc_device_status() == 0
    # sinks never move once written
    for a in range(min(S, T)):
        assert torch.equal(K[:, :, a], ks[a]), "sink slot overwritten"


@pytest.mark.parametrize("table_rows", [8, 200])
def test_streaming_worked_example_positions(table_rows):
    """The pages' example: cache [0,1,2,3,6,7,8] decoding the next token uses positions 0..7.
    With values one-hot per token, the output mixes exactly the tokens 0,1,2,3,6,7,8,9, and the
    logits (rotated at cache positions) equal the oracle's.  With 200 table rows the kernel
    takes the factored rotation (table rows >= one tile of slots)."""
    dev = cuda_or_skip()
    kvc = lib()
    S, W, D = 4, 3, 64
    K = torch.zeros((1, 1, S + W + 1, D), device=dev)
    V = torch.zeros_like(K)
    ks = I.randn((10, 1, 1, D), 61, dev)
    vs = torch.zeros((10, 1, 1, D), device=dev)
    for a in range(10):
        vs[a, 0, 0, a] = 1.0
    q = I.randn((1, 1, D), 62, dev)
    table = kvc.kvc_rope_table(table_rows, D).to(dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    for t in range(10):
        t_dev.fill_(t)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, ks[t], vs[t], t=t_dev, n_sink=S, window=W)
    logits = torch.zeros((1, 1, S + W + 1), device=dev)
    out = kvc.kvc_decode_attn(q, K, V, scale=0.125, rope=kvc.make_rope(S, W, t_dev, table),
                              logits=logits)[0, 0].cpu().numpy()
    assert np.all(out[[4, 5]] == 0) and np.all(out[[0, 1, 2, 3, 6, 7, 8, 9]] > 0)
    tok, cpos, qpos = oracle.stream_window(9, S, W)
    assert list(cpos) == list(range(8)) and qpos == 7
    ref = oracle.stream_decode(9, S, W, f64(q[0, 0]), f64(ks[:, 0, 0]), f64(vs[:, 0, 0]), 0.125)
    assert_close(out, ref, 1e-5, "worked example")
    # logit of each cached token: scale * R(qpos) q . R(cache position) k, at the token's slot
    lg = logits[0, 0].cpu().numpy()
    qr = oracle.rope(f64(q[0, 0]), qpos)
    for a, pos in zip(tok, cpos):
        want = 0.125 * float(np.dot(qr, oracle.rope(f64(ks[a, 0, 0]), int(pos))))
        got = float(lg[oracle.stream_slot(int(a), S, W)])
        assert abs(got - want) <= 1e-5 * max(1.0, abs(want)), f"logit of token {a}"


# (dtype, D, G, S, W, wraps): ALiBi over the sink + ring layout, token by token from empty.
@pytest.mark.parametrize("dtype,D,G,S,W,wraps", [
    (torch.float32, 64, 1, 4, 20, 3),
    (torch.bfloat16, 128, 1, 4, 150, 2),
    (torch.bfloat16, 128, 4, 4, 37, 3),
    (torch.float32, 256, 2, 2, 70, 2),
    (torch.bfloat16, 64, 8, 0, 9, 3),
    (torch.float32, 128, 1, 70, 20, 2),
])
def test_streaming_ring_alibi_matches_oracle_every_step(dtype, D, G, S, W, wraps):
    """Ring append then decode with ALiBi at in-cache positions; every step's output, logits
    (at their slots) and log-sum-exp against the oracle's ALiBi decode from the full history."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv = 2, 2
    Hq = Hkv * G
    T = S + wraps * (W + 1) + 5
    cap = S + W + 1 + 3
    K = torch.zeros((B, Hkv, cap, D), device=dev, dtype=dtype)
    V = torch.zeros_like(K)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, T, 70 + D + W, dev, dtype)
    slopes_h = kvc.kvc_alibi_slopes(Hq)
    slopes = slopes_h.to(dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    alibi = kvc.make_alibi(S, W, t_dev, slopes)
    scale = 1 / math.sqrt(D)
    hk, hv = f64(ks), f64(vs)
    logits = torch.full((B, Hq, cap), float("nan"), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    for t in range(T):
        t_dev.fill_(t)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, ks[t], vs[t], t=t_dev, n_sink=S,
                              window=W)
        out_t = kvc.kvc_decode_attn_alibi(qs[t], K, V, scale=scale, alibi=alibi, logits=logits,
                                          lse=lse)
        t_dev.add_(0)        # a plain kernel: an ordering point after the append (kvc.h)
        out_s = kvc.kvc_decode_attn_alibi(qs[t], K, V, scale=scale, alibi=alibi,
                                          flags=kvc.KVC_DECODE_KV_SETTLED)
        assert torch.equal(out_t, out_s), "settled-cache load order changed the result"
        out, lg, ls = out_t.cpu().numpy(), logits.cpu().numpy(), lse.cpu().numpy()
        tok, _, _ = oracle.stream_window(t, S, W)
        slots = [oracle.stream_slot(int(a), S, W) for a in tok]
        for b in range(B):
            for h in range(Hq):
                ref, ref_lg, ref_lse = oracle.stream_decode_alibi(
                    t, S, W, f64(qs[t, b, h]), hk[:t + 1, b, h // G], hv[:t + 1, b, h // G],
                    scale, float(slopes_h[h]))
                assert_close(out[b, h], ref, TOL[dtype], f"t={t} b={b} h={h}")
                assert_rel(lg[b, h, slots], ref_lg, 1e-5, 1e-4, f"logits t={t} b={b} h={h}")
                assert abs(float(ls[b, h]) - ref_lse) <= 1e-4 * max(1.0, abs(ref_lse))
    assert kvc.kvc_device_status() == 0


def test_alibi_worked_example_continuous_bias():
    """The pages' cache [0,1,2,3,6,7,8] decoding token 9 with q = 0: the logits at the tokens'
    slots are the bias alone, -slope * (7 - r) over in-cache positions r = 0..7, and the output
    mixes only the values of tokens 0,1,2,3,6,7,8,9."""
    dev = cuda_or_skip()
    kvc = lib()
    S, W, D = 4, 3, 64
    K = torch.zeros((1, 1, S + W + 1, D), device=dev)
    V = torch.zeros_like(K)
    ks = I.randn((10, 1, 1, D), 81, dev)
    vs = torch.zeros((10, 1, 1, D), device=dev)
    for a in range(10):
        vs[a, 0, 0, a] = 1.0
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    for t in range(10):
        t_dev.fill_(t)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, ks[t], vs[t], t=t_dev, n_sink=S,
                              window=W)
    slope = 0.375
    slopes = torch.tensor([slope], device=dev)
    logits = torch.zeros((1, 1, S + W + 1), device=dev)
    q = torch.zeros((1, 1, D), device=dev)
    out = kvc.kvc_decode_attn_alibi(q, K, V, scale=0.125, alibi=kvc.make_alibi(S, W, t_dev, slopes),
                                    logits=logits)[0, 0].cpu().numpy()
    assert np.all(out[[4, 5]] == 0) and np.all(out[[0, 1, 2, 3, 6, 7, 8, 9]] > 0)
    tok, cpos, qpos = oracle.stream_window(9, S, W)
    lg = logits[0, 0].cpu().numpy()
    for a, r in zip(tok, cpos):
        want = -slope * (qpos - int(r))
        assert abs(float(lg[oracle.stream_slot(int(a), S, W)]) - want) <= 1e-5, int(a)
    # weights fall off geometrically with the in-cache distance
    w = out[[0, 1, 2, 3, 6, 7, 8, 9]]
    assert np.allclose(w[1:] / w[:-1], math.exp(slope), rtol=1e-5)
