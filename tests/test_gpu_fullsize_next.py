"""GPU parity of ALiBi, DuoAttention, block eviction and grouped-query H2O at the bench
workloads' full sizes, in the launch configuration bench.py times (one layer, same shapes and
calls), on sampled outputs the oracle computes one by one, plus properties that hold at any
size."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, TOL_SPLIT_P, assert_close, cuda_or_skip, f64, lib
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_alibi_full_size_layer():
    """32 heads x batch 16, 4 sinks + W=2044 ring filled from a 4096-token prompt, ALiBi."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["alibi"]
    B, H, D, S, W = w.batch, w.n_heads_kv, w.d_head, w.n_sink, w.window
    slots = S + W + 1
    k_pre, v_pre, text_pos = I.streaming_prefill(w, 0, dev)
    K = torch.zeros((B, H, slots, D), dtype=w.dtype, device=dev)
    V = torch.zeros_like(K)
    ring = [a if a < S else S + (a - S) % (W + 1) for a in text_pos]
    K[:, :, ring] = k_pre
    V[:, :, ring] = v_pre
    slopes_h = kvc.kvc_alibi_slopes(w.n_heads_q)
    t = torch.tensor([w.prompt], dtype=torch.int64, device=dev)
    slopes = slopes_h.to(dev)           # kept alive: the descriptor holds only its address
    alibi = kvc.make_alibi(S, W, t, slopes)
    qs, ks, vs = I.decode_qkv(B, w.n_heads_q, H, D, 3, w.seed, dev, w.dtype)
    ws = kvc.decode_workspace(B, w.n_heads_q, H, D, slots, dev)
    hist_k = {a: k_pre[:, :, i] for i, a in enumerate(text_pos)}
    hist_v = {a: v_pre[:, :, i] for i, a in enumerate(text_pos)}
    sample = [(0, 0), (3, 17), (15, 31), (8, 5)]
    for step in range(3):
        tt = w.prompt + step
        t.fill_(tt)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, ks[step], vs[step], t=t, n_sink=S,
                              window=W)
        hist_k[tt], hist_v[tt] = ks[step], vs[step]
        out = kvc.kvc_decode_attn_alibi(qs[step], K, V, scale=w.scale, alibi=alibi,
                                        ws=ws).cpu().numpy()
        assert np.isfinite(out).all()
        tok, _, _ = oracle.stream_window(tt, S, W)
        for b, h in sample:
            hk = np.zeros((tt + 1, D))
            hv = np.zeros((tt + 1, D))
            for a in tok:
                hk[a] = f64(hist_k[int(a)][b, h])
                hv[a] = f64(hist_v[int(a)][b, h])
            ref, _, _ = oracle.stream_decode_alibi(tt, S, W, f64(qs[step, b, h]), hk, hv,
                                                   w.scale, float(slopes_h[h]))
            assert_close(out[b, h], ref, TOL[w.dtype], f"step {step} ({b},{h})")
    assert kvc.kvc_device_status() == 0


def test_duo_full_size_layer():
    """Batch 1, 32 heads, 131072-token context, 8 retrieval heads (the bench's first layer
    mask), 4 sinks + 64 recent for the others: append and decode, sampled heads of both kinds."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["duo"]
    B, H, D, N, S, W = w.batch, w.n_heads_kv, w.d_head, w.prompt, w.n_sink, w.window
    n_ret = w.extra["n_retrieval"]
    ret_heads = sorted(np.random.default_rng(w.seed).choice(H, n_ret, replace=False).tolist())
    str_heads = [h for h in range(H) if h not in ret_heads]
    hist_k = I.randn((B, H, N + 1, D), 701, dev, w.dtype)
    hist_v = I.randn((B, H, N + 1, D), 702, dev, w.dtype)
    cap = N + 8
    fk = torch.zeros((B, n_ret, cap, D), dtype=w.dtype, device=dev)
    fv = torch.zeros_like(fk)
    fk[:, :, :N] = hist_k[:, ret_heads, :N]
    fv[:, :, :N] = hist_v[:, ret_heads, :N]
    rk = torch.zeros((B, H - n_ret, S + W + 1, D), dtype=w.dtype, device=dev)
    rv = torch.zeros_like(rk)
    keep = list(range(S)) + list(range(N - W, N))
    slots = [oracle.stream_slot(a, S, W) for a in keep]
    rk[:, :, slots] = hist_k[:, str_heads][:, :, keep]
    rv[:, :, slots] = hist_v[:, str_heads][:, :, keep]
    full, ring = kvc.cache_view(fk, fv), kvc.cache_view(rk, rv)
    ln = torch.full((B * n_ret,), N, dtype=torch.int32, device=dev)
    t = torch.tensor([N], dtype=torch.int64, device=dev)
    duo = kvc.Duo(ret_heads, S, W, t)
    kvc.kvc_duo_append(full, ln, ring, duo, hist_k[:, :, N].contiguous(),
                       hist_v[:, :, N].contiguous())
    q = I.randn((B, w.n_heads_q, D), 703, dev, w.dtype)
    ws = torch.zeros(kvc.kvc_decode_attn_duo_workspace_bytes(B, w.n_heads_q, H, D, cap, n_ret) +
                     256, dtype=torch.uint8, device=dev)
    out = kvc.kvc_decode_attn_duo(q, full, ring, duo, scale=w.scale, len=ln, ws=ws).cpu().numpy()
    assert kvc.kvc_device_status() == 0 and np.isfinite(out).all()
    assert ln.cpu().tolist() == [N + 1] * n_ret
    for h in ret_heads[:2] + str_heads[:2] + [str_heads[-1]]:
        ref = oracle.duo_decode(h in ret_heads, N, S, W, f64(q[0, h]), f64(hist_k[0, h]),
                                f64(hist_v[0, h]), w.scale)
        assert_close(out[0, h], ref, TOL[w.dtype], f"head {h}")


def test_paged_full_size_layer():
    """Batch 16, 32 heads, 32-token blocks, 26 full blocks per sequence over a shuffled
    head-major pool: steps of append, decode with logits and the block update; sampled
    sequences teacher-forced (outputs, block-score increments, the released block)."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["paged"]
    B, H, D, bs = w.batch, w.n_heads_kv, w.d_head, w.extra["block_size"]
    nb, recent = -(-w.budget // bs), -(-w.L_local // bs)
    mb, n_pool = nb + 1, B * (nb + 2)
    kp = I.randn((H, n_pool, bs, D), 801, dev, w.dtype)
    vp = I.randn((H, n_pool, bs, D), 802, dev, w.dtype)
    perm = torch.randperm(n_pool, generator=torch.Generator().manual_seed(0))
    table = torch.full((B, mb), -1, dtype=torch.int32, device=dev)
    table[:, :nb] = perm[:B * nb].reshape(B, nb).to(torch.int32).to(dev)
    free = perm[B * nb:].to(torch.int32)
    ids = torch.full((n_pool,), -1, dtype=torch.int32, device=dev)
    ids[:free.numel()] = free.to(dev)
    top = torch.tensor([free.numel()], dtype=torch.int32, device=dev)
    nbl = torch.full((B,), nb, dtype=torch.int32, device=dev)
    ln = torch.full((B,), nb * bs, dtype=torch.int32, device=dev)
    rng = np.random.default_rng(3)
    score = torch.tensor(rng.random((B, mb)) * 40, dtype=torch.float32, device=dev)
    pool, pt = kvc.block_pool_view(kp, vp), kvc.page_table_view(table, nbl, ln, score)
    fp = kvc.free_pool_view(ids, top)
    logits = torch.empty((B, w.n_heads_q, mb * bs), device=dev)
    lse = torch.empty((B, w.n_heads_q), device=dev)
    released = torch.empty(B, dtype=torch.int32, device=dev)
    ws = kvc.decode_workspace(B, w.n_heads_q, H, D, mb * bs, dev)
    qs, ks, vs = I.decode_qkv(B, w.n_heads_q, H, D, 2, w.seed, dev, w.dtype)
    for step in range(2):
        kvc.kvc_paged_append(pool, pt, fp, ks[step], vs[step])
        out = kvc.kvc_decode_attn_paged(qs[step], pool, pt, scale=w.scale, logits=logits,
                                        lse=lse, ws=ws)
        s_before = score.cpu().numpy()
        pre = [x.clone() for x in (table, nbl, ln, score)]
        kvc.kvc_block_accumulate_evict(logits, lse, kvc.page_table_view(*pre), fp, block_size=bs,
                                       budget_blocks=10 ** 6, recent_blocks=recent)
        kvc.kvc_block_accumulate_evict(logits, lse, pt, fp, block_size=bs, budget_blocks=nb,
                                       recent_blocks=recent, released=released)
        assert kvc.kvc_device_status() == 0
        acc, tab0 = pre[3].cpu().numpy(), pre[0].cpu().numpy()
        n0, rel, o = pre[2].cpu().numpy(), released.cpu().numpy(), out.cpu().numpy()
        for b in (0, 9):
            n = int(n0[b])
            blocks = (n + bs - 1) // bs
            Kb = np.concatenate([f64(kp[:, int(tab0[b, i]), :min(bs, n - i * bs)])
                                 for i in range(blocks)], axis=1)
            Vb = np.concatenate([f64(vp[:, int(tab0[b, i]), :min(bs, n - i * bs)])
                                 for i in range(blocks)], axis=1)
            ro, rs, _ = oracle.block_step(f64(qs[step, b]), Kb, Vb, np.zeros(blocks), bs, nb,
                                          recent, w.scale)
            assert_close(o[b], ro, TOL[w.dtype], f"out step {step} b={b}")
            inc = acc[b, :blocks].astype(np.float64) - s_before[b, :blocks]
            tol = 1e-4 * np.abs(rs) + 2.5e-7 * np.abs(acc[b, :blocks]) + 1e-6
            assert np.all(np.abs(inc - rs) <= tol), (step, b)
            assert int(rel[b]) == oracle.block_evict_f32(acc[b, :blocks], nb, recent)
        assert int((rel >= 0).sum()) == (B if step == 0 else 0)   # step 0 opens a block each


def test_h2o_grouped_full_size_layer():
    """Batch 16, 32 query heads over 8 KV heads, budget 819 (410 recent): free-slot append,
    tensor-core decode with logits, grouped update; sampled KV heads teacher-forced."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["h2o_gqa"]
    B, H, D, G = w.batch, w.n_heads_kv, w.d_head, w.group
    cap = w.budget + 1
    Kc = I.randn((B, H, cap, D), 901, dev, w.dtype)
    Vc = I.randn((B, H, cap, D), 902, dev, w.dtype)
    rng = np.random.default_rng(5)
    pos_np = np.full((B, H, cap), -1, dtype=np.int32)
    K_hh = w.budget - w.L_local
    for b in range(B):
        for h in range(H):
            old = np.sort(rng.choice(w.prompt - w.L_local, K_hh, replace=False))
            pos_np[b, h, :w.budget] = np.concatenate([old, np.arange(w.prompt - w.L_local,
                                                                      w.prompt)])
    pos = torch.tensor(pos_np, device=dev)
    sc = torch.tensor(rng.random((B, H, cap)) * 4, dtype=torch.float32, device=dev)
    free = torch.full((B * H,), w.budget, dtype=torch.int32, device=dev)
    t = torch.zeros(1, dtype=torch.int64, device=dev)
    qs, ks, vs = I.decode_qkv(B, w.n_heads_q, H, D, 3, w.seed, dev, w.dtype)
    logits = torch.empty((B, w.n_heads_q, cap), device=dev)
    lse = torch.empty((B, w.n_heads_q), device=dev)
    ws = kvc.decode_workspace(B, w.n_heads_q, H, D, cap, dev)
    worst = 0.0
    for step in range(3):
        tt = w.prompt + step
        t.fill_(tt)
        kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_FREE_SLOT, ks[step], vs[step], t=t,
                              free_slot=free, pos=pos, score=sc)
        K0, V0 = f64(Kc), f64(Vc)
        pos0, s0 = pos.cpu().numpy().astype(np.int64), sc.cpu().numpy().astype(np.float64)
        out = kvc.kvc_decode_attn(qs[step], Kc, Vc, scale=w.scale, n_valid=cap, logits=logits,
                                  lse=lse, ws=ws).cpu().numpy()
        kvc.kvc_h2o_accumulate_evict_gqa(logits, lse, sc, pos, free, n_slots=cap, t=t,
                                         L_local=w.L_local, budget=w.budget)
        assert kvc.kvc_device_status() == 0
        s_gpu, f_gpu = sc.cpu().numpy(), free.cpu().numpy()
        for b, kh in ((0, 0), (7, 3), (15, 7)):
            o_ref, s_ref, _ = oracle.h2o_step_group(f64(qs[step, b, kh * G:(kh + 1) * G]),
                                                    K0[b, kh], V0[b, kh], pos0[b, kh],
                                                    s0[b, kh], tt, w.L_local, w.budget, w.scale)
            worst = max(worst, assert_close(out[b, kh * G:(kh + 1) * G], o_ref, TOL[w.dtype],
                                            f"out ({b},{kh})"))
            assert np.allclose(s_gpu[b, kh], s_ref, rtol=1e-4, atol=1e-5)
            assert oracle.h2o_evict_f32(s_gpu[b, kh], pos0[b, kh], tt, w.L_local) == \
                int(f_gpu[b * H + kh])
    assert worst <= TOL_SPLIT_P, f"tensor-core decode max abs error {worst:.2e}"
    print(f"grouped H2O tensor-core decode: max abs error {worst:.2e}")
