"""GPU parity at the benchmark workloads' full sizes, in the launch configuration bench.py times
(one layer of each workload, same shapes and calls), on sampled outputs the oracle can compute
one by one, plus properties that hold at any size."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (TOL, TOL_SPLIT_P, assert_close, assert_rel, cuda_or_skip, f64, lib,
                         topk_sets_agree)
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_streaming_full_size_layer():
    """32 heads x batch 16, 4 sinks + W=2044 ring filled from a 4096-token prompt, RoPE."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["streaming"]
    B, H, D, S, W = w.batch, w.n_heads_kv, w.d_head, w.n_sink, w.window
    slots = S + W + 1
    k_pre, v_pre, text_pos = I.streaming_prefill(w, 0, dev)
    K = torch.zeros((B, H, slots, D), dtype=w.dtype, device=dev)
    V = torch.zeros_like(K)
    ring = [a if a < S else S + (a - S) % (W + 1) for a in text_pos]
    K[:, :, ring] = k_pre
    V[:, :, ring] = v_pre
    table = kvc.kvc_rope_table(slots, D, w.theta).to(dev)
    t = torch.tensor([w.prompt], dtype=torch.int64, device=dev)
    qs, ks, vs = I.decode_qkv(B, w.n_heads_q, H, D, 3, w.seed, dev, w.dtype)
    rope = kvc.make_rope(S, W, t, table)
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
        out = kvc.kvc_decode_attn(qs[step], K, V, scale=w.scale, rope=rope, ws=ws).cpu().numpy()
        assert np.isfinite(out).all()
        tok, _, _ = oracle.stream_window(tt, S, W)
        for b, h in sample:
            hk = np.zeros((tt + 1, D))
            hv = np.zeros((tt + 1, D))
            for a in tok:
                hk[a] = f64(hist_k[int(a)][b, h])
                hv[a] = f64(hist_v[int(a)][b, h])
            ref = oracle.stream_decode(tt, S, W, f64(qs[step, b, h]), hk, hv, w.scale, w.theta)
            assert_close(out[b, h], ref, TOL[w.dtype], f"step {step} ({b},{h})")
    assert kvc.kvc_device_status() == 0


def test_snapkv_full_size_layer():
    """B=4, 32/8 heads, N=32768, L_obs=32, pool 5, budget 5243: select, compact, decode."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["snapkv"]
    B, Hkv, D, N = w.batch, w.n_heads_kv, w.d_head, w.prompt
    q_obs, k, v = I.snapkv_layer(w, 0, dev)
    n = N - w.L_obs
    scores = torch.empty((B, w.n_heads_q, n), device=dev)
    idx = kvc.kvc_snapkv_select(q_obs, k, seq_len=N, L_obs=w.L_obs, budget=w.budget,
                                scale=w.scale, pool_k=w.pool_k, scores_out=scores)
    assert kvc.kvc_device_status() == 0
    ix, sc = idx.cpu().numpy(), scores.cpu().numpy()
    assert ix.shape == (B, Hkv, w.budget)
    G = w.group
    for b, h in [(0, 0), (3, 7)]:
        row = ix[b, h]
        assert np.all(np.diff(row) > 0) and list(row[-w.L_obs:]) == list(range(n, N))
        replay = oracle.snapkv_stage_f32(sc[b, h * G:(h + 1) * G], w.L_obs, w.budget, w.pool_k)
        assert np.array_equal(replay, row), "stage-exact indices"
        ref_idx, ref_s, ref_score = oracle.snapkv_select(
            f64(q_obs[b, h * G:(h + 1) * G]), f64(k[b, h]), w.budget, w.scale, w.pool_k)
        assert_rel(sc[b, h * G:(h + 1) * G], ref_s[:, :n], 1e-4, 1e-8, "window means")
        topk_sets_agree(row[:w.budget - w.L_obs], ref_idx[:w.budget - w.L_obs], ref_score,
                        w.budget - w.L_obs)
    # every other pair: stage-exact replay, retained count 16% of the prompt
    for b in range(B):
        for h in range(Hkv):
            replay = oracle.snapkv_stage_f32(sc[b, h * G:(h + 1) * G], w.L_obs, w.budget,
                                             w.pool_k)
            assert np.array_equal(replay, ix[b, h])
    cap = w.budget + 4
    Kc = torch.empty((B, Hkv, cap, D), dtype=w.dtype, device=dev)
    Vc = torch.empty_like(Kc)
    lens = torch.zeros(B * Hkv, dtype=torch.int32, device=dev)
    kvc.kvc_compact_gather(k, v, idx, w.budget, Kc, Vc, len_dst=lens)
    assert kvc.kvc_device_status() == 0
    # compaction at full size, bit-exact: every pair's retained rows, in index order, and its
    # length
    assert lens.tolist() == [w.budget] * (B * Hkv)
    sel = idx.long()
    for b in range(B):
        for h in range(Hkv):
            assert torch.equal(Kc[b, h, :w.budget], k[b, h].index_select(0, sel[b, h])), \
                f"compacted K ({b},{h})"
            assert torch.equal(Vc[b, h, :w.budget], v[b, h].index_select(0, sel[b, h])), \
                f"compacted V ({b},{h})"
    qs, ks, vs = I.decode_qkv(B, w.n_heads_q, Hkv, D, 2, w.seed, dev, w.dtype)
    ws = kvc.decode_workspace(B, w.n_heads_q, Hkv, D, cap, dev)
    worst = 0.0
    for step in range(2):
        kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_TAIL, ks[step], vs[step], len=lens)
        out = kvc.kvc_decode_attn(qs[step], Kc, Vc, scale=w.scale, len=lens, ws=ws).cpu().numpy()
        for b, hq in [(0, 0), (2, 13), (3, 31)]:
            kh = hq // G
            Kr = np.concatenate([f64(k[b, kh])[ix[b, kh]], f64(ks[:step + 1, b, kh])])
            Vr = np.concatenate([f64(v[b, kh])[ix[b, kh]], f64(vs[:step + 1, b, kh])])
            ref, _, _ = oracle.attend(f64(qs[step, b, hq]), Kr, Vr, w.scale)
            worst = max(worst, assert_close(out[b, hq], ref, TOL[w.dtype],
                                            f"decode step {step} ({b},{hq})"))
    assert worst <= TOL_SPLIT_P, f"tensor-core decode max abs error {worst:.2e}"
    print(f"SnapKV tensor-core decode: max abs error {worst:.2e}")
    assert kvc.kvc_device_status() == 0


def test_h2o_full_size_layer():
    """B=16, 32 heads, N=4096, budget 819 = 410 recent + 409 heavy: prompt selection, then
    decode steps with accumulate/evict, sampled heads checked teacher-forced."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["h2o"]
    B, H, D, N = w.batch, w.n_heads_kv, w.d_head, w.prompt
    K_hh = w.budget - w.L_local
    q, k, v = I.h2o_layer(w, 0, dev)
    s_full = torch.empty((B, H, N), device=dev)
    idx, score = kvc.kvc_h2o_prefill_select(q, k, seq_len=N, L_local=w.L_local, K_hh=K_hh,
                                            scale=w.scale, s_full=s_full)
    assert kvc.kvc_device_status() == 0
    sf, ix = s_full.cpu().numpy(), idx.cpu().numpy()
    assert np.allclose(sf.sum(axis=-1), N, rtol=1e-3)            # every prompt row sums to 1
    for b in range(B):
        for h in range(H):
            assert np.array_equal(oracle.h2o_prompt_select(sf[b, h].astype(np.float64),
                                                           w.L_local, K_hh), ix[b, h])
    b, h = 5, 11
    ref = oracle.h2o_prompt_scores(f64(q[b, h]), f64(k[b, h]), w.scale)
    assert_rel(sf[b, h], ref, 1e-4, 1e-6, "prompt column sums")
    cap = w.budget + 1
    Kc = torch.zeros((B, H, cap, D), dtype=w.dtype, device=dev)
    Vc = torch.zeros_like(Kc)
    pos = torch.full((B, H, cap), -1, dtype=torch.int32, device=dev)
    sc = torch.zeros((B, H, cap), device=dev)
    kvc.kvc_compact_gather(k, v, idx, w.budget, Kc, Vc, pos_dst=pos)
    sc[:, :, :w.budget] = score
    free = torch.full((B * H,), w.budget, dtype=torch.int32, device=dev)
    t = torch.zeros(1, dtype=torch.int64, device=dev)
    qs, ks, vs = I.decode_qkv(B, H, H, D, 3, w.seed, dev, w.dtype)
    logits = torch.empty((B, H, cap), device=dev)
    lse = torch.empty((B, H), device=dev)
    ws = kvc.decode_workspace(B, H, H, D, cap, dev)
    for step in range(3):
        tt = N + step
        t.fill_(tt)
        kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_FREE_SLOT, ks[step], vs[step], t=t,
                              free_slot=free, pos=pos, score=sc)
        K0, V0 = f64(Kc[b, h]), f64(Vc[b, h])
        pos0, s0 = pos[b, h].cpu().numpy().astype(np.int64), sc[b, h].cpu().numpy().astype(np.float64)
        out = kvc.kvc_decode_attn(qs[step], Kc, Vc, scale=w.scale, n_valid=cap, logits=logits,
                                  lse=lse, ws=ws)
        kvc.kvc_h2o_accumulate_evict(logits, lse, sc, pos, free, n_slots=cap, t=t,
                                     L_local=w.L_local, budget=w.budget)
        o_ref, s_ref, _, _ = oracle.h2o_step(f64(qs[step, b, h]), K0, V0, pos0, s0, tt,
                                             w.L_local, w.budget, w.scale)
        assert_close(out[b, h].cpu().numpy(), o_ref, TOL[w.dtype], f"H2O out step {step}")
        s_gpu = sc[b, h].cpu().numpy()
        assert_rel(s_gpu, s_ref, 1e-4, 1e-6, f"H2O scores step {step}")
        assert oracle.h2o_evict_f32(s_gpu, pos0, tt, w.L_local) == int(free[b * H + h])
    assert kvc.kvc_device_status() == 0


def test_pyramid_full_size_layer():
    """B=2, 24/4 heads, D=256, N=131072, L_obs=64: the first layer's budget (13107), one pair
    against the oracle, every pair stage-exact; then a decode step over the compacted cache."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["pyramid"]
    B, Hkv, D, N, G = w.batch, w.n_heads_kv, w.d_head, w.prompt, w.group
    budget = kvc.kvc_pyramid_budgets(w.layers, w.budget, w.pyramid_ratio, 1)[0]
    assert budget == 13107
    q_obs, k, v = I.pyramid_layer(w, 0, dev)
    n = N - w.L_obs
    scores = torch.empty((B, w.n_heads_q, n), device=dev)
    idx = kvc.kvc_snapkv_select(q_obs, k, seq_len=N, L_obs=w.L_obs, budget=budget,
                                scale=w.scale, pool_k=w.pool_k, scores_out=scores)
    assert kvc.kvc_device_status() == 0
    ix, sc = idx.cpu().numpy(), scores.cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            assert np.array_equal(
                oracle.snapkv_stage_f32(sc[b, h * G:(h + 1) * G], w.L_obs, budget, w.pool_k),
                ix[b, h])
    b, h = 1, 2
    ref_idx, ref_s, ref_score = oracle.snapkv_select(
        f64(q_obs[b, h * G:(h + 1) * G]), f64(k[b, h]), budget, w.scale, w.pool_k)
    assert_rel(sc[b, h * G:(h + 1) * G], ref_s[:, :n], 1e-4, 1e-9, "window means")
    topk_sets_agree(ix[b, h][:budget - w.L_obs], ref_idx[:budget - w.L_obs], ref_score,
                    budget - w.L_obs)
    cap = budget + 2
    Kc = torch.empty((B, Hkv, cap, D), dtype=w.dtype, device=dev)
    Vc = torch.empty_like(Kc)
    lens = torch.zeros(B * Hkv, dtype=torch.int32, device=dev)
    kvc.kvc_compact_gather(k, v, idx, budget, Kc, Vc, len_dst=lens)
    qs, ks, vs = I.decode_qkv(B, w.n_heads_q, Hkv, D, 1, w.seed, dev, w.dtype)
    kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_TAIL, ks[0], vs[0], len=lens)
    out = kvc.kvc_decode_attn(qs[0], Kc, Vc, scale=w.scale, len=lens).cpu().numpy()
    worst = 0.0
    for hq in (0, 11, 23):
        kh = hq // G
        Kr = np.concatenate([f64(k[b, kh])[ix[b, kh]], f64(ks[0, b, kh])[None]])
        Vr = np.concatenate([f64(v[b, kh])[ix[b, kh]], f64(vs[0, b, kh])[None]])
        ref, _, _ = oracle.attend(f64(qs[0, b, hq]), Kr, Vr, w.scale)
        worst = max(worst, assert_close(out[b, hq], ref, TOL[w.dtype], f"decode head {hq}"))
    assert worst <= TOL_SPLIT_P, f"tensor-core decode max abs error {worst:.2e}"
    print(f"long-context tensor-core decode (d_head 256, group 6): max abs error {worst:.2e}")
    assert kvc.kvc_device_status() == 0
