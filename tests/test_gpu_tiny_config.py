"""GPU parity on the tiny fp32 workload at its own configuration, free-running runs and a long
stream, through the C ABI.

- StreamingLLM at the tiny workload's shape: fp32, 8 query heads over 2 KV heads (a group of
  4, so every key reads its RoPE table row), d_head 64, 4 sinks + W = 60, RoPE theta 10000 at
  in-cache positions; the 512-token prompt goes through the ring, then 64 decode steps, every
  step and head against the oracle's decode from the full history ("attention sinks", "como
  funciona"; "Compressão e Poda Dinâmica de KV Cache", StreamingLLM).
- H2O free-running on the tiny workload (budget 102 = 51 recent + 51 heavy hitters, 64 steps):
  the GPU and the oracle each run from the prompt with their own state, and the test reports
  the first step at which the evicted tokens differ; up to it the caches and outputs must
  agree, and the divergence itself must be a near-tie of the oracle's scores ("Compressão e
  Poda Dinâmica de KV Cache", Heavy-Hitter Oracle).
- A 10^4-step StreamingLLM stream (one head, d_head 64): the sinks stay bit-identical to their
  first write, the outputs match the oracle at sampled steps, and no device memory is allocated
  after the first step (the cache is O(S + W), whatever the length).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, assert_close, cuda_or_skip, f64, lib, topk_sets_agree
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_tiny_streaming_rope_at_its_own_config():
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["tiny"]
    B, Hq, Hkv, D, N, S, W = 1, w.n_heads_q, w.n_heads_kv, w.d_head, w.prompt, w.n_sink, w.window
    G = Hq // Hkv
    assert (G, D, S, W, w.dtype) == (4, 64, 4, 60, torch.float32)
    _, k, v = I.prompt_qkv(B, Hq, Hkv, N, D, w.seed, dev, w.dtype)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, w.steps, w.seed, dev, w.dtype)
    K = torch.zeros((B, Hkv, S + W + 1, D), device=dev, dtype=w.dtype)
    V = torch.zeros_like(K)
    table = kvc.kvc_rope_table(S + W + 1, D, w.theta).to(dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    rope = kvc.make_rope(S, W, t_dev, table)
    for a in range(N):                                   # the prompt through the ring
        t_dev.fill_(a)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, k[:, :, a].contiguous(),
                              v[:, :, a].contiguous(), t=t_dev, n_sink=S, window=W)
    hist_k = np.concatenate([f64(k[0]).transpose(1, 0, 2), f64(ks[:, 0])], axis=0)
    hist_v = np.concatenate([f64(v[0]).transpose(1, 0, 2), f64(vs[:, 0])], axis=0)
    worst = 0.0
    for step in range(w.steps):
        t = N + step
        t_dev.fill_(t)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, ks[step], vs[step], t=t_dev, n_sink=S,
                              window=W)
        out = kvc.kvc_decode_attn(qs[step], K, V, scale=w.scale, rope=rope).cpu().numpy()
        for h in range(Hq):
            ref = oracle.stream_decode(t, S, W, f64(qs[step, 0, h]), hist_k[:t + 1, h // G],
                                       hist_v[:t + 1, h // G], w.scale, w.theta)
            worst = max(worst, assert_close(out[0, h], ref, TOL[torch.float32],
                                            f"step {step} head {h}"))
    assert kvc.kvc_device_status() == 0
    # the sinks are the prompt's first tokens, never overwritten
    assert torch.equal(K[:, :, :S], k[:, :, :S])
    print(f"tiny StreamingLLM: max abs error {worst:.2e} over {w.steps} steps x {Hq} heads")


def test_tiny_h2o_free_running_first_divergence():
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["tiny"]
    B, H, N, D = 1, 8, w.prompt, w.d_head
    budget, L_local, steps = w.extra["h2o_budget"], w.L_local, w.steps
    K_hh = budget - L_local
    seed = w.seed + 7
    q, k, v = I.prompt_qkv(B, H, H, N, D, seed, dev, w.dtype)
    scale = w.scale
    # GPU: prompt scores and one-shot compression, then the decode loop on its own state
    idx, score = kvc.kvc_h2o_prefill_select(q, k, seq_len=N, L_local=L_local, K_hh=K_hh,
                                            scale=scale)
    cap = budget + 1
    Kc = torch.zeros((B, H, cap, D), device=dev, dtype=w.dtype)
    Vc = torch.zeros_like(Kc)
    pos = torch.full((B, H, cap), -1, dtype=torch.int32, device=dev)
    sc = torch.zeros((B, H, cap), device=dev)
    kvc.kvc_compact_gather(k, v, idx, budget, Kc, Vc, pos_dst=pos)
    sc[:, :, :budget] = score
    free = torch.full((B * H,), budget, dtype=torch.int32, device=dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    qs, ks, vs = I.decode_qkv(B, H, H, D, steps, seed + 1, dev, w.dtype)
    logits = torch.empty((B, H, cap), device=dev)
    lse = torch.empty((B, H), device=dev)
    # oracle: its own fp64 state from the prompt
    hk, hv = f64(k[0]), f64(v[0])
    o_K = np.zeros((H, cap, D))
    o_V = np.zeros((H, cap, D))
    o_pos = np.full((H, cap), -1, dtype=np.int64)
    o_s = np.zeros((H, cap))
    o_free = np.full(H, budget, dtype=np.int64)
    diverged = {}                                        # head -> first step (-1: the prompt)
    ix = idx.cpu().numpy()
    for h in range(H):
        s_ref = oracle.h2o_prompt_scores(f64(q[0, h]), hk[h], scale)
        keep = oracle.h2o_prompt_select(s_ref, L_local, K_hh)
        o_K[h, :budget], o_V[h, :budget] = hk[h][keep], hv[h][keep]
        o_pos[h, :budget], o_s[h, :budget] = keep, s_ref[keep]
        if not np.array_equal(keep, ix[0, h]):
            topk_sets_agree(ix[0, h][:K_hh], keep[:K_hh], s_ref[:N - L_local], K_hh)
            diverged[h] = -1
    for step in range(steps):
        t = N + step
        t_dev.fill_(t)
        kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_FREE_SLOT, ks[step], vs[step], t=t_dev,
                              free_slot=free, pos=pos, score=sc)
        out = kvc.kvc_decode_attn(qs[step], Kc, Vc, scale=scale, n_valid=cap, logits=logits,
                                  lse=lse)
        kvc.kvc_h2o_accumulate_evict(logits, lse, sc, pos, free, n_slots=cap, t=t_dev,
                                     L_local=L_local, budget=budget)
        o_gpu, f_gpu, p_gpu = out.cpu().numpy(), free.cpu().numpy(), pos.cpu().numpy()
        for h in range(H):
            if h in diverged:
                continue
            f = o_free[h]
            o_K[h, f], o_V[h, f] = f64(ks[step, 0, h]), f64(vs[step, 0, h])
            o_pos[h, f], o_s[h, f] = t, 0.0
            o_ref, s_new, _, ev = oracle.h2o_step(f64(qs[step, 0, h]), o_K[h], o_V[h], o_pos[h],
                                                  o_s[h], t, L_local, budget, scale)
            assert_close(o_gpu[0, h], o_ref, TOL[torch.float32], f"free-running out step {step}")
            o_s[h] = s_new
            if ev != int(f_gpu[h]):
                # a divergence must be decided by rounding: the two evictees' oracle scores
                # lie within a relative 1e-4 of each other
                a, b = int(f_gpu[h]), int(ev)
                assert abs(s_new[a] - s_new[b]) <= 1e-4 * abs(s_new[b]), \
                    f"head {h} step {step}: evicted slot {a} (s={s_new[a]}) vs oracle {b} " \
                    f"(s={s_new[b]})"
                diverged[h] = step
                continue
            o_free[h] = ev
            assert np.array_equal(p_gpu[0, h], o_pos[h]), f"cache positions step {step} head {h}"
    assert kvc.kvc_device_status() == 0
    first = min(diverged.values()) if diverged else None
    print(f"tiny H2O free-running: first divergence step {first} "
          f"({len(diverged)} of {H} heads diverged)")


def test_long_tiny_stream_invariants():
    dev = cuda_or_skip()
    kvc = lib()
    B, H, D, S, W, T = 1, 1, 64, 4, 60, 10000
    dtype = torch.float32
    qs, ks, vs = I.decode_qkv(B, H, H, D, T, 2024, dev, dtype)
    K = torch.zeros((B, H, S + W + 1, D), device=dev, dtype=dtype)
    V = torch.zeros_like(K)
    table = kvc.kvc_rope_table(S + W + 1, D).to(dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    rope = kvc.make_rope(S, W, t_dev, table)
    out = torch.empty((B, H, D), device=dev)
    ws = kvc.decode_workspace(B, H, H, D, S + W + 1, dev)
    scale = 1 / math.sqrt(D)
    hk, hv, hq = f64(ks[:, 0, 0]), f64(vs[:, 0, 0]), f64(qs[:, 0, 0])
    sample = set(range(0, T, 613)) | {S - 1, S, S + W, S + W + 1, T - 1}
    sinks = torch.empty_like(K[:, :, :S])
    allocs = None
    for t in range(T):
        t_dev.fill_(t)
        kvc.kvc_stream_append(K, V, kvc.KVC_APPEND_RING, ks[t], vs[t], t=t_dev, n_sink=S,
                              window=W)
        kvc.kvc_decode_attn(qs[t], K, V, scale=scale, rope=rope, out=out, ws=ws)
        if t == 0:
            torch.cuda.synchronize()
            allocs = torch.cuda.memory_stats(dev)["allocation.all.allocated"]
        if t in sample:
            ref = oracle.stream_decode(t, S, W, hq[t], hk[:t + 1], hv[:t + 1], scale)
            assert_close(out[0, 0].cpu().numpy(), ref, TOL[dtype], f"t={t}")
        if t == S - 1:
            sinks.copy_(K[:, :, :S])
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats(dev)["allocation.all.allocated"] == allocs, \
        "device memory was allocated after the first step"
    assert torch.equal(K[:, :, :S], sinks) and torch.equal(K[0, 0, :S], ks[:S, 0, 0])
    assert kvc.kvc_device_status() == 0
    # the positions stayed within S + W: the ring holds exactly the W + 1 newest tokens
    tok, cpos, qpos = oracle.stream_window(T - 1, S, W)
    assert qpos == S + W and int(cpos.max()) == S + W
    for a in tok[S:]:
        assert torch.equal(K[0, 0, oracle.stream_slot(int(a), S, W)], ks[int(a), 0, 0])
