"""GPU parity: SnapKV selection, compaction and H2O, through the C ABI.

Index contract.  Stage-exact: given the GPU's own fp32 window means (scores_out), the oracle's
fp32 replay of pooling + group max + top-k must give bit-identical indices.  End-to-end: the GPU
index set may differ from the fp64 oracle's only at positions whose oracle score is within a
relative 1e-4 of the k-th threshold.  H2O is checked teacher-forced: every step starts the oracle
from the GPU's state.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (TOL, assert_close, assert_rel, cuda_or_skip, f64, lib,
                         topk_sets_agree)
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _check_snapkv(q_obs, K, seq_len, L_obs, budget, pool_k, scale, kvc, pairs=None,
                  rtol=1e-4):
    dev = q_obs.device
    B, Hq = q_obs.shape[:2]
    Hkv = K.shape[1]
    G = Hq // Hkv
    n = seq_len - L_obs
    scores = torch.empty((B, Hq, n), device=dev)
    idx = kvc.kvc_snapkv_select(q_obs, K, seq_len=seq_len, L_obs=L_obs, budget=budget,
                                scale=scale, pool_k=pool_k, scores_out=scores)
    assert kvc.kvc_device_status() == 0
    idx = idx.cpu().numpy()
    s_gpu = scores.cpu().numpy()
    n_keep = min(budget, seq_len)
    assert idx.shape == (B, Hkv, n_keep)
    pairs = pairs or [(b, h) for b in range(B) for h in range(Hkv)]
    for b, h in pairs:
        row = idx[b, h]
        assert np.all(np.diff(row) > 0), "indices ascending"
        ref_idx, ref_s, ref_score = oracle.snapkv_select(
            f64(q_obs[b, h * G:(h + 1) * G]), f64(K[b, h, :seq_len]), budget, scale, pool_k)
        # window means: fp32 (tensor-core or FMA) against fp64
        assert_rel(s_gpu[b, h * G:(h + 1) * G], ref_s[:, :n], rtol, 1e-7, f"s {b},{h}")
        # stage-exact replay from the GPU's own scores
        replay = oracle.snapkv_stage_f32(s_gpu[b, h * G:(h + 1) * G], L_obs, budget, pool_k)
        assert np.array_equal(replay, row), f"stage-exact indices differ at ({b},{h})"
        # end-to-end against fp64
        if budget < seq_len:
            assert list(row[budget - L_obs:]) == list(range(n, seq_len)), "window kept"
            topk_sets_agree(row[:budget - L_obs], ref_idx[:budget - L_obs], ref_score,
                            budget - L_obs)
        else:
            assert list(row) == list(range(seq_len))
    return idx


def test_snapkv_tiny_workload_fp32():
    """The tiny workload: fp32, Hq=8, Hkv=2, D=64, N=512, L_obs=32, pool 5, budget 128."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["tiny"]
    q, k, v = I.prompt_qkv(1, 8, 2, 512, 64, w.seed, dev, torch.float32)
    _check_snapkv(q[:, :, -32:].contiguous(), k, 512, 32, 128, 5, w.scale, kvc)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,Hq,Hkv,D,N,L_obs,budget", [
    (2, 4, 2, 128, 1000, 20, 200),      # ragged N, window not a multiple of 32
    (1, 6, 1, 256, 777, 64, 300),       # G = 6, D = 256, two tiles per head
    (1, 2, 2, 64, 300, 7, 300),         # budget = N: identity
    (1, 4, 1, 64, 130, 3, 9),           # tiny budget, pool edges
])
def test_snapkv_select_ragged(dtype, B, Hq, Hkv, D, N, L_obs, budget):
    dev = cuda_or_skip()
    kvc = lib()
    q = I.randn((B, Hq, L_obs, D), 70 + N, dev, dtype)
    K = I.randn((B, Hkv, N + 5, D), 71 + N, dev, dtype)      # cap > seq_len
    _check_snapkv(q, K, N, L_obs, budget, 5, 1 / math.sqrt(D), kvc)


@pytest.mark.parametrize("B,Hq,Hkv,D,N,L_obs,budget", [
    (2, 8, 2, 128, 1100, 32, 400),      # the SnapKV workload's group shape, ragged prompt
    (1, 12, 2, 256, 900, 64, 333),      # the long-context group shape (G = 6, D = 256)
    (1, 4, 1, 64, 513, 48, 100),        # heads straddle 32-row chunks of the accumulator
    (1, 2, 1, 128, 4200, 96, 700),      # several pass-1 chunks per row tile
])
def test_snapkv_select_tensor_core_shapes(B, Hq, Hkv, D, N, L_obs, budget):
    """bf16 shapes that take the tcgen05 scoring path (window of at least 32 queries)."""
    dev = cuda_or_skip()
    kvc = lib()
    q = I.randn((B, Hq, L_obs, D), 170 + N, dev, torch.bfloat16)
    K = I.randn((B, Hkv, N, D), 171 + N, dev, torch.bfloat16)
    _check_snapkv(q, K, N, L_obs, budget, 5, 1 / math.sqrt(D), kvc)


@pytest.mark.parametrize("B,Hq,Hkv,D,N,L_obs,budget", [
    (1, 8, 2, 128, 2500, 32, 300),      # one row block of 128 rows per KV head
    (2, 8, 2, 64, 3000, 64, 500),       # two row blocks (heads of 64 rows), d_head 64
    (8, 16, 8, 128, 700, 32, 150),      # 64 pairs, few key chunks
    (1, 4, 1, 128, 40000, 32, 4000),    # one pair, many chunks per pass
])
def test_snapkv_tensor_core_repeated_on_one_workspace(B, Hq, Hkv, D, N, L_obs, budget):
    """bf16 windows whose heads fill whole 128-row blocks (the column-sum pass walks each block's
    key range backwards): three calls in a row on one workspace give the same bits, and the
    selection matches the oracle as for the other shapes."""
    dev = cuda_or_skip()
    kvc = lib()
    q = I.randn((B, Hq, L_obs, D), 400 + N, dev, torch.bfloat16)
    K = I.randn((B, Hkv, N, D), 401 + N, dev, torch.bfloat16)
    ws = kvc._zeroed_workspace(kvc.kvc_snapkv_select_workspace_bytes(B, Hq, Hkv, D, N, L_obs),
                               dev)
    runs = []
    for _ in range(3):
        scores = torch.empty((B, Hq, N - L_obs), device=dev)
        idx = kvc.kvc_snapkv_select(q, K, seq_len=N, L_obs=L_obs, budget=budget,
                                    scale=1 / math.sqrt(D), scores_out=scores, ws=ws)
        assert kvc.kvc_device_status() == 0
        runs.append((idx.cpu(), scores.cpu()))
    for idx, scores in runs[1:]:
        assert torch.equal(idx, runs[0][0]) and torch.equal(scores, runs[0][1])
    pairs = [(0, 0), (B - 1, Hkv - 1)]
    _check_snapkv(q, K, N, L_obs, budget, 5, 1 / math.sqrt(D), kvc, pairs=pairs)


def test_snapkv_tiny_workload_bf16():
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["tiny"]
    q, k, v = I.prompt_qkv(1, 8, 2, 512, 64, w.seed, dev, torch.bfloat16)
    _check_snapkv(q[:, :, -32:].contiguous(), k, 512, 32, 128, 5, w.scale, kvc)


@pytest.mark.parametrize("pool_k", [1, 3, 7, 15])
@pytest.mark.parametrize("dtype,budget", [(torch.bfloat16, 333), (torch.float32, 48)])
def test_snapkv_select_pool_widths(pool_k, dtype, budget):
    """Other pooling widths (zero padding at both ends), and a budget equal to the window
    (nothing kept from the prefix)."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hq, Hkv, D, N, L_obs = 1, 8, 2, 128, 2300, 48
    q = I.randn((B, Hq, L_obs, D), 300 + pool_k, dev, dtype)
    K = I.randn((B, Hkv, N, D), 301 + pool_k, dev, dtype)
    _check_snapkv(q, K, N, L_obs, budget, pool_k, 1 / math.sqrt(D), kvc)


def test_snapkv_ties_across_the_row():
    """All prefix keys identical and a budget that takes ties from several eighths of the row:
    the lowest indices still win."""
    dev = cuda_or_skip()
    kvc = lib()
    D, N, L_obs = 64, 400, 16
    K = I.randn((1, 1, N, D), 91, dev)
    K[0, 0, :N - L_obs] = K[0, 0, 5]
    q = I.randn((1, 2, L_obs, D), 92, dev)
    idx = _check_snapkv(q, K, N, L_obs, 16 + 200, 5, 0.125, kvc)
    assert list(idx[0, 0, :200]) == list(range(2, 202))


def test_snapkv_exact_ties_keep_lowest_index():
    """Identical keys give identical scores: the lower index must win every tie."""
    dev = cuda_or_skip()
    kvc = lib()
    D, N, L_obs = 64, 400, 16
    K = I.randn((1, 1, N, D), 81, dev)
    K[0, 0, :N - L_obs] = K[0, 0, 5]          # every prefix key the same: all scores tie
    q = I.randn((1, 2, L_obs, D), 82, dev)
    idx = _check_snapkv(q, K, N, L_obs, 50, 5, 0.125, kvc)
    # interior pooled scores tie exactly; the two ends lose mass to zero padding
    assert list(idx[0, 0, :34]) == list(range(2, 36))


def test_compact_gather_bit_exact():
    dev = cuda_or_skip()
    kvc = lib()
    B, H, N, D, keep = 2, 3, 500, 128, 77
    K = I.randn((B, H, N, D), 91, dev, torch.bfloat16)
    V = I.randn((B, H, N, D), 92, dev, torch.bfloat16)
    g = torch.Generator().manual_seed(93)
    idx = torch.stack([torch.sort(torch.randperm(N, generator=g)[:keep]).values
                       for _ in range(B * H)]).reshape(B, H, keep).to(torch.int32).to(dev)
    Kd = torch.zeros((B, H, keep + 10, D), device=dev, dtype=torch.bfloat16)
    Vd = torch.zeros_like(Kd)
    pos = torch.zeros((B, H, keep + 10), dtype=torch.int32, device=dev)
    lens = torch.zeros(B * H, dtype=torch.int32, device=dev)
    kvc.kvc_compact_gather(K, V, idx, keep, Kd, Vd, pos_dst=pos, len_dst=lens)
    assert kvc.kvc_device_status() == 0
    il = idx.long()
    assert torch.equal(Kd[:, :, :keep], torch.gather(K, 2, il[..., None].expand(-1, -1, -1, D)))
    assert torch.equal(Vd[:, :, :keep], torch.gather(V, 2, il[..., None].expand(-1, -1, -1, D)))
    assert torch.equal(pos[:, :, :keep], idx) and lens.tolist() == [keep] * (B * H)
    bad = idx.clone()
    bad[1, 2, 5] = N + 3
    kvc.kvc_compact_gather(K, V, bad, keep, Kd, Vd)
    assert kvc.kvc_device_status() == 3      # KVC_DEV_BAD_INDEX, row skipped


def test_snapkv_then_decode_tiny():
    """Select -> compact -> TAIL appends -> decode, against the oracle on the same kept rows."""
    dev = cuda_or_skip()
    kvc = lib()
    w = I.WORKLOADS["tiny"]
    B, Hq, Hkv, D, N = 1, 8, 2, 64, 512
    q, k, v = I.prompt_qkv(B, Hq, Hkv, N, D, w.seed, dev, torch.float32)
    idx = kvc.kvc_snapkv_select(q[:, :, -32:].contiguous(), k, seq_len=N, L_obs=32, budget=128,
                                scale=w.scale)
    cap = 128 + w.steps
    Kc = torch.zeros((B, Hkv, cap, D), device=dev)
    Vc = torch.zeros_like(Kc)
    lens = torch.zeros(B * Hkv, dtype=torch.int32, device=dev)
    kvc.kvc_compact_gather(k, v, idx, 128, Kc, Vc, len_dst=lens)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, w.steps, w.seed, dev)
    kept = idx.cpu().numpy()
    for step in range(w.steps):
        kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_TAIL, ks[step], vs[step], len=lens)
        out = kvc.kvc_decode_attn(qs[step], Kc, Vc, scale=w.scale, len=lens).cpu().numpy()
        if step % 16 == 15 or step == 0:
            for h in range(Hq):
                kh = h // 4
                Kr = np.concatenate([f64(k[0, kh])[kept[0, kh]], f64(ks[:step + 1, 0, kh])])
                Vr = np.concatenate([f64(v[0, kh])[kept[0, kh]], f64(vs[:step + 1, 0, kh])])
                ref, _, _ = oracle.attend(f64(qs[step, 0, h]), Kr, Vr, w.scale)
                assert_close(out[0, h], ref, TOL[torch.float32], f"step {step} head {h}")
    assert lens.tolist() == [128 + w.steps] * Hkv
    assert kvc.kvc_device_status() == 0


# --------------------------------------------------------------------------------- H2O
def _h2o_run(B, H, N, D, budget, L_local, steps, dtype, seed, kvc, dev, check_every=1):
    K_hh = budget - L_local
    q, k, v = I.prompt_qkv(B, H, H, N, D, seed, dev, dtype)
    scale = 1 / math.sqrt(D)
    s_full = torch.empty((B, H, N), device=dev)
    idx, score = kvc.kvc_h2o_prefill_select(q, k, seq_len=N, L_local=L_local, K_hh=K_hh,
                                            scale=scale, s_full=s_full)
    assert kvc.kvc_device_status() == 0
    sf = s_full.cpu().numpy()
    ix = idx.cpu().numpy()
    for b in range(B):
        for h in range(H):
            ref = oracle.h2o_prompt_scores(f64(q[b, h]), f64(k[b, h]), scale)
            assert_rel(sf[b, h], ref, 1e-4, 1e-6, f"prompt scores {b},{h}")
            assert abs(sf[b, h].sum() - N) < 1e-3 * N
            assert np.array_equal(oracle.h2o_prompt_select(sf[b, h].astype(np.float64), L_local,
                                                           K_hh), ix[b, h]), "stage-exact"
            ref_idx = oracle.h2o_prompt_select(ref, L_local, K_hh)
            topk_sets_agree(ix[b, h][:K_hh], ref_idx[:K_hh], ref[:N - L_local], K_hh)
    assert np.allclose(score.cpu().numpy(), np.take_along_axis(sf, ix.astype(np.int64), 2))

    cap = budget + 1
    Kc = torch.zeros((B, H, cap, D), device=dev, dtype=dtype)
    Vc = torch.zeros_like(Kc)
    pos = torch.full((B, H, cap), -1, dtype=torch.int32, device=dev)
    sc = torch.zeros((B, H, cap), device=dev)
    kvc.kvc_compact_gather(k, v, idx, budget, Kc, Vc, pos_dst=pos)
    sc[:, :, :budget] = score
    free = torch.full((B * H,), budget, dtype=torch.int32, device=dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    qs, ks, vs = I.decode_qkv(B, H, H, D, steps, seed + 1, dev, dtype)
    logits = torch.empty((B, H, cap), device=dev)
    lse = torch.empty((B, H), device=dev)
    for step in range(steps):
        t = N + step
        t_dev.fill_(t)
        kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_FREE_SLOT, ks[step], vs[step], t=t_dev,
                              free_slot=free, pos=pos, score=sc)
        check = step % check_every == 0 or step == steps - 1
        if check:
            K0, V0 = f64(Kc), f64(Vc)
            pos0, s0 = pos.cpu().numpy().astype(np.int64), sc.cpu().numpy().astype(np.float64)
        out = kvc.kvc_decode_attn(qs[step], Kc, Vc, scale=scale, n_valid=cap, logits=logits,
                                  lse=lse)
        kvc.kvc_h2o_accumulate_evict(logits, lse, sc, pos, free, n_slots=cap, t=t_dev,
                                     L_local=L_local, budget=budget)
        if not check:
            continue
        o_gpu, s_gpu, f_gpu = out.cpu().numpy(), sc.cpu().numpy(), free.cpu().numpy()
        for b in range(B):
            for h in range(H):
                o_ref, s_ref, _, ev_ref = oracle.h2o_step(
                    f64(qs[step, b, h]), K0[b, h], V0[b, h], pos0[b, h], s0[b, h], t, L_local,
                    budget, scale)
                assert_close(o_gpu[b, h], o_ref, TOL[dtype], f"H2O out step {step}")
                assert_rel(s_gpu[b, h], s_ref, 1e-4, 1e-6, f"H2O s step {step}")
                ev = oracle.h2o_evict_f32(s_gpu[b, h], pos0[b, h], t, L_local)
                assert ev == int(f_gpu[b * H + h]), f"evictee step {step} ({b},{h})"
                kept_pos = set(pos0[b, h]) - {pos0[b, h][ev]}
                assert set(range(t - L_local + 1, t + 1)) <= kept_pos, "recent quota kept"
    assert kvc.kvc_device_status() == 0


def test_h2o_tiny_workload_teacher_forced():
    """The tiny H2O run: fp32, 8 heads, N=512, budget 102 (51 recent + 51 heavy), 64 steps."""
    dev = cuda_or_skip()
    kvc = lib()
    _h2o_run(1, 8, 512, 64, 102, 51, 64, torch.float32, I.WORKLOADS["tiny"].seed + 7, kvc, dev)


def test_h2o_bf16_ragged():
    dev = cuda_or_skip()
    kvc = lib()
    _h2o_run(2, 3, 333, 128, 70, 35, 40, torch.bfloat16, 4321, kvc, dev, check_every=3)


@pytest.mark.parametrize("D", [64, 128])
def test_h2o_bf16_multi_tile_prompt(D):
    """A prompt of several 128-row tiles: causal row and column tiles on the tensor cores
    (resident tile pairs; at d_head 64 one 64-column sub-tile per tile)."""
    dev = cuda_or_skip()
    kvc = lib()
    _h2o_run(1, 2, 700, D, 200, 100, 6, torch.bfloat16, 987, kvc, dev, check_every=2)


def test_h2o_evict_candidates_and_no_candidate_code():
    dev = cuda_or_skip()
    kvc = lib()
    B, H, n = 1, 2, 6
    logits = torch.zeros((B, H, n), device=dev)
    lse = torch.full((B, H), math.log(n), device=dev)        # alpha = 1/6 each
    sc = torch.tensor([[[0.5, 0.2, 0.2, 0.9, 0.2, 0.0], [1, 1, 1, 1, 1, 1]]],
                      dtype=torch.float32, device=dev)
    pos = torch.tensor([[[3, 7, 5, 1, 20, 21], [0, 1, 2, 3, 4, 5]]], dtype=torch.int32,
                       device=dev)
    free = torch.full((2,), -9, dtype=torch.int32, device=dev)
    t = torch.tensor([21], dtype=torch.int64, device=dev)
    kvc.kvc_h2o_accumulate_evict(logits, lse, sc, pos, free, n_slots=n, t=t, L_local=2, budget=5)
    assert kvc.kvc_device_status() == 0
    assert int(free[0]) == 1               # tie at 0.2+1/6: larger position 7 is evicted
    assert int(free[1]) == 5               # all tie: the largest candidate position (5 <= 19)
    t.fill_(2)                             # row 0 now has no position <= t - L_local = 0
    pos[0, 0] = torch.tensor([3, 7, 5, 9, 20, 21], dtype=torch.int32)
    kvc.kvc_h2o_accumulate_evict(logits, lse, sc, pos, free, n_slots=n, t=t, L_local=2, budget=5)
    assert kvc.kvc_device_status() == 6    # KVC_DEV_NO_CANDIDATE (row 0)
    assert int(free[1]) == 0               # row 1: position 0 is the only candidate


@pytest.mark.parametrize("dtype,G,D", [(torch.bfloat16, 4, 128), (torch.float32, 2, 64),
                                       (torch.bfloat16, 8, 64)])
def test_h2o_grouped_query_steps_teacher_forced(dtype, G, D):
    """H2O on a grouped-query cache: free-slot append, decode (tensor cores for bf16 groups)
    with logits, then the grouped score update; every step from the GPU's own state: output,
    scores (the sum over the group's heads) and the evicted slot, exactly, given the GPU's
    fp32 scores."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, N, budget, L_local, steps = 2, 2, 300, 70, 35, 24
    Hq = Hkv * G
    cap = budget + 1
    rng = np.random.default_rng(60 + G + D)
    Kc = I.randn((B, Hkv, cap, D), 61 + G, dev, dtype)
    Vc = I.randn((B, Hkv, cap, D), 62 + G, dev, dtype)
    pos_np = np.full((B, Hkv, cap), -1, dtype=np.int32)
    for b in range(B):
        for h in range(Hkv):
            old = np.sort(rng.choice(N - L_local, budget - L_local, replace=False))
            pos_np[b, h, :budget] = np.concatenate([old, np.arange(N - L_local, N)])
    pos = torch.tensor(pos_np, device=dev)
    sc = torch.tensor(rng.random((B, Hkv, cap)) * 3, dtype=torch.float32, device=dev)
    free = torch.full((B * Hkv,), budget, dtype=torch.int32, device=dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, steps, 63 + G, dev, dtype)
    logits = torch.empty((B, Hq, cap), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    scale = 1 / math.sqrt(D)
    for step in range(steps):
        t = N + step
        t_dev.fill_(t)
        kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_FREE_SLOT, ks[step], vs[step], t=t_dev,
                              free_slot=free, pos=pos, score=sc)
        K0, V0 = f64(Kc), f64(Vc)
        pos0, s0 = pos.cpu().numpy().astype(np.int64), sc.cpu().numpy().astype(np.float64)
        out = kvc.kvc_decode_attn(qs[step], Kc, Vc, scale=scale, n_valid=cap, logits=logits,
                                  lse=lse)
        kvc.kvc_h2o_accumulate_evict_gqa(logits, lse, sc, pos, free, n_slots=cap, t=t_dev,
                                         L_local=L_local, budget=budget)
        assert kvc.kvc_device_status() == 0
        o_gpu, s_gpu, f_gpu = out.cpu().numpy(), sc.cpu().numpy(), free.cpu().numpy()
        for b in range(B):
            for kh in range(Hkv):
                qg = f64(qs[step, b, kh * G:(kh + 1) * G])
                o_ref, s_ref, _ = oracle.h2o_step_group(qg, K0[b, kh], V0[b, kh], pos0[b, kh],
                                                        s0[b, kh], t, L_local, budget, scale)
                assert_close(o_gpu[b, kh * G:(kh + 1) * G], o_ref, TOL[dtype],
                             f"out step {step} ({b},{kh})")
                assert_rel(s_gpu[b, kh], s_ref, 1e-4, 1e-5, f"s step {step} ({b},{kh})")
                ev = oracle.h2o_evict_f32(s_gpu[b, kh], pos0[b, kh], t, L_local)
                assert ev == int(f_gpu[b * Hkv + kh]), f"evictee step {step} ({b},{kh})"


@pytest.mark.parametrize("dtype,G", [(torch.float32, 1), (torch.bfloat16, 4)])
def test_h2o_streamed_prompt_teacher_forced(dtype, G):
    """The streamed-prompt reading of H2O: the prompt goes through the decode-time step token
    by token from an empty cache, eviction active as soon as the cache exceeds the budget.
    Tail appends fill the cache (len counts the tokens), then each token takes the slot the
    previous step freed; decode and score update run over the tokens held so far.  Every step
    from the GPU's own state against the oracle's step: output, scores, evictee (exact, given
    the GPU's fp32 scores)."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, D, N, budget, L_local = 2, 2, 64, 150, 48, 24
    Hq = Hkv * G
    cap = budget + 1
    Kc = torch.zeros((B, Hkv, cap, D), device=dev, dtype=dtype)
    Vc = torch.zeros_like(Kc)
    pos = torch.full((B, Hkv, cap), -1, dtype=torch.int32, device=dev)
    sc = torch.zeros((B, Hkv, cap), device=dev)
    ln = torch.zeros(B * Hkv, dtype=torch.int32, device=dev)
    free = torch.zeros(B * Hkv, dtype=torch.int32, device=dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, N, 77 + G, dev, dtype)
    logits = torch.empty((B, Hq, cap), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    scale = 1 / math.sqrt(D)
    n_evicted = 0
    for t in range(N):
        t_dev.fill_(t)
        n = min(t + 1, cap)
        if t < cap:
            kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_TAIL, ks[t], vs[t], t=t_dev, len=ln,
                                  pos=pos, score=sc)
        else:
            kvc.kvc_stream_append(Kc, Vc, kvc.KVC_APPEND_FREE_SLOT, ks[t], vs[t], t=t_dev,
                                  free_slot=free, pos=pos, score=sc)
        K0, V0 = f64(Kc), f64(Vc)
        pos0, s0 = pos.cpu().numpy().astype(np.int64), sc.cpu().numpy().astype(np.float64)
        out = kvc.kvc_decode_attn(qs[t], Kc, Vc, scale=scale, n_valid=n, logits=logits, lse=lse)
        kvc.kvc_h2o_accumulate_evict_gqa(logits, lse, sc, pos, free, n_slots=n, t=t_dev,
                                         L_local=L_local, budget=budget)
        assert kvc.kvc_device_status() == 0, f"t={t}"
        o_gpu, s_gpu, f_gpu = out.cpu().numpy(), sc.cpu().numpy(), free.cpu().numpy()
        for b in range(B):
            for kh in range(Hkv):
                qg = f64(qs[t, b, kh * G:(kh + 1) * G])
                o_ref, s_ref, ev_ref = oracle.h2o_step_group(qg, K0[b, kh, :n], V0[b, kh, :n],
                                                             pos0[b, kh, :n], s0[b, kh, :n], t,
                                                             L_local, budget, scale)
                assert_close(o_gpu[b, kh * G:(kh + 1) * G], o_ref, TOL[dtype], f"out t={t}")
                assert_rel(s_gpu[b, kh, :n], s_ref, 1e-4, 1e-5, f"s t={t} ({b},{kh})")
                if n > budget:
                    ev = oracle.h2o_evict_f32(s_gpu[b, kh, :n], pos0[b, kh, :n], t, L_local)
                    assert ev == int(f_gpu[b * Hkv + kh]), f"evictee t={t} ({b},{kh})"
                    n_evicted += 1
                else:
                    assert ev_ref == -1
    assert n_evicted == B * Hkv * (N - budget)
    # the cache ends with the L_local newest prompt tokens and budget - L_local older ones
    p_end = pos.cpu().numpy()
    for b in range(B):
        for kh in range(Hkv):
            held = sorted(int(x) for x in p_end[b, kh])
            assert held[-L_local:] == list(range(N - L_local, N))


@pytest.mark.parametrize("dtype,D,G", [(torch.float32, 64, 4), (torch.bfloat16, 128, 4),
                                       (torch.bfloat16, 128, 2)])
def test_h2o_prompt_select_grouped_query(dtype, D, G):
    """H2O's prompt compression on a grouped-query cache: each KV head's column sums added over
    its query heads (against the oracle, relative 1e-4; G * N in total), the kept positions
    bit-exact given the GPU's scores, the kept scores gathered from them."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, N, L_local, K_hh = 2, 2, 333, 40, 60
    Hq = Hkv * G
    q, k, v = I.prompt_qkv(B, Hq, Hkv, N, D, 123 + D + G, dev, dtype)
    scale = 1 / math.sqrt(D)
    s_full = torch.empty((B, Hkv, N), device=dev)
    idx, score = kvc.kvc_h2o_prefill_select_gqa(q, k, seq_len=N, L_local=L_local, K_hh=K_hh,
                                                scale=scale, s_full=s_full)
    assert kvc.kvc_device_status() == 0
    sf, ix, sc = s_full.cpu().numpy(), idx.cpu().numpy(), score.cpu().numpy()
    for b in range(B):
        for kh in range(Hkv):
            ref = oracle.h2o_prompt_scores_group(f64(q[b, kh * G:(kh + 1) * G]), f64(k[b, kh]),
                                                 scale)
            assert_rel(sf[b, kh], ref, 1e-4, 1e-5, f"group column sums ({b},{kh})")
            assert abs(float(sf[b, kh].sum()) - G * N) < 1e-3 * G * N
            assert np.array_equal(oracle.h2o_prompt_select(sf[b, kh].astype(np.float64), L_local,
                                                           K_hh), ix[b, kh]), "stage-exact"
            assert np.array_equal(sc[b, kh], sf[b, kh][ix[b, kh]])
            # end to end against the oracle's own selection: the recent quota exactly, the heavy
            # hitters except where the oracle scores tie within the band of the K_hh-th
            ref_idx = oracle.h2o_prompt_select(ref, L_local, K_hh)
            assert list(ix[b, kh][K_hh:]) == list(ref_idx[K_hh:]) == list(range(N - L_local, N))
            topk_sets_agree(ix[b, kh][:K_hh], ref_idx[:K_hh], ref[:N - L_local], K_hh)
