"""GPU parity: block-level eviction over page tables (paged append, paged decode attention,
block score accumulation and release), through the C ABI, against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, assert_close, assert_rel, cuda_or_skip, f64, lib
from kv_cache_compression_kvc_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _gather(k_pool, v_pool, table, n, bs):
    """K, V [Hkv, n, D] of one sequence in page-table order (host arrays)."""
    nb = (n + bs - 1) // bs
    ks, vs = [], []
    for i in range(nb):
        fill = min(bs, n - i * bs)
        ks.append(k_pool[:, table[i], :fill])
        vs.append(v_pool[:, table[i], :fill])
    D = k_pool.shape[-1]
    if not ks:
        return np.zeros((k_pool.shape[0], 0, D)), np.zeros((k_pool.shape[0], 0, D))
    return np.concatenate(ks, axis=1), np.concatenate(vs, axis=1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D,G,bs", [(64, 1, 16), (128, 1, 32), (128, 4, 16), (256, 2, 32),
                                    (64, 8, 32)])
def test_paged_decode_matches_oracle(dtype, D, G, bs):
    """Random page tables over a shuffled pool: ragged lengths (empty, one token, partial and
    full last blocks, the whole table), logits at logical slots and log-sum-exp."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, mb = 5, 2, 9
    Hq = Hkv * G
    n_pool = B * mb + 3
    seed = 200 + D + G + bs
    kp = I.randn((Hkv, n_pool, bs, D), seed, dev, dtype)
    vp = I.randn((Hkv, n_pool, bs, D), seed + 1, dev, dtype)
    q = I.randn((B, Hq, D), seed + 2, dev, dtype)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(n_pool)[:B * mb].reshape(B, mb)
    lens = np.array([0, 1, bs * 3, bs * 4 + 5, mb * bs])
    table = torch.tensor(perm, dtype=torch.int32, device=dev)
    nbl = torch.tensor((lens + bs - 1) // bs, dtype=torch.int32, device=dev)
    ln = torch.tensor(lens, dtype=torch.int32, device=dev)
    score = torch.zeros((B, mb), device=dev)
    pool = kvc.block_pool_view(kp, vp)
    pt = kvc.page_table_view(table, nbl, ln, score)
    scale = 1 / math.sqrt(D)
    logits = torch.full((B, Hq, mb * bs), float("nan"), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    out = kvc.kvc_decode_attn_paged(q, pool, pt, scale=scale, logits=logits, lse=lse)
    out2 = kvc.kvc_decode_attn_paged(q, pool, pt, scale=scale, flags=kvc.KVC_DECODE_KV_SETTLED)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    assert torch.equal(out, out2)
    kph, vph, qh = f64(kp), f64(vp), f64(q)
    o, lg, ls = out.cpu().numpy(), logits.cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        K, V = _gather(kph, vph, perm[b], int(lens[b]), bs)
        for h in range(Hq):
            ro, rl, rls = oracle.attend(qh[b, h], K[h // G], V[h // G], scale)
            assert_close(o[b, h], ro, TOL[dtype], f"out b={b} h={h}")
            if lens[b] == 0:
                assert np.all(o[b, h] == 0) and math.isinf(float(ls[b, h]))
                continue
            assert_close(lg[b, h, :lens[b]], rl, 1e-4, f"logits b={b} h={h}")
            assert abs(float(ls[b, h]) - rls) <= 1e-4 * max(1.0, abs(rls))


@pytest.mark.parametrize("dtype,D,G,bs,budget,recent", [
    (torch.float32, 64, 2, 16, 4, 2),
    (torch.bfloat16, 128, 1, 32, 3, 1),
    (torch.bfloat16, 64, 4, 16, 5, 3),
])
def test_block_eviction_steps_teacher_forced(dtype, D, G, bs, budget, recent):
    """Token by token from empty caches: paged append, paged decode with logits, then the block
    update.  Every step is checked from the GPU's own state: the output against the oracle's
    block step, the accumulated scores (a second call on a copy of the state with no budget
    gives them before the release) against the oracle's, and the released block exactly
    against the oracle's decision on those fp32 scores; the table, scores, lengths and free
    stack after the release must be the pre-release state with that one block moved out."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv = 3, 2
    Hq = Hkv * G
    mb = budget + 1
    n_pool = B * mb + 2
    T = (budget + 3) * bs + 5
    scale = 1 / math.sqrt(D)
    kp = torch.zeros((Hkv, n_pool, bs, D), device=dev, dtype=dtype)
    vp = torch.zeros_like(kp)
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, T, 300 + D + bs, dev, dtype)
    rng = np.random.default_rng(5)
    ids = torch.tensor(rng.permutation(n_pool), dtype=torch.int32, device=dev)
    top = torch.tensor([n_pool], dtype=torch.int32, device=dev)
    table = torch.full((B, mb), -1, dtype=torch.int32, device=dev)
    nbl = torch.zeros(B, dtype=torch.int32, device=dev)
    ln = torch.zeros(B, dtype=torch.int32, device=dev)
    score = torch.zeros((B, mb), device=dev)
    pos = torch.full((n_pool, bs), -1, dtype=torch.int32, device=dev)
    t_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    pool = kvc.block_pool_view(kp, vp)
    pt = kvc.page_table_view(table, nbl, ln, score)
    fp = kvc.free_pool_view(ids, top)
    logits = torch.zeros((B, Hq, mb * bs), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    released = torch.empty(B, dtype=torch.int32, device=dev)
    n_released = 0
    for t in range(T):
        t_dev.fill_(t)
        kvc.kvc_paged_append(pool, pt, fp, ks[t], vs[t], t=t_dev, pos=pos)
        out = kvc.kvc_decode_attn_paged(qs[t], pool, pt, scale=scale, logits=logits, lse=lse)
        s_before = score.cpu().numpy()               # after the append, before accumulation
        pre = [x.clone() for x in (table, nbl, ln, score)]
        pre_top = top.clone()
        pt_copy = kvc.page_table_view(*pre)
        kvc.kvc_block_accumulate_evict(logits, lse, pt_copy, fp, block_size=bs,
                                       budget_blocks=10 ** 6, recent_blocks=recent)
        kvc.kvc_block_accumulate_evict(logits, lse, pt, fp, block_size=bs, budget_blocks=budget,
                                       recent_blocks=recent, released=released)
        assert kvc.kvc_device_status() == 0, f"t={t}"
        acc = pre[3].cpu().numpy()                   # GPU scores after accumulation
        tab0, nb0, n0 = pre[0].cpu().numpy(), pre[1].cpu().numpy(), pre[2].cpu().numpy()
        rel = released.cpu().numpy()
        kph, vph = f64(kp), f64(vp)
        o = out.cpu().numpy()
        for b in range(B):
            nb, n = int(nb0[b]), int(n0[b])
            assert nb == (n + bs - 1) // bs and 0 < n <= mb * bs
            K, V = _gather(kph, vph, tab0[b], n, bs)
            # the oracle's step from zero scores gives this step's increments
            ro, rs, _ = oracle.block_step(f64(qs[t, b]), K, V, np.zeros(nb), bs, budget, recent,
                                          scale)
            assert_close(o[b], ro, TOL[dtype], f"out t={t} b={b}")
            inc = acc[b, :nb].astype(np.float64) - s_before[b, :nb]
            tol = 1e-4 * np.abs(rs) + 2.5e-7 * np.abs(acc[b, :nb]) + 1e-6
            assert np.all(np.abs(inc - rs) <= tol), (t, b, inc, rs)
            want = oracle.block_evict_f32(acc[b, :nb], budget, recent)
            assert int(rel[b]) == want, (t, b, int(rel[b]), want)
            # state after the release
            tab1, sc1 = table[b].cpu().numpy(), score[b].cpu().numpy()
            if want < 0:
                assert np.array_equal(tab1[:nb], tab0[b, :nb]) and int(nbl[b]) == nb
                assert np.array_equal(sc1[:nb], acc[b, :nb]) and int(ln[b]) == n
            else:
                n_released += 1
                keep = [i for i in range(nb) if i != want]
                assert np.array_equal(tab1[:nb - 1], tab0[b, keep])
                assert np.array_equal(sc1[:nb - 1], acc[b, keep])
                assert int(nbl[b]) == nb - 1 and int(ln[b]) == n - bs
        # pushes: the released physical ids are on the stack above the old top
        n_push = int((rel >= 0).sum())
        assert int(top) == int(pre_top) + n_push
        pushed = sorted(ids[int(pre_top):int(top)].cpu().tolist())
        assert pushed == sorted(int(tab0[b, rel[b]]) for b in range(B) if rel[b] >= 0)
    assert n_released > 0
    # every physical block is in exactly one place: a page table or the free stack
    live = [int(x) for b in range(B) for x in table[b, :int(nbl[b])].cpu().tolist()]
    free = ids[:int(top)].cpu().tolist()
    assert sorted(live + free) == list(range(n_pool))
    # the positions in each table are increasing text positions ending at the last token
    pos_h = pos.cpu().numpy()
    for b in range(B):
        seq = []
        for i in range(int(nbl[b])):
            fill = min(bs, int(ln[b]) - i * bs)
            seq += pos_h[int(table[b, i]), :fill].tolist()
        assert seq == sorted(seq) and seq[-1] == T - 1 and len(seq) == int(ln[b])


def test_block_scores_accumulate_like_the_oracle():
    """Several steps with no release: the GPU's block scores against the oracle's running block
    scores (relative 1e-4), on grouped-query heads with a partly filled last block."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, G, D, bs, mb = 2, 2, 4, 64, 16, 6
    Hq = Hkv * G
    n_pool = B * mb
    dtype = torch.float32
    kp = torch.zeros((Hkv, n_pool, bs, D), device=dev, dtype=dtype)
    vp = torch.zeros_like(kp)
    T = mb * bs - 3
    qs, ks, vs = I.decode_qkv(B, Hq, Hkv, D, T, 401, dev, dtype)
    ids = torch.arange(n_pool, dtype=torch.int32, device=dev)
    top = torch.tensor([n_pool], dtype=torch.int32, device=dev)
    table = torch.full((B, mb), -1, dtype=torch.int32, device=dev)
    nbl = torch.zeros(B, dtype=torch.int32, device=dev)
    ln = torch.zeros(B, dtype=torch.int32, device=dev)
    score = torch.zeros((B, mb), device=dev)
    pool, pt = kvc.block_pool_view(kp, vp), kvc.page_table_view(table, nbl, ln, score)
    fp = kvc.free_pool_view(ids, top)
    logits = torch.zeros((B, Hq, mb * bs), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    s_ref = [np.zeros(0) for _ in range(B)]
    scale = 1 / math.sqrt(D)
    for t in range(T):
        kvc.kvc_paged_append(pool, pt, fp, ks[t], vs[t])
        kvc.kvc_decode_attn_paged(qs[t], pool, pt, scale=scale, logits=logits, lse=lse)
        kvc.kvc_block_accumulate_evict(logits, lse, pt, fp, block_size=bs, budget_blocks=mb,
                                       recent_blocks=1)
        kph, vph = f64(kp), f64(vp)
        tab = table.cpu().numpy()
        for b in range(B):
            n = t + 1
            nb = (n + bs - 1) // bs
            s_ref[b] = np.concatenate([s_ref[b], np.zeros(nb - len(s_ref[b]))])
            K, V = _gather(kph, vph, tab[b], n, bs)
            _, s_ref[b], ev = oracle.block_step(f64(qs[t, b]), K, V, s_ref[b], bs, mb, 1, scale)
            assert ev == -1
    assert kvc.kvc_device_status() == 0
    for b in range(B):
        nb = len(s_ref[b])
        assert_rel(score[b, :nb].cpu().numpy(), s_ref[b], 1e-4, 1e-5, f"scores b={b}")
        assert abs(float(score[b, :nb].sum()) - Hq * T) <= 1e-3 * Hq * T


def test_paged_append_reports_an_empty_pool():
    """A sequence that needs a block when the free stack is empty is skipped and the device
    code says so (a range check, not a fault); the others are appended."""
    dev = cuda_or_skip()
    kvc = lib()
    B, Hkv, D, bs, mb = 2, 1, 64, 16, 2
    kp = torch.zeros((Hkv, 1, bs, D), device=dev)
    vp = torch.zeros_like(kp)
    ids = torch.tensor([0], dtype=torch.int32, device=dev)
    top = torch.tensor([1], dtype=torch.int32, device=dev)
    table = torch.full((B, mb), -1, dtype=torch.int32, device=dev)
    nbl = torch.zeros(B, dtype=torch.int32, device=dev)
    ln = torch.zeros(B, dtype=torch.int32, device=dev)
    score = torch.zeros((B, mb), device=dev)
    pool, pt = kvc.block_pool_view(kp, vp), kvc.page_table_view(table, nbl, ln, score)
    fp = kvc.free_pool_view(ids, top)
    k = torch.ones((B, Hkv, D), device=dev)
    kvc.kvc_paged_append(pool, pt, fp, k, k)
    assert kvc.kvc_device_status() == 10                 # KVC_DEV_POOL_EMPTY
    assert sorted(ln.cpu().tolist()) == [0, 1] and int(top) == 0


@pytest.mark.parametrize("dtype,budget,recent", [(torch.float32, 7, 2), (torch.bfloat16, 5, 1),
                                                 (torch.bfloat16, 40, 3)])
def test_block_prompt_select_matches_oracle(dtype, budget, recent):
    """The prompt's one-shot block compression: integer-valued per-token scores make every block
    sum exact (ties included), so the kept blocks, their order and scores must equal the
    oracle's, the pool blocks must hold the kept prompt rows bit for bit, the free stack must
    have given each sequence distinct ids, and a decode over the result must equal attention
    over the kept tokens.  budget 40 keeps the whole 19-block prompt."""
    dev = cuda_or_skip()
    kvc = lib()
    B, H, D, N, bs = 2, 3, 64, 300, 16
    nblk = (N + bs - 1) // bs
    n_keep = min(budget, nblk)
    mb = max(budget, nblk) + 1
    n_pool = B * mb + 3
    rng = np.random.default_rng(budget)
    s_np = rng.integers(0, 4, size=(B, H, N)).astype(np.float32)
    s = torch.tensor(s_np, device=dev)
    kpr = I.randn((B, H, N + 5, D), 41, dev, dtype)
    vpr = I.randn((B, H, N + 5, D), 42, dev, dtype)
    kp = torch.zeros((H, n_pool, bs, D), device=dev, dtype=dtype)
    vp = torch.zeros_like(kp)
    ids = torch.tensor(rng.permutation(n_pool), dtype=torch.int32, device=dev)
    top = torch.tensor([n_pool], dtype=torch.int32, device=dev)
    table = torch.full((B, mb), -1, dtype=torch.int32, device=dev)
    nbl = torch.zeros(B, dtype=torch.int32, device=dev)
    ln = torch.zeros(B, dtype=torch.int32, device=dev)
    score = torch.zeros((B, mb), device=dev)
    pool, pt = kvc.block_pool_view(kp, vp), kvc.page_table_view(table, nbl, ln, score)
    fp = kvc.free_pool_view(ids, top)
    kvc.kvc_block_prompt_select(s, kpr, vpr, pool, pt, fp, seq_len=N, budget_blocks=budget,
                                recent_blocks=recent)
    assert kvc.kvc_device_status() == 0
    assert nbl.cpu().tolist() == [n_keep] * B
    assert ln.cpu().tolist() == [(n_keep - 1) * bs + (N - (nblk - 1) * bs)] * B
    assert int(top) == n_pool - B * n_keep
    tab, sc = table.cpu().numpy(), score.cpu().numpy()
    used = tab[:, :n_keep].flatten().tolist()
    assert len(set(used)) == len(used) and set(used) <= set(ids.cpu().tolist()[int(top):])
    kp_h, vp_h, kpr_h, vpr_h = kp.cpu(), vp.cpu(), kpr.cpu(), vpr.cpu()
    q = I.randn((B, H, D), 43, dev, dtype)
    out = kvc.kvc_decode_attn_paged(q, pool, pt, scale=1 / math.sqrt(D)).cpu().numpy()
    for b in range(B):
        keep, bsc = oracle.block_prompt_select(s_np[b].astype(np.float64), bs, budget, recent)
        assert len(keep) == n_keep
        assert np.array_equal(sc[b, :n_keep], bsc[keep].astype(np.float32))
        toks = []
        for e, i in enumerate(keep):
            fill = min(bs, N - i * bs)
            phys = int(tab[b, e])
            assert torch.equal(kp_h[:, phys, :fill], kpr_h[b, :, i * bs:i * bs + fill])
            assert torch.equal(vp_h[:, phys, :fill], vpr_h[b, :, i * bs:i * bs + fill])
            toks += list(range(i * bs, i * bs + fill))
        for h in range(H):
            ref, _, _ = oracle.attend(f64(q[b, h]), f64(kpr[b, h, toks]), f64(vpr[b, h, toks]),
                                      1 / math.sqrt(D))
            assert_close(out[b, h], ref, TOL[dtype], f"decode over the kept prompt b={b} h={h}")
