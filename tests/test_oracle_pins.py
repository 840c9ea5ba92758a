"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: a worked example the pages
print (tests/golden/), a closed form, an invariant, a library routine on a special case, or
brute force on tiny inputs.  The cases are chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, a flipped tie rule) fails one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _sdpa(Q, K, V, scale, causal=True):
    """Library attention (torch, fp64) over [n, D] rows."""
    q = torch.from_numpy(np.asarray(Q, dtype=np.float64))[None, None]
    k = torch.from_numpy(np.asarray(K, dtype=np.float64))[None, None]
    v = torch.from_numpy(np.asarray(V, dtype=np.float64))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    return o[0, 0].numpy()


def _causal_probs(Q, K, scale):
    """Library softmax (torch, fp64) of the causal score matrix, rows = queries."""
    q = torch.from_numpy(np.asarray(Q, dtype=np.float64))
    k = torch.from_numpy(np.asarray(K, dtype=np.float64))
    s = (q @ k.T) * scale
    n, m = s.shape
    # query r sits at text position (m - n + r)
    mask = torch.arange(m)[None, :] > (m - n + torch.arange(n))[:, None]
    s = s.masked_fill(mask, float("-inf"))
    return torch.softmax(s, dim=-1).numpy()


def _rope_complex(x, pos, theta=10000.0):
    """RoPE as a complex multiplication: pair (x_i, x_{i+D/2}) times exp(i*pos*theta^(-2i/D))."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    z = x[..., :h] + 1j * x[..., h:]
    w = np.exp(1j * pos * theta ** (-2.0 * np.arange(h) / D))
    r = z * w
    return np.concatenate([r.real, r.imag], axis=-1)


# ---------------------------------------------------------------------------- memory model
def test_kv_bytes_worked_example():
    g = _golden("kv_bytes_qwen.json")
    for c in g["cases"]:
        got = oracle.kv_bytes(c["n_layers"], c["n_heads_kv"], c["d_head"], c["seq_len"],
                              c["bytes"], c["batch"])
        assert got == c["expect"], c["what"]
    # the page's two headline figures in binary units
    assert oracle.kv_bytes(64, 4, 256, 262144, 2, 1) == 64 * 2**30
    assert oracle.kv_bytes(16, 4, 256, 262144, 2, 1) == 16 * 2**30


def test_kv_bytes_scales_with_batch_and_is_linear():
    base = oracle.kv_bytes(32, 8, 128, 1000, 2, 1)
    assert oracle.kv_bytes(32, 8, 128, 1000, 2, 16) == 16 * base
    assert oracle.kv_bytes(32, 8, 128, 2000, 2, 1) == 2 * base


# ---------------------------------------------------------------------------- PyramidKV
@pytest.mark.parametrize("n_layers,target", [(16, 8192), (32, 5243), (7, 1001), (2, 3), (5, 0)])
def test_pyramid_total_and_linear_shape(n_layers, target):
    b = oracle.pyramid_budgets(n_layers, target, 4, 1)
    # sum_l B_l = N_L * B_target, exactly (Alocação piramidal com o PyramidKV)
    assert int(b.sum()) == n_layers * target
    # linear decrease: each B_l within one slot of the exact rational ramp
    exact = [2 * target * (4 * (n_layers - 1 - l) + l) / (5 * (n_layers - 1))
             for l in range(n_layers)]
    assert all(abs(int(bl) - e) < 1.0 for bl, e in zip(b, exact))
    assert all(b[i] >= b[i + 1] for i in range(n_layers - 1))


def test_pyramid_long_context_workload():
    b = oracle.pyramid_budgets(16, 8192, 4, 1)
    assert int(b.sum()) == 131072
    assert b[0] == 13107 and b[-1] == 3277            # 1.6x and 0.4x of 8192, ratio 4
    diffs = np.diff(b.astype(np.int64))
    assert diffs.min() >= -656 and diffs.max() <= -654  # constant step 655.36 up to rounding


def test_pyramid_degenerate():
    assert list(oracle.pyramid_budgets(1, 77, 4, 1)) == [77]
    assert list(oracle.pyramid_budgets(6, 50, 1, 1)) == [50] * 6      # ratio 1: uniform
    up = oracle.pyramid_budgets(5, 100, 1, 4)                        # ratio < 1: increasing
    assert int(up.sum()) == 500 and all(up[i] <= up[i + 1] for i in range(4))


# ---------------------------------------------------------------------------- RoPE
def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(1)
    for D in (8, 64, 128):
        x = rng.standard_normal(D)
        for pos in (0, 1, 7, 2048, 100003):
            # the angle pos*theta^(-2i/D) carries ~1e-16 relative rounding on either side
            tol = 1e-13 * max(1, pos) * math.sqrt(D)
            assert np.allclose(oracle.rope(x, pos), _rope_complex(x, pos), atol=tol, rtol=0)


def test_rope_basis_vector_and_invariants():
    D = 16
    e0 = np.zeros(D); e0[0] = 1.0
    y = oracle.rope(e0, 1)
    assert y[0] == pytest.approx(math.cos(1.0)) and y[D // 2] == pytest.approx(math.sin(1.0))
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    assert np.allclose(oracle.rope(q, 0), q)
    assert np.linalg.norm(oracle.rope(k, 12345)) == pytest.approx(np.linalg.norm(k))
    # (R(a)q).(R(b)k) depends only on a - b
    d1 = oracle.rope(q, 10) @ oracle.rope(k, 3)
    d2 = oracle.rope(q, 107) @ oracle.rope(k, 100)
    assert d1 == pytest.approx(d2, abs=1e-10)


# ---------------------------------------------------------------------------- attention
def test_attend_single_key_returns_value():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal(8), rng.standard_normal((1, 8)), rng.standard_normal((1, 8))
    out, logits, lse = oracle.attend(q, k, v, 0.5)
    assert np.array_equal(out, v[0])
    assert lse == pytest.approx(0.5 * float(q @ k[0]))
    assert logits[0] == pytest.approx(0.5 * float(q @ k[0]))


def test_attend_empty_cache():
    out, logits, lse = oracle.attend(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert np.all(out == 0) and lse == -math.inf and logits.shape == (0,)


def test_attend_softmax_rows_sum_to_one_and_match_library():
    rng = np.random.default_rng(4)
    D, n = 32, 57
    q, K, V = rng.standard_normal(D), rng.standard_normal((n, D)), rng.standard_normal((n, D))
    out, logits, lse = oracle.attend(q, K, V, 1 / math.sqrt(D))
    assert np.exp(logits - lse).sum() == pytest.approx(1.0, abs=1e-13)
    ref = _sdpa(q[None], K, V, 1 / math.sqrt(D), causal=False)[0]
    assert np.allclose(out, ref, atol=1e-12, rtol=0)


def test_decode_is_exact_causal_attention():
    """Incremental decode over a growing cache reproduces every row of causal attention."""
    rng = np.random.default_rng(5)
    N, D = 48, 16
    Q, K, V = (rng.standard_normal((N, D)) for _ in range(3))
    full = _sdpa(Q, K, V, 1 / math.sqrt(D), causal=True)
    for t in range(N):
        o, _, _ = oracle.attend(Q[t], K[:t + 1], V[:t + 1], 1 / math.sqrt(D))
        assert np.max(np.abs(o - full[t])) <= 1e-12


# ---------------------------------------------------------------------------- StreamingLLM
def test_stream_positions_worked_example():
    g = _golden("stream_positions.json")
    tok, cpos, qpos = oracle.stream_window(g["t"], g["S"], g["W"])
    assert list(tok) == g["attended_tokens"]
    assert list(cpos) == g["positions"]
    assert qpos == g["query_position"]
    assert list(tok[:-1]) == g["cached_tokens"]


def test_stream_positions_never_exceed_window_long_stream():
    S, W = 4, 60
    for t in (0, 3, 4, 63, 64, 65, 1000, 4_000_000):
        tok, cpos, qpos = oracle.stream_window(t, S, W)
        assert len(tok) == min(t + 1, S + W + 1)          # O(W + 4) memory
        assert qpos == min(t, S + W) and cpos.max() == qpos
        assert list(tok[:min(S, t + 1)]) == list(range(min(S, t + 1)))   # sinks fixed


def test_stream_ring_slots_never_clobber_live_tokens():
    S, W = 4, 5
    for t in range(0, 60):
        tok, _, _ = oracle.stream_window(t, S, W)
        slots = [oracle.stream_slot(int(a), S, W) for a in tok]
        assert len(set(slots)) == len(slots)              # attended tokens own distinct slots
        assert all(0 <= s < S + W + 1 for s in slots)
        assert oracle.stream_slot(t, S, W) == slots[-1]


def test_stream_decode_without_eviction_is_rotated_causal_attention():
    rng = np.random.default_rng(6)
    S, W, D, N = 4, 30, 16, 30
    Qp, Kp, V = (rng.standard_normal((N, D)) for _ in range(3))
    scale = 1 / math.sqrt(D)
    Qr = np.stack([_rope_complex(Qp[i], i) for i in range(N)])
    Kr = np.stack([_rope_complex(Kp[i], i) for i in range(N)])
    full = _sdpa(Qr, Kr, V, scale, causal=True)
    for t in range(N):                                     # S + W >= t: nothing evicted
        o = oracle.stream_decode(t, S, W, Qp[t], Kp, V, scale)
        assert np.max(np.abs(o - full[t])) <= 1e-10


def test_stream_decode_with_eviction_uses_cache_positions():
    rng = np.random.default_rng(7)
    S, W, D, t = 4, 3, 8, 9
    Kp, V = rng.standard_normal((t + 1, D)), rng.standard_normal((t + 1, D))
    q = rng.standard_normal(D)
    scale = 1 / math.sqrt(D)
    kept = [0, 1, 2, 3, 6, 7, 8, 9]                        # the worked example's cache + token
    Kr = np.stack([_rope_complex(Kp[a], p) for p, a in enumerate(kept)])
    ref = _sdpa(_rope_complex(q, 7)[None], Kr, V[kept], scale, causal=False)[0]
    o = oracle.stream_decode(t, S, W, q, Kp, V, scale)
    assert np.max(np.abs(o - ref)) <= 1e-12
    # text positions (the wrong reading) give a different answer
    Kt = np.stack([_rope_complex(Kp[a], a) for a in kept])
    wrong = _sdpa(_rope_complex(q, 9)[None], Kt, V[kept], scale, causal=False)[0]
    assert np.max(np.abs(o - wrong)) > 1e-6


def test_window_attention_special_case():
    """S = 0: plain window attention over the W most recent tokens plus the current one."""
    tok, cpos, qpos = oracle.stream_window(20, 0, 5)
    assert list(tok) == list(range(15, 21)) and qpos == 5


def test_alibi_worked_example_bias_is_continuous():
    """The pages' cache [0,1,2,3,6,7,8] decoding token 9 under ALiBi: with q = 0 the logits are
    the bias alone, -slope * (7 - r) over in-cache positions r = 0..7 -- one unbroken line, not
    the text distances 9,8,7,6,3,2,1,0 with their jump over the evicted tokens 4 and 5."""
    g = _golden("stream_positions.json")
    S, W, t, D = g["S"], g["W"], g["t"], 8
    rng = np.random.default_rng(31)
    hk, hv = rng.standard_normal((t + 1, D)), rng.standard_normal((t + 1, D))
    slope = 0.375
    _, logits, lse = oracle.stream_decode_alibi(t, S, W, np.zeros(D), hk, hv, 0.5, slope)
    qp = g["query_position"]
    want = [-slope * (qp - p) for p in g["positions"]]
    assert list(logits) == want                               # exact: 0 * anything + bias
    text = [-slope * (t - a) for a in g["attended_tokens"]]
    assert list(logits) != text
    rho = math.exp(-slope)                                    # log of a geometric sum
    assert abs(lse - math.log((1 - rho ** 8) / (1 - rho))) <= 1e-14


def test_alibi_geometric_closed_form_after_eviction():
    """Equal keys make the weights proportional to rho^distance (rho = e^-slope) over the
    n = S + W + 1 attended tokens: the mean in-cache position has a closed form."""
    S, W, D, t = 4, 20, 6, 100
    rng = np.random.default_rng(32)
    k = rng.standard_normal(D)
    hk = np.tile(k, (t + 1, 1))
    hv = np.zeros((t + 1, D))
    hv[:, 0] = 1.0
    for a in range(t + 1):                                    # in-cache position of token a
        hv[a, 1] = a if a < S else (S + a - (t - W) if a >= t - W else -1e9)
    slope, n = 0.3, S + W + 1
    out, _, _ = oracle.stream_decode_alibi(t, S, W, rng.standard_normal(D), hk, hv, 0.25, slope)
    rho = math.exp(-slope)
    mean_d = rho * (1 - n * rho ** (n - 1) + (n - 1) * rho ** n) / ((1 - rho) * (1 - rho ** n))
    assert abs(out[0] - 1.0) <= 1e-14
    assert abs(out[1] - ((n - 1) - mean_d)) <= 1e-12


def test_alibi_reduces_to_library_attention():
    """Slope 0: window attention over the attended tokens.  No eviction (t <= S + W): in-cache
    and text positions coincide, so ALiBi is causal attention with the additive bias
    -slope * (t - j) (library attention with a float mask)."""
    rng = np.random.default_rng(33)
    S, W, D = 4, 9, 16
    T = 40
    hk, hv = rng.standard_normal((T, D)), rng.standard_normal((T, D))
    q = rng.standard_normal(D)
    scale = 1 / math.sqrt(D)
    t = T - 1
    tok, _, _ = oracle.stream_window(t, S, W)
    o, _, _ = oracle.stream_decode_alibi(t, S, W, q, hk, hv, scale, 0.0)
    ref = _sdpa(q[None], hk[tok], hv[tok], scale, causal=False)[0]
    assert np.max(np.abs(o - ref)) <= 1e-12
    slope, t = 0.125, S + W                                   # the last step with no eviction
    o, _, _ = oracle.stream_decode_alibi(t, 4, W, q, hk, hv, scale, slope)
    bias = torch.tensor([[-slope * (t - j) for j in range(t + 1)]], dtype=torch.float64)
    qq = torch.from_numpy(q)[None, None, None]
    kk = torch.from_numpy(hk[:t + 1])[None, None]
    vv = torch.from_numpy(hv[:t + 1])[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=bias,
                                                           scale=scale)[0, 0, 0].numpy()
    assert np.max(np.abs(o - ref)) <= 1e-12


def test_alibi_steep_slope_attends_to_the_newest_token():
    rng = np.random.default_rng(34)
    S, W, D, t = 4, 7, 8, 30
    hk, hv = rng.standard_normal((t + 1, D)), rng.standard_normal((t + 1, D))
    o, _, _ = oracle.stream_decode_alibi(t, S, W, 0.1 * rng.standard_normal(D), hk, hv, 0.1, 80.0)
    assert np.max(np.abs(o - hv[t])) <= 1e-12


# ---------------------------------------------------------------------------- top-k
def _brute_topk(score, k):
    n = len(score)
    keep = [i for i in range(n)
            if sum(1 for j in range(n) if score[j] > score[i] or (score[j] == score[i] and j < i)) < k]
    return keep


def test_topk_rank_count_with_ties():
    rng = np.random.default_rng(8)
    for trial in range(200):
        n = int(rng.integers(1, 24))
        score = rng.integers(0, 5, size=n).astype(np.float64)      # many ties
        k = int(rng.integers(0, n + 2))
        got = oracle.topk_ascending(score, k)
        assert list(got) == _brute_topk(score, min(k, n))


def test_topk_exhaustive_tiny():
    for n in range(1, 7):
        for score in itertools.product([0.0, 1.0, 2.0], repeat=n):
            for k in range(n + 1):
                assert list(oracle.topk_ascending(np.array(score), k)) == _brute_topk(score, k)


# ---------------------------------------------------------------------------- SnapKV
def test_snapkv_obs_scores_match_library_softmax_and_sum_to_one():
    rng = np.random.default_rng(9)
    N, L, D = 70, 9, 16
    Q, K = rng.standard_normal((L, D)), rng.standard_normal((N, D))
    s = oracle.snapkv_obs_scores(Q, K, 1 / math.sqrt(D))
    P = _causal_probs(Q, K, 1 / math.sqrt(D))
    assert np.allclose(s, P.mean(axis=0), atol=1e-14, rtol=0)
    assert s.sum() == pytest.approx(1.0, abs=1e-13)           # mean of L rows summing to 1
    # the last window query sees every key, the first sees N-L+1 keys
    assert np.all(s[N - L + 1:] > 0) and np.all(s >= 0)


def test_pool1d_matches_convolution():
    rng = np.random.default_rng(10)
    for n in (1, 2, 4, 5, 13, 100):
        s = rng.random(n)
        for k in (1, 3, 5, 7):
            ref = np.convolve(s, np.ones(k) / k, mode="full")[(k - 1) // 2:(k - 1) // 2 + n]
            assert np.allclose(oracle.pool1d(s, k), ref, atol=1e-15, rtol=0)


def test_snapkv_select_identity_when_budget_covers_prompt():
    rng = np.random.default_rng(11)
    N, L, D, G = 40, 8, 8, 2
    idx, _, _ = oracle.snapkv_select(rng.standard_normal((G, L, D)), rng.standard_normal((N, D)),
                                     budget=N, scale=0.3)
    assert list(idx) == list(range(N))
    idx, _, _ = oracle.snapkv_select(rng.standard_normal((G, L, D)), rng.standard_normal((N, D)),
                                     budget=N + 5, scale=0.3)
    assert list(idx) == list(range(N))


def test_snapkv_select_plain_per_head_topk_special_case():
    """pool 1 and one head per group reduce steps 3-4 to a plain top-k of the window means."""
    rng = np.random.default_rng(12)
    N, L, D, budget = 64, 6, 8, 20
    Q, K = rng.standard_normal((1, L, D)), rng.standard_normal((N, D))
    idx, s, _ = oracle.snapkv_select(Q, K, budget, 0.35, pool_k=1)
    P = _causal_probs(Q[0], K, 0.35).mean(axis=0)
    expect = _brute_topk(P[:N - L], budget - L) + list(range(N - L, N))
    assert list(idx) == expect


def test_snapkv_select_group_max_and_pooling():
    rng = np.random.default_rng(13)
    N, L, D, G, budget = 90, 8, 8, 3, 30
    Q, K = rng.standard_normal((G, L, D)), rng.standard_normal((N, D))
    idx, s, score = oracle.snapkv_select(Q, K, budget, 0.4, pool_k=5)
    n = N - L
    pooled = [np.convolve(_causal_probs(Q[g], K, 0.4).mean(axis=0)[:n], np.ones(5) / 5,
                          mode="full")[2:2 + n] for g in range(G)]
    ref_score = np.max(np.stack(pooled), axis=0)
    assert np.allclose(score, ref_score, atol=1e-15, rtol=0)
    assert list(idx) == _brute_topk(ref_score, budget - L) + list(range(n, N))
    assert len(idx) == budget and np.all(np.diff(idx) > 0)


def test_snapkv_retention_figure():
    g = _golden("snapkv_retention.json")
    assert g["budget"] == math.ceil(g["fraction"] * g["N"])
    assert g["selected_prefix"] == g["budget"] - g["L_obs"]


def test_snapkv_stage_f32_replays_in_single_precision():
    rng = np.random.default_rng(14)
    G, n, L, budget = 2, 50, 4, 20
    s = rng.random((G, n)).astype(np.float32)
    s[:, 10:14] = s[:, 10:11]                       # plateaus: ties after pooling
    idx = oracle.snapkv_stage_f32(s, L, budget)
    pooled = []
    for g in range(G):
        row = np.zeros(n, dtype=np.float32)
        for i in range(n):
            acc = np.float32(0.0)
            for j in range(i - 2, i + 3):
                if 0 <= j < n:
                    acc = np.float32(acc + s[g, j])
            row[i] = np.float32(acc / np.float32(5.0))
        pooled.append(row)
    score = np.max(np.stack(pooled), axis=0)
    assert list(idx) == _brute_topk(score.astype(np.float64), budget - L) + list(range(n, n + L))


# ---------------------------------------------------------------------------- H2O
def test_h2o_prompt_scores_are_causal_column_sums():
    rng = np.random.default_rng(15)
    N, D = 33, 8
    Q, K = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    s = oracle.h2o_prompt_scores(Q, K, 0.3)
    P = _causal_probs(Q, K, 0.3)
    assert np.allclose(s, P.sum(axis=0), atol=1e-13, rtol=0)
    assert s.sum() == pytest.approx(N, abs=1e-11)           # every row sums to 1


def test_h2o_prompt_select_recent_quota_plus_heavy_hitters():
    rng = np.random.default_rng(16)
    for trial in range(50):
        N = int(rng.integers(5, 40))
        L_local, K_hh = int(rng.integers(0, 6)), int(rng.integers(0, 6))
        s = rng.integers(0, 4, size=N).astype(np.float64)
        idx = oracle.h2o_prompt_select(s, L_local, K_hh)
        if N <= L_local + K_hh:
            assert list(idx) == list(range(N))
            continue
        old = N - L_local
        assert list(idx) == _brute_topk(s[:old], K_hh) + list(range(old, N))


def _run_h2o(N, steps, D, budget, L_local, seed):
    """Oracle H2O over a prompt and `steps` decode tokens; returns the per-step records."""
    rng = np.random.default_rng(seed)
    T = N + steps
    Q, K, V = (rng.standard_normal((T, D)) for _ in range(3))
    scale = 1 / math.sqrt(D)
    s_prompt = oracle.h2o_prompt_scores(Q[:N], K[:N], scale)
    K_hh = budget - L_local
    kept = list(oracle.h2o_prompt_select(s_prompt, L_local, K_hh))
    evicted_mass = float(s_prompt.sum() - s_prompt[kept].sum())
    pos = kept[:]
    s = [float(s_prompt[j]) for j in kept]
    records = []
    for t in range(N, T):
        pos.append(t); s.append(0.0)                       # append with s = 0
        out, s_new, alpha, ev = oracle.h2o_step(Q[t], K[pos], V[pos], pos, s, t, L_local,
                                                 budget, scale)
        records.append((t, list(pos), list(s_new), ev, out, Q, K, V))
        s = list(s_new)
        if ev >= 0:
            evicted_mass += s[ev]
            del pos[ev]; del s[ev]
    return records, pos, s, evicted_mass, (Q, K, V, scale)


def test_h2o_mass_invariant_and_recent_quota():
    N, steps, D, budget, L_local = 40, 25, 8, 12, 6
    records, pos, s, evicted_mass, _ = _run_h2o(N, steps, D, budget, L_local, seed=17)
    assert sum(s) + evicted_mass == pytest.approx(N + steps, abs=1e-9)
    assert len(pos) == budget
    T = N + steps
    assert set(range(T - L_local, T)) <= set(pos)          # guaranteed recent quota


def test_h2o_eviction_is_the_pages_partition_rule():
    """After each step the cache is: the L_local newest tokens plus the K_HH largest-score
    historical tokens (ties keep the lower position) -- a selection, not an argmin."""
    N, steps, D, budget, L_local = 30, 30, 8, 10, 4
    records, *_ = _run_h2o(N, steps, D, budget, L_local, seed=18)
    for (t, pos, s_new, ev, *_rest) in records:
        recent = [p for p in pos if p > t - L_local]
        hist = [(s_new[i], p) for i, p in enumerate(pos) if p <= t - L_local]
        hist_sorted = sorted(hist, key=lambda e: (-e[0], e[1]))
        keep_hist = {p for _, p in hist_sorted[:budget - L_local]}
        keep = set(recent) | keep_hist
        assert len(pos) == budget + 1 and ev >= 0
        assert set(pos) - {pos[ev]} == keep


def test_h2o_no_eviction_gives_causal_column_sums():
    rng = np.random.default_rng(19)
    N, steps, D = 12, 10, 8
    T = N + steps
    Q, K, V = (rng.standard_normal((T, D)) for _ in range(3))
    scale = 1 / math.sqrt(D)
    s = list(oracle.h2o_prompt_scores(Q[:N], K[:N], scale))
    pos = list(range(N))
    outs = []
    for t in range(N, T):
        pos.append(t); s.append(0.0)
        out, s_new, _, ev = oracle.h2o_step(Q[t], K[pos], V[pos], pos, s, t, 3, 10 ** 6, scale)
        assert ev == -1
        s = list(s_new); outs.append(out)
    P = _causal_probs(Q, K, scale)
    assert np.allclose(s, P.sum(axis=0), atol=1e-12, rtol=0)
    full = _sdpa(Q, K, V, scale, causal=True)
    assert np.allclose(np.stack(outs), full[N:], atol=1e-12, rtol=0)


def test_h2o_evict_ties_evict_larger_position():
    s = np.array([0.5, 0.2, 0.2, 0.9, 0.2], dtype=np.float32)
    pos = np.array([3, 7, 5, 1, 20])
    assert oracle.h2o_evict_f32(s, pos, t=20, L_local=2) == 1       # pos 7 of the 0.2 ties
    assert oracle.h2o_evict_f32(s, pos, t=20, L_local=14) == 2      # pos 7 protected now
    assert oracle.h2o_evict_f32(s, pos, t=20, L_local=30) == -1     # nothing historical


def test_h2o_step_exact_tie_evicts_larger_position():
    """Two historical slots with identical keys and scores tie exactly; the larger position
    leaves (the lower index is kept, as in every top-k here)."""
    rng = np.random.default_rng(20)
    D = 8
    K = rng.standard_normal((6, D)); V = rng.standard_normal((6, D))
    K[1] = K[3]                                           # identical keys: identical attention
    pos = [0, 2, 5, 9, 11, 12]
    s = [3.0, 0.25, 1.0, 0.25, 0.5, 0.0]                  # slots 1 and 3 tie before and after
    q = rng.standard_normal(D)
    _, s_new, alpha, ev = oracle.h2o_step(q, K, V, pos, s, 12, 2, 5, 0.3)
    assert s_new[1] == s_new[3]
    lowest = min(range(4), key=lambda j: (s_new[j], -pos[j]))
    assert ev == lowest == 3


def test_pyramid_equal_remainders_round_lower_layer_first():
    # ratio 3 over 3 layers with B_target 1: exact budgets 1.5, 1, 0.5 -- one slot to place,
    # two equal remainders; the reading gives it to the lower layer.
    assert list(oracle.pyramid_budgets(3, 1, 3, 1)) == [2, 1, 0]


def test_snapkv_stage_f32_divides_after_summing():
    """The fp32 replay divides the pooled sum by k (an IEEE division), which is not the same
    as multiplying by a rounded 1/k: find two sums that only one of the two rules separates."""
    a = np.float32(1.5)             # a/5 lands in [0.25, 0.5), where its ulp is 2^-25 > ulp(a)/5
    found = None
    for _ in range(100000):
        b = np.nextafter(a, np.float32(2.0), dtype=np.float32)
        div_tie = np.float32(a / np.float32(5)) == np.float32(b / np.float32(5))
        mul_tie = np.float32(a * np.float32(0.2)) == np.float32(b * np.float32(0.2))
        if div_tie != mul_tie:
            found = (a, b, div_tie)
            break
        a = b
    assert found is not None
    a, b, div_tie = found
    n, L = 16, 2
    s = np.zeros((1, n), dtype=np.float32)
    s[0, 2], s[0, 11] = a, b            # pooled sums: a at positions 0..4, b at 9..13
    idx = oracle.snapkv_stage_f32(s, L, budget=L + 1)
    expect_first = 0 if div_tie else 9  # tie keeps the lower index; else b's window wins
    assert list(idx) == [expect_first, n, n + 1]


# ---------------------------------------------------------------------------- block eviction
def test_block_step_with_one_token_blocks_is_h2o():
    """Blocks of one token and one head: the block scores are H2O's per-token scores, the
    recent-block quota is H2O's recent quota (the newest tokens sit at consecutive positions),
    and the released block is H2O's evicted token -- including an exact tie among candidates,
    which releases the newer one."""
    rng = np.random.default_rng(41)
    D, L_local, budget = 8, 3, 6
    n = budget + 1
    K, V = rng.standard_normal((n, D)), rng.standard_normal((n, D))
    t = 50
    pos = np.array([2, 5, 9, 11, t - 2, t - 1, t])
    for q, s0 in ((rng.standard_normal(D), rng.random(n)),
                  (np.zeros(D), np.array([0.5, 0.25, 0.25, 0.25, 0.1, 0.2, 0.0]))):
        o_h, s_h, _, ev_h = oracle.h2o_step(q, K, V, pos, s0, t, L_local, budget, 0.3)
        o_b, s_b, ev_b = oracle.block_step(q[None], K[None], V[None], s0, 1, budget, L_local, 0.3)
        assert ev_b == ev_h and np.array_equal(s_b, s_h) and np.array_equal(o_b[0], o_h)
    assert ev_b == 3                      # uniform attention: ties 1,2,3 -> the newest goes


def test_block_score_is_the_sum_of_its_token_scores():
    """Score(block) = sum of s_t over its tokens ([KVC] block-level eviction), s_t summed over
    the query heads: blocks of 4 against blocks of 1 on the same grouped-query inputs, several
    steps with no release, the last block partly filled."""
    rng = np.random.default_rng(42)
    Hq, Hkv, D, bs = 4, 2, 8, 4
    s1 = np.zeros(0)
    s4 = np.zeros(0)
    for n_tok in (9, 10, 11, 12, 13):
        K, V = rng.standard_normal((Hkv, n_tok, D)), rng.standard_normal((Hkv, n_tok, D))
        q = rng.standard_normal((Hq, D))
        s1 = np.concatenate([s1, np.zeros(n_tok - len(s1))])
        s4 = np.concatenate([s4, np.zeros((n_tok + bs - 1) // bs - len(s4))])
        _, s1, e1 = oracle.block_step(q, K, V, s1, 1, 100, 1, 0.35)
        _, s4, e4 = oracle.block_step(q, K, V, s4, bs, 100, 1, 0.35)
        assert e1 == e4 == -1
        pad = np.concatenate([s1, np.zeros(len(s4) * bs - len(s1))])
        assert np.max(np.abs(pad.reshape(-1, bs).sum(axis=1) - s4)) <= 1e-12


def test_block_step_against_library_softmax_brute_force():
    rng = np.random.default_rng(43)
    Hq, Hkv, D, bs, n_tok = 4, 2, 8, 4, 23          # 6 blocks, the last holds 3 tokens
    budget, recent = 5, 2
    G = Hq // Hkv
    K, V = rng.standard_normal((Hkv, n_tok, D)), rng.standard_normal((Hkv, n_tok, D))
    q = rng.standard_normal((Hq, D))
    s0 = rng.random(6) * 3
    scale = 1 / math.sqrt(D)
    out, s_new, ev = oracle.block_step(q, K, V, s0, bs, budget, recent, scale)
    want = s0.copy()
    for h in range(Hq):
        lg = torch.from_numpy(K[h // G] @ q[h] * scale)
        a = torch.softmax(lg, dim=0).numpy()
        want += np.concatenate([a, np.zeros(6 * bs - n_tok)]).reshape(6, bs).sum(axis=1)
        ref = _sdpa(q[h][None], K[h // G], V[h // G], scale, causal=False)[0]
        assert np.max(np.abs(out[h] - ref)) <= 1e-12
    assert np.max(np.abs(s_new - want)) <= 1e-12
    assert abs((s_new - s0).sum() - Hq) <= 1e-12          # every head's attention sums to 1
    cands = sorted(range(6 - recent), key=lambda i: (want[i], -i))
    assert ev == cands[0]


def test_block_release_rules():
    s = np.array([0.5, 0.25, 0.25, 0.9, 0.0, 0.0], dtype=np.float32)
    assert oracle.block_evict_f32(s, 6, 2) == -1            # within budget: nothing released
    assert oracle.block_evict_f32(s, 5, 2) == 2             # tie 1/2: the newer goes
    assert oracle.block_evict_f32(s, 5, 1) == 4             # recent quota of one block
    assert oracle.block_evict_f32(s, 5, 5) == 0             # only the oldest is a candidate


# ---------------------------------------------------------------------------- grouped-query H2O
def test_h2o_group_of_one_is_h2o():
    rng = np.random.default_rng(51)
    n, D, t, L_local, budget = 9, 8, 40, 3, 8
    K, V = rng.standard_normal((n, D)), rng.standard_normal((n, D))
    pos = np.array([0, 5, 7, 12, 20, 30, 38, 39, 40])
    s0 = rng.random(n)
    q = rng.standard_normal(D)
    o1, s1, _, e1 = oracle.h2o_step(q, K, V, pos, s0, t, L_local, budget, 0.3)
    og, sg, eg = oracle.h2o_step_group(q[None], K, V, pos, s0, t, L_local, budget, 0.3)
    assert eg == e1 and np.array_equal(sg, s1) and np.array_equal(og[0], o1)


def test_h2o_group_sums_the_heads_attention():
    """Library softmax per query head, summed over the group; the increments total G; the
    evicted row is the brute-force minimum over the candidates (ties: larger position)."""
    rng = np.random.default_rng(52)
    G, n, D, t, L_local, budget = 4, 12, 8, 60, 4, 11
    K, V = rng.standard_normal((n, D)), rng.standard_normal((n, D))
    pos = np.array([1, 3, 9, 10, 14, 22, 31, 44, 57, 58, 59, 60])
    q = rng.standard_normal((G, D))
    s0 = rng.random(n) * 2
    scale = 1 / math.sqrt(D)
    out, s_new, ev = oracle.h2o_step_group(q, K, V, pos, s0, t, L_local, budget, scale)
    want = s0.copy()
    for g in range(G):
        want += torch.softmax(torch.from_numpy(K @ q[g] * scale), dim=0).numpy()
        ref = _sdpa(q[g][None], K, V, scale, causal=False)[0]
        assert np.max(np.abs(out[g] - ref)) <= 1e-12
    assert np.max(np.abs(s_new - want)) <= 1e-12
    assert abs((s_new - s0).sum() - G) <= 1e-12
    cands = [j for j in range(n) if pos[j] <= t - L_local]
    assert ev == sorted(cands, key=lambda j: (want[j], -pos[j]))[0]
    # one head of the group alone gives different scores: every head counts
    _, s_one, ev_one = oracle.h2o_step_group(q[:1], K, V, pos, s0, t, L_local, budget, scale)
    assert not np.allclose(s_one, s_new)


# ---------------------------------------------------------------------------- DuoAttention
def test_duo_memory_saving_matches_the_pages():
    """[KVC] DuoAttention: retrieval heads are 20-30 % of the heads and the method saves up to
    70 % of the KV memory at 128k tokens: with 30 % retrieval heads (a 4 + 64 token buffer for
    the others) the saving is 70 % to within 0.1 %, with 20 % it is 80 %; no streaming heads is
    the plain memory formula."""
    g = _golden("duo_memory.json")
    N, S, W = g["seq_len"], g["n_sink"], g["window"]
    full = oracle.kv_bytes(32, 10, 128, N, 2, 1)
    for c in g["cases"]:
        duo = oracle.duo_kv_bytes(32, c["n_retrieval"], c["n_streaming"], 128, N, S, W, 2, 1)
        assert abs((1 - duo / full) - c["saving"]) < 1e-3, c["what"]
    assert oracle.duo_kv_bytes(32, 10, 0, 128, N, S, W, 2, 1) == full
    # a streaming head's buffer is constant: O(1) in the sequence length
    a = oracle.duo_kv_bytes(1, 0, 1, 128, 10 ** 6, S, W, 2, 1)
    assert a == oracle.duo_kv_bytes(1, 0, 1, 128, 10 ** 4, S, W, 2, 1) == 2 * 128 * 2 * (S + W + 1)


def test_duo_heads_against_library_attention():
    """A retrieval head is causal attention over the whole history; a streaming head is
    attention over the sinks, the window and the token itself (torch SDPA on those rows); while
    the history fits the buffer the two agree."""
    rng = np.random.default_rng(71)
    D, S, W, T = 16, 4, 6, 40
    hk, hv = rng.standard_normal((T, D)), rng.standard_normal((T, D))
    q = rng.standard_normal(D)
    scale = 1 / math.sqrt(D)
    t = T - 1
    o_r = oracle.duo_decode(True, t, S, W, q, hk, hv, scale)
    assert np.max(np.abs(o_r - _sdpa(q[None], hk, hv, scale, causal=False)[0])) <= 1e-12
    o_s = oracle.duo_decode(False, t, S, W, q, hk, hv, scale)
    keep = list(range(S)) + list(range(t - W, t + 1))
    assert np.max(np.abs(o_s - _sdpa(q[None], hk[keep], hv[keep], scale, causal=False)[0])) <= 1e-12
    assert np.max(np.abs(o_s - o_r)) > 1e-6
    for t in (0, 3, S + W):
        a = oracle.duo_decode(True, t, S, W, q, hk, hv, scale)
        b = oracle.duo_decode(False, t, S, W, q, hk, hv, scale)
        assert np.max(np.abs(a - b)) <= 1e-15


def test_block_prompt_select_one_token_blocks_is_h2o_prompt_select():
    rng = np.random.default_rng(81)
    N, L_local, K_hh = 200, 30, 45
    s = rng.random(N) * 3
    s[[10, 11, 12]] = 1.5                                    # exact ties among candidates
    keep, sc = oracle.block_prompt_select(s[None], 1, L_local + K_hh, L_local)
    assert np.array_equal(keep, oracle.h2o_prompt_select(s, L_local, K_hh))
    assert np.array_equal(sc, s)


def test_block_prompt_select_block_scores_and_rules():
    """Uniform scores give H * block_size per block (the partial last block: H * its tokens);
    the recent blocks are always kept, the rest by score with ties to the lower index; a
    prompt within the budget keeps every block."""
    H, N, bs = 3, 70, 16                                     # 5 blocks, the last holds 6 tokens
    keep, sc = oracle.block_prompt_select(np.ones((H, N)), bs, 3, 1)
    assert list(sc) == [48.0, 48.0, 48.0, 48.0, 18.0]
    assert list(keep) == [0, 1, 4]                           # ties: lower indices, + newest
    s = np.zeros((H, N))
    s[1, 20] = 5.0                                           # block 1
    s[2, 50:53] = 1.0                                        # block 3
    keep, _ = oracle.block_prompt_select(s, bs, 3, 1)
    assert list(keep) == [1, 3, 4]
    keep, _ = oracle.block_prompt_select(s, bs, 2, 2)
    assert list(keep) == [3, 4]                              # only the recent blocks
    keep, _ = oracle.block_prompt_select(s, bs, 5, 1)
    assert list(keep) == [0, 1, 2, 3, 4]


def test_h2o_prompt_scores_group():
    """A group of one is H2O's prompt scores; the group's sum is the sum of library causal
    softmax columns over its heads; every head's rows sum to one, so the total is G * N."""
    rng = np.random.default_rng(91)
    G, N, D = 3, 40, 8
    Q, K = rng.standard_normal((G, N, D)), rng.standard_normal((N, D))
    scale = 1 / math.sqrt(D)
    one = oracle.h2o_prompt_scores_group(Q[:1], K, scale)
    assert np.array_equal(one, oracle.h2o_prompt_scores(Q[0], K, scale))
    s = oracle.h2o_prompt_scores_group(Q, K, scale)
    want = sum(_causal_probs(Q[g], K, scale).sum(axis=0) for g in range(G))
    assert np.max(np.abs(s - want)) <= 1e-12
    assert abs(s.sum() - G * N) <= 1e-9
