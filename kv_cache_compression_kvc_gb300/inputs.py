"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and shapes them (sink boosts, needle runs, heavy-tailed
key scales); it holds none of the method's arithmetic, and both the CUDA path and the CPU oracle
receive exactly the tensors it makes.  There is no model and no dataset: queries, keys and
values are N(0, 1) draws, shaped as described below (the recipe is also in the design notes).

Workloads (sizes as stated by the benchmark configuration):
  tiny        fp32, B=1, Hq=8, Hkv=2, D=64, N=512; keys 0-3 boosted by +3 toward the group's
              mean query (attention sinks); SnapKV L_obs=32, pool 5, budget 128; StreamingLLM
              4 sinks + W=60, RoPE theta 10000, 64 decode steps; H2O budget 102 (51 recent).
  streaming   Llama-2-7B attention shape: 32 layers, MHA 32 heads, D=128, bf16, B=16; cache of
              4 sinks + a ring of W=2044 filled from a 4096-token prompt; 1024 decode steps.
  snapkv      32 layers, Hq=32, Hkv=8, D=128, bf16, B=4, N=32768; L_obs=32, pool 5, budget
              5243 per KV head; 2% of positions per head boosted x4 toward the observation
              queries in runs of 3-8 tokens; 256 decode steps.
  h2o         32 layers, MHA 32 heads, D=128, bf16, B=16, N=4096; budget 819 = 410 recent +
              409 heavy hitters; keys scaled per position by a Zipf(1.1) draw on {1..8}; 512 steps.
  pyramid     16 layers, Hq=24, Hkv=4, D=256, bf16, B=2, N=131072; L_obs=64, pool 5; budgets
              fall linearly (ratio 4) around a mean of 8192; sink-boosted keys 0-3; 256 steps.
  alibi       the streaming shape with ALiBi at in-cache positions in place of RoPE (slopes
              2^(-8(h+1)/32) for the 32 heads); same cache, prompt and steps.
  paged       the h2o shape with block-level eviction: blocks of 32 tokens, 26 blocks (832
              tokens, >= the 819 budget) per sequence, the 13 newest (>= 410 recent tokens)
              protected; pools of N(0,1) keys and values.
  h2o_gqa     the h2o shape on a grouped-query cache: 32 query heads over 8 KV heads; caches of
              N(0,1) keys/values at the 410 newest and 409 random older prompt positions.
  duo         DuoAttention at 128k tokens: 32 layers, MHA 32 heads, D=128, bf16, batch 1; per
              layer a seeded fixed choice of 8 retrieval heads (25 %) with full caches of N(0,1)
              keys/values, the other 24 with 4 sinks + 64 recent tokens; 256 steps.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    n_heads_q: int
    n_heads_kv: int
    d_head: int
    prompt: int
    steps: int
    dtype: torch.dtype
    seed: int
    n_sink: int = 4
    window: int = 0
    L_obs: int = 0
    pool_k: int = 5
    budget: int = 0
    L_local: int = 0
    theta: float = 10000.0
    pyramid_ratio: int = 4
    extra: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.n_heads_q // self.n_heads_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_head)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 8, 2, 64, 512, 64, torch.float32, 1235, n_sink=4, window=60,
                     L_obs=32, budget=128, L_local=51, extra={"h2o_budget": 102}),
    "streaming": Workload("streaming", 32, 16, 32, 32, 128, 4096, 1024, torch.bfloat16, 1236,
                          n_sink=4, window=2044),
    "snapkv": Workload("snapkv", 32, 4, 32, 8, 128, 32768, 256, torch.bfloat16, 1237, L_obs=32,
                       budget=5243),
    "h2o": Workload("h2o", 32, 16, 32, 32, 128, 4096, 512, torch.bfloat16, 1238, budget=819,
                    L_local=410),
    "pyramid": Workload("pyramid", 16, 2, 24, 4, 256, 131072, 256, torch.bfloat16, 1239,
                        L_obs=64, budget=8192),
    "alibi": Workload("alibi", 32, 16, 32, 32, 128, 4096, 1024, torch.bfloat16, 1240,
                      n_sink=4, window=2044),
    "paged": Workload("paged", 32, 16, 32, 32, 128, 4096, 512, torch.bfloat16, 1241,
                      budget=819, L_local=410, extra={"block_size": 32}),
    "h2o_gqa": Workload("h2o_gqa", 32, 16, 32, 8, 128, 4096, 512, torch.bfloat16, 1242,
                        budget=819, L_local=410),
    "duo": Workload("duo", 32, 1, 32, 32, 128, 131072, 256, torch.bfloat16, 1243, n_sink=4,
                    window=64, extra={"n_retrieval": 8}),
}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """N(0,1) draws in fp32 from a seeded generator, then cast to `dtype`."""
    g = generator(seed, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def unit_mean_direction(q: torch.Tensor) -> torch.Tensor:
    """Unit vector along the mean of query rows q[..., n, D] (over n), fp32."""
    m = q.float().mean(dim=-2)
    return m / m.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def boost_positions(k: torch.Tensor, positions, direction: torch.Tensor, c: float) -> None:
    """In place: k[b, h, p, :] += c * sqrt(D) * direction[b, h, :] for p in positions.

    k: [B, H, N, D]; direction: [B, H, D] unit vectors.  The sqrt(D) makes the logit shift of a
    query aligned with the direction about c (logits are scaled by 1/sqrt(D))."""
    D = k.shape[-1]
    pos = torch.as_tensor(positions, device=k.device, dtype=torch.long)
    add = (c * math.sqrt(D)) * direction.to(k.device).float()[:, :, None, :]
    k[:, :, pos, :] = (k[:, :, pos, :].float() + add).to(k.dtype)


def needle_runs(n_prefix: int, target: int, seed: int, lo: int = 3, hi: int = 8):
    """Non-overlapping, non-adjacent runs of lo..hi tokens with uniform starts in
    [0, n_prefix - len], drawn until `target` positions are covered (the last run may be cut
    short to hit the count exactly)."""
    rng = np.random.default_rng(seed)
    target = min(int(target), n_prefix // 2)
    taken = np.zeros(n_prefix, dtype=bool)
    count = 0
    while count < target:
        ln = int(rng.integers(lo, hi + 1))
        ln = min(ln, target - count)
        start = int(rng.integers(0, n_prefix - ln + 1))
        if taken[max(0, start - 1):start + ln + 1].any():
            continue
        taken[start:start + ln] = True
        count += ln
    return np.nonzero(taken)[0]


def zipf_scales(n: int, a: float, kmax: int, seed: int) -> np.ndarray:
    """n draws from P(k) proportional to k^-a on {1..kmax}."""
    rng = np.random.default_rng(seed)
    ks = np.arange(1, kmax + 1, dtype=np.float64)
    p = ks ** (-a)
    p /= p.sum()
    return rng.choice(ks, size=n, p=p).astype(np.float32)


# ------------------------------------------------------------------------------------------
def prompt_qkv(B, Hq, Hkv, N, D, seed, device="cpu", dtype=torch.float32, sink_boost=3.0,
               n_sink=4):
    """Prompt Q [B,Hq,N,D], K, V [B,Hkv,N,D]; keys 0..n_sink-1 boosted toward the group's mean
    prompt query (attention sinks)."""
    q = randn((B, Hq, N, D), seed * 3 + 0, device)
    k = randn((B, Hkv, N, D), seed * 3 + 1, device)
    v = randn((B, Hkv, N, D), seed * 3 + 2, device)
    if sink_boost and n_sink:
        G = Hq // Hkv
        qg = q.reshape(B, Hkv, G * N, D)
        boost_positions(k, range(min(n_sink, N)), unit_mean_direction(qg), sink_boost)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def decode_qkv(B, Hq, Hkv, D, steps, seed, device="cpu", dtype=torch.float32):
    """Per-step decode inputs: q [steps,B,Hq,D], k/v [steps,B,Hkv,D] (no model: N(0,1))."""
    q = randn((steps, B, Hq, D), seed * 5 + 0, device, dtype)
    k = randn((steps, B, Hkv, D), seed * 5 + 1, device, dtype)
    v = randn((steps, B, Hkv, D), seed * 5 + 2, device, dtype)
    return q, k, v


def snapkv_layer(w: Workload, layer: int, device="cpu", N: Optional[int] = None,
                 batch: Optional[int] = None):
    """One layer's SnapKV prompt: Q_obs [B,Hq,L_obs,D], K, V [B,Hkv,N,D] with needle runs."""
    N = N or w.prompt
    B = batch or w.batch
    seed = w.seed * 1000 + layer
    D, Hq, Hkv = w.d_head, w.n_heads_q, w.n_heads_kv
    q_obs = randn((B, Hq, w.L_obs, D), seed * 3 + 0, device)
    k = randn((B, Hkv, N, D), seed * 3 + 1, device)
    v = randn((B, Hkv, N, D), seed * 3 + 2, device)
    direction = unit_mean_direction(q_obs.reshape(B, Hkv, w.group * w.L_obs, D))
    for b in range(B):
        for h in range(Hkv):
            pos = needle_runs(N - w.L_obs, round(0.02 * N), seed * 7919 + b * 131 + h)
            boost_positions(k[b:b + 1, h:h + 1], pos, direction[b:b + 1, h:h + 1], 4.0)
    return q_obs.to(w.dtype), k.to(w.dtype), v.to(w.dtype)


def pyramid_layer(w: Workload, layer: int, device="cpu", N: Optional[int] = None,
                  batch: Optional[int] = None):
    """One layer's long-context prompt: Q_obs, K, V with sink-boosted keys 0-3."""
    N = N or w.prompt
    B = batch or w.batch
    seed = w.seed * 1000 + layer
    D, Hq, Hkv = w.d_head, w.n_heads_q, w.n_heads_kv
    q_obs = randn((B, Hq, w.L_obs, D), seed * 3 + 0, device)
    k = randn((B, Hkv, N, D), seed * 3 + 1, device)
    v = randn((B, Hkv, N, D), seed * 3 + 2, device)
    direction = unit_mean_direction(q_obs.reshape(B, Hkv, w.group * w.L_obs, D))
    boost_positions(k, range(w.n_sink), direction, 3.0)
    return q_obs.to(w.dtype), k.to(w.dtype), v.to(w.dtype)


def h2o_layer(w: Workload, layer: int, device="cpu", N: Optional[int] = None,
              batch: Optional[int] = None):
    """One layer's H2O prompt Q, K, V [B,H,N,D]; keys scaled per (batch, position) by Zipf(1.1)."""
    N = N or w.prompt
    B = batch or w.batch
    seed = w.seed * 1000 + layer
    D, H = w.d_head, w.n_heads_q
    q = randn((B, H, N, D), seed * 3 + 0, device)
    k = randn((B, H, N, D), seed * 3 + 1, device)
    v = randn((B, H, N, D), seed * 3 + 2, device)
    sc = torch.from_numpy(zipf_scales(B * N, 1.1, 8, seed * 7 + 5)).reshape(B, 1, N, 1)
    k = k * sc.to(device)
    return q.to(w.dtype), k.to(w.dtype), v.to(w.dtype)


def streaming_prefill(w: Workload, layer: int, device="cpu", batch: Optional[int] = None,
                      heads: Optional[int] = None):
    """Pre-rotation K, V of the prompt tokens a StreamingLLM cache still holds after a
    w.prompt-token prefill: sinks 0..S-1 and the window prompt-W .. prompt-1, as
    [B, H, S+W, D] (sinks first, then the window in text order), with the sinks boosted toward
    the mean of 64 reference queries.  Returns (k, v, text_positions)."""
    B = batch or w.batch
    H = heads or w.n_heads_kv
    D, S, W, N = w.d_head, w.n_sink, w.window, w.prompt
    seed = w.seed * 1000 + layer
    n = S + W
    k = randn((B, H, n, D), seed * 3 + 1, device)
    v = randn((B, H, n, D), seed * 3 + 2, device)
    qref = randn((B, H, 64, D), seed * 3 + 0, device)
    boost_positions(k, range(S), unit_mean_direction(qref), 3.0)
    text_pos = list(range(S)) + list(range(N - W, N))
    return k.to(w.dtype), v.to(w.dtype), text_pos
