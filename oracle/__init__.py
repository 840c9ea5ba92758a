"""CPU oracle for KV-cache compression and decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The product library never calls it, and it shares no code with the CUDA path:
the arithmetic lives in ``kvc_oracle.c`` (plain C, double precision, scalar loops), compiled
with gcc into ``oracle/_build/``.  This module only marshals numpy arrays.

Functions (each follows the page passage cited in ``kvc_oracle.c``):
  kv_bytes, pyramid_budgets, rope, attend, stream_window, stream_slot, stream_decode,
  stream_decode_alibi, topk_ascending, snapkv_obs_scores, pool1d, snapkv_select, snapkv_stage_f32,
  h2o_prompt_scores, h2o_prompt_scores_group, h2o_prompt_select, h2o_step, h2o_step_group,
  h2o_evict_f32, block_step, block_evict_f32,
  duo_decode, duo_kv_bytes, block_prompt_select.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against values the pages
print, closed forms, invariants, library routines on special cases or brute force on tiny
inputs (``tests/test_oracle_pins.py``).  The attention-quality numbers the pages quote
(perplexity, task accuracy, speedups) need model weights and datasets: parity unpinned, and not
computed here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkvc_oracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add, so x86 and Arm builds round identically.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (a few seconds); returns the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_f64 = ctypes.c_double
_ptr = ctypes.c_void_p

_SIGS = {
    "orc_kv_bytes": (_u64, [_u64] * 6),
    "orc_pyramid_budgets": (ctypes.c_int, [ctypes.c_int, _i64, _i64, _i64, _ptr]),
    "orc_rope": (None, [ctypes.c_int, _f64, _i64, _ptr, _ptr]),
    "orc_attend": (None, [ctypes.c_int, ctypes.c_int, _f64, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "orc_stream_window": (ctypes.c_int, [_i64, ctypes.c_int, ctypes.c_int, _ptr, _ptr, _ptr]),
    "orc_stream_slot": (_i64, [_i64, ctypes.c_int, ctypes.c_int]),
    "orc_stream_decode": (None, [_i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64, _f64,
                                 _ptr, _ptr, _ptr, _ptr]),
    "orc_stream_decode_alibi": (None, [_i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64,
                                       _f64, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "orc_topk_ascending": (None, [ctypes.c_int, ctypes.c_int, _ptr, _ptr]),
    "orc_snapkv_obs_scores": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64, _ptr,
                                     _ptr, _ptr]),
    "orc_pool1d": (None, [ctypes.c_int, ctypes.c_int, _ptr, _ptr]),
    "orc_snapkv_select": (ctypes.c_int, [ctypes.c_int] * 6 + [_f64, _ptr, _ptr, _ptr, _ptr,
                                                               _ptr]),
    "orc_snapkv_stage_f32": (ctypes.c_int, [ctypes.c_int] * 5 + [_ptr, _ptr]),
    "orc_h2o_prompt_scores": (None, [ctypes.c_int, ctypes.c_int, _f64, _ptr, _ptr, _ptr]),
    "orc_h2o_prompt_select": (ctypes.c_int, [ctypes.c_int] * 3 + [_ptr, _ptr]),
    "orc_h2o_prompt_scores_group": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64, _ptr,
                                           _ptr, _ptr]),
    "orc_h2o_step": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _f64, _ptr, _ptr, _ptr, _ptr,
                                    _ptr, _i64, ctypes.c_int, ctypes.c_int, _ptr, _ptr]),
    "orc_h2o_evict_f32": (ctypes.c_int, [ctypes.c_int, _ptr, _ptr, _i64, ctypes.c_int]),
    "orc_h2o_step_group": (ctypes.c_int, [ctypes.c_int] * 3 + [_f64, _ptr, _ptr, _ptr, _ptr,
                                                               _ptr, _i64, ctypes.c_int,
                                                               ctypes.c_int, _ptr]),
    "orc_block_step": (ctypes.c_int, [ctypes.c_int] * 5 + [_f64, _ptr, _ptr, _ptr, _ptr,
                                                           ctypes.c_int, ctypes.c_int, _ptr]),
    "orc_block_evict_f32": (ctypes.c_int, [ctypes.c_int, _ptr, ctypes.c_int, ctypes.c_int]),
    "orc_duo_decode": (None, [ctypes.c_int, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              _f64, _ptr, _ptr, _ptr, _ptr]),
    "orc_duo_kv_bytes": (_u64, [_u64] * 9),
    "orc_block_prompt_select": (ctypes.c_int, [ctypes.c_int] * 3 + [_ptr, ctypes.c_int,
                                                                   ctypes.c_int, _ptr, _ptr]),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            handle = ctypes.CDLL(build())
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _f(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _opt(a):
    return None if a is None else _p(a)


# --------------------------------------------------------------------------------------------
def kv_bytes(n_layers, n_heads_kv, d_head, seq_len, bytes_per_elem, batch) -> int:
    return int(lib().orc_kv_bytes(n_layers, n_heads_kv, d_head, seq_len, bytes_per_elem, batch))


def pyramid_budgets(n_layers: int, b_target: int, ratio_num: int = 4, ratio_den: int = 1):
    out = np.zeros(max(n_layers, 1), dtype=np.int64)
    rc = lib().orc_pyramid_budgets(n_layers, b_target, ratio_num, ratio_den, _p(out))
    if rc != 0:
        raise ValueError("invalid pyramid arguments")
    return out[:n_layers]


def rope(x, pos: int, theta: float = 10000.0) -> np.ndarray:
    x = _f(x)
    y = np.empty_like(x)
    lib().orc_rope(x.shape[-1], theta, int(pos), _p(x), _p(y))
    return y


def attend(q, K, V, scale: float):
    """o, logits, lse of one query over n keys (rows of K, V)."""
    q, K, V = _f(q), _f(K).reshape(-1, len(q)), _f(V).reshape(-1, len(q))
    n, D = K.shape
    out = np.empty(D)
    logits = np.empty(max(n, 1))
    lse = np.empty(1)
    lib().orc_attend(n, D, scale, _p(q), _p(K), _p(V), _p(out), _p(logits), _p(lse))
    return out, logits[:n], float(lse[0])


def stream_window(t: int, S: int, W: int):
    """(text positions, in-cache positions, query position) attended when decoding token t."""
    tok = np.empty(S + W + 1, dtype=np.int64)
    cpos = np.empty(S + W + 1, dtype=np.int64)
    q = np.empty(1, dtype=np.int64)
    n = lib().orc_stream_window(int(t), S, W, _p(tok), _p(cpos), _p(q))
    return tok[:n].copy(), cpos[:n].copy(), int(q[0])


def stream_slot(a: int, S: int, W: int) -> int:
    return int(lib().orc_stream_slot(int(a), S, W))


def stream_decode(t: int, S: int, W: int, q_pre, hist_k, hist_v, scale: float,
                  theta: float = 10000.0) -> np.ndarray:
    q_pre = _f(q_pre)
    D = q_pre.shape[0]
    hk, hv = _f(hist_k), _f(hist_v)
    assert hk.shape[0] >= t + 1 and hv.shape[0] >= t + 1 and hk.shape[1] == D
    out = np.empty(D)
    lib().orc_stream_decode(int(t), S, W, D, theta, scale, _p(q_pre), _p(hk), _p(hv), _p(out))
    return out


def stream_decode_alibi(t: int, S: int, W: int, q, hist_k, hist_v, scale: float, slope: float):
    """StreamingLLM decode with ALiBi at in-cache positions -> (out, logits in rank order, lse)."""
    q = _f(q)
    D = q.shape[0]
    hk, hv = _f(hist_k), _f(hist_v)
    assert hk.shape[0] >= t + 1 and hv.shape[0] >= t + 1 and hk.shape[1] == D
    out = np.empty(D)
    logits = np.empty(S + W + 1)
    lse = np.empty(1)
    lib().orc_stream_decode_alibi(int(t), S, W, D, float(slope), float(scale), _p(q), _p(hk),
                                  _p(hv), _p(out), _p(logits), _p(lse))
    n = min(int(t) + 1, S + W + 1)
    return out, logits[:n].copy(), float(lse[0])


def topk_ascending(score, k: int) -> np.ndarray:
    score = _f(score)
    n = score.shape[0]
    kk = max(0, min(k, n))
    idx = np.empty(max(kk, 1), dtype=np.int32)
    lib().orc_topk_ascending(n, k, _p(score), _p(idx))
    return idx[:kk]


def snapkv_obs_scores(Qobs, K, scale: float) -> np.ndarray:
    Qobs, K = _f(Qobs), _f(K)
    L_obs, D = Qobs.shape
    N = K.shape[0]
    s = np.empty(N)
    lib().orc_snapkv_obs_scores(L_obs, N, D, scale, _p(Qobs), _p(K), _p(s))
    return s


def pool1d(s, k: int = 5) -> np.ndarray:
    s = _f(s)
    p = np.empty(max(s.shape[0], 1))
    lib().orc_pool1d(s.shape[0], k, _p(s), _p(p))
    return p[:s.shape[0]]


def snapkv_select(Qobs, K, budget: int, scale: float, pool_k: int = 5):
    """Qobs [G, L_obs, D], K [N, D] -> (idx, s [G, N], score [N-L_obs])."""
    Qobs, K = _f(Qobs), _f(K)
    G, L_obs, D = Qobs.shape
    N = K.shape[0]
    idx = np.empty(max(N, budget, 1), dtype=np.int32)
    s = np.empty((G, N))
    score = np.empty(max(N - L_obs, 1))
    kept = lib().orc_snapkv_select(G, L_obs, N, D, pool_k, budget, scale, _p(Qobs), _p(K),
                                   _p(idx), _p(s), _p(score))
    if kept < 0:
        raise ValueError("invalid SnapKV arguments")
    return idx[:kept].copy(), s, score[:N - L_obs].copy()


def snapkv_stage_f32(s_f32, L_obs: int, budget: int, pool_k: int = 5) -> np.ndarray:
    """Pool + group max + top-k replayed in fp32 from given fp32 column means [G, n_prefix]."""
    s = np.ascontiguousarray(np.asarray(s_f32, dtype=np.float32))
    G, n = s.shape
    idx = np.empty(max(n + L_obs, budget, 1), dtype=np.int32)
    kept = lib().orc_snapkv_stage_f32(G, n, pool_k, L_obs, budget, _p(s), _p(idx))
    if kept < 0:
        raise ValueError("invalid SnapKV arguments")
    return idx[:kept].copy()


def h2o_prompt_scores(Q, K, scale: float) -> np.ndarray:
    Q, K = _f(Q), _f(K)
    N, D = Q.shape
    s = np.empty(N)
    lib().orc_h2o_prompt_scores(N, D, scale, _p(Q), _p(K), _p(s))
    return s


def h2o_prompt_scores_group(Q, K, scale: float) -> np.ndarray:
    """Q [G, N, D] the group's query heads, K [N, D] -> s [N] summed over the group."""
    Q, K = _f(Q), _f(K)
    G, N, D = Q.shape
    s = np.empty(N)
    lib().orc_h2o_prompt_scores_group(G, N, D, scale, _p(Q), _p(K), _p(s))
    return s


def h2o_prompt_select(s, L_local: int, K_hh: int) -> np.ndarray:
    s = _f(s)
    N = s.shape[0]
    idx = np.empty(max(N, 1), dtype=np.int32)
    n = lib().orc_h2o_prompt_select(N, L_local, K_hh, _p(s), _p(idx))
    return idx[:n].copy()


def h2o_step(q, K, V, pos, s, t: int, L_local: int, budget: int, scale: float):
    """One decode step; returns (out, s_new, alpha, evicted slot or -1).  s is not modified."""
    q, K, V = _f(q), _f(K), _f(V)
    n, D = K.shape
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    s_new = _f(s).copy()
    out = np.empty(D)
    alpha = np.empty(max(n, 1))
    ev = lib().orc_h2o_step(n, D, scale, _p(q), _p(K), _p(V), _p(pos), _p(s_new), int(t),
                            L_local, budget, _p(out), _p(alpha))
    return out, s_new, alpha[:n].copy(), int(ev)


def h2o_step_group(q, K, V, pos, s, t: int, L_local: int, budget: int, scale: float):
    """One decode step of a grouped-query KV head: q [G, D]; returns (out [G, D], s_new,
    evicted slot or -1).  s is not modified."""
    q, K, V = _f(q), _f(K), _f(V)
    G, D = q.shape
    n = K.shape[0]
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    s_new = _f(s).copy()
    out = np.empty((G, D))
    ev = lib().orc_h2o_step_group(G, n, D, scale, _p(q), _p(K), _p(V), _p(pos), _p(s_new),
                                  int(t), L_local, budget, _p(out))
    return out, s_new, int(ev)


def h2o_evict_f32(s_f32, pos, t: int, L_local: int) -> int:
    s = np.ascontiguousarray(np.asarray(s_f32, dtype=np.float32))
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    return int(lib().orc_h2o_evict_f32(s.shape[0], _p(s), _p(pos), int(t), L_local))


def block_step(q, K, V, score, bs: int, budget_blocks: int, recent_blocks: int, scale: float):
    """One block-eviction decode step of one sequence.  q [Hq, D]; K, V [Hkv, n_tok, D] in
    page-table order; score [nb] (not modified).  Returns (out [Hq, D], score_new, released
    block index or -1)."""
    q, K, V = _f(q), _f(K), _f(V)
    Hq, D = q.shape
    Hkv, n_tok = K.shape[0], K.shape[1]
    nb = (n_tok + bs - 1) // bs
    s_new = _f(score).copy()
    assert s_new.shape[0] == nb
    out = np.empty((Hq, D))
    ev = lib().orc_block_step(Hq, Hkv, D, n_tok, bs, scale, _p(q), _p(K), _p(V), _p(s_new),
                              budget_blocks, recent_blocks, _p(out))
    return out, s_new, int(ev)


def block_evict_f32(score_f32, budget_blocks: int, recent_blocks: int) -> int:
    s = np.ascontiguousarray(np.asarray(score_f32, dtype=np.float32))
    return int(lib().orc_block_evict_f32(s.shape[0], _p(s), budget_blocks, recent_blocks))


def duo_decode(retrieval: bool, t: int, S: int, W: int, q, hist_k, hist_v, scale: float):
    """DuoAttention decode of one head at text position t: full history for a retrieval head,
    the StreamingLLM set (sinks + window + t) for a streaming head."""
    q = _f(q)
    D = q.shape[0]
    hk, hv = _f(hist_k), _f(hist_v)
    assert hk.shape[0] >= t + 1 and hv.shape[0] >= t + 1 and hk.shape[1] == D
    out = np.empty(D)
    lib().orc_duo_decode(int(bool(retrieval)), int(t), S, W, D, float(scale), _p(q), _p(hk),
                         _p(hv), _p(out))
    return out


def duo_kv_bytes(n_layers, n_retrieval, n_streaming, d_head, seq_len, n_sink, window,
                 bytes_per_elem, batch) -> int:
    return int(lib().orc_duo_kv_bytes(n_layers, n_retrieval, n_streaming, d_head, seq_len,
                                      n_sink, window, bytes_per_elem, batch))


def block_prompt_select(s, bs: int, budget_blocks: int, recent_blocks: int):
    """s [H, N] per-token scores -> (kept block indices ascending, block scores [nblk])."""
    s = _f(s)
    H, N = s.shape
    nblk = (N + bs - 1) // bs
    keep = np.empty(max(nblk, 1), dtype=np.int32)
    sc = np.empty(max(nblk, 1))
    n = lib().orc_block_prompt_select(H, N, bs, _p(s), budget_blocks, recent_blocks, _p(sc),
                                      _p(keep))
    return keep[:n].copy(), sc[:nblk].copy()
