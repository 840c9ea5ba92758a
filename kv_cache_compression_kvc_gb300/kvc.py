"""Python binding of libkvc (include/kvc.h): same names as the C entry points.

Argument marshalling only: torch tensors are turned into device pointers, sizes and strides,
and every step runs in the library's CUDA kernels on the current torch stream.  PyTorch only
provides device memory and streams.  There is no fallback: if libkvc.so has not been built (see
``kv_cache_compression_kvc_gb300.build``) or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

KVC_OK = 0
KVC_F32, KVC_BF16 = 0, 1
KVC_APPEND_TAIL, KVC_APPEND_RING, KVC_APPEND_FREE_SLOT = 0, 1, 2
KVC_DECODE_KV_SETTLED = 1
KVC_DECODE_BALANCE = 2
KVC_DECODE_TEST_STARVE = 0x80000000
STATUS_NAMES = {0: "KVC_OK", 1: "KVC_ERR_INVALID_ARG", 2: "KVC_ERR_SHAPE", 3: "KVC_ERR_ALIGN",
                4: "KVC_ERR_CAPACITY", 5: "KVC_ERR_CUDA", 6: "KVC_ERR_WORKSPACE",
                7: "KVC_ERR_DEVICE"}


class KvcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class kvc_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("n_heads_kv", ctypes.c_int32),
                ("cap", ctypes.c_int32), ("d_head", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("stride_b", ctypes.c_int64),
                ("stride_h", ctypes.c_int64), ("stride_slot", ctypes.c_int64)]


class kvc_rope(ctypes.Structure):
    _fields_ = [("n_sink", ctypes.c_int32), ("window", ctypes.c_int32),
                ("t", ctypes.c_void_p), ("cos_sin", ctypes.c_void_p),
                ("n_pos", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class kvc_alibi(ctypes.Structure):
    _fields_ = [("n_sink", ctypes.c_int32), ("window", ctypes.c_int32),
                ("t", ctypes.c_void_p), ("slopes", ctypes.c_void_p)]


class kvc_block_pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("n_blocks", ctypes.c_int32), ("n_heads_kv", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("d_head", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class kvc_page_table(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("n_blocks", ctypes.c_void_p),
                ("len", ctypes.c_void_p), ("score", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("max_blocks", ctypes.c_int32)]


class kvc_free_pool(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("top", ctypes.c_void_p),
                ("capacity", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class kvc_duo(ctypes.Structure):
    _fields_ = [("n_retrieval", ctypes.c_int32), ("n_sink", ctypes.c_int32),
                ("window", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("retrieval_heads", ctypes.c_void_p), ("t", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_SZ = ctypes.c_size_t
_U32 = ctypes.c_uint32
_F32 = ctypes.c_float
_CACHE_P = ctypes.POINTER(kvc_cache)
_ROPE_P = ctypes.POINTER(kvc_rope)
_ALIBI_P = ctypes.POINTER(kvc_alibi)
_POOL_P = ctypes.POINTER(kvc_block_pool)
_PT_P = ctypes.POINTER(kvc_page_table)
_FREE_P = ctypes.POINTER(kvc_free_pool)
_DUO_P = ctypes.POINTER(kvc_duo)

# name -> (restype, argtypes); every symbol declared in include/kvc.h
SIGNATURES = {
    "kvc_last_error": (ctypes.c_char_p, []),
    "kvc_device_status": (_I32, [_P, ctypes.POINTER(_I32)]),
    "kvc_kv_bytes": (_U64, [_U64] * 6),
    "kvc_pyramid_budgets": (_I32, [_I32, _I64, _I64, _I64, _P]),
    "kvc_rope_table": (_I32, [_I32, _I32, ctypes.c_double, _P]),
    "kvc_snapkv_select_workspace_bytes": (_SZ, [_I32] * 6),
    "kvc_snapkv_select": (_I32, [_P, _CACHE_P, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P, _P,
                                 _SZ, _P]),
    "kvc_compact_gather": (_I32, [_CACHE_P, _P, _I64, _I32, _CACHE_P, _P, _I64, _P, _P]),
    "kvc_stream_append": (_I32, [_CACHE_P, _I32, _P, _P, _P, _P, _I32, _I32, _P, _P, _I64, _P,
                                 _I64, _P]),
    "kvc_position_advance": (_I32, [_P, _I64, _P]),
    "kvc_decode_attn_workspace_bytes": (_SZ, [_I32] * 5),
    "kvc_decode_attn": (_I32, [_P, _I32, _CACHE_P, _P, _I32, _ROPE_P, _F32, _P, _P, _I64, _P,
                               _P, _SZ, _P]),
    "kvc_decode_attn_ex": (_I32, [_P, _I32, _CACHE_P, _P, _I32, _ROPE_P, _F32, _P, _P, _I64,
                                  _P, _P, _SZ, _U32, _P]),
    "kvc_decode_attn_alibi": (_I32, [_P, _I32, _CACHE_P, _ALIBI_P, _F32, _P, _P, _I64, _P, _P,
                                     _SZ, _U32, _P]),
    "kvc_alibi_slopes": (_I32, [_I32, _P]),
    "kvc_duo_kv_bytes": (_U64, [_U64] * 9),
    "kvc_duo_append": (_I32, [_CACHE_P, _P, _CACHE_P, _DUO_P, _P, _P, _P]),
    "kvc_decode_attn_duo_workspace_bytes": (_SZ, [_I32] * 6),
    "kvc_decode_attn_duo": (_I32, [_P, _I32, _CACHE_P, _P, _I32, _CACHE_P, _DUO_P, _F32, _P, _P,
                                   _I64, _P, _P, _SZ, _U32, _P]),
    "kvc_paged_append": (_I32, [_POOL_P, _PT_P, _FREE_P, _P, _P, _P, _P, _P]),
    "kvc_decode_attn_paged": (_I32, [_P, _I32, _POOL_P, _PT_P, _F32, _P, _P, _I64, _P, _P, _SZ,
                                     _U32, _P]),
    "kvc_block_prompt_select_workspace_bytes": (_SZ, [_I32] * 4),
    "kvc_block_prompt_select": (_I32, [_P, _I64, _CACHE_P, _I32, _POOL_P, _PT_P, _FREE_P, _I32,
                                       _I32, _P, _SZ, _P]),
    "kvc_block_accumulate_evict": (_I32, [_P, _I64, _P, _I32, _I32, _PT_P, _FREE_P, _I32, _I32,
                                          _P, _P]),
    "kvc_decode_attn_noalloc": (_I32, [_P, _I32, _CACHE_P, _P, _I32, _ROPE_P, _F32, _P, _P,
                                       _I64, _P, _P]),
    "kvc_h2o_accumulate_evict": (_I32, [_P, _I64, _P, _P, _P, _I64, _P, _I32, _I32, _I32, _P,
                                        _I32, _I32, _P]),
    "kvc_h2o_accumulate_evict_gqa": (_I32, [_P, _I64, _P, _P, _P, _I64, _P, _I32, _I32, _I32,
                                            _I32, _P, _I32, _I32, _P]),
    "kvc_h2o_prefill_workspace_bytes": (_SZ, [_I32] * 4),
    "kvc_h2o_prefill_gqa_workspace_bytes": (_SZ, [_I32] * 5),
    "kvc_h2o_prefill_select_gqa": (_I32, [_P, _I32, _CACHE_P, _I32, _I32, _I32, _F32, _P, _P, _P,
                                          _P, _SZ, _P]),
    "kvc_h2o_prefill_select": (_I32, [_P, _CACHE_P, _I32, _I32, _I32, _F32, _P, _P, _P, _P,
                                      _SZ, _P]),
}

_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libkvc.so (built in-tree).  Raises if it is missing: there is no fallback path."""
    global _lib
    with _lib_lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libkvc.so not found at {path}: build it with "
                                   "kv_cache_compression_kvc_gb300.build.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int):
    if status != KVC_OK:
        raise KvcError(status, load().kvc_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return KVC_F32
    if dt == torch.bfloat16:
        return KVC_BF16
    raise TypeError(f"unsupported element type {dt} (float32 or bfloat16)")


def cache_view(k: torch.Tensor, v: Optional[torch.Tensor] = None) -> kvc_cache:
    """Describe K (and V) tensors shaped [batch, n_heads_kv, cap, d_head] (d_head contiguous)."""
    if k.dim() != 4 or k.stride(3) != 1:
        raise ValueError("cache tensors are [batch, n_heads_kv, cap, d_head], d_head contiguous")
    if v is not None and (v.shape != k.shape or v.stride() != k.stride() or v.dtype != k.dtype):
        raise ValueError("k and v must have the same shape, strides and dtype")
    c = kvc_cache()
    c.k = k.data_ptr()
    c.v = v.data_ptr() if v is not None else None
    c.dtype = _dtype_code(k.dtype)
    c.batch, c.n_heads_kv, c.cap, c.d_head = (int(x) for x in k.shape)
    c.stride_b, c.stride_h, c.stride_slot = k.stride(0), k.stride(1), k.stride(2)
    c._keep = (k, v)                # the descriptor holds their addresses: keep them alive
    return c


# ------------------------------------------------------------------------------------------
def kvc_last_error() -> str:
    return load().kvc_last_error().decode()


def kvc_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device range-check code."""
    code = _I32(0)
    st = load().kvc_device_status(_stream(stream), ctypes.byref(code))
    if st not in (KVC_OK, 7):
        _check(st)
    return int(code.value)


def kvc_kv_bytes(n_layers, n_heads_kv, d_head, seq_len, bytes_per_elem, batch) -> int:
    return int(load().kvc_kv_bytes(n_layers, n_heads_kv, d_head, seq_len, bytes_per_elem, batch))


def kvc_pyramid_budgets(n_layers: int, b_target: int, ratio_num: int = 4, ratio_den: int = 1):
    out = (ctypes.c_int64 * n_layers)()
    _check(load().kvc_pyramid_budgets(n_layers, b_target, ratio_num, ratio_den, out))
    return [int(x) for x in out]


def kvc_rope_table(n_pos: int, d_head: int, theta: float = 10000.0) -> torch.Tensor:
    """Host fp32 table [n_pos, 2, d_head/2] (cosines, then sines); upload it for decode."""
    out = torch.empty((n_pos, 2, d_head // 2), dtype=torch.float32)
    _check(load().kvc_rope_table(n_pos, d_head, theta, _ptr(out)))
    return out


def _zeroed_workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    return torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)


def _ws_ptr(ws: Optional[torch.Tensor]):
    """256-byte aligned pointer inside a workspace tensor and the bytes available after it."""
    if ws is None:
        return None, 0
    base = ws.data_ptr()
    aligned = (base + 255) & ~255
    return ctypes.c_void_p(aligned), ws.numel() * ws.element_size() - (aligned - base)


# ------------------------------------------------------------------------------------------
def kvc_decode_attn_workspace_bytes(batch, n_heads_q, n_heads_kv, d_head, cap) -> int:
    return int(load().kvc_decode_attn_workspace_bytes(batch, n_heads_q, n_heads_kv, d_head, cap))


def decode_workspace(batch, n_heads_q, n_heads_kv, d_head, cap, device) -> Optional[torch.Tensor]:
    """A zero-filled workspace for kvc_decode_attn (zeroed once; the kernel keeps it zeroed)."""
    return _zeroed_workspace(
        kvc_decode_attn_workspace_bytes(batch, n_heads_q, n_heads_kv, d_head, cap), device)


def make_rope(n_sink: int, window: int, t: torch.Tensor, cos_sin: torch.Tensor) -> kvc_rope:
    r = kvc_rope()
    r.n_sink, r.window = n_sink, window
    r.t = t.data_ptr()
    r.cos_sin = cos_sin.data_ptr()
    r.n_pos = cos_sin.shape[0]
    r._keep = (t, cos_sin)          # the descriptor holds their addresses: keep them alive
    return r


def kvc_decode_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                    scale: float, len: Optional[torch.Tensor] = None,
                    n_valid: Optional[int] = None, rope: Optional[kvc_rope] = None,
                    out: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    stream=None, cache: Optional[kvc_cache] = None) -> torch.Tensor:
    """q [B, Hq, D] -> out [B, Hq, D] fp32 (see kvc.h for valid slots and logits layout)."""
    c = cache if cache is not None else cache_view(k_cache, v_cache)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(B, Hq, c.n_heads_kv, D, c.cap, q.device)
    wp, wb = _ws_ptr(ws)
    lstride = logits.stride(-2) if logits is not None else 0
    _check(load().kvc_decode_attn(
        _ptr(q), Hq, ctypes.byref(c), _ptr(len), -1 if n_valid is None else int(n_valid),
        ctypes.byref(rope) if rope is not None else None, float(scale), _ptr(out),
        _ptr(logits), lstride, _ptr(lse), wp, wb, _stream(stream)))
    return out


def kvc_decode_attn_ex(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                       scale: float, flags: int = 0, len: Optional[torch.Tensor] = None,
                       n_valid: Optional[int] = None, rope: Optional[kvc_rope] = None,
                       out: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                       stream=None, cache: Optional[kvc_cache] = None) -> torch.Tensor:
    """kvc_decode_attn with flags (KVC_DECODE_KV_SETTLED: see kvc.h for the caller's promise)."""
    c = cache if cache is not None else cache_view(k_cache, v_cache)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(B, Hq, c.n_heads_kv, D, c.cap, q.device)
    wp, wb = _ws_ptr(ws)
    lstride = logits.stride(-2) if logits is not None else 0
    _check(load().kvc_decode_attn_ex(
        _ptr(q), Hq, ctypes.byref(c), _ptr(len), -1 if n_valid is None else int(n_valid),
        ctypes.byref(rope) if rope is not None else None, float(scale), _ptr(out),
        _ptr(logits), lstride, _ptr(lse), wp, wb, int(flags), _stream(stream)))
    return out


def kvc_alibi_slopes(n_heads: int) -> torch.Tensor:
    """Host fp32 [n_heads]: 2^(-8 (h+1) / n_heads) (power-of-two head counts)."""
    out = torch.empty(n_heads, dtype=torch.float32)
    _check(load().kvc_alibi_slopes(n_heads, _ptr(out)))
    return out


def make_alibi(n_sink: int, window: int, t: torch.Tensor, slopes: torch.Tensor) -> kvc_alibi:
    a = kvc_alibi()
    a.n_sink, a.window = n_sink, window
    a.t = t.data_ptr()
    a.slopes = slopes.data_ptr()
    a._keep = (t, slopes)           # the descriptor holds their addresses: keep them alive
    return a


def kvc_decode_attn_alibi(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                          scale: float, alibi: kvc_alibi, flags: int = 0,
                          out: Optional[torch.Tensor] = None,
                          logits: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                          stream=None, cache: Optional[kvc_cache] = None) -> torch.Tensor:
    """StreamingLLM decode with ALiBi at in-cache positions: q [B, Hq, D] -> out [B, Hq, D]."""
    c = cache if cache is not None else cache_view(k_cache, v_cache)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(B, Hq, c.n_heads_kv, D, c.cap, q.device)
    wp, wb = _ws_ptr(ws)
    lstride = logits.stride(-2) if logits is not None else 0
    _check(load().kvc_decode_attn_alibi(
        _ptr(q), Hq, ctypes.byref(c), ctypes.byref(alibi), float(scale), _ptr(out),
        _ptr(logits), lstride, _ptr(lse), wp, wb, int(flags), _stream(stream)))
    return out


def block_pool_view(k_pool: torch.Tensor, v_pool: torch.Tensor) -> kvc_block_pool:
    """Describe a block pool: K and V tensors [n_heads_kv, n_blocks, block_size, d_head]
    (head-major), contiguous."""
    if k_pool.dim() != 4 or not k_pool.is_contiguous() or v_pool.shape != k_pool.shape or \
            not v_pool.is_contiguous() or v_pool.dtype != k_pool.dtype:
        raise ValueError("block pools are contiguous [n_heads_kv, n_blocks, block_size, d_head]")
    c = kvc_block_pool()
    c.k, c.v = k_pool.data_ptr(), v_pool.data_ptr()
    c.dtype = _dtype_code(k_pool.dtype)
    c.n_heads_kv, c.n_blocks, c.block_size, c.d_head = (int(x) for x in k_pool.shape)
    c._keep = (k_pool, v_pool)
    return c


def page_table_view(table: torch.Tensor, n_blocks: torch.Tensor, len: torch.Tensor,
                    score: torch.Tensor) -> kvc_page_table:
    """table int32 [batch, max_blocks], n_blocks / len int32 [batch], score fp32
    [batch, max_blocks], all contiguous."""
    B, mb = table.shape
    if table.dtype != torch.int32 or n_blocks.dtype != torch.int32 or len.dtype != torch.int32 \
            or score.dtype != torch.float32 or tuple(score.shape) != (B, mb) or \
            not (table.is_contiguous() and score.is_contiguous()):
        raise ValueError("page table: int32 table [B, max_blocks], int32 n_blocks/len [B], "
                         "fp32 score [B, max_blocks]")
    c = kvc_page_table()
    c.table, c.n_blocks, c.len, c.score = (table.data_ptr(), n_blocks.data_ptr(), len.data_ptr(),
                                           score.data_ptr())
    c.batch, c.max_blocks = B, mb
    c._keep = (table, n_blocks, len, score)
    return c


def free_pool_view(ids: torch.Tensor, top: torch.Tensor) -> kvc_free_pool:
    """ids int32 [capacity] (a stack, ids[:top]), top int32 [1]."""
    c = kvc_free_pool()
    c.ids, c.top = ids.data_ptr(), top.data_ptr()
    c.capacity = ids.numel()
    c._keep = (ids, top)
    return c


def kvc_paged_append(pool: kvc_block_pool, pt: kvc_page_table, free_pool: kvc_free_pool,
                     k_new: torch.Tensor, v_new: torch.Tensor, *,
                     t: Optional[torch.Tensor] = None, pos: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    _check(load().kvc_paged_append(ctypes.byref(pool), ctypes.byref(pt), ctypes.byref(free_pool),
                                   _ptr(k_new), _ptr(v_new), _ptr(t), _ptr(pos),
                                   _stream(stream)))


def kvc_decode_attn_paged(q: torch.Tensor, pool: kvc_block_pool, pt: kvc_page_table, *,
                          scale: float, flags: int = 0, out: Optional[torch.Tensor] = None,
                          logits: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """q [B, Hq, D] -> out [B, Hq, D] fp32 over each sequence's page table."""
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(B, Hq, pool.n_heads_kv, D, pt.max_blocks * pool.block_size,
                              q.device)
    wp, wb = _ws_ptr(ws)
    lstride = logits.stride(-2) if logits is not None else 0
    _check(load().kvc_decode_attn_paged(
        _ptr(q), Hq, ctypes.byref(pool), ctypes.byref(pt), float(scale), _ptr(out),
        _ptr(logits), lstride, _ptr(lse), wp, wb, int(flags), _stream(stream)))
    return out


def kvc_block_prompt_select(s: torch.Tensor, k_prompt: torch.Tensor, v_prompt: torch.Tensor,
                            pool: kvc_block_pool, pt: kvc_page_table, free_pool: kvc_free_pool, *,
                            seq_len: int, budget_blocks: int, recent_blocks: int,
                            ws: Optional[torch.Tensor] = None, stream=None) -> None:
    """s [B, Hkv, >= seq_len] per-token prompt scores; k/v_prompt [B, Hkv, cap, D]."""
    c = cache_view(k_prompt, v_prompt)
    if ws is None:
        ws = _zeroed_workspace(int(load().kvc_block_prompt_select_workspace_bytes(
            pt.batch, seq_len, pool.block_size, budget_blocks)), s.device)
    wp, wb = _ws_ptr(ws)
    _check(load().kvc_block_prompt_select(
        _ptr(s), s.stride(-2), ctypes.byref(c), int(seq_len), ctypes.byref(pool),
        ctypes.byref(pt), ctypes.byref(free_pool), int(budget_blocks), int(recent_blocks), wp, wb,
        _stream(stream)))


def kvc_block_accumulate_evict(logits: torch.Tensor, lse: torch.Tensor, pt: kvc_page_table,
                               free_pool: kvc_free_pool, *, block_size: int, budget_blocks: int,
                               recent_blocks: int, released: Optional[torch.Tensor] = None,
                               stream=None) -> None:
    """logits [B, Hq, >= max_blocks*block_size], lse [B, Hq]."""
    B, Hq = lse.shape
    _check(load().kvc_block_accumulate_evict(
        _ptr(logits), logits.stride(-2), _ptr(lse), Hq, int(block_size), ctypes.byref(pt),
        ctypes.byref(free_pool), int(budget_blocks), int(recent_blocks), _ptr(released),
        _stream(stream)))


class Duo:
    """A kvc_duo descriptor with the host array of retrieval heads it points to kept alive."""

    def __init__(self, retrieval_heads, n_sink: int, window: int, t: torch.Tensor):
        heads = [int(h) for h in retrieval_heads]
        self._heads = (ctypes.c_int32 * max(1, len(heads)))(*heads)
        self.desc = kvc_duo()
        self.desc.n_retrieval = len(heads)
        self.desc.n_sink, self.desc.window = n_sink, window
        self.desc.retrieval_heads = ctypes.cast(self._heads, ctypes.c_void_p)
        self.desc.t = t.data_ptr()
        self._t = t                     # the descriptor holds its address: keep it alive


def kvc_duo_kv_bytes(n_layers, n_retrieval, n_streaming, d_head, seq_len, n_sink, window,
                     bytes_per_elem, batch) -> int:
    return int(load().kvc_duo_kv_bytes(n_layers, n_retrieval, n_streaming, d_head, seq_len,
                                       n_sink, window, bytes_per_elem, batch))


def kvc_duo_append(full: kvc_cache, len: torch.Tensor, ring: kvc_cache, duo: Duo,
                   k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    _check(load().kvc_duo_append(ctypes.byref(full), _ptr(len), ctypes.byref(ring),
                                 ctypes.byref(duo.desc), _ptr(k_new), _ptr(v_new),
                                 _stream(stream)))


def kvc_decode_attn_duo_workspace_bytes(batch, n_heads_q, n_heads_kv, d_head, cap,
                                        n_retrieval) -> int:
    return int(load().kvc_decode_attn_duo_workspace_bytes(batch, n_heads_q, n_heads_kv, d_head,
                                                          cap, n_retrieval))


def kvc_decode_attn_duo(q: torch.Tensor, full: kvc_cache, ring: kvc_cache, duo: Duo, *,
                        scale: float, len: Optional[torch.Tensor] = None,
                        n_valid: Optional[int] = None, flags: int = 0,
                        out: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """q [B, Hq, D] (model head order) -> out [B, Hq, D] fp32."""
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = _zeroed_workspace(kvc_decode_attn_duo_workspace_bytes(
            B, Hq, full.n_heads_kv + ring.n_heads_kv, D, full.cap, duo.desc.n_retrieval),
            q.device)
    wp, wb = _ws_ptr(ws)
    lstride = logits.stride(-2) if logits is not None else 0
    _check(load().kvc_decode_attn_duo(
        _ptr(q), Hq, ctypes.byref(full), _ptr(len), -1 if n_valid is None else int(n_valid),
        ctypes.byref(ring), ctypes.byref(duo.desc), float(scale), _ptr(out), _ptr(logits),
        lstride, _ptr(lse), wp, wb, int(flags), _stream(stream)))
    return out


def kvc_decode_attn_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                            scale: float, len: Optional[torch.Tensor] = None,
                            n_valid: Optional[int] = None, rope: Optional[kvc_rope] = None,
                            out: Optional[torch.Tensor] = None,
                            logits: Optional[torch.Tensor] = None,
                            lse: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """kvc_decode_attn without a workspace (the library's fixed 8 MiB scratch is used)."""
    c = cache_view(k_cache, v_cache)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    lstride = logits.stride(-2) if logits is not None else 0
    _check(load().kvc_decode_attn_noalloc(
        _ptr(q), Hq, ctypes.byref(c), _ptr(len), -1 if n_valid is None else int(n_valid),
        ctypes.byref(rope) if rope is not None else None, float(scale), _ptr(out),
        _ptr(logits), lstride, _ptr(lse), _stream(stream)))
    return out


def kvc_stream_append(k_cache: torch.Tensor, v_cache: torch.Tensor, policy: int,
                      k_new: torch.Tensor, v_new: torch.Tensor, *,
                      t: Optional[torch.Tensor] = None, len: Optional[torch.Tensor] = None,
                      n_sink: int = 0, window: int = 0,
                      free_slot: Optional[torch.Tensor] = None,
                      pos: Optional[torch.Tensor] = None, score: Optional[torch.Tensor] = None,
                      stream=None, cache: Optional[kvc_cache] = None) -> None:
    c = cache if cache is not None else cache_view(k_cache, v_cache)
    _check(load().kvc_stream_append(
        ctypes.byref(c), policy, _ptr(k_new), _ptr(v_new), _ptr(t), _ptr(len), n_sink, window,
        _ptr(free_slot), _ptr(pos), pos.stride(-2) if pos is not None else 0, _ptr(score),
        score.stride(-2) if score is not None else 0, _stream(stream)))


def kvc_position_advance(t: torch.Tensor, delta: int = 1, stream=None) -> None:
    _check(load().kvc_position_advance(_ptr(t), int(delta), _stream(stream)))


def kvc_compact_gather(k_src: torch.Tensor, v_src: torch.Tensor, idx: torch.Tensor, n_keep: int,
                       k_dst: torch.Tensor, v_dst: torch.Tensor, *,
                       pos_dst: Optional[torch.Tensor] = None,
                       len_dst: Optional[torch.Tensor] = None, stream=None) -> None:
    src, dst = cache_view(k_src, v_src), cache_view(k_dst, v_dst)
    _check(load().kvc_compact_gather(
        ctypes.byref(src), _ptr(idx), idx.stride(-2), int(n_keep), ctypes.byref(dst),
        _ptr(pos_dst), pos_dst.stride(-2) if pos_dst is not None else 0, _ptr(len_dst),
        _stream(stream)))


def kvc_snapkv_select_workspace_bytes(batch, n_heads_q, n_heads_kv, d_head, seq_len, L_obs):
    return int(load().kvc_snapkv_select_workspace_bytes(batch, n_heads_q, n_heads_kv, d_head,
                                                        seq_len, L_obs))


def kvc_snapkv_select(q_obs: torch.Tensor, k_prompt: torch.Tensor, *, seq_len: int, L_obs: int,
                      budget: int, scale: float, pool_k: int = 5,
                      idx_out: Optional[torch.Tensor] = None,
                      scores_out: Optional[torch.Tensor] = None,
                      ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q_obs [B, Hq, L_obs, D]; k_prompt [B, Hkv, cap, D] -> idx [B, Hkv, min(budget, seq_len)]."""
    c = cache_view(k_prompt)
    B, Hq = q_obs.shape[0], q_obs.shape[1]
    n_keep = min(budget, seq_len)
    if idx_out is None:
        idx_out = torch.empty((B, c.n_heads_kv, n_keep), dtype=torch.int32, device=q_obs.device)
    if ws is None:
        ws = _zeroed_workspace(kvc_snapkv_select_workspace_bytes(
            B, Hq, c.n_heads_kv, c.d_head, seq_len, L_obs), q_obs.device)
    wp, wb = _ws_ptr(ws)
    _check(load().kvc_snapkv_select(
        _ptr(q_obs), ctypes.byref(c), Hq, seq_len, L_obs, pool_k, budget, float(scale),
        _ptr(idx_out), _ptr(scores_out), wp, wb, _stream(stream)))
    return idx_out


def kvc_h2o_accumulate_evict(logits: torch.Tensor, lse: torch.Tensor, score: torch.Tensor,
                             pos: torch.Tensor, free_slot: torch.Tensor, *, n_slots: int,
                             t: torch.Tensor, L_local: int, budget: int, stream=None) -> None:
    """logits [B, H, >=n_slots], lse [B, H], score/pos [B, H, stride], free_slot [B, H]."""
    B, H = lse.shape
    if score.stride(-2) != pos.stride(-2):
        raise ValueError("score and pos must share a row stride")
    _check(load().kvc_h2o_accumulate_evict(
        _ptr(logits), logits.stride(-2), _ptr(lse), _ptr(score), _ptr(pos), score.stride(-2),
        _ptr(free_slot), B, H, int(n_slots), _ptr(t), int(L_local), int(budget),
        _stream(stream)))


def kvc_h2o_accumulate_evict_gqa(logits: torch.Tensor, lse: torch.Tensor, score: torch.Tensor,
                                 pos: torch.Tensor, free_slot: torch.Tensor, *, n_slots: int,
                                 t: torch.Tensor, L_local: int, budget: int,
                                 stream=None) -> None:
    """logits [B, Hq, >=n_slots], lse [B, Hq]; score/pos [B, Hkv, stride], free_slot [B, Hkv]."""
    B, Hq = lse.shape
    Hkv = score.shape[1]
    if score.stride(-2) != pos.stride(-2):
        raise ValueError("score and pos must share a row stride")
    _check(load().kvc_h2o_accumulate_evict_gqa(
        _ptr(logits), logits.stride(-2), _ptr(lse), _ptr(score), _ptr(pos), score.stride(-2),
        _ptr(free_slot), B, Hq, Hkv, int(n_slots), _ptr(t), int(L_local), int(budget),
        _stream(stream)))


def kvc_h2o_prefill_workspace_bytes(batch, n_heads, d_head, seq_len) -> int:
    return int(load().kvc_h2o_prefill_workspace_bytes(batch, n_heads, d_head, seq_len))


def kvc_h2o_prefill_select(q: torch.Tensor, k_prompt: torch.Tensor, *, seq_len: int,
                           L_local: int, K_hh: int, scale: float,
                           idx_out: Optional[torch.Tensor] = None,
                           score_out: Optional[torch.Tensor] = None,
                           s_full: Optional[torch.Tensor] = None,
                           ws: Optional[torch.Tensor] = None, stream=None):
    """q [B, H, N, D]; k_prompt [B, H, cap, D] -> (idx [B, H, n_keep], score [B, H, n_keep])."""
    c = cache_view(k_prompt)
    B, H = q.shape[0], q.shape[1]
    n_keep = min(seq_len, K_hh + L_local)
    if idx_out is None:
        idx_out = torch.empty((B, H, n_keep), dtype=torch.int32, device=q.device)
    if score_out is None:
        score_out = torch.empty((B, H, n_keep), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = _zeroed_workspace(kvc_h2o_prefill_workspace_bytes(B, H, c.d_head, seq_len), q.device)
    wp, wb = _ws_ptr(ws)
    _check(load().kvc_h2o_prefill_select(
        _ptr(q), ctypes.byref(c), seq_len, L_local, K_hh, float(scale), _ptr(idx_out),
        _ptr(score_out), _ptr(s_full), wp, wb, _stream(stream)))
    return idx_out, score_out


def kvc_h2o_prefill_gqa_workspace_bytes(batch, n_heads_kv, d_head, seq_len, dtype) -> int:
    return int(load().kvc_h2o_prefill_gqa_workspace_bytes(batch, n_heads_kv, d_head, seq_len,
                                                           dtype))


def kvc_h2o_prefill_select_gqa(q: torch.Tensor, k_prompt: torch.Tensor, *, seq_len: int,
                               L_local: int, K_hh: int, scale: float,
                               idx_out: Optional[torch.Tensor] = None,
                               score_out: Optional[torch.Tensor] = None,
                               s_full: Optional[torch.Tensor] = None,
                               ws: Optional[torch.Tensor] = None, stream=None):
    """q [B, Hq, N, D]; k_prompt [B, Hkv, cap, D] -> (idx [B, Hkv, n_keep], score [B, Hkv, n_keep])."""
    c = cache_view(k_prompt)
    B, Hq = q.shape[0], q.shape[1]
    # the library reads q as a contiguous [batch][Hq][seq_len][d_head] array of the prompt's type
    # and writes batch * Hkv * seq_len floats to s_full: check both before handing over pointers
    if q.dim() != 4 or not q.is_contiguous() or q.dtype != k_prompt.dtype or \
            tuple(q.shape) != (c.batch, Hq, int(seq_len), c.d_head):
        raise ValueError(f"q must be a contiguous {k_prompt.dtype} tensor "
                         f"[{c.batch}, n_heads_q, {seq_len}, {c.d_head}], got "
                         f"{q.dtype} {tuple(q.shape)}")
    if s_full is not None and (s_full.dtype != torch.float32 or not s_full.is_contiguous() or
                               tuple(s_full.shape) != (c.batch, c.n_heads_kv, int(seq_len))):
        raise ValueError(f"s_full must be a contiguous float32 tensor "
                         f"[{c.batch}, {c.n_heads_kv}, {seq_len}]")
    n_keep = min(seq_len, K_hh + L_local)
    if idx_out is None:
        idx_out = torch.empty((B, c.n_heads_kv, n_keep), dtype=torch.int32, device=q.device)
    if score_out is None:
        score_out = torch.empty((B, c.n_heads_kv, n_keep), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = _zeroed_workspace(kvc_h2o_prefill_gqa_workspace_bytes(
            B, c.n_heads_kv, c.d_head, seq_len, c.dtype), q.device)
    wp, wb = _ws_ptr(ws)
    _check(load().kvc_h2o_prefill_select_gqa(
        _ptr(q), Hq, ctypes.byref(c), seq_len, L_local, K_hh, float(scale), _ptr(idx_out),
        _ptr(score_out), _ptr(s_full), wp, wb, _stream(stream)))
    return idx_out, score_out
