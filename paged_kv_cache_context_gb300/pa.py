"""Python binding of the C ABI in include/pa.h (argument marshalling only).

Every function takes torch CUDA tensors, passes their device pointers and
sizes to the same-named C entry point of ``libpagedattn.so`` on the current
torch stream, and raises ``PagedAttentionError`` on a non-zero status. All
computation runs in the library's CUDA kernels; there is no fallback: if the
library is missing, loading fails loudly.

The sizes the C calls receive are read from the tensors' shapes, so before a
call the binding checks what the C side cannot see: that every tensor is a
CUDA tensor on one device (the library takes raw device pointers) and that
the shapes and element types of the arguments agree with each other. A
mismatch raises ``ValueError`` and nothing is enqueued.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpagedattn.so")

# enums of include/pa.h
PA_F32, PA_BF16, PA_F16 = 0, 1, 2
PA_KV_AUTO, PA_KV_FP8_E4M3, PA_KV_INT8 = 0, 1, 2
PA_ERR_DEVICE = -9
DEVERR_BITS = {1: "slot", 2: "block_id", 4: "context_len", 8: "timeout", 16: "seq"}

_DTYPE = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float16: PA_F16}
_KV = {"auto": PA_KV_AUTO, "fp8_e4m3": PA_KV_FP8_E4M3, "int8": PA_KV_INT8}

_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "paged_kv_cache_context_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "pa_slot_mapping": [P, P, P, P, I, I, I, I, I, P],
            "pa_reshape_and_cache": [P, P, P, P, P, I, I, I, I, I, I, I, F, F, P],
            "pa_decode": [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, F, F, P, Z, P],
            "pa_decode_plan": [I, I, I, I, I, I, I, P, P],
            "pa_decode_workspace_size": [I, I, I, I, I, I, I],
            "pa_decode_partials": [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, F,
                                   F, I, I, P],
            "pa_reduce": [P, P, P, P, I, I, I, I, I, P],
            "pa_decode_balanced": [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, F, F, P,
                                   Z, P, P],
            "pa_decode_workspace_clear": [P, Z, P],
            "pa_decode_cascade_workspace_size": [I, I, I, I, I, I],
            "pa_decode_cascade": [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, Z, P],
            "pa_decode_cascade_fp8": [P, P, P, P, P, P, I, I, I, I, I, I, I, F, F, F, I, I, P, Z,
                                      P],
            "pa_decode_cascade_int8": [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, Z,
                                       P],
            "pa_copy_blocks": [P, P, P, I, I, I, I, I, I, P],
            "pa_block_budget": [I, ctypes.c_double, Z, I, I, I, I, I, I],
            "pa_reshape_and_cache_int8": [P, P, P, P, P, P, P, I, I, I, I, I, I, P],
            "pa_decode_int8": [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, Z, P],
            "pa_prefill": [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P],
            "pa_prefill_int8": [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P],
            "pa_prefill_fp8": [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, F, F, I, P],
            "pa_decode_static_scratch": [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, F,
                                         F, P],
            "pa_get_device_error": [P, P],
            "pa_status_string": [I],
            "pa_version": [],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = I
        L.pa_decode_workspace_size.restype = Z
        L.pa_decode_cascade_workspace_size.restype = Z
        L.pa_block_budget.restype = ctypes.c_int64
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_test_set_unarmed_page.argtypes = [I]
        L.pa_test_set_unarmed_page.restype = None
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(status).decode()


def version() -> int:
    return lib().pa_version()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _is_device_tensor(t: torch.Tensor) -> bool:
    return t.is_cuda


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _on_device(**named):
    """Every tensor argument is a CUDA tensor, all on one device."""
    dev = None
    for name, t in named.items():
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name}: expected a torch tensor")
        if not _is_device_tensor(t):
            raise ValueError(f"{name}: must be a CUDA tensor (the library takes device pointers)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name}: every tensor must be on {dev}")


def _shape(name: str, t: torch.Tensor, shape):
    if t.shape != shape:
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dtype(name: str, t: torch.Tensor, dt: torch.dtype):
    if t.dtype != dt:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dt}")


_CACHE_DTYPE = {"fp8_e4m3": torch.uint8, "int8": torch.int8}


def _check_caches(k_cache, v_cache, num_kv_heads: int, head_dim: int, dtype: torch.dtype):
    _need(k_cache.dim() == 4, "k_cache: expected [num_blocks, num_kv_heads, block_size, D]")
    _shape("v_cache", v_cache, k_cache.shape)
    if k_cache.shape[1] != num_kv_heads or k_cache.shape[3] != head_dim:
        raise ValueError(f"k_cache: shape {tuple(k_cache.shape)} does not hold {num_kv_heads} "
                         f"kv heads of dimension {head_dim}")
    _dtype("k_cache", k_cache, dtype)
    _dtype("v_cache", v_cache, dtype)


def _check_scales(k_scales, v_scales, k_cache):
    for name, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _shape(name, t, k_cache.shape[:3])
        _dtype(name, t, torch.float32)


def _check_decode_args(out, query, k_cache, v_cache, block_tables, context_lens,
                       num_kv_heads: int, cache_dtype: torch.dtype):
    _need(query.dim() == 3, "query: expected [num_seqs, num_heads, head_dim]")
    S, Hq, D = query.shape
    _shape("out", out, query.shape)
    _dtype("out", out, query.dtype)
    _check_caches(k_cache, v_cache, num_kv_heads, D, cache_dtype)
    if block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError(f"block_tables: expected [{S}, max_blocks_per_seq]")
    _dtype("block_tables", block_tables, torch.int32)
    _shape("context_lens", context_lens, (S,))
    _dtype("context_lens", context_lens, torch.int32)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(rc: int, what: str):
    if rc != 0:
        raise PagedAttentionError(rc, what)


def slot_mapping(out: torch.Tensor, block_tables: torch.Tensor, seq_idx: Optional[torch.Tensor],
                 positions: torch.Tensor, block_size: int, window: int = 0, stream=None):
    """pa_slot_mapping: out[t] = cache slot of token t (ring-aware)."""
    _on_device(out=out, block_tables=block_tables, seq_idx=seq_idx, positions=positions)
    _need(block_tables.dim() == 2, "block_tables: expected [num_seqs, max_blocks_per_seq]")
    _dtype("block_tables", block_tables, torch.int32)
    _dtype("positions", positions, torch.int32)
    _shape("out", out, (positions.numel(),))
    _dtype("out", out, torch.int64)
    if seq_idx is not None:
        _shape("seq_idx", seq_idx, (positions.numel(),))
        _dtype("seq_idx", seq_idx, torch.int32)
    S, MB = block_tables.shape
    _check(lib().pa_slot_mapping(_ptr(out), _ptr(block_tables), _ptr(seq_idx), _ptr(positions),
                                 positions.numel(), S, MB, block_size, window, _stream(stream)),
           "pa_slot_mapping")


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping_: torch.Tensor, kv_dtype: str = "auto",
                      k_scale: float = 1.0, v_scale: float = 1.0, stream=None):
    """pa_reshape_and_cache: key/value [T, Hkv, D] into caches [NB, Hkv, bs, D]."""
    _on_device(key=key, value=value, k_cache=k_cache, v_cache=v_cache,
               slot_mapping=slot_mapping_)
    _need(key.dim() == 3, "key: expected [num_tokens, num_kv_heads, head_dim]")
    _shape("value", value, key.shape)
    _dtype("value", value, key.dtype)
    _check_caches(k_cache, v_cache, key.shape[1], key.shape[2],
                  _CACHE_DTYPE.get(kv_dtype, key.dtype))
    _shape("slot_mapping", slot_mapping_, (key.shape[0],))
    _dtype("slot_mapping", slot_mapping_, torch.int64)
    T, H, D = key.shape
    NB, _, bs, _ = k_cache.shape
    _check(lib().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(slot_mapping_), T, H, D, bs, NB, _DTYPE[key.dtype],
                                      _KV[kv_dtype], k_scale, v_scale, _stream(stream)),
           "pa_reshape_and_cache")


def reshape_and_cache_int8(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                           slot_mapping_: torch.Tensor, stream=None):
    """pa_reshape_and_cache_int8: key/value [T, Hkv, D] into int8 caches
    [NB, Hkv, bs, D] and fp32 row scales [NB, Hkv, bs]."""
    _on_device(key=key, value=value, k_cache=k_cache, v_cache=v_cache, k_scales=k_scales,
               v_scales=v_scales, slot_mapping=slot_mapping_)
    _need(key.dim() == 3, "key: expected [num_tokens, num_kv_heads, head_dim]")
    _shape("value", value, key.shape)
    _dtype("value", value, key.dtype)
    _check_caches(k_cache, v_cache, key.shape[1], key.shape[2], torch.int8)
    _check_scales(k_scales, v_scales, k_cache)
    _shape("slot_mapping", slot_mapping_, (key.shape[0],))
    _dtype("slot_mapping", slot_mapping_, torch.int64)
    T, H, D = key.shape
    NB, _, bs, _ = k_cache.shape
    _check(lib().pa_reshape_and_cache_int8(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(k_scales), _ptr(v_scales), _ptr(slot_mapping_),
                                           T, H, D, bs, NB, _DTYPE[key.dtype], _stream(stream)),
           "pa_reshape_and_cache_int8")


def decode_int8(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                v_cache: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int,
                scale: float, window: int = 0, workspace: Optional[torch.Tensor] = None,
                stream=None):
    """pa_decode_int8: pa_decode over an INT8 cache with per-row scales."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache, k_scales=k_scales,
               v_scales=v_scales, block_tables=block_tables, context_lens=context_lens,
               workspace=workspace)
    _check_decode_args(out, query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       torch.int8)
    _check_scales(k_scales, v_scales, k_cache)
    S, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_int8(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                _ptr(k_scales), _ptr(v_scales), _ptr(block_tables),
                                _ptr(context_lens), S, Hq, num_kv_heads, D, bs, NB, MB, scale,
                                window, _DTYPE[query.dtype], _ptr(workspace), ws_bytes,
                                _stream(stream)), "pa_decode_int8")


def prefill(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
            v_cache: torch.Tensor, block_tables: torch.Tensor, cu_q: torch.Tensor,
            context_lens: torch.Tensor, num_kv_heads: int, max_q_len: int, scale: float,
            stream=None):
    """pa_prefill: causal attention of query [T, Hq, D] (the last tokens of each
    sequence's context, offsets cu_q [S + 1]) over the paged cache."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, cu_q=cu_q, context_lens=context_lens)
    _need(query.dim() == 3, "query: expected [num_tokens, num_heads, head_dim]")
    _shape("out", out, query.shape)
    _dtype("out", out, query.dtype)
    _check_caches(k_cache, v_cache, num_kv_heads, query.shape[2], query.dtype)
    _need(block_tables.dim() == 2, "block_tables: expected [num_seqs, max_blocks_per_seq]")
    _dtype("block_tables", block_tables, torch.int32)
    S = block_tables.shape[0]
    _shape("cu_q", cu_q, (S + 1,))
    _dtype("cu_q", cu_q, torch.int32)
    _shape("context_lens", context_lens, (S,))
    _dtype("context_lens", context_lens, torch.int32)
    T, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    S, MB = block_tables.shape
    _check(lib().pa_prefill(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                            _ptr(block_tables), _ptr(cu_q), _ptr(context_lens), T, S, Hq,
                            num_kv_heads, D, bs, NB, MB, max_q_len, scale, _DTYPE[query.dtype],
                            _stream(stream)), "pa_prefill")


def prefill_int8(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                 block_tables: torch.Tensor, cu_q: torch.Tensor, context_lens: torch.Tensor,
                 num_kv_heads: int, max_q_len: int, scale: float, stream=None):
    """pa_prefill_int8: pa_prefill over an INT8 cache with per-row scales."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache, k_scales=k_scales,
               v_scales=v_scales, block_tables=block_tables, cu_q=cu_q,
               context_lens=context_lens)
    _need(query.dim() == 3, "query: expected [num_tokens, num_heads, head_dim]")
    _shape("out", out, query.shape)
    _dtype("out", out, query.dtype)
    _check_caches(k_cache, v_cache, num_kv_heads, query.shape[2], torch.int8)
    _check_scales(k_scales, v_scales, k_cache)
    _need(block_tables.dim() == 2, "block_tables: expected [num_seqs, max_blocks_per_seq]")
    _dtype("block_tables", block_tables, torch.int32)
    S = block_tables.shape[0]
    _shape("cu_q", cu_q, (S + 1,))
    _dtype("cu_q", cu_q, torch.int32)
    _shape("context_lens", context_lens, (S,))
    _dtype("context_lens", context_lens, torch.int32)
    T, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    S, MB = block_tables.shape
    _check(lib().pa_prefill_int8(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(k_scales), _ptr(v_scales), _ptr(block_tables), _ptr(cu_q),
                                 _ptr(context_lens), T, S, Hq, num_kv_heads, D, bs, NB, MB,
                                 max_q_len, scale, _DTYPE[query.dtype], _stream(stream)),
           "pa_prefill_int8")


def prefill_fp8(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                v_cache: torch.Tensor, block_tables: torch.Tensor, cu_q: torch.Tensor,
                context_lens: torch.Tensor, num_kv_heads: int, max_q_len: int, scale: float,
                k_scale: float, v_scale: float, stream=None):
    """pa_prefill_fp8: pa_prefill over an FP8 E4M3 cache (uint8 codes) with
    per-tensor scales."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, cu_q=cu_q, context_lens=context_lens)
    _need(query.dim() == 3, "query: expected [num_tokens, num_heads, head_dim]")
    _shape("out", out, query.shape)
    _dtype("out", out, query.dtype)
    _check_caches(k_cache, v_cache, num_kv_heads, query.shape[2], torch.uint8)
    _need(block_tables.dim() == 2, "block_tables: expected [num_seqs, max_blocks_per_seq]")
    _dtype("block_tables", block_tables, torch.int32)
    S = block_tables.shape[0]
    _shape("cu_q", cu_q, (S + 1,))
    _dtype("cu_q", cu_q, torch.int32)
    _shape("context_lens", context_lens, (S,))
    _dtype("context_lens", context_lens, torch.int32)
    T, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    S, MB = block_tables.shape
    _check(lib().pa_prefill_fp8(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_tables), _ptr(cu_q), _ptr(context_lens), T, S, Hq,
                                num_kv_heads, D, bs, NB, MB, max_q_len, scale, k_scale, v_scale,
                                _DTYPE[query.dtype], _stream(stream)), "pa_prefill_fp8")


def decode_plan(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                block_size: int, max_blocks_per_seq: int, window: int = 0) -> Tuple[int, int]:
    """pa_decode_plan: (num_splits, pages_per_split)."""
    ns, pps = ctypes.c_int(), ctypes.c_int()
    _check(lib().pa_decode_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, window, ctypes.addressof(ns),
                                ctypes.addressof(pps)), "pa_decode_plan")
    return ns.value, pps.value


def decode_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                          block_size: int, max_blocks_per_seq: int, window: int = 0) -> int:
    return int(lib().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                              block_size, max_blocks_per_seq, window))


def decode(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int,
           scale: float, window: int = 0, kv_dtype: str = "auto", k_scale: float = 1.0,
           v_scale: float = 1.0, workspace: Optional[torch.Tensor] = None, stream=None):
    """pa_decode: out [S, Hq, D] = paged attention of query [S, Hq, D]."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, context_lens=context_lens, workspace=workspace)
    _check_decode_args(out, query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       _CACHE_DTYPE.get(kv_dtype, query.dtype))
    S, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                           _ptr(block_tables), _ptr(context_lens), S, Hq, num_kv_heads, D, bs, NB,
                           MB, scale, window, _DTYPE[query.dtype], _KV[kv_dtype], k_scale,
                           v_scale, _ptr(workspace), ws_bytes, _stream(stream)), "pa_decode")


def decode_balanced(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                    num_kv_heads: int, scale: float, workspace: torch.Tensor, window: int = 0,
                    kv_dtype: str = "auto", k_scale: float = 1.0, v_scale: float = 1.0,
                    stream=None) -> int:
    """pa_decode_balanced: the balanced path's decode launch (arrival counters
    must be zero: see decode_workspace_clear); returns num_ctas."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, context_lens=context_lens, workspace=workspace)
    _check_decode_args(out, query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       _CACHE_DTYPE.get(kv_dtype, query.dtype))
    S, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    n = ctypes.c_int()
    _check(lib().pa_decode_balanced(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_tables), _ptr(context_lens), S, Hq, num_kv_heads,
                                    D, bs, NB, MB, scale, window, _DTYPE[query.dtype],
                                    _KV[kv_dtype], k_scale, v_scale, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    ctypes.addressof(n), _stream(stream)), "pa_decode_balanced")
    return n.value


def decode_workspace_clear(workspace: torch.Tensor, stream=None):
    """pa_decode_workspace_clear: zero the balanced path's arrival counters."""
    _on_device(workspace=workspace)
    _check(lib().pa_decode_workspace_clear(_ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _stream(stream)), "pa_decode_workspace_clear")


def decode_cascade_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int,
                                  head_dim: int, block_size: int, prefix_pages: int) -> int:
    return int(lib().pa_decode_cascade_workspace_size(num_seqs, num_heads, num_kv_heads,
                                                      head_dim, block_size, prefix_pages))


def decode_cascade(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                   num_kv_heads: int, scale: float, prefix_pages: int,
                   workspace: torch.Tensor, stream=None):
    """pa_decode_cascade: decode of a batch sharing its first prefix_pages blocks."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, context_lens=context_lens, workspace=workspace)
    _check_decode_args(out, query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       query.dtype)
    S, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    _check(lib().pa_decode_cascade(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(block_tables), _ptr(context_lens), S, Hq, num_kv_heads, D,
                                   bs, NB, MB, scale, _DTYPE[query.dtype], prefix_pages,
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "pa_decode_cascade")


def decode_cascade_fp8(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, block_tables: torch.Tensor,
                       context_lens: torch.Tensor, num_kv_heads: int, scale: float,
                       k_scale: float, v_scale: float, prefix_pages: int,
                       workspace: torch.Tensor, stream=None):
    """pa_decode_cascade_fp8: pa_decode_cascade over an FP8 E4M3 cache (uint8
    codes) with per-tensor scales."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, context_lens=context_lens, workspace=workspace)
    _check_decode_args(out, query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       torch.uint8)
    S, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    _check(lib().pa_decode_cascade_fp8(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_tables), _ptr(context_lens), S, Hq,
                                       num_kv_heads, D, bs, NB, MB, scale, k_scale, v_scale,
                                       _DTYPE[query.dtype], prefix_pages, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "pa_decode_cascade_fp8")


def decode_cascade_int8(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                        v_cache: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                        block_tables: torch.Tensor, context_lens: torch.Tensor,
                        num_kv_heads: int, scale: float, prefix_pages: int,
                        workspace: torch.Tensor, stream=None):
    """pa_decode_cascade_int8: pa_decode_cascade over an INT8 cache with per-row
    scales."""
    _on_device(out=out, query=query, k_cache=k_cache, v_cache=v_cache, k_scales=k_scales,
               v_scales=v_scales, block_tables=block_tables, context_lens=context_lens,
               workspace=workspace)
    _check_decode_args(out, query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       torch.int8)
    _check_scales(k_scales, v_scales, k_cache)
    S, Hq, D = query.shape
    NB, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    _check(lib().pa_decode_cascade_int8(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(k_scales), _ptr(v_scales), _ptr(block_tables),
                                        _ptr(context_lens), S, Hq, num_kv_heads, D, bs, NB, MB,
                                        scale, _DTYPE[query.dtype], prefix_pages,
                                        _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "pa_decode_cascade_int8")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_pairs: torch.Tensor,
                stream=None):
    """pa_copy_blocks: block_pairs int32 [n, 2] = (source, destination)."""
    _on_device(k_cache=k_cache, v_cache=v_cache, block_pairs=block_pairs)
    _need(k_cache.dim() == 4, "k_cache: expected [num_blocks, num_kv_heads, block_size, D]")
    _shape("v_cache", v_cache, k_cache.shape)
    _dtype("v_cache", v_cache, k_cache.dtype)
    _need(block_pairs.dim() == 2 and block_pairs.shape[1] == 2, "block_pairs: expected [n, 2]")
    _dtype("block_pairs", block_pairs, torch.int32)
    NB, H, bs, D = k_cache.shape
    _check(lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs),
                                block_pairs.shape[0], H, D, bs, NB, k_cache.element_size(),
                                _stream(stream)), "pa_copy_blocks")


PA_BUDGET_MB, PA_BUDGET_FRACTION, PA_BUDGET_CONTEXT = 0, 1, 2


def block_budget(num_layers: int, num_kv_heads: int, head_dim: int, block_size: int,
                 dtype: torch.dtype, kv_dtype: str = "auto", *, mb: Optional[float] = None,
                 fraction: Optional[float] = None, context_tokens: Optional[int] = None,
                 available_bytes: Optional[int] = None) -> int:
    """pa_block_budget: cache blocks for a budget given as exactly one of mb,
    fraction (of available_bytes, by default the device's free memory) or
    context_tokens."""
    given = [x is not None for x in (mb, fraction, context_tokens)]
    if sum(given) != 1:
        raise ValueError("give exactly one of mb, fraction, context_tokens")
    if fraction is not None and available_bytes is None:
        available_bytes = torch.cuda.mem_get_info()[0]
    kind, amount = ((PA_BUDGET_MB, mb) if mb is not None else
                    (PA_BUDGET_FRACTION, fraction) if fraction is not None else
                    (PA_BUDGET_CONTEXT, context_tokens))
    n = lib().pa_block_budget(kind, float(amount), int(available_bytes or 0), num_layers,
                              num_kv_heads, head_dim, block_size, _DTYPE[dtype], _KV[kv_dtype])
    if n < 0:
        raise PagedAttentionError(int(n), "pa_block_budget")
    return int(n)


def decode_partials(tmp_out: torch.Tensor, max_logits: torch.Tensor, exp_sums: torch.Tensor,
                    query: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int,
                    scale: float, num_splits: int, pages_per_split: int, window: int = 0,
                    kv_dtype: str = "auto", k_scale: float = 1.0, v_scale: float = 1.0,
                    stream=None):
    """pa_decode_partials: split partials tmp_out [S, Hq, NS, D], max_logits and
    exp_sums [S, Hq, NS]."""
    _on_device(tmp_out=tmp_out, max_logits=max_logits, exp_sums=exp_sums, query=query,
               k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               context_lens=context_lens)
    _check_decode_args(query, query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       _CACHE_DTYPE.get(kv_dtype, query.dtype))
    S, Hq, D = query.shape
    _shape("tmp_out", tmp_out, (S, Hq, num_splits, D))
    for name, t in (("max_logits", max_logits), ("exp_sums", exp_sums)):
        _shape(name, t, (S, Hq, num_splits))
        _dtype(name, t, torch.float32)
    _dtype("tmp_out", tmp_out, torch.float32)
    NB, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    _check(lib().pa_decode_partials(_ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums),
                                    _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_tables), _ptr(context_lens), S, Hq, num_kv_heads,
                                    D, bs, NB, MB, scale, window, _DTYPE[query.dtype],
                                    _KV[kv_dtype], k_scale, v_scale, num_splits,
                                    pages_per_split, _stream(stream)), "pa_decode_partials")


def reduce(out: torch.Tensor, tmp_out: torch.Tensor, max_logits: torch.Tensor,
           exp_sums: torch.Tensor, stream=None):
    """pa_reduce: LSE combination of [S, Hq, NS, D] partials into out [S, Hq, D]."""
    _on_device(out=out, tmp_out=tmp_out, max_logits=max_logits, exp_sums=exp_sums)
    _need(tmp_out.dim() == 4, "tmp_out: expected [num_seqs, num_heads, num_splits, D]")
    S, Hq, NS, D = tmp_out.shape
    _shape("out", out, (S, Hq, D))
    _dtype("tmp_out", tmp_out, torch.float32)
    for name, t in (("max_logits", max_logits), ("exp_sums", exp_sums)):
        _shape(name, t, (S, Hq, NS))
        _dtype(name, t, torch.float32)
    _check(lib().pa_reduce(_ptr(out), _ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums), S, Hq,
                           D, NS, _DTYPE[out.dtype], _stream(stream)), "pa_reduce")


def test_set_unarmed_page(page: int) -> None:
    """pa_test_set_unarmed_page: test hook; the producer of every CTA of later
    decodes stops before arming its page number ``page`` (negative: off)."""
    lib().pa_test_set_unarmed_page(int(page))


def get_device_error(stream=None) -> int:
    """pa_get_device_error: synchronise, return and clear the device error bits."""
    bits = ctypes.c_uint32()
    rc = lib().pa_get_device_error(_stream(stream), ctypes.addressof(bits))
    if rc not in (0, PA_ERR_DEVICE):
        raise PagedAttentionError(rc, "pa_get_device_error")
    return bits.value
