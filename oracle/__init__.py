"""CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; the library package never imports
it. The arithmetic lives in ``pa_oracle.c`` (plain C, fp64); this module only
marshals torch CPU tensors into it.

Functions follow the web pages on the subject:
  * "PagedAttention in mistral.rs" -- blocked K/V pool, block size = tokens per
    block, FP8 E4M3 cache ("KV Cache Quantization").
  * "Optimization plans" (mistral.rs discussion #46) -- reshape_and_cache.
  * "Rolling buffer cache" (llama.cpp discussion #3581) -- slot i mod W.
  * "libmir-metal trace/kv.rs" -- INT8 pages with one FP32 scale per token
    and head.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import build as _build

# element codes of the oracle's own C interface
_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
_E4M3 = 3
_I8 = 4

_lib = None
_i64 = ctypes.c_int64
_int = ctypes.c_int
_flt = ctypes.c_float
_dbl = ctypes.c_double
_ptr = ctypes.c_void_p


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_set_threads.restype = _int
        L.oracle_set_threads.argtypes = [_int]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [_flt]
        L.oracle_e4m3_decode.restype = _flt
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode_array.argtypes = [_ptr, _ptr, _i64]
        L.oracle_e4m3_decode_array.argtypes = [_ptr, _ptr, _i64]
        L.oracle_slot_mapping.restype = _i64
        L.oracle_slot_mapping.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _int, _int, _int, _int]
        L.oracle_reshape_and_cache.restype = _i64
        L.oracle_reshape_and_cache.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _i64, _int, _int,
                                               _int, _i64, _int, _int, _flt, _flt]
        L.oracle_decode_partial.restype = _int
        L.oracle_decode_partial.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                            _int, _int, _int, _int, _int, _int, _i64, _int,
                                            _dbl, _int, _int, _int, _flt, _flt, _ptr, _ptr,
                                            _i64, _i64]
        L.oracle_decode_rows.restype = _i64
        L.oracle_decode_rows.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _int, _int, _int,
                                         _int, _int, _i64, _int, _dbl, _int, _int, _int, _flt,
                                         _flt, _ptr, _ptr, _ptr, _i64]
        L.oracle_int8_quantise_row.argtypes = [_ptr, _int, _ptr, _ptr]
        L.oracle_prefill_rows.restype = _i64
        L.oracle_prefill_rows.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _ptr, _ptr, _ptr, _int,
                                          _int, _int, _int, _int, _i64, _int, _dbl, _int, _int,
                                          _flt, _flt, _ptr, _ptr]
        L.oracle_reshape_and_cache_int8.restype = _i64
        L.oracle_reshape_and_cache_int8.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                                    _i64, _int, _int, _int, _i64, _int]
        L.oracle_reduce.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _int, _int]
        _lib = L
    return _lib


def _cpu(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu" or not t.is_contiguous():
        t = t.detach().to("cpu").contiguous()
    return t


def _p(t) -> int:
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _cache_code(cache: torch.Tensor, kv_dtype: str) -> int:
    if kv_dtype == "int8":
        assert cache.dtype == torch.int8
        return _I8
    if kv_dtype == "fp8_e4m3":
        assert cache.dtype == torch.uint8
        return _E4M3
    return _CODE[cache.dtype]


# ---------------------------------------------------------------- FP8 E4M3
def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """E4M3 code of every binary32 value (round to nearest even, saturate at 448)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_p(x), _p(out), x.size)
    return out


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """Exact binary32 value of every E4M3 code (NaN for S.1111.111)."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float32)
    lib().oracle_e4m3_decode_array(_p(b), _p(out), b.size)
    return out


# ---------------------------------------------------------------- INT8 rows
def int8_quantise_rows(x: np.ndarray):
    """INT8 per-row quantisation of a [rows, n] binary32 array: (codes int8
    [rows, n], scales float32 [rows])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, n = x.shape
    codes = np.empty((rows, n), dtype=np.int8)
    scales = np.empty(rows, dtype=np.float32)
    for r in range(rows):
        lib().oracle_int8_quantise_row(_p(x[r]), n, _p(codes[r]), _p(scales[r:r + 1]))
    return codes, scales


# ---------------------------------------------------------------- slot mapping
def slot_mapping(block_tables: torch.Tensor, seq_idx, positions: torch.Tensor,
                 block_size: int, window: int = 0):
    """int64 slot of each token; returns (slots, number of out-of-range tokens)."""
    bt = _cpu(block_tables).to(torch.int32)
    pos = _cpu(positions).to(torch.int32)
    sq = None if seq_idx is None else _cpu(seq_idx).to(torch.int32)
    out = torch.empty(pos.numel(), dtype=torch.int64)
    bad = lib().oracle_slot_mapping(_p(out), _p(bt), None if sq is None else _p(sq), _p(pos),
                                    pos.numel(), bt.shape[0], bt.shape[1], block_size, window)
    return out, int(bad)


# ---------------------------------------------------------------- write
def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping_, block_size: int,
                      kv_dtype: str = "auto", k_scale: float = 1.0, v_scale: float = 1.0) -> int:
    """Write key/value [T, Hkv, D] into the CPU caches [NB, Hkv, bs, D] in place.

    Returns the number of tokens whose slot was beyond the pool."""
    key, value = _cpu(key), _cpu(value)
    sm = _cpu(slot_mapping_).to(torch.int64)
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous()
    assert v_cache.device.type == "cpu" and v_cache.is_contiguous()
    T, H, D = key.shape
    code = _cache_code(k_cache, kv_dtype)
    if code != _E4M3:
        assert k_cache.dtype == key.dtype
    bad = lib().oracle_reshape_and_cache(_p(key), _p(value), _p(k_cache), _p(v_cache), _p(sm),
                                         T, H, D, block_size, k_cache.shape[0], _CODE[key.dtype],
                                         code, k_scale, v_scale)
    return int(bad)


def reshape_and_cache_int8(key, value, k_cache, v_cache, k_scales, v_scales, slot_mapping_,
                           block_size: int) -> int:
    """INT8 write of key/value [T, Hkv, D] into int8 caches [NB, Hkv, bs, D] and
    fp32 scales [NB, Hkv, bs] (CPU tensors, in place). Returns the number of
    tokens whose slot was beyond the pool."""
    key, value = _cpu(key), _cpu(value)
    sm = _cpu(slot_mapping_).to(torch.int64)
    for t, dt in ((k_cache, torch.int8), (v_cache, torch.int8), (k_scales, torch.float32),
                  (v_scales, torch.float32)):
        assert t.device.type == "cpu" and t.is_contiguous() and t.dtype == dt
    T, H, D = key.shape
    bad = lib().oracle_reshape_and_cache_int8(_p(key), _p(value), _p(k_cache), _p(v_cache),
                                              _p(k_scales), _p(v_scales), _p(sm), T, H, D,
                                              block_size, k_cache.shape[0], _CODE[key.dtype])
    return int(bad)


# ---------------------------------------------------------------- decode
def _row_scales(kv_dtype, k_scales, v_scales):
    if kv_dtype != "int8":
        return None, None
    ks, vs = _cpu(k_scales), _cpu(v_scales)
    assert ks.dtype == torch.float32 and vs.dtype == torch.float32
    return ks, vs


def set_threads(n: int) -> int:
    """Host threads of the oracle's parallel loops (n > 0 sets it); returns the
    previous setting. Timing only: results do not depend on it."""
    return int(lib().oracle_set_threads(int(n)))


def decode(query, k_cache, v_cache, block_tables, context_lens, num_kv_heads: int,
           block_size: int, scale: float, window: int = 0, kv_dtype: str = "auto",
           k_scale: float = 1.0, v_scale: float = 1.0, rows=None, k_scales=None,
           v_scales=None) -> np.ndarray:
    """fp64 attention output [S, Hq, D]; with ``rows`` (s*Hq+h indices) only those
    rows are computed (the others stay NaN). An "int8" cache takes its per-row
    scales k_scales / v_scales [NB, Hkv, bs]."""
    q = _cpu(query)
    kc, vc = _cpu(k_cache), _cpu(v_cache)
    ks, vs = _row_scales(kv_dtype, k_scales, v_scales)
    bt = _cpu(block_tables).to(torch.int32)
    cl = _cpu(context_lens).to(torch.int32)
    S, Hq, D = q.shape
    out = np.full((S, Hq, D), np.nan, dtype=np.float64)
    r = None
    if rows is not None:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    bad = lib().oracle_decode_rows(_p(out), _p(q), _p(kc), _p(vc), _p(bt), _p(cl), S, Hq,
                                   num_kv_heads, D, block_size, kc.shape[0], bt.shape[1],
                                   float(np.float32(scale)), window, _CODE[q.dtype],
                                   _cache_code(kc, kv_dtype), k_scale, v_scale,
                                   None if ks is None else _p(ks), None if vs is None else _p(vs),
                                   None if r is None else _p(r), 0 if r is None else r.size)
    if bad:
        raise ValueError(f"oracle decode: {bad} rows met a block id outside the pool")
    return out


def decode_partial(query, k_cache, v_cache, block_tables, context_lens, s: int, h: int,
                   num_kv_heads: int, block_size: int, scale: float, tok_begin: int,
                   tok_end: int, window: int = 0, kv_dtype: str = "auto",
                   k_scale: float = 1.0, v_scale: float = 1.0, k_scales=None, v_scales=None):
    """(o [D] fp64, m, l) of head h of sequence s over slots [tok_begin, tok_end)."""
    q = _cpu(query)
    kc, vc = _cpu(k_cache), _cpu(v_cache)
    ks, vs = _row_scales(kv_dtype, k_scales, v_scales)
    bt = _cpu(block_tables).to(torch.int32)
    cl = _cpu(context_lens).to(torch.int32)
    S, Hq, D = q.shape
    o = np.zeros(D, dtype=np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    rc = lib().oracle_decode_partial(_p(o), ctypes.addressof(m), ctypes.addressof(l), _p(q),
                                     _p(kc), _p(vc), _p(bt), _p(cl), s, h, Hq, num_kv_heads, D,
                                     block_size, kc.shape[0], bt.shape[1],
                                     float(np.float32(scale)), window, _CODE[q.dtype],
                                     _cache_code(kc, kv_dtype), k_scale, v_scale,
                                     None if ks is None else _p(ks),
                                     None if vs is None else _p(vs), tok_begin, tok_end)
    if rc:
        raise ValueError("oracle decode_partial: block id outside the pool")
    return o, m.value, l.value


# ---------------------------------------------------------------- prefill
def prefill(query, q_seq, q_pos, k_cache, v_cache, block_tables, num_kv_heads: int,
            block_size: int, scale: float, kv_dtype: str = "auto", k_scale: float = 1.0,
            v_scale: float = 1.0, k_scales=None, v_scales=None):
    """Causal multi-query attention over the paged cache: query [T, Hq, D], token
    t of sequence q_seq[t] at position q_pos[t] attends to positions
    0..q_pos[t]. Returns (out [T, Hq, D] fp64, number of bad rows)."""
    q = _cpu(query)
    qs = _cpu(q_seq).to(torch.int32)
    qp = _cpu(q_pos).to(torch.int32)
    kc, vc = _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_tables).to(torch.int32)
    ks, vs = _row_scales(kv_dtype, k_scales, v_scales)
    T, Hq, D = q.shape
    out = np.empty((T, Hq, D), dtype=np.float64)
    bad = lib().oracle_prefill_rows(_p(out), _p(q), _p(qs), _p(qp), T, _p(kc), _p(vc), _p(bt),
                                    bt.shape[0], Hq, num_kv_heads, D, block_size, kc.shape[0],
                                    bt.shape[1], float(np.float32(scale)), _CODE[q.dtype],
                                    _cache_code(kc, kv_dtype), k_scale, v_scale,
                                    None if ks is None else _p(ks),
                                    None if vs is None else _p(vs))
    return out, int(bad)


# ---------------------------------------------------------------- reduce
def reduce(tmp_out, max_logits, exp_sums) -> np.ndarray:
    """LSE combination: tmp_out [..., NS, D], max_logits/exp_sums [..., NS] -> [..., D]."""
    o = np.ascontiguousarray(np.asarray(tmp_out, dtype=np.float64))
    m = np.ascontiguousarray(np.asarray(max_logits, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(exp_sums, dtype=np.float64))
    NS, D = o.shape[-2], o.shape[-1]
    lead = o.shape[:-2]
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (D,), dtype=np.float64)
    lib().oracle_reduce(_p(out), _p(o), _p(m), _p(l), rows, D, NS)
    return out
