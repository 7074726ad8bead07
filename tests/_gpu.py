"""GPU-side test helpers: build caches and run decode through the C ABI binding,
and compare against oracle results with the stated tolerances.

Tolerances (decode output, from the method's statement):
  * fp32 output: per (sequence, head) row, max |gpu - oracle| <= 1e-3 * max(max |oracle|, 1e-6)
  * bf16 / f16 output: max |gpu - oracle| <= 2e-2 over all elements
The write, the slot mapping and the FP8 encode are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_context_gb300 import pa
from paged_kv_cache_context_gb300 import workloads as wl

DEV = "cuda"
FP32_REL_TOL = 1e-3
HALF_ABS_TOL = 2e-2


def to_dev(t):
    return t.to(DEV, non_blocking=False).contiguous()


def gpu_slot_mapping(case, seq, pos):
    sm = torch.empty(pos.numel(), dtype=torch.int64, device=DEV)
    pa.slot_mapping(sm, to_dev(case.block_tables), None if seq is None else to_dev(seq),
                    to_dev(pos), case.block_size, case.window)
    return sm


def gpu_caches(case, with_new: bool = True):
    """Caches on the GPU, written by pa_slot_mapping + pa_reshape_and_cache."""
    kc, vc = wl.empty_caches(case, device=DEV)
    for a, b in case.pre_chunks:
        if b <= a:
            continue
        sm = gpu_slot_mapping(case, case.pre_seq[a:b], case.pre_pos[a:b])
        pa.reshape_and_cache(to_dev(case.pre_key[a:b]), to_dev(case.pre_value[a:b]), kc, vc, sm,
                             case.kv_dtype, case.k_scale, case.v_scale)
    if with_new:
        sm = gpu_slot_mapping(case, None, case.new_pos)
        pa.reshape_and_cache(to_dev(case.new_key), to_dev(case.new_value), kc, vc, sm,
                             case.kv_dtype, case.k_scale, case.v_scale)
    return kc, vc


def gpu_decode(case, kc, vc, split: bool = True, context_lens=None, block_tables=None):
    out = torch.empty(case.num_seqs, case.num_heads, case.head_dim, dtype=case.q_dtype,
                      device=DEV)
    ws = None
    if split:
        nbytes = pa.decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                          case.head_dim, case.block_size,
                                          case.max_blocks_per_seq, case.window)
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    pa.decode(out, to_dev(case.query), kc, vc,
              to_dev(case.block_tables if block_tables is None else block_tables),
              to_dev(case.context_lens if context_lens is None else context_lens),
              case.num_kv_heads, case.scale, case.window, case.kv_dtype, case.k_scale,
              case.v_scale, ws)
    return out


def assert_close(case, got: torch.Tensor, ref: np.ndarray, rows=None, what=""):
    """Compare GPU output [S, Hq, D] with oracle fp64 output (only ``rows`` =
    s*Hq+h indices when given)."""
    g = got.detach().float().cpu().double().numpy().reshape(-1, case.head_dim)
    r = ref.reshape(-1, case.head_dim)
    idx = np.arange(g.shape[0]) if rows is None else np.asarray(rows)
    g, r = g[idx], r[idx]
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    if case.q_dtype == torch.float32:
        bound = FP32_REL_TOL * np.maximum(np.abs(r).max(axis=1), 1e-6)
        worst = (err.max(axis=1) / bound).max()
        assert worst <= 1.0, f"{what}: fp32 row error {worst:.3g} x tolerance"
    else:
        assert err.max() <= HALF_ABS_TOL, f"{what}: max abs error {err.max():.3g}"
    return float(err.max())


def bits(t: torch.Tensor) -> torch.Tensor:
    """Integer view for bitwise comparison (NaN payloads included)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def device_errors() -> int:
    return pa.get_device_error()


def gpu_int8_caches(case):
    """INT8 caches and row scales on the GPU (pa_slot_mapping +
    pa_reshape_and_cache_int8), written in the same order as the oracle's."""
    kc, vc = wl.empty_caches(case, device=DEV)
    ks, vs = wl.empty_scales(case, device=DEV)
    steps = [(case.pre_seq[a:b], case.pre_pos[a:b], case.pre_key[a:b], case.pre_value[a:b])
             for a, b in case.pre_chunks if b > a]
    steps.append((None, case.new_pos, case.new_key, case.new_value))
    for seq, pos, key, val in steps:
        sm = gpu_slot_mapping(case, seq, pos)
        pa.reshape_and_cache_int8(to_dev(key), to_dev(val), kc, vc, ks, vs, sm)
    return kc, vc, ks, vs
