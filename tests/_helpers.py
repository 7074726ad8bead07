"""Shared test helpers: building caches with the oracle, dense references.

Nothing here computes the method on the GPU side; the dense references use
PyTorch float64 library routines (matmul, softmax) on the raw per-position
rows the generator drew.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_context_gb300 import workloads as wl


def oracle_caches(case: wl.DecodeCase, with_new: bool = True):
    """CPU caches holding the case's rows, written by the oracle's own slot
    mapping and reshape_and_cache (pre-step chunks in order, then the new
    tokens)."""
    kc, vc = wl.empty_caches(case)
    for a, b in case.pre_chunks:
        if b <= a:
            continue
        sm, bad = oracle.slot_mapping(case.block_tables, case.pre_seq[a:b], case.pre_pos[a:b],
                                      case.block_size, case.window)
        assert bad == 0
        assert oracle.reshape_and_cache(case.pre_key[a:b], case.pre_value[a:b], kc, vc, sm,
                                        case.block_size, case.kv_dtype, case.k_scale,
                                        case.v_scale) == 0
    if with_new:
        sm, bad = oracle.slot_mapping(case.block_tables, None, case.new_pos, case.block_size,
                                      case.window)
        assert bad == 0
        assert oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, sm,
                                        case.block_size, case.kv_dtype, case.k_scale,
                                        case.v_scale) == 0
    return kc, vc


def sampled_seqs(case: wl.DecodeCase, count: int = 4, seed: int = 7):
    """The longest and the shortest context and seeded random others, sorted:
    the sequences a full-size test checks against the oracle row by row."""
    lens = case.context_lens.tolist()
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    g = torch.Generator().manual_seed(seed)
    while len(pick) < min(count, case.num_seqs):
        pick.add(int(torch.randint(0, case.num_seqs, (1,), generator=g)))
    return sorted(pick)


def oracle_caches_for(case: wl.DecodeCase, seqs):
    """CPU caches holding only the rows of the listed sequences (each written by
    its own oracle calls: slot mapping, then reshape_and_cache; a shared prefix
    comes with every sequence that uses it)."""
    kc, vc = wl.empty_caches(case)
    for s in seqs:
        pos, key, val = case.tokens_of(s)
        sm, bad = oracle.slot_mapping(case.block_tables, torch.full_like(pos, s), pos,
                                      case.block_size, case.window)
        assert bad == 0
        assert oracle.reshape_and_cache(key, val, kc, vc, sm, case.block_size, case.kv_dtype,
                                        case.k_scale, case.v_scale) == 0
    return kc, vc


def oracle_int8_caches(case: wl.DecodeCase):
    """INT8 caches and their per-row scales (kc, vc, ks, vs), written by the
    oracle's slot mapping and INT8 write in the same order as oracle_caches."""
    kc, vc = wl.empty_caches(case)
    ks, vs = wl.empty_scales(case)
    steps = [(case.pre_seq[a:b], case.pre_pos[a:b], case.pre_key[a:b], case.pre_value[a:b])
             for a, b in case.pre_chunks if b > a]
    steps.append((None, case.new_pos, case.new_key, case.new_value))
    for seq, pos, key, val in steps:
        sm, bad = oracle.slot_mapping(case.block_tables, seq, pos, case.block_size, case.window)
        assert bad == 0
        assert oracle.reshape_and_cache_int8(key, val, kc, vc, ks, vs, sm, case.block_size) == 0
    return kc, vc, ks, vs


def oracle_decode(case: wl.DecodeCase, kc, vc, rows=None, context_lens=None, k_scales=None,
                  v_scales=None):
    return oracle.decode(case.query, kc, vc, case.block_tables,
                         case.context_lens if context_lens is None else context_lens,
                         case.num_kv_heads, case.block_size, case.scale, case.window,
                         case.kv_dtype, case.k_scale, case.v_scale, rows=rows,
                         k_scales=k_scales, v_scales=v_scales)


def torch_dequant(x: torch.Tensor, scale: float) -> torch.Tensor:
    """Library-routine FP8 round trip: x / scale in fp32, saturate, PyTorch's
    E4M3 cast, back to fp32 times the scale (fp32)."""
    y = x.float() / torch.tensor(scale, dtype=torch.float32)
    q = torch.clamp(y, -448.0, 448.0).to(torch.float8_e4m3fn).float()
    return q * torch.tensor(scale, dtype=torch.float32)


def torch_int8_dequant(x: torch.Tensor) -> torch.Tensor:
    """Library-routine INT8 per-row round trip over the last dimension, fp32:
    scale = max|x| / 127, round(x / scale) (ties to even) clamped to +-127,
    times the scale; a zero scale gives zeros."""
    x = x.float()
    scale = x.abs().amax(dim=-1, keepdim=True) / torch.tensor(127.0)
    safe = torch.where(scale == 0, torch.ones_like(scale), scale)
    q = torch.clamp(torch.round(x / safe), -127, 127)
    q = torch.where(scale == 0, torch.zeros_like(q), q)
    return q * scale


def attended_rows(case: wl.DecodeCase, s: int):
    """Raw key/value rows [L, Hkv, D] of the positions sequence s attends (its
    last L_s positions, latest write of each), in position order."""
    n = int(case.context_lens[s])
    L = case.attended(s)
    pos, key, val = case.tokens_of(s)
    last = {}
    for i, p in enumerate(pos.tolist()):
        last[p] = i
    idx = torch.tensor([last[p] for p in range(n - L, n)], dtype=torch.int64)
    return key[idx], val[idx]


def dense_reference(case: wl.DecodeCase, s: int, h: int) -> np.ndarray:
    """softmax(q K^T * scale) V in float64 over the positions sequence s attends,
    from the raw rows the generator drew."""
    if case.attended(s) == 0:
        return np.zeros(case.head_dim)
    key, val = attended_rows(case, s)
    g = h // (case.num_heads // case.num_kv_heads)
    K = key[:, g].float()
    V = val[:, g].float()
    if case.kv_dtype == "fp8_e4m3":
        K = torch_dequant(K, case.k_scale)
        V = torch_dequant(V, case.v_scale)
    if case.kv_dtype == "int8":
        K = torch_int8_dequant(K)
        V = torch_int8_dequant(V)
    q = case.query[s, h].cpu().float().double()
    logits = (K.double() @ q) * float(np.float32(case.scale))
    p = torch.softmax(logits, dim=0)
    return (p @ V.double()).numpy()
