"""Seeded synthetic inputs for paged decode attention.

This module draws the inputs both the CUDA library and the CPU oracle consume:
context lengths, the assignment of physical cache blocks to sequences (block
tables), and the query / key / value values, plus the list of which
(sequence, position) every key/value row belongs to. It holds none of the
method's arithmetic: slot addresses, the cache write, FP8 quantisation and the
attention itself are computed by the library and, independently, by the
oracle.

Draw order for a seed: lengths -> pool permutation -> q -> K -> V.

Workload shapes (all block_size 32, fp32 accumulation, values N(0, 1)):
  tiny         2 seqs, 4 = 4 heads, D 64, fp32, lengths {17, 45}, pool of 8 blocks
  mistral_bf16 32 seqs, 32 q / 8 kv heads, D 128, bf16, lengths U[512, 4096]
  ring_bf16    8 seqs, same heads, W = 4096 rolling buffer (128 blocks per seq),
               absolute positions U[4096, 32768]
  fp8_phi3     64 seqs, 32 = 32 heads, D 96, K/V fp32 -> FP8 E4M3 cache with
               per-tensor scales amax/448, bf16 query and output, lengths U[1024, 8192]
  prefix_bf16  128 seqs, 32 q / 8 kv heads, D 128, bf16, a 2048-token prefix held
               in 64 blocks shared by every table, unique suffixes of 0-512 tokens
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import torch

INT32_POISON = -1  # block-table entries a sequence does not own


@dataclasses.dataclass
class DecodeCase:
    """One batch of paged decode inputs."""

    name: str
    seed: int
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    window: int
    q_dtype: torch.dtype
    kv_dtype: str  # "auto", "fp8_e4m3" or "int8" (per-token/head scales)
    kv_src_dtype: torch.dtype  # dtype of the key/value rows before the cache write
    scale: float
    context_lens: torch.Tensor  # int32 [S], including the new token
    block_tables: torch.Tensor  # int32 [S, MB]; -1 where a sequence owns no block
    num_blocks: int
    shared_prefix_tokens: int  # positions < this are stored once, under sequence 0
    # rows in the cache before the step: token i is (pre_seq[i], pre_pos[i])
    pre_seq: torch.Tensor  # int32 [T0]
    pre_pos: torch.Tensor  # int32 [T0]
    pre_key: torch.Tensor  # [T0, Hkv, D] kv_src_dtype
    pre_value: torch.Tensor
    pre_chunks: List[Tuple[int, int]]  # token ranges written by separate calls, in order
    # the step: one new token per sequence at position n_s - 1 (-1 if n_s == 0)
    new_pos: torch.Tensor  # int32 [S]
    new_key: torch.Tensor  # [S, Hkv, D] kv_src_dtype
    new_value: torch.Tensor
    query: torch.Tensor  # [S, Hq, D] q_dtype
    k_scale: float
    v_scale: float

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def cache_dtype(self) -> torch.dtype:
        if self.kv_dtype == "int8":
            return torch.int8
        return torch.uint8 if self.kv_dtype == "fp8_e4m3" else self.q_dtype

    @property
    def cache_shape(self) -> Tuple[int, int, int, int]:
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def attended(self, s: int) -> int:
        """Number of tokens sequence s attends to (window-limited context)."""
        n = int(self.context_lens[s])
        return min(n, self.window) if self.window > 0 else n

    def tokens_of(self, s: int):
        """(positions, key rows, value rows) of every token of sequence s, in the
        order they are written (prefix rows shared through sequence 0 included,
        the step's new token last)."""
        pre_seq = self.pre_seq.cpu()
        pre_pos = self.pre_pos.cpu()
        sel = pre_seq == s
        if self.shared_prefix_tokens and s != 0:
            sel = sel | ((pre_seq == 0) & (pre_pos < self.shared_prefix_tokens))
        idx = torch.nonzero(sel).flatten()
        pos = pre_pos[idx]
        didx = idx.to(self.pre_key.device)
        key = self.pre_key[didx].cpu()
        val = self.pre_value[didx].cpu()
        if int(self.new_pos[s]) >= 0:
            pos = torch.cat([pos, self.new_pos.cpu()[s:s + 1]])
            key = torch.cat([key, self.new_key.cpu()[s:s + 1]])
            val = torch.cat([val, self.new_value.cpu()[s:s + 1]])
        return pos, key, val

    def kv_bytes(self) -> int:
        """Key+value cache bytes the decode must read (attended tokens only;
        an INT8 cache adds each row's 4-byte scale)."""
        elem = (1 if self.kv_dtype in ("fp8_e4m3", "int8")
                else torch.finfo(self.q_dtype).bits // 8)
        row = self.head_dim * elem + (4 if self.kv_dtype == "int8" else 0)
        tokens = sum(self.attended(s) for s in range(self.num_seqs))
        return tokens * self.num_kv_heads * 2 * row


def _normal(g: torch.Generator, shape, dtype, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    return x.to(dtype)


def make_case(name: str, seed: int, num_seqs: int, num_heads: int, num_kv_heads: int,
              head_dim: int, block_size: int = 32, *, lens: Optional[Sequence[int]] = None,
              len_range: Optional[Tuple[int, int]] = None, window: int = 0,
              q_dtype: torch.dtype = torch.bfloat16, kv_dtype: str = "auto",
              kv_src_dtype: Optional[torch.dtype] = None, scale: Optional[float] = None,
              extra_blocks: int = 0, shared_prefix_blocks: int = 0,
              suffix_range: Optional[Tuple[int, int]] = None,
              max_blocks_per_seq: Optional[int] = None, ring_overwrite: bool = False,
              value_device: str = "cpu") -> DecodeCase:
    """Draw one paged decode batch.

    lens / len_range   context lengths (including the step's new token), given or
                       drawn uniformly from [lo, hi].
    window             rolling-buffer span W (0 = none); a sequence owns at most
                       W / block_size blocks.
    shared_prefix_blocks  every table starts with the same blocks, holding a
                       common prefix of that many full blocks; the length of
                       sequence s is then prefix + U[suffix_range] + 1.
    ring_overwrite     write every position from 0 (in calls of at most W
                       consecutive positions) instead of only the last W, so
                       the rolling buffer is overwritten before the step.
    value_device       where q/K/V are drawn; a CUDA device draws them with a
                       CUDA generator seeded alike (fast for full-size batches).
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    S, bs = num_seqs, block_size
    prefix_tokens = shared_prefix_blocks * bs

    # 1. lengths
    if lens is not None:
        n_list = [int(v) for v in lens]
        assert len(n_list) == S
    elif shared_prefix_blocks:
        lo, hi = suffix_range
        n_list = [prefix_tokens + int(v) + 1
                  for v in torch.randint(lo, hi + 1, (S,), generator=g)]
    else:
        lo, hi = len_range
        n_list = [int(v) for v in torch.randint(lo, hi + 1, (S,), generator=g)]

    # blocks owned by each sequence (a ring owns at most W / bs of them)
    def pages(nv: int) -> int:
        p = -(-nv // bs)
        return min(p, window // bs) if window > 0 else p

    own = [pages(v) for v in n_list]
    if shared_prefix_blocks:
        own = [p - shared_prefix_blocks for p in own]
        assert all(p >= 1 for p in own)
    if max_blocks_per_seq is None:
        if window > 0:
            max_blocks_per_seq = window // bs
        else:
            if shared_prefix_blocks:
                hi_len = prefix_tokens + suffix_range[1] + 1
            elif len_range is not None and lens is None:
                hi_len = len_range[1]
            else:
                hi_len = max(n_list) if n_list else 1
            max_blocks_per_seq = max(1, -(-hi_len // bs))
    MB = max_blocks_per_seq
    NB = shared_prefix_blocks + sum(own) + extra_blocks

    # 2. pool permutation: blocks are handed out in this order
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((S, MB), INT32_POISON, dtype=torch.int32)
    shared = perm[:shared_prefix_blocks]
    cur = shared_prefix_blocks
    for s in range(S):
        row = torch.cat([shared, perm[cur:cur + own[s]]])
        cur += own[s]
        assert row.numel() <= MB, (row.numel(), MB)
        tables[s, :row.numel()] = row

    # which (sequence, position) rows are in the cache before the step
    pre_seq: List[int] = []
    pre_pos: List[int] = []
    chunks: List[Tuple[int, int]] = []
    if ring_overwrite and window > 0:
        # all positions, in calls of at most W consecutive positions per sequence
        rounds = max((max(v - 1, 0) + window - 1) // window for v in n_list) if S else 0
        for k in range(rounds):
            start = len(pre_seq)
            for s in range(S):
                for p in range(k * window, min((k + 1) * window, n_list[s] - 1)):
                    pre_seq.append(s)
                    pre_pos.append(p)
            chunks.append((start, len(pre_seq)))
    else:
        for s in range(S):
            first = max(0, n_list[s] - window) if window > 0 else 0
            if shared_prefix_blocks and s != 0:
                first = max(first, prefix_tokens)
            last = n_list[s] - 1
            if last > first:
                pre_seq.extend([s] * (last - first))
                pre_pos.extend(range(first, last))
        chunks.append((0, len(pre_seq)))
    T0 = len(pre_seq)

    # 3-5. values
    gv = g if value_device == "cpu" else torch.Generator(device=value_device).manual_seed(seed)
    kv_src = kv_src_dtype or (torch.float32 if kv_dtype == "fp8_e4m3" else q_dtype)
    q = _normal(gv, (S, num_heads, head_dim), q_dtype, value_device)
    k_all = _normal(gv, (T0 + S, num_kv_heads, head_dim), kv_src, value_device)
    v_all = _normal(gv, (T0 + S, num_kv_heads, head_dim), kv_src, value_device)

    new_pos = torch.tensor([v - 1 for v in n_list], dtype=torch.int32)
    k_scale = v_scale = 1.0
    if kv_dtype == "fp8_e4m3":
        # per-tensor scales amax / 448 over every row written, in fp32
        live = (new_pos >= 0).to(k_all.device)
        for which, t in (("k", k_all), ("v", v_all)):
            amax = torch.zeros((), dtype=torch.float32, device=t.device)
            if T0:
                amax = torch.maximum(amax, t[:T0].float().abs().max())
            if bool(live.any()):
                amax = torch.maximum(amax, t[T0:][live].float().abs().max())
            sc = float(amax / 448.0) if float(amax) > 0 else 1.0
            if which == "k":
                k_scale = sc
            else:
                v_scale = sc

    return DecodeCase(
        name=name, seed=seed, num_seqs=S, num_heads=num_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, window=window, q_dtype=q_dtype, kv_dtype=kv_dtype,
        kv_src_dtype=kv_src, scale=scale if scale is not None else 1.0 / math.sqrt(head_dim),
        context_lens=torch.tensor(n_list, dtype=torch.int32), block_tables=tables,
        num_blocks=NB, shared_prefix_tokens=prefix_tokens,
        pre_seq=torch.tensor(pre_seq, dtype=torch.int32),
        pre_pos=torch.tensor(pre_pos, dtype=torch.int32),
        pre_key=k_all[:T0], pre_value=v_all[:T0], pre_chunks=chunks, new_pos=new_pos,
        new_key=k_all[T0:], new_value=v_all[T0:], query=q,
        k_scale=float(torch.tensor(k_scale, dtype=torch.float32)),
        v_scale=float(torch.tensor(v_scale, dtype=torch.float32)))


def cache_poison(case: DecodeCase) -> int:
    """Bit pattern the caches hold before any write (a NaN of the cache's
    element type), so that a stray read of an unwritten row shows up."""
    if case.kv_dtype == "fp8_e4m3":
        return 0x7F
    if case.kv_dtype == "int8":
        return -128  # a code the INT8 quantiser never writes
    return {torch.float32: 0x7FC00000, torch.bfloat16: 0x7FC0, torch.float16: 0x7E00}[case.q_dtype]


def empty_caches(case: DecodeCase, device: str = "cpu"):
    """Key and value caches [NB, Hkv, bs, D] filled with the poison pattern."""
    dt = case.cache_dtype
    pat = cache_poison(case)
    if dt in (torch.uint8, torch.int8):
        k = torch.full(case.cache_shape, pat, dtype=dt, device=device)
    else:
        itype = {torch.float32: torch.int32, torch.bfloat16: torch.int16,
                 torch.float16: torch.int16}[dt]
        k = torch.full(case.cache_shape, pat, dtype=itype, device=device).view(dt)
    return k, k.clone()


def empty_scales(case: DecodeCase, device: str = "cpu"):
    """Per-row fp32 scales [NB, Hkv, bs] of an INT8 cache, K and V, filled with
    NaN before any write."""
    k = torch.full(case.cache_shape[:3], float("nan"), dtype=torch.float32, device=device)
    return k, k.clone()


def prefill_queries(case: DecodeCase, per_seq: int, seed: int, device: str = "cpu"):
    """Query rows for a prefill chunk: the last min(per_seq, n_s) positions of
    every sequence, in sequence order. Returns (query [T, Hq, D] of q_dtype,
    q_seq int32 [T], q_pos int32 [T]); values N(0, 1) from their own seed."""
    seqs, pos = [], []
    for s in range(case.num_seqs):
        n = int(case.context_lens[s])
        for p in range(max(0, n - per_seq), n):
            seqs.append(s)
            pos.append(p)
    g = torch.Generator().manual_seed(seed)
    q = _normal(g, (len(pos), case.num_heads, case.head_dim), case.q_dtype, "cpu").to(device)
    return (q, torch.tensor(seqs, dtype=torch.int32), torch.tensor(pos, dtype=torch.int32))


# ------------------------------------------------------------------ named workloads
CONFIG_NAMES = ("tiny", "mistral_bf16", "ring_bf16", "fp8_phi3", "prefix_bf16")


def config(name: str, value_device: str = "cpu", seed: Optional[int] = None) -> DecodeCase:
    """The five named workloads at their full sizes."""
    kw = dict(value_device=value_device)
    if name == "tiny":
        return make_case(name, seed or 1001, 2, 4, 4, 64, lens=[17, 45], q_dtype=torch.float32,
                         extra_blocks=5, **kw)
    if name == "mistral_bf16":
        return make_case(name, seed or 1002, 32, 32, 8, 128, len_range=(512, 4096), **kw)
    if name == "ring_bf16":
        return make_case(name, seed or 1003, 8, 32, 8, 128, len_range=(4096, 32768),
                         window=4096, **kw)
    if name == "fp8_phi3":
        return make_case(name, seed or 1004, 64, 32, 32, 96, len_range=(1024, 8192),
                         kv_dtype="fp8_e4m3", kv_src_dtype=torch.float32, **kw)
    if name == "prefix_bf16":
        return make_case(name, seed or 1005, 128, 32, 8, 128, shared_prefix_blocks=64,
                         suffix_range=(0, 512), **kw)
    raise KeyError(name)


def scaled_config(name: str, seqs: int, len_div: int, seed: Optional[int] = None) -> DecodeCase:
    """A named workload with fewer sequences and lengths divided by len_div, for
    element-by-element checks against the oracle within seconds."""
    if name == "mistral_bf16":
        return make_case(name + "_small", seed or 2002, seqs, 32, 8, 128,
                         len_range=(512 // len_div, 4096 // len_div),
                         max_blocks_per_seq=4096 // 32)
    if name == "ring_bf16":
        w = 4096 // len_div
        return make_case(name + "_small", seed or 2003, seqs, 32, 8, 128,
                         len_range=(w, 8 * w), window=w)
    if name == "fp8_phi3":
        return make_case(name + "_small", seed or 2004, seqs, 32, 32, 96,
                         len_range=(1024 // len_div, 8192 // len_div), kv_dtype="fp8_e4m3",
                         kv_src_dtype=torch.float32, max_blocks_per_seq=8192 // 32)
    if name == "prefix_bf16":
        return make_case(name + "_small", seed or 2005, seqs, 32, 8, 128,
                         shared_prefix_blocks=max(1, 64 // len_div),
                         suffix_range=(0, 512 // len_div))
    raise KeyError(name)
