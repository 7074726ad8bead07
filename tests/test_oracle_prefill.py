"""Pins of the oracle's multi-query (prefill) attention over the paged cache.

"PagedAttention in mistral.rs" runs a prefill phase next to the paged decode
("FlashAttention V2/V3 + PagedAttention") and lists speculative decoding: both
attend several query tokens of one sequence to its paged K/V at once. The
oracle reads that as causal attention: the token at position p sees the
positions 0..p of its sequence. These tests hold it against PyTorch float64
softmax attention with an explicit causal mask over the raw rows (a library
routine), the single-position closed form, the decode of the last token, and
the handling of padding and bad rows.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import (attended_rows, oracle_caches, oracle_decode, oracle_int8_caches,
                      torch_dequant, torch_int8_dequant)
from paged_kv_cache_context_gb300 import workloads as wl


def dense_causal(case, query, q_seq, q_pos):
    """float64 softmax(q K^T * scale) V of every query token over the raw rows
    of positions 0..p of its sequence."""
    G = case.num_heads // case.num_kv_heads
    out = np.zeros(tuple(query.shape), dtype=np.float64)
    sc = float(np.float32(case.scale))
    for t in range(query.shape[0]):
        s, p = int(q_seq[t]), int(q_pos[t])
        key, val = attended_rows(case, s)  # positions 0 .. n_s - 1 (no window)
        K, V = key[:p + 1].float(), val[:p + 1].float()
        if case.kv_dtype == "int8":
            K, V = torch_int8_dequant(K), torch_int8_dequant(V)
        if case.kv_dtype == "fp8_e4m3":
            K, V = torch_dequant(K, case.k_scale), torch_dequant(V, case.v_scale)
        for h in range(case.num_heads):
            q = query[t, h].float().double()
            logits = (K[:, h // G].double() @ q) * sc
            w = torch.softmax(logits, dim=0)
            out[t, h] = (w @ V[:, h // G].double()).numpy()
    return out


@pytest.mark.parametrize("D,Hq,Hkv,bs,qd,per_seq", [
    (64, 8, 2, 16, torch.float32, 5),
    (128, 8, 8, 32, torch.bfloat16, 40),    # chunks that cross block boundaries
    (96, 12, 4, 32, torch.float16, 100),    # whole contexts for the short sequences
])
def test_prefill_equals_dense_causal_attention(D, Hq, Hkv, bs, qd, per_seq):
    case = wl.make_case(f"pf{D}", 90 + D, 4, Hq, Hkv, D, bs, lens=[1, 7, 33, 95], q_dtype=qd,
                        extra_blocks=3)
    kc, vc = oracle_caches(case)
    query, q_seq, q_pos = wl.prefill_queries(case, per_seq, seed=91 + D)
    out, bad = oracle.prefill(query, q_seq, q_pos, kc, vc, case.block_tables, Hkv, bs,
                              case.scale)
    assert bad == 0
    ref = dense_causal(case, query, q_seq, q_pos)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


def test_prefill_over_an_int8_cache():
    case = wl.make_case("pf_i8", 92, 3, 8, 2, 64, lens=[3, 40, 70], kv_dtype="int8")
    kc, vc, ks, vs = oracle_int8_caches(case)
    query, q_seq, q_pos = wl.prefill_queries(case, 20, seed=93)
    out, bad = oracle.prefill(query, q_seq, q_pos, kc, vc, case.block_tables, 2, 32, case.scale,
                              "int8", k_scales=ks, v_scales=vs)
    assert bad == 0
    ref = dense_causal(case, query, q_seq, q_pos)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


def test_prefill_over_an_fp8_cache():
    """An FP8 E4M3 cache with per-tensor scales: the dense reference takes the
    rows through PyTorch's E4M3 cast (a library routine) and back times the
    scale in fp32."""
    case = wl.make_case("pf_e4", 94, 3, 8, 2, 64, lens=[3, 40, 70], kv_dtype="fp8_e4m3",
                        kv_src_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    query, q_seq, q_pos = wl.prefill_queries(case, 20, seed=95)
    out, bad = oracle.prefill(query, q_seq, q_pos, kc, vc, case.block_tables, 2, 32, case.scale,
                              "fp8_e4m3", case.k_scale, case.v_scale)
    assert bad == 0
    ref = dense_causal(case, query, q_seq, q_pos)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


def test_position_zero_returns_its_value_row_and_the_last_token_is_the_decode():
    case = wl.make_case("pf_last", 94, 3, 4, 2, 64, lens=[1, 30, 64], q_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    # the decode's own query at each sequence's last position
    q = case.query.clone()
    q_seq = torch.arange(3, dtype=torch.int32)
    q_pos = case.context_lens - 1
    out, bad = oracle.prefill(q, q_seq, q_pos, kc, vc, case.block_tables, 2, 32, case.scale)
    assert bad == 0
    np.testing.assert_array_equal(out, oracle_decode(case, kc, vc))
    # position 0 sees one row: its value row, whatever the query
    q0 = torch.randn(1, 4, 64, generator=torch.Generator().manual_seed(95))
    out0, _ = oracle.prefill(q0, torch.tensor([2], dtype=torch.int32),
                             torch.tensor([0], dtype=torch.int32), kc, vc, case.block_tables, 2,
                             32, case.scale)
    key, val = attended_rows(case, 2)
    for h in range(4):
        np.testing.assert_array_equal(out0[0, h], val[0, h // 2].double().numpy())


def test_padding_and_out_of_range_rows():
    case = wl.make_case("pf_bad", 96, 2, 4, 4, 64, lens=[10, 20], q_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    q = torch.randn(4, 4, 64, generator=torch.Generator().manual_seed(97))
    q_seq = torch.tensor([0, 1, 5, 1], dtype=torch.int32)             # sequence 5 does not exist
    q_pos = torch.tensor([-1, 3, 2, case.max_blocks_per_seq * 32], dtype=torch.int32)
    out, bad = oracle.prefill(q, q_seq, q_pos, kc, vc, case.block_tables, 4, 32, case.scale)
    assert np.all(out[0] == 0)
    assert np.isfinite(out[1]).all()
    assert np.isnan(out[2]).all() and np.isnan(out[3]).all()
    assert bad == 2 * 4
