"""GPU parity of pa_prefill (causal multi-query attention over the paged
cache) against the oracle's prefill, element by element within the bf16 /
f16 output tolerance.

"PagedAttention in mistral.rs" runs a prefill phase beside the paged decode
("FlashAttention V2/V3 + PagedAttention") and lists speculative decoding:
several query tokens of a sequence attend to its paged K/V at once. The
chunks below cross block boundaries and 64-row query tiles, include a single
query token, whole contexts (q_len = n) and every group size bucket, and the
device-side checks (offsets that do not fit, a chunk longer than its context,
a bad block id) are exercised without any out-of-range access.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import DEV, device_errors, gpu_caches, gpu_int8_caches, to_dev
from _helpers import oracle_caches
from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 2e-2  # bf16 / f16 output: max |gpu - oracle|


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    pa.lib()
    device_errors()


def chunk(case, per_seq, seed):
    query, q_seq, q_pos = wl.prefill_queries(case, per_seq, seed)
    q_lens = [int((q_seq == s).sum()) for s in range(case.num_seqs)]
    cu = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    return query, q_seq, q_pos, cu, max(q_lens)


def gpu_prefill(case, kg, vg, query, cu, max_q, block_tables=None, context_lens=None):
    out = torch.full(tuple(query.shape), float("nan"), dtype=case.q_dtype, device=DEV)
    pa.prefill(out, to_dev(query), kg, vg,
               to_dev(case.block_tables if block_tables is None else block_tables), to_dev(cu),
               to_dev(case.context_lens if context_lens is None else context_lens),
               case.num_kv_heads, max_q, case.scale)
    return out


@pytest.mark.parametrize("D,Hq,Hkv,bs,qd,per_seq", [
    (128, 32, 8, 32, torch.bfloat16, 16),    # G 4: 64 query rows per kv head
    (128, 32, 8, 16, torch.float16, 100),    # 400 rows: seven 64-row tiles, bs 16
    (64, 16, 16, 64, torch.bfloat16, 7),     # G 1, bs 64
    (64, 12, 4, 32, torch.float16, 300),     # G 3; short contexts taken whole (q_len = n)
    (128, 8, 1, 32, torch.bfloat16, 1),      # G 8, one query token (the decode's shape)
    (128, 16, 16, 32, torch.bfloat16, 65),   # G 1, 65 rows: a one-row second tile
    (64, 16, 2, 16, torch.float16, 33),      # G 8, 264 rows
])
def test_prefill_matches_oracle(D, Hq, Hkv, bs, qd, per_seq):
    case = wl.make_case(f"pf{D}_{Hq}_{Hkv}_{bs}", 120 + D + Hq + bs, 9, Hq, Hkv, D, bs,
                        len_range=(1, 500), q_dtype=qd, extra_blocks=3)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    query, q_seq, q_pos, cu, max_q = chunk(case, per_seq, 121 + D + per_seq)
    out = gpu_prefill(case, kg, vg, query, cu, max_q)
    torch.cuda.synchronize()
    assert device_errors() == 0
    ref, bad = oracle.prefill(query, q_seq, q_pos, ko, vo, case.block_tables, Hkv, bs,
                              case.scale)
    assert bad == 0
    g = out.float().cpu().double().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref).max()
    assert err <= TOL, f"max abs error {err:.3g}"


def test_prefill_last_token_equals_the_decode_oracle():
    """A chunk of one token per sequence at its last position is the decode
    step; the prefill kernel's answer matches the oracle's decode."""
    from _helpers import oracle_decode
    case = wl.make_case("pf_dec", 131, 6, 32, 8, 128, len_range=(1, 300),
                        q_dtype=torch.bfloat16)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    cu = torch.arange(case.num_seqs + 1, dtype=torch.int32)
    out = gpu_prefill(case, kg, vg, case.query.cpu(), cu, 1)
    ref = oracle_decode(case, ko, vo)
    err = np.abs(out.float().cpu().double().numpy() - ref).max()
    assert err <= TOL, err
    assert device_errors() == 0


def test_prefill_device_checks():
    """Offsets that do not fit flag PA_DEVERR_SEQ and leave that sequence
    unwritten; a chunk longer than its context flags PA_DEVERR_CONTEXT_LEN and
    gives zero rows; a block id outside the pool flags PA_DEVERR_BLOCK_ID and
    reads as zeros. The other sequences keep the oracle's answer."""
    case = wl.make_case("pf_bad", 132, 4, 8, 2, 64, lens=[40, 70, 9, 100],
                        q_dtype=torch.bfloat16, extra_blocks=2)
    bs = case.block_size
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    query, q_seq, q_pos, cu, max_q = chunk(case, 8, 133)
    assert cu.tolist() == [0, 8, 16, 24, 32] and max_q == 8
    ref, _ = oracle.prefill(query, q_seq, q_pos, ko, vo, case.block_tables, 2, bs, case.scale)
    device_errors()

    def close(g, rows):
        return np.abs(g[rows] - ref[rows]).max() <= TOL

    # sequence 1 claims rows [8, 17): 9 tokens, above max_q_len = 8
    cu_bad = cu.clone()
    cu_bad[2] = 17
    out = gpu_prefill(case, kg, vg, query, cu_bad, max_q)
    torch.cuda.synchronize()
    assert device_errors() & 16
    g = out.float().cpu().double().numpy()
    assert np.isnan(g[8:17]).all()  # not written
    assert close(g, np.r_[0:8, 24:32])

    # sequence 2's context (5 tokens) is shorter than its chunk of 8
    cl = case.context_lens.clone()
    cl[2] = 5
    out = gpu_prefill(case, kg, vg, query, cu, max_q, context_lens=cl)
    torch.cuda.synchronize()
    assert device_errors() & 4
    g = out.float().cpu().double().numpy()
    assert (g[16:24] == 0).all()
    assert close(g, np.r_[0:16, 24:32])

    # a block id outside the pool in sequence 3's table
    bt = case.block_tables.clone()
    bt[3, 0] = case.num_blocks + 5
    out = gpu_prefill(case, kg, vg, query, cu, max_q, block_tables=bt)
    torch.cuda.synchronize()
    assert device_errors() & 2
    g = out.float().cpu().double().numpy()
    assert np.isfinite(g).all()
    assert close(g, np.r_[0:24])


# ------------------------------------------------------------ INT8 cache
@pytest.mark.parametrize("D,Hq,Hkv,bs,qd,per_seq", [
    (128, 32, 8, 32, torch.bfloat16, 16),    # G 4
    (128, 16, 2, 16, torch.float16, 100),    # G 8, bs 16, several row tiles
    (64, 16, 16, 64, torch.bfloat16, 7),     # G 1, bs 64, D 64
    (64, 12, 4, 32, torch.float16, 300),     # G 3; short contexts taken whole
    (128, 8, 1, 32, torch.bfloat16, 1),      # one query token
])
def test_prefill_int8_matches_oracle(D, Hq, Hkv, bs, qd, per_seq):
    """pa_prefill_int8 against the oracle's prefill over the same INT8 codes
    and row scales; rows past each context hold code -128 and NaN scales
    (never written), which must not reach the output."""
    from _helpers import oracle_int8_caches
    case = wl.make_case(f"pf8_{D}_{Hq}_{Hkv}_{bs}", 140 + D + Hq + bs, 9, Hq, Hkv, D, bs,
                        len_range=(1, 500), q_dtype=qd, kv_dtype="int8", extra_blocks=3)
    kg, vg, ksg, vsg = gpu_int8_caches(case)
    ko, vo, kso, vso = oracle_int8_caches(case)
    assert torch.equal(kg.cpu(), ko) and torch.equal(vg.cpu(), vo)
    query, q_seq, q_pos, cu, max_q = chunk(case, per_seq, 141 + D + per_seq)
    out = torch.full(tuple(query.shape), float("nan"), dtype=qd, device=DEV)
    pa.prefill_int8(out, to_dev(query), kg, vg, ksg, vsg, to_dev(case.block_tables), to_dev(cu),
                    to_dev(case.context_lens), Hkv, max_q, case.scale)
    torch.cuda.synchronize()
    assert device_errors() == 0
    ref, bad = oracle.prefill(query, q_seq, q_pos, ko, vo, case.block_tables, Hkv, bs,
                              case.scale, "int8", k_scales=kso, v_scales=vso)
    assert bad == 0
    g = out.float().cpu().double().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref).max()
    assert err <= TOL, f"max abs error {err:.3g}"


def test_prefill_int8_flags_a_bad_block_and_keeps_the_rest():
    """A block id outside the pool in one sequence's table reads as zeros
    (flagged); the other sequences keep the oracle's answer."""
    from _helpers import oracle_int8_caches
    case = wl.make_case("pf8_bad", 150, 4, 8, 2, 64, lens=[40, 70, 9, 100],
                        q_dtype=torch.bfloat16, kv_dtype="int8", extra_blocks=2)
    kg, vg, ksg, vsg = gpu_int8_caches(case)
    ko, vo, kso, vso = oracle_int8_caches(case)
    query, q_seq, q_pos, cu, max_q = chunk(case, 8, 151)
    ref, _ = oracle.prefill(query, q_seq, q_pos, ko, vo, case.block_tables, 2,
                            case.block_size, case.scale, "int8", k_scales=kso, v_scales=vso)
    device_errors()
    bt = case.block_tables.clone()
    bt[3, 0] = case.num_blocks + 5
    out = torch.full(tuple(query.shape), float("nan"), dtype=torch.bfloat16, device=DEV)
    pa.prefill_int8(out, to_dev(query), kg, vg, ksg, vsg, to_dev(bt), to_dev(cu),
                    to_dev(case.context_lens), 2, max_q, case.scale)
    torch.cuda.synchronize()
    assert device_errors() & 2
    g = out.float().cpu().double().numpy()
    assert np.isfinite(g).all()
    assert np.abs(g[0:24] - ref[0:24]).max() <= TOL


# ------------------------------------------------------------ FP8 cache
@pytest.mark.parametrize("D,Hq,Hkv,bs,qd,per_seq", [
    (128, 32, 8, 32, torch.bfloat16, 16),    # G 4
    (128, 16, 2, 16, torch.float16, 100),    # G 8, bs 16, several row tiles
    (64, 16, 16, 64, torch.bfloat16, 7),     # G 1, bs 64, D 64
    (64, 12, 4, 32, torch.float16, 300),     # G 3; short contexts taken whole
    (128, 8, 1, 32, torch.bfloat16, 1),      # one query token
])
def test_prefill_fp8_matches_oracle(D, Hq, Hkv, bs, qd, per_seq):
    """pa_prefill_fp8 against the oracle's prefill over the same E4M3 codes
    and per-tensor scales ("PagedAttention in mistral.rs", KV Cache
    Quantization); the caches are written by pa_reshape_and_cache and equal
    the oracle's byte for byte."""
    case = wl.make_case(f"pfe_{D}_{Hq}_{Hkv}_{bs}", 160 + D + Hq + bs, 9, Hq, Hkv, D, bs,
                        len_range=(1, 500), q_dtype=qd, kv_dtype="fp8_e4m3", extra_blocks=3)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    assert torch.equal(kg.cpu(), ko) and torch.equal(vg.cpu(), vo)
    query, q_seq, q_pos, cu, max_q = chunk(case, per_seq, 161 + D + per_seq)
    out = torch.full(tuple(query.shape), float("nan"), dtype=qd, device=DEV)
    pa.prefill_fp8(out, to_dev(query), kg, vg, to_dev(case.block_tables), to_dev(cu),
                   to_dev(case.context_lens), Hkv, max_q, case.scale, case.k_scale, case.v_scale)
    torch.cuda.synchronize()
    assert device_errors() == 0
    ref, bad = oracle.prefill(query, q_seq, q_pos, ko, vo, case.block_tables, Hkv, bs,
                              case.scale, "fp8_e4m3", case.k_scale, case.v_scale)
    assert bad == 0
    g = out.float().cpu().double().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref).max()
    assert err <= TOL, f"max abs error {err:.3g}"


def test_prefill_fp8_flags_a_bad_block_and_keeps_the_rest():
    """A block id outside the pool in one sequence's table reads as zeros
    (flagged); the other sequences keep the oracle's answer."""
    case = wl.make_case("pfe_bad", 170, 4, 8, 2, 64, lens=[40, 70, 9, 100],
                        q_dtype=torch.bfloat16, kv_dtype="fp8_e4m3", extra_blocks=2)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    query, q_seq, q_pos, cu, max_q = chunk(case, 8, 171)
    ref, _ = oracle.prefill(query, q_seq, q_pos, ko, vo, case.block_tables, 2,
                            case.block_size, case.scale, "fp8_e4m3", case.k_scale, case.v_scale)
    device_errors()
    bt = case.block_tables.clone()
    bt[3, 0] = case.num_blocks + 5
    out = torch.full(tuple(query.shape), float("nan"), dtype=torch.bfloat16, device=DEV)
    pa.prefill_fp8(out, to_dev(query), kg, vg, to_dev(bt), to_dev(cu), to_dev(case.context_lens),
                   2, max_q, case.scale, case.k_scale, case.v_scale)
    torch.cuda.synchronize()
    assert device_errors() & 2
    g = out.float().cpu().double().numpy()
    assert np.isfinite(g).all()
    assert np.abs(g[0:24] - ref[0:24]).max() <= TOL
