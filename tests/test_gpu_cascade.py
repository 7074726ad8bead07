"""GPU parity of the shared-prefix cascade decode (pa_decode_cascade) and of
block copies (pa_copy_blocks).

Pages: "PagedAttention in mistral.rs" (prefix caching: a prefix's KV state is
kept in the paged cache and reused by later sequences), "libmir-metal
trace/kv.rs" (copy-on-write block maps). The cascade computes exactly what
decode computes, so it is compared with the oracle's decode element by
element, within the bf16 / f16 output tolerance.
"""
import numpy as np
import pytest
import torch

from _gpu import (DEV, assert_close, bits, device_errors, gpu_caches, gpu_decode,
                  gpu_int8_caches, to_dev)
from _helpers import (oracle_caches, oracle_caches_for, oracle_decode, oracle_int8_caches,
                      sampled_seqs)
from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    pa.lib()
    device_errors()


def cascade(case, kg, vg, prefix_pages, block_tables=None, context_lens=None):
    out = torch.full((case.num_seqs, case.num_heads, case.head_dim), float("nan"),
                     dtype=case.q_dtype, device=DEV)
    nbytes = pa.decode_cascade_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                              case.head_dim, case.block_size, prefix_pages)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    pa.decode_cascade(out, to_dev(case.query), kg, vg,
                      to_dev(case.block_tables if block_tables is None else block_tables),
                      to_dev(case.context_lens if context_lens is None else context_lens),
                      case.num_kv_heads, case.scale, prefix_pages, ws)
    return out


@pytest.mark.parametrize("D,Hq,Hkv,bs,qd,prefix_blocks,suffix", [
    (128, 32, 8, 32, torch.bfloat16, 8, (0, 64)),    # the prefix_bf16 shape, scaled
    (128, 32, 8, 32, torch.float16, 3, (1, 100)),
    (64, 16, 16, 16, torch.bfloat16, 9, (0, 40)),    # G = 1, bs 16, a ragged last tile
    (128, 16, 2, 64, torch.bfloat16, 2, (0, 200)),   # G = 8, bs 64
    (64, 12, 4, 32, torch.float16, 5, (0, 31)),      # G = 3 (not a power of two)
])
def test_cascade_matches_oracle(D, Hq, Hkv, bs, qd, prefix_blocks, suffix):
    case = wl.make_case(f"casc{D}_{Hq}_{Hkv}_{bs}", 300 + D + Hq + bs, 21, Hq, Hkv, D, bs,
                        q_dtype=qd, shared_prefix_blocks=prefix_blocks, suffix_range=suffix,
                        extra_blocks=2)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    ref = oracle_decode(case, ko, vo)
    out = cascade(case, kg, vg, prefix_blocks)
    assert_close(case, out, ref, what=f"cascade {case.name}")
    assert device_errors() == 0


def test_cascade_with_part_of_the_prefix_and_many_query_tiles():
    """Treating only the first pages of a longer shared prefix as the prefix
    is still exact (the rest is decoded as each sequence's own pages); 150
    sequences x 4 heads span several 64-row query tiles."""
    case = wl.make_case("casc_part", 311, 150, 16, 4, 128, q_dtype=torch.bfloat16,
                        shared_prefix_blocks=6, suffix_range=(0, 90))
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    ref = oracle_decode(case, ko, vo)
    for pp in (1, 4, 6):
        assert_close(case, cascade(case, kg, vg, pp), ref, what=f"cascade prefix_pages={pp}")
    assert device_errors() == 0


def test_cascade_full_size_prefix_workload():
    """prefix_bf16 at its full size (128 sequences, a 2048-token shared
    prefix: several prefix ranges and one suffix CTA per sequence and kv head,
    as the benchmark's cascade path runs it): every query head of the
    longest, the shortest and two random sequences against the oracle, and
    every row of the batch within the bf16 tolerance of pa_decode."""
    case = wl.config("prefix_bf16", value_device=DEV)
    kg, vg = gpu_caches(case)
    out = cascade(case, kg, vg, 64)
    torch.cuda.synchronize()
    assert device_errors() == 0
    assert torch.isfinite(out.float()).all()
    seqs = sampled_seqs(case)
    ko, vo = oracle_caches_for(case, seqs)
    rows = [s * case.num_heads + h for s in seqs for h in range(case.num_heads)]
    ref = oracle_decode(case, ko, vo, rows=rows)
    assert_close(case, out, ref, rows=rows, what="cascade prefix_bf16, sampled rows")
    dec = gpu_decode(case, kg, vg)
    diff = (out.float() - dec.float()).abs().max().item()
    assert diff <= 2e-2, diff
    assert device_errors() == 0


def test_cascade_flags_broken_preconditions():
    case = wl.make_case("casc_bad", 312, 5, 8, 2, 64, q_dtype=torch.bfloat16,
                        shared_prefix_blocks=4, suffix_range=(1, 20), extra_blocks=3)
    kg, vg = gpu_caches(case)
    bt = case.block_tables.clone()
    bt[3, 1] = bt[3, 1] + 1 if int(bt[3, 1]) + 1 < case.num_blocks else 0  # row 3 disagrees
    out = cascade(case, kg, vg, 4, block_tables=bt)
    torch.cuda.synchronize()
    assert device_errors() & 2
    cl = case.context_lens.clone()
    cl[1] = 4 * 32 - 1  # shorter than the prefix
    cascade(case, kg, vg, 4, context_lens=cl)
    assert device_errors() & 4
    assert torch.isfinite(out.float()).all()


def cascade_8bit(case, caches, prefix_pages, context_lens=None):
    """pa_decode_cascade_fp8 / _int8 on the case's 8-bit caches."""
    out = torch.full((case.num_seqs, case.num_heads, case.head_dim), float("nan"),
                     dtype=case.q_dtype, device=DEV)
    nbytes = pa.decode_cascade_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                              case.head_dim, case.block_size, prefix_pages)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    cl = to_dev(case.context_lens if context_lens is None else context_lens)
    if case.kv_dtype == "fp8_e4m3":
        kg, vg = caches
        pa.decode_cascade_fp8(out, to_dev(case.query), kg, vg, to_dev(case.block_tables), cl,
                              case.num_kv_heads, case.scale, case.k_scale, case.v_scale,
                              prefix_pages, ws)
    else:
        kg, vg, ksg, vsg = caches
        pa.decode_cascade_int8(out, to_dev(case.query), kg, vg, ksg, vsg,
                               to_dev(case.block_tables), cl, case.num_kv_heads, case.scale,
                               prefix_pages, ws)
    return out


@pytest.mark.parametrize("kv", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("D,Hq,Hkv,bs,qd,prefix_blocks,suffix", [
    (128, 32, 8, 32, torch.bfloat16, 8, (0, 64)),    # the prefix_bf16 shape, scaled
    (64, 16, 16, 16, torch.float16, 9, (0, 40)),     # G = 1, bs 16, a ragged last tile
    (128, 16, 2, 64, torch.bfloat16, 2, (0, 200)),   # G = 8, bs 64
    (64, 12, 4, 32, torch.bfloat16, 5, (0, 31)),     # G = 3 (not a power of two)
])
def test_cascade_8bit_matches_oracle(kv, D, Hq, Hkv, bs, qd, prefix_blocks, suffix):
    """The cascade over an FP8 E4M3 cache (per-tensor scales) or an INT8 cache
    (per-row scales): the oracle's decode over the same codes, element by
    element within the bf16 / f16 output tolerance."""
    case = wl.make_case(f"casc8{kv}{D}_{Hq}_{Hkv}_{bs}", 330 + D + Hq + bs, 21, Hq, Hkv, D, bs,
                        q_dtype=qd, kv_dtype=kv, shared_prefix_blocks=prefix_blocks,
                        suffix_range=suffix, extra_blocks=2)
    if kv == "int8":
        caches = gpu_int8_caches(case)
        ko, vo, kso, vso = oracle_int8_caches(case)
        ref = oracle_decode(case, ko, vo, k_scales=kso, v_scales=vso)
    else:
        caches = gpu_caches(case)
        ko, vo = oracle_caches(case)
        ref = oracle_decode(case, ko, vo)
    out = cascade_8bit(case, caches, prefix_blocks)
    assert_close(case, out, ref, what=f"cascade {case.name}")
    assert device_errors() == 0


@pytest.mark.parametrize("kv", ["fp8_e4m3", "int8"])
def test_cascade_8bit_full_size_prefix_workload(kv):
    """prefix_bf16's shape (128 sequences, a 2048-token shared prefix) over an
    8-bit cache: every query head of sampled sequences against the oracle."""
    case = wl.make_case(f"prefix_{kv}", 340, 128, 32, 8, 128, q_dtype=torch.bfloat16,
                        kv_dtype=kv, shared_prefix_blocks=64, suffix_range=(0, 512),
                        value_device=DEV)
    caches = gpu_int8_caches(case) if kv == "int8" else gpu_caches(case)
    out = cascade_8bit(case, caches, 64)
    torch.cuda.synchronize()
    assert device_errors() == 0
    assert torch.isfinite(out.float()).all()
    seqs = sampled_seqs(case)
    rows = [s * case.num_heads + h for s in seqs for h in range(case.num_heads)]
    if kv == "int8":
        ko, vo, kso, vso = oracle_int8_caches(case)
        ref = oracle_decode(case, ko, vo, rows=rows, k_scales=kso, v_scales=vso)
    else:
        ko, vo = oracle_caches_for(case, seqs)
        ref = oracle_decode(case, ko, vo, rows=rows)
    assert_close(case, out, ref, rows=rows, what=f"cascade {kv} prefix workload, sampled rows")


def test_cascade_8bit_flags_broken_preconditions():
    case = wl.make_case("casc8_bad", 350, 5, 8, 2, 64, q_dtype=torch.bfloat16,
                        kv_dtype="fp8_e4m3", shared_prefix_blocks=4, suffix_range=(1, 20),
                        extra_blocks=3)
    caches = gpu_caches(case)
    cl = case.context_lens.clone()
    cl[1] = 4 * 32 - 1  # shorter than the prefix
    out = cascade_8bit(case, caches, 4, context_lens=cl)
    torch.cuda.synchronize()
    assert device_errors() & 4
    assert torch.isfinite(out.float()).all()


def test_copy_blocks_is_exact_and_touches_nothing_else():
    for dt, elem in ((torch.bfloat16, 2), (torch.uint8, 1), (torch.float32, 4)):
        g = torch.Generator().manual_seed(313)
        shape = (12, 4, 32, 64)
        if dt == torch.uint8:
            kc = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
        else:
            kc = torch.randn(shape, generator=g).to(dt)
        vc = kc.flip(0).clone()
        pairs = torch.tensor([[1, 7], [3, 0], [11, 5]], dtype=torch.int32)
        want_k, want_v = kc.clone(), vc.clone()
        for s, d in pairs.tolist():
            want_k[d] = kc[s]
            want_v[d] = vc[s]
        kg, vg = kc.to(DEV), vc.to(DEV)
        pa.copy_blocks(kg, vg, pairs.to(DEV))
        assert torch.equal(bits(kg.cpu()), bits(want_k)) and torch.equal(bits(vg.cpu()),
                                                                          bits(want_v))
        assert device_errors() == 0
    bad = torch.tensor([[2, 12], [4, 6]], dtype=torch.int32, device=DEV)
    before = kg.clone()
    pa.copy_blocks(kg, vg, bad)
    assert device_errors() & 2
    want = before.clone()
    want[6] = before[4]
    assert torch.equal(bits(kg.cpu()), bits(want.cpu()))


def test_cascade_when_some_contexts_end_at_the_prefix():
    """A context exactly as long as the prefix has no page of its own: its
    output is the prefix's attention alone."""
    import dataclasses
    case = wl.make_case("casc_end", 314, 7, 8, 2, 128, q_dtype=torch.bfloat16,
                        shared_prefix_blocks=3, suffix_range=(0, 50))
    kg, vg = gpu_caches(case)
    cl = case.context_lens.clone()
    cl[::2] = 3 * 32
    short = dataclasses.replace(case, context_lens=cl)
    ko, vo = oracle_caches(case)
    ref = oracle_decode(short, ko, vo)
    assert_close(short, cascade(short, kg, vg, 3), ref, what="cascade, empty suffixes")
    assert device_errors() == 0
