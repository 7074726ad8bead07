"""GPU parity of the INT8 per-token/head cache: the write (codes and fp32 row
scales, bit for bit) and the decode (element by element against the oracle,
within the bf16 / f16 output tolerance), through the C ABI.

Page: "libmir-metal trace/kv.rs" (packed INT8 pages with per-token/head FP32
scales, dequantised inside the paged attention).
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import DEV, assert_close, bits, device_errors, gpu_slot_mapping, to_dev
from _helpers import oracle_decode, oracle_int8_caches
from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    pa.lib()
    device_errors()


def gpu_int8_caches(case):
    """INT8 caches and row scales on the GPU, written by pa_slot_mapping and
    pa_reshape_and_cache_int8 in the same order as the oracle's."""
    kc, vc = wl.empty_caches(case, device=DEV)
    ks, vs = wl.empty_scales(case, device=DEV)
    steps = [(case.pre_seq[a:b], case.pre_pos[a:b], case.pre_key[a:b], case.pre_value[a:b])
             for a, b in case.pre_chunks if b > a]
    steps.append((None, case.new_pos, case.new_key, case.new_value))
    for seq, pos, key, val in steps:
        sm = gpu_slot_mapping(case, seq, pos)
        pa.reshape_and_cache_int8(to_dev(key), to_dev(val), kc, vc, ks, vs, sm)
    return kc, vc, ks, vs


def gpu_decode_int8(case, kc, vc, ks, vs, balanced=True):
    out = torch.full((case.num_seqs, case.num_heads, case.head_dim), float("nan"),
                     dtype=case.q_dtype, device=DEV)
    ws = None
    if balanced:
        n = pa.decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                     case.head_dim, case.block_size, case.max_blocks_per_seq,
                                     case.window)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    pa.decode_int8(out, to_dev(case.query), kc, vc, ks, vs, to_dev(case.block_tables),
                   to_dev(case.context_lens), case.num_kv_heads, case.scale, case.window, ws)
    return out


@pytest.mark.parametrize("src", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 96, 128])
def test_int8_write_bit_exact_whole_pool(src, D):
    case = wl.make_case("w8", 60 + D, 5, 8, 4, D, len_range=(1, 150), q_dtype=torch.bfloat16,
                        kv_dtype="int8", kv_src_dtype=src, extra_blocks=6)
    kg, vg, ksg, vsg = gpu_int8_caches(case)
    ko, vo, kso, vso = oracle_int8_caches(case)
    assert torch.equal(kg.cpu(), ko) and torch.equal(vg.cpu(), vo)
    assert torch.equal(bits(ksg), bits(kso)) and torch.equal(bits(vsg), bits(vso))
    assert device_errors() == 0


def test_int8_write_padding_zero_rows_and_bad_slots():
    case = wl.make_case("w8z", 61, 3, 4, 2, 64, lens=[5, 40, 70], kv_dtype="int8",
                        extra_blocks=2)
    kc, vc = wl.empty_caches(case, device=DEV)
    ks, vs = wl.empty_scales(case, device=DEV)
    key = torch.randn(4, 2, 64, generator=torch.Generator().manual_seed(62)).to(torch.bfloat16)
    key[1] = 0  # an all-zero row: scale 0, codes 0
    val = key.flip(0).contiguous()
    cap = case.num_blocks * 32
    slots = torch.tensor([3, 7, -1, cap], dtype=torch.int64)
    pa.reshape_and_cache_int8(to_dev(key), to_dev(val), kc, vc, ks, vs, to_dev(slots))
    torch.cuda.synchronize()
    assert device_errors() & 1  # slot beyond the pool
    ko, vo = wl.empty_caches(case)
    kso, vso = wl.empty_scales(case)
    assert oracle.reshape_and_cache_int8(key, val, ko, vo, kso, vso, slots, 32) == 1
    assert torch.equal(kc.cpu(), ko) and torch.equal(vc.cpu(), vo)
    assert torch.equal(bits(ks), bits(kso)) and torch.equal(bits(vs), bits(vso))
    assert float(ks[0, 0, 7]) == 0.0 and torch.all(kc[0, :, 7] == 0)


@pytest.mark.parametrize("D,Hq,Hkv,bs,qd", [
    (128, 32, 8, 32, torch.bfloat16),   # G = 4, the mistral shape
    (128, 32, 8, 16, torch.float16),
    (96, 16, 16, 32, torch.bfloat16),   # G = 1, D 96 (two-code pieces)
    (64, 16, 2, 64, torch.bfloat16),    # G = 8, bs 64
    (64, 12, 4, 32, torch.float16),     # G = 3
    (128, 8, 4, 64, torch.float16),     # G = 2
    (128, 8, 8, 32, torch.bfloat16),    # G = 1, swizzled rows
    (96, 32, 4, 16, torch.float16),     # G = 8, bs 16: four pages per iteration
])
def test_int8_decode_matches_oracle_both_modes(D, Hq, Hkv, bs, qd):
    case = wl.make_case(f"d8_{D}_{Hq}_{Hkv}_{bs}", 70 + D + Hq + bs, 23, Hq, Hkv, D, bs,
                        len_range=(1, 700), q_dtype=qd, kv_dtype="int8", extra_blocks=3)
    kg, vg, ksg, vsg = gpu_int8_caches(case)
    ko, vo, kso, vso = oracle_int8_caches(case)
    ref = oracle_decode(case, ko, vo, k_scales=kso, v_scales=vso)
    for balanced in (True, False):
        out = gpu_decode_int8(case, kg, vg, ksg, vsg, balanced)
        assert_close(case, out, ref, what=f"int8 decode balanced={balanced}")
    assert device_errors() == 0


def test_int8_decode_ring_and_empty_contexts():
    case = wl.make_case("d8_ring", 81, 6, 16, 4, 128, lens=[0, 1, 64, 65, 300, 1000],
                        window=128, ring_overwrite=True, kv_dtype="int8")
    kg, vg, ksg, vsg = gpu_int8_caches(case)
    ko, vo, kso, vso = oracle_int8_caches(case)
    ref = oracle_decode(case, ko, vo, k_scales=kso, v_scales=vso)
    for balanced in (True, False):
        out = gpu_decode_int8(case, kg, vg, ksg, vsg, balanced)
        assert_close(case, out, ref, what="int8 ring")
        assert torch.all(out[0] == 0)
    assert device_errors() == 0


def test_int8_decode_full_size_mistral_shape_sampled_rows():
    """The mistral_bf16 batch (32 sequences of 512-4096 tokens, 32 q / 8 kv
    heads, D 128) held as an INT8 cache: sampled rows against the oracle."""
    base = wl.config("mistral_bf16")
    case = wl.make_case("mistral_int8", base.seed, 32, 32, 8, 128, len_range=(512, 4096),
                        kv_dtype="int8")
    kg, vg, ksg, vsg = gpu_int8_caches(case)
    out = gpu_decode_int8(case, kg, vg, ksg, vsg)
    rng = np.random.default_rng(82)
    rows = np.sort(rng.choice(case.num_seqs * case.num_heads, 48, replace=False))
    ko, vo, kso, vso = oracle_int8_caches(case)
    ref = oracle_decode(case, ko, vo, rows=rows, k_scales=kso, v_scales=vso)
    assert_close(case, out, ref, rows=rows, what="int8 full size")
    assert device_errors() == 0


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 8, 2), (128, 16, 4)])  # plain / swizzled staged rows
def test_int8_decode_never_reads_rows_past_the_context(D, Hq, Hkv):
    """Unwritten rows hold code -128 and NaN scales; the output stays finite
    and equal to the oracle's."""
    case = wl.make_case(f"d8_stale{D}", 83, 9, Hq, Hkv, D, len_range=(1, 100), kv_dtype="int8",
                        extra_blocks=4)
    kg, vg, ksg, vsg = gpu_int8_caches(case)
    assert torch.isnan(ksg).any()
    ko, vo, kso, vso = oracle_int8_caches(case)
    ref = oracle_decode(case, ko, vo, k_scales=kso, v_scales=vso)
    assert_close(case, gpu_decode_int8(case, kg, vg, ksg, vsg), ref, what="int8 stale rows")
    assert device_errors() == 0
