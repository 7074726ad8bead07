"""GPU parity of the cache write path (reshape_and_cache, FP8 E4M3 encode) and
of the ring-aware slot mapping: bit-exact against the oracle.

"Optimization plans" (mistral.rs discussion #46) traces junk output to a wrong
reshape_and_cache, so these run before any decode parity test.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import DEV, bits, device_errors, gpu_caches, gpu_slot_mapping, to_dev
from _helpers import oracle_caches
from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    pa.lib()
    device_errors()


def test_slot_mapping_bit_exact_paged_and_ring():
    for case in (wl.make_case("p", 21, 6, 8, 2, 64, len_range=(1, 300), extra_blocks=4),
                 wl.make_case("r", 22, 5, 8, 2, 64, lens=[3, 64, 65, 129, 400], window=64,
                              ring_overwrite=True),
                 wl.make_case("b16", 23, 4, 4, 4, 64, 16, len_range=(1, 90))):
        for a, b in case.pre_chunks:
            seq, pos = case.pre_seq[a:b], case.pre_pos[a:b]
            want, bad = oracle.slot_mapping(case.block_tables, seq, pos, case.block_size,
                                            case.window)
            got = gpu_slot_mapping(case, seq, pos).cpu()
            assert bad == 0 and torch.equal(got, want)
        want, _ = oracle.slot_mapping(case.block_tables, None, case.new_pos, case.block_size,
                                      case.window)
        assert torch.equal(gpu_slot_mapping(case, None, case.new_pos).cpu(), want)
    assert device_errors() == 0


def test_slot_mapping_padding_and_bad_sequence():
    case = wl.make_case("p", 24, 3, 4, 4, 64, lens=[10, 40, 70])
    pos = torch.tensor([-1, 5, 69, 3 * 32], dtype=torch.int32)
    seq = torch.tensor([0, 7, 2, 2], dtype=torch.int32)  # seq 7 does not exist
    got = gpu_slot_mapping(case, seq, pos).cpu()
    want, bad = oracle.slot_mapping(case.block_tables, seq, pos, 32, 0)
    assert torch.equal(got, want) and bad == 2
    assert got[0] == -1 and got[1] == -1 and got[3] == -1
    assert device_errors() == 16


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 96, 128])
def test_auto_write_bit_exact_whole_pool(dtype, D):
    case = wl.make_case("w", 30 + D, 5, 8, 4, D, len_range=(1, 150), q_dtype=dtype,
                        extra_blocks=6)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    assert torch.equal(bits(kg), bits(ko)) and torch.equal(bits(vg), bits(vo))
    assert device_errors() == 0


@pytest.mark.parametrize("src", [torch.float32, torch.bfloat16, torch.float16])
def test_fp8_write_bit_exact_whole_pool(src):
    case = wl.make_case("w8", 40, 6, 8, 8, 96, len_range=(1, 200), q_dtype=torch.bfloat16,
                        kv_dtype="fp8_e4m3", kv_src_dtype=src, extra_blocks=5)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    assert torch.equal(kg.cpu(), ko) and torch.equal(vg.cpu(), vo)
    assert device_errors() == 0


def test_fp8_encode_every_fp32_bit_pattern():
    """All 2^32 binary32 patterns through pa_reshape_and_cache (scale 1), in
    chunks of 2^28, against the oracle's E4M3 encoder, byte for byte (NaN codes
    and signs included)."""
    D, bs = 128, 32
    chunk = 1 << 28
    T = chunk // D
    slots = torch.arange(T, dtype=torch.int64, device=DEV)
    kc = torch.empty(T // bs, 1, bs, D, dtype=torch.uint8, device=DEV)
    vc = torch.empty_like(kc)
    for start in range(0, 1 << 32, chunk):
        pat = torch.arange(start, start + chunk, dtype=torch.int64, device=DEV)
        pat = torch.where(pat >= 1 << 31, pat - (1 << 32), pat)  # same 32 bits, signed
        x = pat.to(torch.int32).view(torch.float32).view(T, 1, D)
        pa.reshape_and_cache(x, x, kc, vc, slots, "fp8_e4m3", 1.0, 1.0)
        got = kc.view(-1).cpu().numpy()
        host = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        want = oracle.e4m3_encode(host)
        if not np.array_equal(got, want):
            i = np.flatnonzero(got != want)[:5]
            raise AssertionError(f"patterns {host.view(np.uint32)[i]}: gpu {got[i]} oracle {want[i]}")
        assert torch.equal(kc, vc)
    assert device_errors() == 0


def test_fp8_division_by_scale_is_ieee():
    """Random values and awkward scales: the quantised code is E4M3(x / s) with
    a correctly rounded binary32 division."""
    g = torch.Generator().manual_seed(41)
    x = (torch.randn(4096, 1, 64, generator=g) * 300).float()
    for s in (0.7, 1.0 / 3.0, 2.2e-3, 1e-30, 3.1e7):
        s = float(np.float32(s))
        slots = torch.arange(4096, dtype=torch.int64)
        kc = torch.zeros(128, 1, 32, 64, dtype=torch.uint8)
        vc = torch.zeros_like(kc)
        oracle.reshape_and_cache(x, x, kc, vc, slots, 32, "fp8_e4m3", s, s)
        kg = torch.zeros_like(kc, device=DEV)
        vg = torch.zeros_like(kg)
        pa.reshape_and_cache(to_dev(x), to_dev(x), kg, vg, to_dev(slots), "fp8_e4m3", s, s)
        assert torch.equal(kg.cpu(), kc)
    assert device_errors() == 0


def test_write_skips_padding_and_flags_out_of_range():
    case = wl.make_case("pad", 42, 3, 4, 2, 64, lens=[5, 40, 70], q_dtype=torch.float32)
    kg, vg = wl.empty_caches(case, device=DEV)
    before = bits(kg).clone()
    cap = case.num_blocks * 32
    slots = torch.tensor([-1, cap, cap + 77], dtype=torch.int64, device=DEV)
    pa.reshape_and_cache(to_dev(case.new_key), to_dev(case.new_value), kg, vg, slots)
    assert torch.equal(bits(kg), before)
    assert device_errors() == 1
    assert device_errors() == 0  # reading clears the word
