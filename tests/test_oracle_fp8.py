"""Pins of the oracle's FP8 E4M3 encoder/decoder ("PagedAttention in mistral.rs",
KV Cache Quantization: the cache may be stored as F8E4M3).

The oracle's encoder is written from the format definition; here it is held
against PyTorch's own float8_e4m3fn conversion (a library routine), against
the format's fixed points, and against round-to-nearest-even tie rules.
"""
import os

import numpy as np
import pytest
import torch

import oracle

E4M3_MAX = 448.0
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def torch_e4m3(x: np.ndarray) -> np.ndarray:
    """Library routine: saturate, then PyTorch's round-to-nearest-even cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return torch.clamp(t, -E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def compare_codes(x, mine, ref):
    nan_in = np.isnan(x)
    # NaN inputs: any NaN code is a NaN; the oracle keeps the sign (0x7F | sign)
    assert np.all((mine[nan_in] & 0x7F) == 0x7F)
    bad = (~nan_in) & (mine != ref)
    if bad.any():
        i = np.flatnonzero(bad)[:8]
        raise AssertionError(f"mismatch at {x[i]!r}: oracle {mine[i]} torch {ref[i]}")


@pytest.mark.parametrize("sign", [0, 1])
def test_encode_matches_torch_every_pattern_in_rounding_range(sign):
    """Every binary32 pattern with |x| in [2^-11, 2^10): all patterns whose
    E4M3 rounding is not trivially 0 or 448 (below 2^-10 everything rounds to
    zero, above 464 everything saturates)."""
    lo = (116 << 23) | (sign << 31)
    hi = (137 << 23) | (sign << 31)
    step = 1 << 26
    for start in range(lo, hi, step):
        bits = np.arange(start, min(start + step, hi), dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        compare_codes(x, oracle.e4m3_encode(x), torch_e4m3(x))


def test_encode_matches_torch_strided_all_patterns():
    """A stride-251 sweep of all 2^32 patterns: zeros, subnormals, huge values,
    infinities and NaNs of both signs."""
    bits = (np.arange(0, (1 << 32) // 251 + 1, dtype=np.uint64) * 251).astype(np.uint32)
    specials = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000,
                         0xFFC00000, 0x7F7FFFFF, 0xFF7FFFFF, 0x00000001, 0x80000001,
                         0x43E00000, 0x43E80000, 0x43E7FFFF, 0xC3E80000],
                        dtype=np.uint32)
    bits = np.concatenate([bits, specials])
    x = bits.view(np.float32)
    compare_codes(x, oracle.e4m3_encode(x), torch_e4m3(x))


def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]


def test_format_fixed_points():
    """E4M3: bias 7, 3 fraction bits, largest finite 448, smallest subnormal 2^-9."""
    dec = {int(c): float(v) for c, v in enumerate(oracle.e4m3_decode(np.arange(256, dtype=np.uint8)))}
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert dec[0x38] == 1.0  # exponent field 7 = bias
    assert dec[0x08] == 2.0 ** -6  # smallest normal
    assert dec[0x01] == 2.0 ** -9  # smallest subnormal
    assert dec[0x07] == 7 * 2.0 ** -9  # largest subnormal
    assert dec[0x00] == 0.0 and np.signbit(dec[0x80])
    enc = oracle.e4m3_encode(np.array([448.0, 1e9, np.inf, -np.inf, -0.0, 0.0, np.nan, -np.nan],
                                      dtype=np.float32))
    assert list(enc[:6]) == [0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00]
    assert enc[6] == 0x7F and enc[7] == 0xFF


def test_every_code_round_trips():
    """decode then encode gives the same code for all 256 codes (both zeros,
    both NaNs included)."""
    codes = np.arange(256, dtype=np.uint8)
    again = oracle.e4m3_encode(oracle.e4m3_decode(codes))
    assert np.array_equal(again, codes)


def test_ties_round_to_even_code():
    """Midpoints between neighbouring positive codes go to the code with an
    even last bit; a hair above/below goes to the nearer code."""
    vals = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)
    for c in range(0, 0x7E):
        a, b = vals[c], vals[c + 1]
        mid = np.float32((a + b) / 2)
        assert float(mid) == (a + b) / 2  # exactly representable
        want = c if c % 2 == 0 else c + 1
        got = oracle.e4m3_encode(np.array([mid, -mid], dtype=np.float32))
        assert got[0] == want and got[1] == (want | 0x80), (c, a, b)
        up = np.nextafter(mid, np.float32(np.inf))
        dn = np.nextafter(mid, np.float32(0))
        assert oracle.e4m3_encode(np.array([up, dn], dtype=np.float32)).tolist() == [c + 1, c]
    # above the largest code: 464 is the midpoint to the (absent) next value and
    # still gives 448; everything larger saturates as well
    assert oracle.e4m3_encode(np.array([463.99997, 464.0, 464.00003, 3e38],
                                       dtype=np.float32)).tolist() == [0x7E] * 4


def test_fp8_cache_is_half_of_16bit_cache():
    """KV Cache Quantization: an FP8 cache takes half the bytes of a 16-bit one
    (one byte per element instead of two), for the same pool shape."""
    from paged_kv_cache_context_gb300 import workloads as wl
    with open(os.path.join(GOLDEN, "capacity.txt")) as f:
        gold = {l.split()[0]: float(l.split()[1]) for l in f if l.strip() and l[0] != "#"}
    a = wl.make_case("a", 1, 2, 4, 4, 64, lens=[40, 70], q_dtype=torch.bfloat16)
    b = wl.make_case("b", 1, 2, 4, 4, 64, lens=[40, 70], q_dtype=torch.bfloat16,
                     kv_dtype="fp8_e4m3")
    ka, _ = wl.empty_caches(a)
    kb, _ = wl.empty_caches(b)
    assert ka.shape == kb.shape
    ratio = (kb.numel() * kb.element_size()) / (ka.numel() * ka.element_size())
    assert ratio == gold["fp8_over_fp16_bytes"]
