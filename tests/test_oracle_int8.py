"""Pins of the oracle's INT8 per-token/head cache.

"libmir-metal trace/kv.rs" names a KV cache of packed INT8 pages with one FP32
scale per token and head, dequantised inside the paged attention. The oracle
reads that as symmetric per-row quantisation: scale = max|x| / 127, code =
round-to-nearest-even(x / scale) clamped to +-127, value = code * scale. These
tests hold it against closed forms (rows whose scale is exactly 1, all-zero
rows, the largest element landing on +-127), the half-step error bound that
any correct rounding quantiser meets, PyTorch's own rounding as a library
routine, and dense float64 attention over PyTorch-dequantised rows.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import dense_reference, oracle_decode, oracle_int8_caches, torch_int8_dequant
from paged_kv_cache_context_gb300 import workloads as wl


def test_rows_with_unit_scale_round_half_to_even():
    x = np.array([[127, -127, 0.5, 1.5, 2.5, -0.5, -2.5, 3.49, 126.5, -0.0]], np.float32)
    codes, scales = oracle.int8_quantise_rows(x)
    assert scales.tolist() == [1.0]
    assert codes.tolist() == [[127, -127, 0, 2, 2, 0, -2, 3, 126, 0]]


def test_zero_and_underflowing_rows_store_zero_codes():
    x = np.zeros((2, 16), np.float32)
    x[1, 3] = np.float32(1e-44)  # max / 127 underflows to zero
    codes, scales = oracle.int8_quantise_rows(x)
    assert np.all(codes == 0) and np.all(scales == 0)


def test_scale_is_max_over_127_and_the_largest_element_is_127():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((400, 96)) * np.exp(rng.uniform(-40, 40, (400, 1)))).astype(np.float32)
    codes, scales = oracle.int8_quantise_rows(x)
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(scales, (amax / np.float32(127)).astype(np.float32))
    i = np.abs(x).argmax(axis=1)
    top = codes[np.arange(400), i].astype(np.int32)
    assert np.all(np.abs(top) == 127)
    assert np.all(np.sign(top) == np.sign(x[np.arange(400), i]))
    assert codes.min() >= -127


def test_dequantised_values_are_within_half_a_step():
    """|code * scale - x| <= scale / 2 (plus the binary32 rounding of x / scale
    and of the product); a wrong divisor (128, 255) or truncation fails it."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((300, 128)).astype(np.float32) * np.float32(3.7)
    codes, scales = oracle.int8_quantise_rows(x)
    deq = codes.astype(np.float64) * scales[:, None].astype(np.float64)
    err = np.abs(deq - x.astype(np.float64))
    bound = scales[:, None].astype(np.float64) * (0.5 + 2.0 ** -16)
    assert np.all(err <= bound)
    # the grid is used, not wasted: the error reaches ~ half a step somewhere
    assert err.max() > 0.4 * scales.max()


def test_rows_match_library_rounding():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((200, 64)).astype(np.float32)
    x[:20] *= np.float32(1e-30)
    x[20:40] *= np.float32(1e30)
    codes, scales = oracle.int8_quantise_rows(x)
    deq = codes.astype(np.float32) * scales[:, None]
    assert np.array_equal(deq, torch_int8_dequant(torch.from_numpy(x)).numpy())


def test_write_places_codes_and_scales_per_row_and_leaves_the_rest():
    case = wl.make_case("w_i8", 41, 4, 8, 2, 64, lens=[1, 30, 33, 70], q_dtype=torch.bfloat16,
                        kv_dtype="int8", extra_blocks=3)
    kc, vc, ks, vs = oracle_int8_caches(case)
    written = torch.zeros(case.num_blocks, 32, dtype=torch.bool)
    for s in range(case.num_seqs):
        pos, key, val = case.tokens_of(s)
        sm, _ = oracle.slot_mapping(case.block_tables, torch.full_like(pos, s), pos, 32)
        for i, slot in enumerate(sm.tolist()):
            b, r = divmod(slot, 32)
            written[b, r] = True
            for cache, sc, x in ((kc, ks, key[i]), (vc, vs, val[i])):
                xf = x.float()
                want_scale = xf.abs().amax(dim=-1) / torch.tensor(127.0)
                assert torch.equal(sc[b, :, r], want_scale)
                want = torch.clamp(torch.round(xf / want_scale[:, None]), -127, 127).to(torch.int8)
                assert torch.equal(cache[b, :, r], want)
    rest = kc.permute(0, 2, 1, 3)[~written]
    assert torch.all(rest == -128)
    assert torch.all(torch.isnan(ks.permute(0, 2, 1)[~written]))
    bad = torch.tensor([case.num_blocks * 32])
    assert oracle.reshape_and_cache_int8(case.new_key[:1], case.new_value[:1], kc, vc, ks, vs,
                                         bad, 32) == 1


@pytest.mark.parametrize("D,Hq,Hkv,bs,window", [(64, 8, 2, 32, 0), (96, 4, 4, 16, 0),
                                               (128, 16, 2, 32, 64)])
def test_int8_decode_equals_dense_over_library_dequantised_rows(D, Hq, Hkv, bs, window):
    lens = [1, 17, 64, 100, 150] if window else [1, 31, 33, 90]
    case = wl.make_case(f"i8_{D}", 42 + D, len(lens), Hq, Hkv, D, bs, lens=lens,
                        q_dtype=torch.bfloat16, kv_dtype="int8", window=window, extra_blocks=2)
    kc, vc, ks, vs = oracle_int8_caches(case)
    out = oracle_decode(case, kc, vc, k_scales=ks, v_scales=vs)
    for s in range(case.num_seqs):
        for h in range(case.num_heads):
            ref = dense_reference(case, s, h)
            np.testing.assert_allclose(out[s, h], ref, rtol=0,
                                       atol=1e-12 * max(1.0, np.abs(ref).max()))


def test_per_row_scales_are_read_per_row():
    """Scaling one cached row's K scale changes that row's logit only: with a
    single attended row the output is that row's dequantised V, whatever K."""
    case = wl.make_case("i8_one", 43, 2, 4, 1, 64, lens=[1, 2], q_dtype=torch.float32,
                        kv_dtype="int8")
    kc, vc, ks, vs = oracle_int8_caches(case)
    out = oracle_decode(case, kc, vc, k_scales=ks, v_scales=vs)
    b = int(case.block_tables[0, 0])
    want = (vc[b, 0, 0].float() * vs[b, 0, 0]).double()  # one binary32 multiply
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], want.numpy())
    ks2 = ks.clone()
    b1 = int(case.block_tables[1, 0])
    ks2[b1, 0, 1] *= 3
    out2 = oracle_decode(case, kc, vc, k_scales=ks2, v_scales=vs)
    np.testing.assert_array_equal(out2[0], out[0])
    assert not np.allclose(out2[1], out[1])
