"""GPU parity of paged decode (pa_decode, pa_decode_partials, pa_reduce) against
the oracle, element by element, on the named workloads at reduced sizes and on
random shapes that span several pages, splits and a ragged tail.

Pages: "PagedAttention in mistral.rs" (blocked cache, FP8 E4M3 cache),
"Rolling buffer cache" (slot i mod W, attend the last W positions).
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import (DEV, assert_close, bits, device_errors, gpu_caches, gpu_decode, to_dev)
from _helpers import oracle_caches, oracle_decode
from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    pa.lib()
    device_errors()


def check_case(case, splits=(True, False)):
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    assert torch.equal(bits(kg), bits(ko)) and torch.equal(bits(vg), bits(vo)), "cache write"
    ref = oracle_decode(case, ko, vo)
    for split in splits:
        out = gpu_decode(case, kg, vg, split=split)
        assert_close(case, out, ref, what=f"{case.name} split={split}")
    assert device_errors() == 0


def test_tiny_workload():
    check_case(wl.config("tiny"))


@pytest.mark.parametrize("name,seqs,div", [("mistral_bf16", 6, 8), ("ring_bf16", 3, 16),
                                           ("fp8_phi3", 6, 8), ("prefix_bf16", 8, 8)])
def test_named_workloads_scaled(name, seqs, div):
    check_case(wl.scaled_config(name, seqs, div))


def test_ring_with_overwrites():
    check_case(wl.make_case("ringow", 51, 4, 16, 4, 128, lens=[5, 256, 257, 1000], window=256,
                            ring_overwrite=True))


SHAPES = [  # (D, Hq, Hkv, bs, q dtype, kv)
    (64, 4, 4, 32, torch.float32, "auto"),
    (96, 8, 8, 32, torch.bfloat16, "auto"),
    (128, 16, 2, 32, torch.bfloat16, "auto"),   # G = 8
    (128, 12, 4, 32, torch.float16, "auto"),    # G = 3 (padded to 4)
    (64, 16, 8, 16, torch.bfloat16, "auto"),    # G = 2, bs 16
    (128, 8, 8, 64, torch.float32, "auto"),     # bs 64
    (96, 32, 32, 32, torch.bfloat16, "fp8_e4m3"),
    (128, 32, 8, 32, torch.bfloat16, "fp8_e4m3"),
    (64, 14, 2, 16, torch.float32, "fp8_e4m3"),  # G = 7
    (96, 6, 6, 64, torch.float16, "fp8_e4m3"),
    (128, 40, 5, 32, torch.float16, "auto"),    # G = 8
    # tensor-core consumers with other stage counts and slice layouts
    (64, 16, 4, 32, torch.bfloat16, "auto"),    # G = 4, D 64: 7 stages
    (64, 32, 4, 16, torch.float16, "auto"),     # G = 8, bs 16: 4 pages per iteration
    (128, 32, 8, 64, torch.bfloat16, "auto"),   # G = 4, bs 64: one page per iteration
    # FP8 tensor-core consumers: every head_dim, group bucket and slice layout
    (64, 16, 8, 16, torch.bfloat16, "fp8_e4m3"),   # G = 2, bs 16: 4 pages per iteration
    (128, 16, 2, 64, torch.float16, "fp8_e4m3"),   # G = 8, bs 64: one page per iteration
    (96, 24, 8, 32, torch.bfloat16, "fp8_e4m3"),   # G = 3 (bucket 4)
    (128, 8, 8, 16, torch.bfloat16, "fp8_e4m3"),   # G = 1, D 128
    (64, 40, 5, 64, torch.float16, "fp8_e4m3"),    # G = 8, D 64
]


@pytest.mark.parametrize("D,Hq,Hkv,bs,qd,kv", SHAPES)
def test_random_shapes_and_edge_lengths(D, Hq, Hkv, bs, qd, kv):
    MB = 24
    ns, pps = pa.decode_plan(1, Hq, Hkv, D, bs, MB, 0)
    edge = {1, bs - 1, bs, bs + 1, 2 * bs + 3, MB * bs, MB * bs - 1}
    if ns > 1:
        edge |= {pps * bs - 1, pps * bs, pps * bs + 1}
    lens = sorted(x for x in edge if 1 <= x <= MB * bs)
    case = wl.make_case(f"shape{D}_{Hq}_{Hkv}_{bs}", 60 + D + Hq + bs, len(lens), Hq, Hkv, D, bs,
                        lens=lens, q_dtype=qd, kv_dtype=kv,
                        kv_src_dtype=torch.float32 if kv != "auto" else None,
                        max_blocks_per_seq=MB, extra_blocks=3)
    check_case(case)


def test_many_splits_forced_through_partials_and_reduce():
    """pa_decode_partials with a fine explicit plan, then pa_reduce, equals the
    oracle; every partial equals the oracle's partial over its slot range."""
    case = wl.make_case("parts", 70, 3, 8, 2, 128, lens=[1, 300, 777], q_dtype=torch.float32,
                        max_blocks_per_seq=25)
    kg, vg = gpu_caches(case)
    ko, vo = oracle_caches(case)
    S, Hq, D = case.num_seqs, case.num_heads, case.head_dim
    pps = 3
    ns = -(-case.max_blocks_per_seq // pps)
    tmp = torch.full((S, Hq, ns, D), float("nan"), device=DEV)
    ml = torch.empty(S, Hq, ns, device=DEV)
    es = torch.empty(S, Hq, ns, device=DEV)
    pa.decode_partials(tmp, ml, es, to_dev(case.query), kg, vg, to_dev(case.block_tables),
                       to_dev(case.context_lens), case.num_kv_heads, case.scale, ns, pps)
    tmp_c, ml_c, es_c = tmp.cpu().double().numpy(), ml.cpu().double().numpy(), es.cpu().double().numpy()
    for s in range(S):
        for h in range(Hq):
            for i in range(ns):
                o, m, l = oracle.decode_partial(case.query, ko, vo, case.block_tables,
                                                case.context_lens, s, h, case.num_kv_heads, 32,
                                                case.scale, i * pps * 32, (i + 1) * pps * 32)
                if l == 0:
                    assert ml_c[s, h, i] == -np.inf and es_c[s, h, i] == 0
                    assert np.isnan(tmp_c[s, h, i]).all()  # left untouched
                    continue
                assert abs(ml_c[s, h, i] - m) <= 1e-4 * max(1, abs(m))
                assert abs(es_c[s, h, i] - l) <= 1e-4 * l
                np.testing.assert_allclose(tmp_c[s, h, i], o, rtol=0,
                                           atol=1e-3 * max(np.abs(o).max(), 1e-6))
    out = torch.empty(S, Hq, D, device=DEV)
    pa.reduce(out, tmp, ml, es)
    assert_close(case, out, oracle_decode(case, ko, vo), what="partials+reduce")
    assert device_errors() == 0


@pytest.mark.parametrize("odt,NS", [(torch.float32, 7), (torch.bfloat16, 7), (torch.float16, 7),
                                    (torch.float32, 8), (torch.bfloat16, 13), (torch.float32, 40)])
def test_reduce_matches_oracle_on_generated_partials(odt, NS):
    """pa_reduce on seeded partials (some splits empty with NaN garbage rows):
    up to 8 splits are loaded in one round, more in rounds of 8."""
    g = torch.Generator().manual_seed(80 + NS)
    S, Hq, D = 5, 6, 96
    o = torch.randn(S, Hq, NS, D, generator=g)
    m = torch.randn(S, Hq, NS, generator=g) * 5
    l = torch.rand(S, Hq, NS, generator=g) * 10 + 0.1
    empty = torch.rand(S, Hq, NS, generator=g) < 0.3
    empty[0, 0, :] = True  # a row with no tokens at all
    m[empty] = -float("inf")
    l[empty] = 0
    o[empty] = float("nan")
    out = torch.empty(S, Hq, D, dtype=odt, device=DEV)
    pa.reduce(out, to_dev(o), to_dev(m), to_dev(l))
    ref = oracle.reduce(o.numpy(), m.numpy(), l.numpy())
    got = out.float().cpu().double().numpy()
    tol = 2e-2 if odt != torch.float32 else 1e-5
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= tol
    assert np.all(got[0, 0] == 0)


def test_single_token_returns_value_row_exactly():
    for dt in (torch.float32, torch.bfloat16):
        case = wl.make_case("one", 90, 4, 8, 2, 128, lens=[1, 1, 1, 1], q_dtype=dt)
        kg, vg = gpu_caches(case)
        out = gpu_decode(case, kg, vg).cpu()
        want = case.new_value.repeat_interleave(4, dim=1)
        assert torch.equal(bits(out), bits(want))


def test_fp8_single_token_is_dequantised_value():
    case = wl.make_case("one8", 91, 2, 4, 4, 96, lens=[1, 1], q_dtype=torch.float32,
                        kv_dtype="fp8_e4m3", kv_src_dtype=torch.float32)
    kg, vg = gpu_caches(case)
    out = gpu_decode(case, kg, vg).cpu().double().numpy()
    ko, vo = oracle_caches(case)
    np.testing.assert_allclose(out, oracle_decode(case, ko, vo), rtol=1e-6, atol=0)


def test_empty_context_and_poisoned_tails_give_finite_output():
    case = wl.make_case("empty", 92, 4, 8, 8, 64, lens=[0, 1, 31, 33], q_dtype=torch.bfloat16,
                        extra_blocks=4)
    kg, vg = gpu_caches(case)
    for split in (True, False):
        out = gpu_decode(case, kg, vg, split=split).cpu()
        assert torch.all(out[0] == 0)
        assert torch.isfinite(out.float()).all()
    check_case(case)


def test_block_relabelling_gives_bit_identical_output():
    case = wl.make_case("relabel", 93, 6, 16, 4, 128, len_range=(1, 700), extra_blocks=9,
                        max_blocks_per_seq=22)
    kg, vg = gpu_caches(case)
    out = gpu_decode(case, kg, vg)
    perm = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(94))
    k2 = torch.empty_like(kg)
    v2 = torch.empty_like(vg)
    k2[to_dev(perm)] = kg
    v2[to_dev(perm)] = vg
    bt = case.block_tables.clone()
    owned = bt >= 0
    bt[owned] = perm[bt[owned].long()].to(torch.int32)
    out2 = gpu_decode(case, k2, v2, block_tables=bt)
    assert torch.equal(bits(out), bits(out2))
    assert device_errors() == 0


def test_bad_block_id_and_context_len_are_flagged_not_faulted():
    case = wl.make_case("bad", 95, 3, 8, 2, 64, lens=[40, 70, 10], q_dtype=torch.float32)
    kg, vg = gpu_caches(case)
    bt = case.block_tables.clone()
    bt[1, 1] = case.num_blocks + 1000
    out = gpu_decode(case, kg, vg, block_tables=bt)
    torch.cuda.synchronize()
    assert device_errors() & 2
    cl = case.context_lens.clone()
    cl[2] = case.max_blocks_per_seq * 32 + 500
    gpu_decode(case, kg, vg, context_lens=cl)
    assert device_errors() & 4
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------ balanced path cuts
def test_balanced_one_context_cut_across_every_cta():
    """A single 98k-token context: every persistent CTA holds a piece of it,
    and the CTA whose piece arrives last combines all of them."""
    case = wl.make_case("long", 96, 1, 4, 1, 128, lens=[98_000], q_dtype=torch.float32,
                        max_blocks_per_seq=-(-98_000 // 32))
    check_case(case, splits=(True,))


def test_balanced_thousands_of_tiny_contexts_with_empty_ones():
    g = torch.Generator().manual_seed(97)
    lens = torch.randint(0, 41, (3000,), generator=g)
    lens[::7] = 0  # empty sequences interleaved
    case = wl.make_case("tiny_many", 98, 3000, 8, 2, 64, lens=lens.tolist(),
                        q_dtype=torch.bfloat16, max_blocks_per_seq=2)
    check_case(case)


@pytest.mark.parametrize("lens,Hkv", [([1, 70, 0, 129, 64], 2),  # fewer pages than CTAs
                                      ([17, 200, 33], 1), ([0, 0, 0], 4), ([300], 8)])
def test_balanced_fewer_pages_than_ctas(lens, Hkv):
    """With fewer pages than persistent CTAs a CTA holds one page or none:
    a cut context's pieces sit in every CTA its pages map to, with empty CTAs
    between them; all-empty batches write zero rows only."""
    case = wl.make_case(f"thin{Hkv}", 100 + Hkv, len(lens), 2 * Hkv, Hkv, 96, lens=lens,
                        q_dtype=torch.float16, max_blocks_per_seq=10, extra_blocks=2)
    check_case(case, splits=(True,))


def test_balanced_launch_without_clear_after_a_clean_launch():
    """A launch that raised no device error leaves the arrival counters zero,
    so pa_decode_balanced may follow it without a clear; and clear + balanced
    gives bit-for-bit what pa_decode gives."""
    case = wl.make_case("two", 99, 9, 32, 8, 128, len_range=(1, 3000), max_blocks_per_seq=94)
    kg, vg = gpu_caches(case)
    ref = gpu_decode(case, kg, vg, split=True)
    nbytes = pa.decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                      case.head_dim, case.block_size, case.max_blocks_per_seq)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    pa.decode_workspace_clear(ws)
    for _ in range(3):
        out = torch.full_like(ref, float("nan"))
        n = pa.decode_balanced(out, to_dev(case.query), kg, vg, to_dev(case.block_tables),
                               to_dev(case.context_lens), case.num_kv_heads, case.scale, ws)
        assert n > 0
        assert torch.equal(bits(out), bits(ref))
    assert torch.all(ws[:3840] == 0)
    assert device_errors() == 0
