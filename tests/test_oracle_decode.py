"""Pins of the oracle's paged write, gather, attention and split reduction.

Each test holds the oracle against something other than itself: PyTorch
float64 softmax attention over the raw rows (a library routine), special cases
with closed forms, invariances the method must have, and the worked examples
the pages print (tests/golden).

Pages: "PagedAttention in mistral.rs" (blocked pool, block size, FP8 cache),
"Optimization plans" (reshape_and_cache), "Rolling buffer cache" (slot i mod W).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from _helpers import attended_rows, dense_reference, oracle_caches, oracle_decode
from paged_kv_cache_context_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def all_rows_close(case, out, tol=1e-12):
    for s in range(case.num_seqs):
        for h in range(case.num_heads):
            ref = dense_reference(case, s, h)
            np.testing.assert_allclose(out[s, h], ref, rtol=0, atol=tol * max(1.0, np.abs(ref).max()),
                                       err_msg=f"s={s} h={h}")


# ------------------------------------------------------------ c1 / c5: attention
def test_tiny_workload_matches_dense_attention():
    """The tiny workload (2 seqs, lengths 17 and 45, shuffled pool of 8 blocks,
    new token written by reshape_and_cache) equals dense softmax attention."""
    case = wl.config("tiny")
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    all_rows_close(case, out)


@pytest.mark.parametrize("bs", [16, 32])
def test_paged_equals_dense_for_every_length_residue(bs):
    """Random tables and every n mod bs residue (n = 1 .. 3*bs+1)."""
    lens = list(range(1, 3 * bs + 2))
    case = wl.make_case("res", 11 + bs, len(lens), 2, 1, 64, bs, lens=lens,
                        q_dtype=torch.float32, extra_blocks=7)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    all_rows_close(case, out)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_half_precision_inputs_widen_exactly(dtype):
    case = wl.make_case("half", 5, 3, 8, 2, 128, lens=[1, 33, 70], q_dtype=dtype)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    all_rows_close(case, out)


# ------------------------------------------------------------ c2: single token
def test_single_token_returns_its_value_row_exactly():
    case = wl.make_case("one", 3, 4, 4, 2, 64, lens=[1, 1, 1, 1], q_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    for s in range(4):
        for h in range(4):
            v = case.new_value[s, h // 2].double().numpy()
            assert np.array_equal(out[s, h], v)


# ------------------------------------------------------------ c3: uniform keys
def test_equal_keys_or_zero_scale_give_mean_of_values():
    case = wl.make_case("uni", 4, 2, 4, 4, 64, lens=[29, 77], q_dtype=torch.float32)
    # all keys of each (sequence, head) the same row
    case.pre_key[:] = case.new_key[0]
    case.new_key[:] = case.new_key[0]
    kc, vc = oracle_caches(case)
    for c in (case, None):
        if c is None:  # scale 0 with arbitrary keys
            c = wl.make_case("uni0", 4, 2, 4, 4, 64, lens=[29, 77], q_dtype=torch.float32,
                             scale=0.0)
            kc, vc = oracle_caches(c)
        out = oracle_decode(c, kc, vc)
        for s in range(2):
            _, val = attended_rows(c, s)
            for h in range(4):
                mean = val[:, h].double().mean(0).numpy()
                np.testing.assert_allclose(out[s, h], mean, rtol=0, atol=1e-13)


def test_empty_context_gives_zero():
    case = wl.make_case("empty", 6, 3, 4, 4, 64, lens=[0, 5, 0], q_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    all_rows_close(case, out)


# ------------------------------------------------------------ c4: relabelling
def test_block_relabelling_is_bit_invariant():
    case = wl.make_case("perm", 7, 5, 8, 2, 64, len_range=(1, 200), q_dtype=torch.float32,
                        extra_blocks=9)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    g = torch.Generator().manual_seed(70)
    perm = torch.randperm(case.num_blocks, generator=g)  # old id -> new id
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt = case.block_tables.clone()
    owned = bt >= 0
    bt[owned] = perm[bt[owned].long()].to(torch.int32)
    out2 = oracle.decode(case.query, kc2, vc2, bt, case.context_lens, case.num_kv_heads,
                         case.block_size, case.scale)
    assert np.array_equal(out, out2)


# ------------------------------------------------------------ c6: rolling buffer
def test_ring_with_overwrites_equals_dense_over_last_window():
    """Every position is written at slot p mod W (later rounds overwrite);
    decode attends exactly the last W positions."""
    W = 64
    case = wl.make_case("ring", 8, 4, 4, 2, 64, lens=[10, 64, 65, 300], window=W,
                        q_dtype=torch.float32, ring_overwrite=True)
    assert len(case.pre_chunks) > 1  # overwrites really happen
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    all_rows_close(case, out)


def test_attention_is_invariant_under_key_permutation():
    """Attention is a set operation: permuting the (key, value) rows of the
    context (what a ring's physical visit order does) leaves it unchanged."""
    case = wl.make_case("kperm", 9, 2, 4, 4, 64, lens=[70, 41], q_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    g = torch.Generator().manual_seed(90)
    for s in range(2):
        n = int(case.context_lens[s])
        p = torch.randperm(n, generator=g)
        key, val = attended_rows(case, s)
        # a fresh contiguous single-sequence cache holding the permuted rows
        c1 = wl.make_case("kperm1", 1, 1, 4, 4, 64, lens=[n], q_dtype=torch.float32)
        c1.query = case.query[s:s + 1].clone()
        sm = torch.cat([c1.pre_pos, c1.new_pos])
        k1, v1 = wl.empty_caches(c1)
        slots, _ = oracle.slot_mapping(c1.block_tables, torch.zeros(n, dtype=torch.int32), sm,
                                       c1.block_size)
        oracle.reshape_and_cache(key[p], val[p], k1, v1, slots, c1.block_size)
        o1 = oracle.decode(c1.query, k1, v1, c1.block_tables, c1.context_lens, 4, 32, case.scale)
        np.testing.assert_allclose(o1[0], out[s], rtol=0, atol=1e-13)


def test_ring_slot_mapping_golden_w3():
    """The rolling buffer's worked example (W = 3): slot = position mod 3."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "ring_w3.txt")) if l[0] != "#" and l.strip()]
    W, bs = map(int, rows[0])
    pos = torch.tensor([int(r[0]) for r in rows[1:]], dtype=torch.int32)
    want = [int(r[1]) for r in rows[1:]]
    # block size 1 and an identity table: the slot is the ring position itself
    tables = torch.arange(W, dtype=torch.int32)[None, :]
    slots, bad = oracle.slot_mapping(tables, torch.zeros_like(pos), pos, bs, W)
    assert bad == 0 and slots.tolist() == want


def test_ring_slots_form_a_bijection_per_window():
    """Any W consecutive positions occupy all W ring slots once; positions W
    apart share a slot; padding positions map to -1."""
    W, bs = 128, 32
    case = wl.make_case("rb", 12, 3, 4, 4, 64, lens=[W, W, W], window=W, q_dtype=torch.float32)
    for start in (0, 5, 1000):
        pos = torch.arange(start, start + W, dtype=torch.int32)
        seq = torch.full_like(pos, 1)
        slots, bad = oracle.slot_mapping(case.block_tables, seq, pos, bs, W)
        owned = set()
        for b in case.block_tables[1].tolist():
            owned.update(range(b * bs, b * bs + bs))
        assert bad == 0 and sorted(slots.tolist()) == sorted(owned)
        s2, _ = oracle.slot_mapping(case.block_tables, seq, pos + W, bs, W)
        assert torch.equal(slots, s2)
    s3, bad = oracle.slot_mapping(case.block_tables, None, torch.tensor([-1, 0, -5], dtype=torch.int32), bs, W)
    assert bad == 0 and s3.tolist()[0] == -1 and s3.tolist()[2] == -1


def test_ring_memory_is_one_eighth_at_32k():
    """Rolling buffer cache: at 32k tokens with W = 4096 the cache is 8x smaller."""
    gold = {l.split()[0]: float(l.split()[1])
            for l in open(os.path.join(GOLDEN, "capacity.txt")) if l.strip() and l[0] != "#"}
    n, W = int(gold["ring_tokens"]), int(gold["ring_window"])
    # 1 head, D 64, no values needed beyond the layout
    full = wl.make_case("full", 1, 1, 1, 1, 64, lens=[n], q_dtype=torch.bfloat16)
    ring = wl.make_case("ring", 1, 1, 1, 1, 64, lens=[n], window=W, q_dtype=torch.bfloat16)
    assert full.num_blocks / ring.num_blocks == gold["ring_memory_reduction"]
    assert int(gold["default_block_size"]) == full.block_size == ring.block_size


# ------------------------------------------------------------ c7: GQA
def test_grouped_heads_equal_repeated_kv_heads():
    case = wl.make_case("gqa", 13, 3, 8, 2, 64, lens=[5, 40, 97], q_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    G = 4
    kr = kc.repeat_interleave(G, dim=1).contiguous()
    vr = vc.repeat_interleave(G, dim=1).contiguous()
    out_mha = oracle.decode(case.query, kr, vr, case.block_tables, case.context_lens, 8,
                            case.block_size, case.scale)
    assert np.array_equal(out, out_mha)


# ------------------------------------------------------------ c8: split + reduce
def test_split_partials_reduce_to_unsplit_result():
    case = wl.make_case("split", 14, 2, 4, 2, 64, lens=[150, 33], q_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    full = oracle_decode(case, kc, vc)
    g = torch.Generator().manual_seed(140)
    for s in range(2):
        n = int(case.context_lens[s])
        for h in range(4):
            cuts = sorted(set(torch.randint(0, n + 1, (4,), generator=g).tolist()) | {0, n})
            segs = list(zip(cuts[:-1], cuts[1:])) + [(n, n + 40)]  # last one empty
            parts = [oracle.decode_partial(case.query, kc, vc, case.block_tables,
                                           case.context_lens, s, h, 2, 32, case.scale, a, b)
                     for a, b in segs]
            o = np.stack([p[0] for p in parts])
            m = np.array([p[1] for p in parts])
            l = np.array([p[2] for p in parts])
            assert l[-1] == 0 and m[-1] == -np.inf
            red = oracle.reduce(o[None], m[None], l[None])[0]
            np.testing.assert_allclose(red, full[s, h], rtol=0, atol=1e-13)
            # one split is the identity; an empty split changes nothing
            one = oracle.decode_partial(case.query, kc, vc, case.block_tables, case.context_lens,
                                        s, h, 2, 32, case.scale, 0, n)
            r1 = oracle.reduce(one[0][None, None], [[one[1]]], [[one[2]]])[0]
            np.testing.assert_allclose(r1, full[s, h], rtol=0, atol=1e-15)
            r2 = oracle.reduce(np.stack([one[0], np.full_like(one[0], np.nan)])[None],
                               [[one[1], -np.inf]], [[one[2], 0.0]])[0]
            assert np.array_equal(r1, r2)


def test_reduce_all_empty_is_zero():
    o = np.full((1, 3, 8), np.nan)
    assert np.all(oracle.reduce(o, [[-np.inf] * 3], [[0.0] * 3]) == 0)


# ------------------------------------------------------------ FP8 pipeline
def test_fp8_decode_equals_dense_over_library_dequantised_rows():
    case = wl.make_case("f8", 15, 3, 4, 4, 96, lens=[1, 31, 100], q_dtype=torch.bfloat16,
                        kv_dtype="fp8_e4m3", kv_src_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    out = oracle_decode(case, kc, vc)
    all_rows_close(case, out)


# ------------------------------------------------------------ c11 / write
def test_auto_write_copies_bits_and_leaves_other_rows():
    case = wl.make_case("w", 16, 3, 4, 2, 64, lens=[3, 40, 70], q_dtype=torch.bfloat16,
                        extra_blocks=3)
    kc, vc = wl.empty_caches(case)
    sm, _ = oracle.slot_mapping(case.block_tables, None, case.new_pos, 32)
    sm[1] = -1  # padding token: skipped
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, sm, 32)
    written = torch.zeros(case.num_blocks, 32, dtype=torch.bool)
    for t in (0, 2):
        b, r = divmod(int(sm[t]), 32)
        assert torch.equal(kc[b, :, r].view(torch.int16), case.new_key[t].view(torch.int16))
        assert torch.equal(vc[b, :, r].view(torch.int16), case.new_value[t].view(torch.int16))
        written[b, r] = True
    poison = wl.cache_poison(case)
    rest = kc.view(torch.int16).permute(0, 2, 1, 3)[~written]
    assert torch.all(rest == poison)
    assert oracle.reshape_and_cache(case.new_key[:1], case.new_value[:1], kc, vc,
                                    torch.tensor([case.num_blocks * 32]), 32) == 1


def test_fp8_write_matches_library_cast():
    case = wl.make_case("w8", 17, 4, 4, 4, 96, lens=[1, 30, 64, 90], q_dtype=torch.bfloat16,
                        kv_dtype="fp8_e4m3", kv_src_dtype=torch.float32)
    kc, vc = oracle_caches(case)
    for s in range(4):
        pos, key, val = case.tokens_of(s)
        sm, _ = oracle.slot_mapping(case.block_tables, torch.full_like(pos, s), pos, 32)
        for i, slot in enumerate(sm.tolist()):
            b, r = divmod(slot, 32)
            for cache, x, sc in ((kc, key[i], case.k_scale), (vc, val[i], case.v_scale)):
                y = x.float() / torch.tensor(sc, dtype=torch.float32)
                want = torch.clamp(y, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
                assert torch.equal(cache[b, :, r], want)


def test_fp8_write_nan_keeps_the_input_sign():
    """A NaN input is stored as the NaN code with the input's own sign (the
    sign of a NaN quotient x / scale is not fixed by IEEE 754)."""
    x = torch.tensor([float("nan"), -float("nan"), 1.0, -0.0]).view(1, 1, 4).repeat(1, 1, 2)
    x = x.reshape(1, 1, 8).float()
    kc = torch.zeros(1, 1, 32, 8, dtype=torch.uint8)
    vc = torch.zeros_like(kc)
    for scale in (1.0, 0.37, 3.0e5):
        oracle.reshape_and_cache(x, x, kc, vc, torch.tensor([0]), 32, "fp8_e4m3", scale, scale)
        assert kc[0, 0, 0, 0] == 0x7F and kc[0, 0, 0, 1] == 0xFF
        assert kc[0, 0, 0, 3] == 0x80
