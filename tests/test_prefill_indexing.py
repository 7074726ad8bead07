"""The paged prefill kernel's index arithmetic, restated on the CPU.

The kernel runs one CTA per (query tile, kv head, sequence), the tile 256
rows (two 128-row MMA tiles) over a 16-bit cache and 128 over an 8-bit one; its rows
are the (token, head-in-group) pairs r = i * G + j of one sequence's chunk,
token i sitting at position n - q_len + i. It streams keys of positions
[0, kv_end) in 64-token tiles, with kv_end one past the position of the
tile's last row, and masks key t for a row at position pos when t > pos.
These tests restate that arithmetic (the formulas of the kernel's row, head,
position, kv_end, page and address computations) and check, over random
batches, that every global read and write stays inside its buffer and that
the (row, key) pairs attended are exactly the causal ones.
"""
import random

import pytest

TILE = 64


def kernel_accesses(q_lens, ctx, G, Hkv, Hq, bs, MB, NB, D, tables, ROWS=256):
    """Per CTA of the grid: the query / output rows it touches, the cache
    element offsets it reads and the (token, head, key) triples it attends,
    following the kernel's formulas."""
    cu = [0]
    for q in q_lens:
        cu.append(cu[-1] + q)
    T = cu[-1]
    max_q = max(q_lens)
    tiles = (max_q * G + ROWS - 1) // ROWS
    rows_touched, reads, pairs = [], [], set()
    for s in range(len(q_lens)):
        q0, q_len, n = cu[s], cu[s + 1] - cu[s], ctx[s]
        assert 0 <= q0 <= T - q_len and q_len <= max_q
        rows_total = q_len * G
        for g in range(Hkv):
            for qt in range(tiles):
                if qt * ROWS >= rows_total:
                    continue
                assert q_len <= n <= MB * bs
                pos0 = n - q_len
                r_last = min(qt * ROWS + ROWS, rows_total) - 1
                kv_end = pos0 + r_last // G + 1
                for rr in range(ROWS):
                    r = qt * ROWS + rr
                    if r < rows_total:
                        row = (q0 + r // G) * Hq + g * G + r % G
                        rows_touched.append(row)
                        pos = pos0 + r // G
                        for t in range(kv_end):
                            if t <= pos:
                                pairs.add((q0 + r // G, g * G + r % G, t))
                for tile in range((kv_end + TILE - 1) // TILE):
                    for rr in range(TILE):
                        t = tile * TILE + rr
                        if t < kv_end:
                            assert t // bs < MB
                            b = tables[s][t // bs]
                            for c in (0, D // 8 - 1):  # first and last 16-byte chunk
                                off = ((b * Hkv + g) * bs + t % bs) * D * 2 + c * 16
                                reads.append((off, off + 16))
    return T, rows_touched, reads, pairs


@pytest.mark.parametrize("rows", [256, 128])
@pytest.mark.parametrize("seed", range(4))
def test_accesses_in_bounds_and_attention_is_causal(seed, rows):
    rng = random.Random(seed)
    for _ in range(25):
        S = rng.randint(1, 5)
        Hkv = rng.choice([1, 2, 4])
        G = rng.choice([1, 2, 3, 4, 8])
        Hq, bs, D = Hkv * G, rng.choice([16, 32, 64]), rng.choice([64, 128])
        q_lens = [rng.choice([0, 1, 2, 7, 33, 70]) for _ in range(S)]
        if max(q_lens) == 0:
            q_lens[0] = 1
        ctx = [q + rng.choice([0, 1, 40, 130]) for q in q_lens]
        MB = max((c + bs - 1) // bs for c in ctx) + rng.randint(0, 2)
        NB = S * MB + 1
        pool = list(range(NB))
        rng.shuffle(pool)
        tables = [pool[s * MB:(s + 1) * MB] for s in range(S)]
        T, touched, reads, pairs = kernel_accesses(q_lens, ctx, G, Hkv, Hq, bs, MB, NB, D,
                                                   tables, rows)
        # every output row written once, inside [T][Hq]
        assert sorted(touched) == list(range(T * Hq))
        cache_bytes = NB * Hkv * bs * D * 2
        assert all(0 <= a and b <= cache_bytes for a, b in reads)
        # exactly the causal pairs: token i of sequence s (position n - q_len + i)
        # with every key position 0 .. that position
        want = set()
        cu = 0
        for s in range(S):
            for i in range(q_lens[s]):
                p = ctx[s] - q_lens[s] + i
                for h in range(Hq):
                    for t in range(p + 1):
                        want.add((cu + i, h, t))
            cu += q_lens[s]
        assert pairs == want


def test_every_row_sees_position_zero_in_the_first_tile():
    """The online softmax needs a finite maximum after the first tile: every
    row's position is >= 0, so key 0 (in tile 0) is always attended."""
    for q_len in (1, 5, 64, 200):
        for extra in (0, 1, 100):
            n = q_len + extra
            for i in range(q_len):
                assert n - q_len + i >= 0
