"""The balanced decode path's partition arithmetic, restated on the CPU.

The persistent decode kernel cuts the pages of all (sequence, kv head)
segments, taken in (sequence, kv head, page) order, P pages in total, into C
equal ranges [c*P/C, (c+1)*P/C). A segment cut by range boundaries leaves one
partial per CTA it touches: in slot 1 if the piece does not start the CTA's
range, else slot 0. Each cut piece adds its page count to the counter of the
CTA that holds the segment's last page, and the piece that completes the count
enumerates the segment's pieces by arithmetic alone. These tests restate that
integer arithmetic (the formulas of the kernel's range_lo, cta_of and
piece_index, and the producer's piece bookkeeping) and check, over random
batches, that the enumeration finds exactly the pieces the producers write and
that the counts add up to the segment's pages.
"""
import random

import pytest


def range_lo(c, P, C):
    return c * P // C


def cta_of(x, P, C):
    return ((x + 1) * C - 1) // P


def piece_index(j, seg0, P, C, c_first, first_in_slot1):
    cc = c_first + j if P >= C else cta_of(seg0 + j, P, C)
    return cc, (1 if (j == 0 and first_in_slot1) else 0)


def segments(pages_per_seq, Hkv):
    out, x = [], 0
    for pg in pages_per_seq:
        for _ in range(Hkv):
            if pg > 0:
                out.append((x, pg))
                x += pg
    return out, x


def walk(pages_per_seq, Hkv, C):
    """What the CTAs' producers do: per CTA the pieces of its range, with the
    slot, the head/tail role and the counter each cut piece adds to."""
    segs, P = segments(pages_per_seq, Hkv)
    cut_pieces = {}   # (cta, slot) -> segment index
    counts = {}       # (segment, counter index) -> pages added
    for c in range(C):
        a, b = range_lo(c, P, C), range_lo(c + 1, P, C)
        k = 0
        for si, (s0, n) in enumerate(segs):
            ps, pe = max(a, s0), min(b, s0 + n)
            if ps >= pe:
                continue
            length, pg = pe - ps, ps - s0
            whole = pg == 0 and pg + length == n
            if not whole:
                tail = k + length == b - a
                assert tail or k == 0, "a cut piece starts or ends the CTA's range"
                slot = 1 if k > 0 else 0
                assert (c, slot) not in cut_pieces
                cut_pieces[(c, slot)] = si
                seg0 = a + k - pg
                assert seg0 == s0
                key = (si, cta_of(seg0 + n - 1, P, C))
                counts[key] = counts.get(key, 0) + length
            k += length
        assert k == b - a
    return segs, P, cut_pieces, counts


@pytest.mark.parametrize("seed", range(6))
def test_enumeration_finds_exactly_the_written_pieces(seed):
    rng = random.Random(seed)
    for _ in range(200):
        S = rng.randint(1, 40)
        Hkv = rng.choice([1, 2, 4, 8, 32])
        C = rng.choice([1, 2, 3, 7, 152, 456, 608, 760, 912])
        mx = rng.choice([1, 2, 5, 40, 300])
        pages = [rng.randint(0, mx) for _ in range(S)]
        segs, P, cut_pieces, counts = walk(pages, Hkv, C)
        for si, (s0, n) in enumerate(segs):
            mine = sorted(k for k, v in cut_pieces.items() if v == si)
            if not mine:
                continue
            c_first = cta_of(s0, P, C)
            first_in_slot1 = s0 != range_lo(c_first, P, C)
            m = cta_of(s0 + n - 1, P, C) - c_first + 1 if P >= C else n
            found = sorted(piece_index(j, s0, P, C, c_first, first_in_slot1) for j in range(m))
            assert found == mine
            # every piece counts into one counter, and the counts complete it
            assert counts[(si, cta_of(s0 + n - 1, P, C))] == n


def test_counter_index_is_unique_per_cut_segment():
    """Two cut segments never share a counter: a counter is indexed by the CTA
    holding the segment's last page, and that page is the first page of the
    CTA's range whenever the segment started in an earlier CTA."""
    rng = random.Random(7)
    for _ in range(2000):
        pages = [rng.randint(0, 90) for _ in range(rng.randint(1, 30))]
        Hkv, C = rng.choice([1, 4, 8]), rng.choice([5, 152, 456, 608, 760, 912])
        _, _, _, counts = walk(pages, Hkv, C)
        idx = [c for (_, c) in counts]
        assert len(idx) == len(set(idx))


def test_equal_shares():
    for P in (1, 7, 455, 456, 18_432, 147_456):
        for C in (456, 608, 760, 912):
            sizes = [range_lo(c + 1, P, C) - range_lo(c, P, C) for c in range(C)]
            assert sum(sizes) == P and max(sizes) - min(sizes) <= 1
