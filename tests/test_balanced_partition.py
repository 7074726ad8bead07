"""The balanced decode path's partition arithmetic, restated on the CPU.

The persistent decode kernel cuts the pages of all (sequence, kv head)
segments, taken in (sequence, kv head, page) order, P pages in total, into C
contiguous ranges, CTA c's share proportional to w(c) = 1000 - step * (c // rs)
(rs CTAs per launch rank; step 0, equal shares, when P < 2C), so that
lo(c) = P * cum(c) // T with cum(c) the weights of CTAs below c and T = cum(C).
A segment cut by range boundaries leaves one
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


class Ranges:
    def __init__(self, P, C, rs=152, step=0):
        self.P, self.C, self.rs = P, C, rs
        self.step = step if P >= 2 * C else 0
        self.T = self.cum(C)

    def w(self, r):
        return 1000 - self.step * r

    def cum(self, c):
        R = c // self.rs
        return self.rs * (R * 1000 - self.step * (R * (R - 1) // 2)) + (c - R * self.rs) * self.w(R)

    def lo(self, c):
        return self.P * self.cum(c) // self.T

    def of(self, x):
        y = ((x + 1) * self.T - 1) // self.P
        b0 = 0
        while True:
            b1 = min(b0 + self.rs, self.C)
            if b1 == self.C or self.cum(b1) > y:
                return b0 + (y - self.cum(b0)) // self.w(b0 // self.rs)
            b0 += self.rs


def piece_index(j, seg0, rg, c_first, first_in_slot1):
    cc = c_first + j if rg.P >= rg.C else rg.of(seg0 + j)
    return cc, (1 if (j == 0 and first_in_slot1) else 0)


def segments(pages_per_seq, Hkv):
    out, x = [], 0
    for pg in pages_per_seq:
        for _ in range(Hkv):
            if pg > 0:
                out.append((x, pg))
                x += pg
    return out, x


def walk(pages_per_seq, Hkv, C, rs, step):
    """What the CTAs' producers do: per CTA the pieces of its range, with the
    slot, the head/tail role and the counter each cut piece adds to."""
    segs, P = segments(pages_per_seq, Hkv)
    rg = Ranges(P, C, rs, step)
    cut_pieces = {}   # (cta, slot) -> segment index
    counts = {}       # (segment, counter index) -> pages added
    for c in range(C):
        a, b = rg.lo(c), rg.lo(c + 1)
        if rg.P >= 2 * rg.C:
            assert b > a, "with P >= 2C every CTA gets a page"
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
                key = (si, rg.of(seg0 + n - 1))
                counts[key] = counts.get(key, 0) + length
            k += length
        assert k == b - a
    return segs, rg, cut_pieces, counts


def random_batch(rng):
    S = rng.randint(1, 40)
    Hkv = rng.choice([1, 2, 4, 8, 32])
    C = rng.choice([1, 2, 3, 7, 152, 456, 608])
    rs = rng.choice([C, 152, max(1, C // 3), 5])
    ranks = -(-C // rs)
    step = rng.choice([0, 130, 500]) // max(1, ranks - 1)
    mx = rng.choice([1, 2, 5, 40, 300])
    return [rng.randint(0, mx) for _ in range(S)], Hkv, C, rs, step


@pytest.mark.parametrize("seed", range(6))
def test_enumeration_finds_exactly_the_written_pieces(seed):
    rng = random.Random(seed)
    for _ in range(200):
        pages, Hkv, C, rs, step = random_batch(rng)
        segs, rg, cut_pieces, counts = walk(pages, Hkv, C, rs, step)
        for si, (s0, n) in enumerate(segs):
            mine = sorted(k for k, v in cut_pieces.items() if v == si)
            if not mine:
                continue
            c_first = rg.of(s0)
            first_in_slot1 = s0 != rg.lo(c_first)
            m = rg.of(s0 + n - 1) - c_first + 1 if rg.P >= rg.C else n
            found = sorted(piece_index(j, s0, rg, c_first, first_in_slot1) for j in range(m))
            assert found == mine
            # every piece counts into one counter, and the counts complete it
            assert counts[(si, rg.of(s0 + n - 1))] == n


def test_counter_index_is_unique_per_cut_segment():
    """Two cut segments never share a counter: a counter is indexed by the CTA
    holding the segment's last page, and that page is the first page of the
    CTA's range whenever the segment started in an earlier CTA."""
    rng = random.Random(7)
    for _ in range(1000):
        pages, Hkv, C, rs, step = random_batch(rng)
        _, _, _, counts = walk(pages, Hkv, C, rs, step)
        idx = [c for (_, c) in counts]
        assert len(idx) == len(set(idx))


def test_shares():
    """Equal shares (to one page) without a step; with one, shares that fall
    rank by rank in the ratio of the weights, and of() inverts lo()."""
    for P in (1, 7, 455, 456, 912, 18_432, 147_456):
        for C, rs, step in ((456, 152, 0), (608, 152, 0), (456, 152, 65), (608, 152, 43)):
            rg = Ranges(P, C, rs, step)
            sizes = [rg.lo(c + 1) - rg.lo(c) for c in range(C)]
            assert sum(sizes) == P and min(sizes) >= 0
            if rg.step == 0:
                assert max(sizes) - min(sizes) <= 1
            else:
                for r in range(C // rs):
                    share = sum(sizes[r * rs:(r + 1) * rs])
                    assert abs(share - P * rs * rg.w(r) / rg.T) <= 1
            for x in range(0, P, max(1, P // 997)):
                c = rg.of(x)
                assert rg.lo(c) <= x < rg.lo(c + 1)
