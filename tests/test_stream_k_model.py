"""Invariants of the stream-K work split of the W8A8 tensor-core kernel,
checked on the CPU against a restatement of its segment arithmetic.

The kernel (``Work`` in ``csrc/w8a8_fused.cu``) gives unit u of U the
iterations [total * u // U, total * (u + 1) // U) of the tile-major order
(total = tiles * nkb), cut at tile boundaries into (tile, kb_lo, kb_hi)
segments.  A segment with kb_lo > 0 is parked for the tile's owner; the
unit holding k-block 0 of a tile whose range ends inside it (kb_hi < nkb)
owns it and adds the parts of the units u + 1, u + 2, ... whose first
iteration lies inside the tile.  These tests check, for many shapes, that
the segments cover every (tile, k-block) exactly once, that each unit parks
at most one part (its first segment, so one workspace slot per unit
suffices), that an owner's contributor list is exactly the set of units that
parked a part of its tile, and that every wait points to a later unit (no
cycle).  The planner only runs stream-K with tiles > U; the protocol holds
more generally (tiles < U, several contributors per tile), which is covered
too.
"""

from __future__ import annotations

import pytest


def segments(tiles: int, nkb: int, u: int, units: int):
    total = tiles * nkb
    cur, end = total * u // units, total * (u + 1) // units
    out = []
    while cur < end:
        t = cur // nkb
        lo = cur - t * nkb
        hi = min(nkb, end - t * nkb)
        out.append((t, lo, hi))
        cur = t * nkb + hi
    return out


def contributors(tiles: int, nkb: int, u: int, units: int, tile: int):
    total = tiles * nkb
    q, out = u + 1, []
    while q < units and total * q // units < (tile + 1) * nkb:
        out.append(q)
        q += 1
    return out


def check(tiles: int, nkb: int, units: int):
    owner_of = {}
    parked = {}
    covered = set()
    for u in range(units):
        segs = segments(tiles, nkb, u, units)
        assert segs, "every unit gets work when total >= units"
        for i, (t, lo, hi) in enumerate(segs):
            assert 0 <= lo < hi <= nkb
            for kb in range(lo, hi):
                assert (t, kb) not in covered
                covered.add((t, kb))
            if lo > 0:
                assert i == 0, "a parked part is the unit's first segment"
                assert u not in parked
                parked[u] = t
            elif hi < nkb:
                assert i == len(segs) - 1, "an owned split tile is the unit's last segment"
                owner_of[t] = u
    assert len(covered) == tiles * nkb
    for t, u in owner_of.items():
        got = contributors(tiles, nkb, u, units, t)
        assert got == sorted(q for q, tt in parked.items() if tt == t)
        assert all(q > u for q in got)
    for q, t in parked.items():
        assert t in owner_of and owner_of[t] < q


@pytest.mark.parametrize("tiles", [1, 2, 3, 5, 19, 20, 76, 77, 80, 88, 150, 160, 192, 1216])
@pytest.mark.parametrize("nkb", [1, 2, 3, 17, 40, 97, 152, 153])
def test_stream_k_segments(tiles, nkb):
    for units in (2, 3, 7, 74, 76):
        if units <= tiles * nkb:
            check(tiles, nkb, units)


def test_planner_regime_has_one_contributor_per_tile():
    """With more tiles than units (the only regime the planner uses) every
    unit's range spans at least one whole tile's k-blocks, so a split tile has
    exactly one parked part."""
    for tiles in (77, 80, 88, 160, 200):
        for nkb in (17, 40, 152):
            units = 76
            for u in range(units):
                for t, lo, hi in segments(tiles, nkb, u, units):
                    if lo == 0 and hi < nkb:
                        assert len(contributors(tiles, nkb, u, units, t)) == 1
