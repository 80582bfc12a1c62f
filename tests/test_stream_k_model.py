"""Invariants of the stream-K work split of the W8A8 tensor-core kernel,
checked on the CPU against a restatement of its segment arithmetic.

The kernel (``Work`` in ``csrc/w8a8_fused.cu``) gives unit u of U the
iterations [total * u // U, total * (u + 1) // U) of the tile-major order
(total = tiles * nkb), cut at tile boundaries into (tile, kb_lo, kb_hi)
segments that the unit processes from the END of its range backwards.  A
segment with kb_hi < nkb (the unit does not hold the tile's last k-block) is
parked for the tile's finisher; the unit holding the last k-block of a tile
whose first k-blocks belong to others (kb_lo > 0) finishes it, adding the
parts of the units u - 1, u - 2, ... whose ranges reach into the tile.

These tests check, for many shapes, that the segments cover every (tile,
k-block) exactly once; that each unit parks at most one part, as the FIRST
segment it processes (so one workspace slot per unit suffices, and the part
is parked before the unit waits for anything); that a finished split tile is
the LAST segment its finisher processes; that a finisher's contributor list
is exactly the set of units that parked a part of its tile; and that every
wait points to an earlier unit.  Earlier units are dispatched no later than
the waiting one and park before they wait themselves, so no wait depends on
a unit that might not be resident yet.  The planner only runs stream-K with
tiles > U; the protocol holds more generally (tiles < U, several
contributors per tile), which is covered too.
"""

from __future__ import annotations

import pytest


def unit_range(tiles: int, nkb: int, u: int, units: int):
    total = tiles * nkb
    return total * u // units, total * (u + 1) // units


def segments(tiles: int, nkb: int, u: int, units: int):
    """The unit's segments in the order it processes them (range end first)."""
    lo_bound, end = unit_range(tiles, nkb, u, units)
    out = []
    while end > lo_bound:
        t = (end - 1) // nkb
        lo = max(lo_bound, t * nkb) - t * nkb
        hi = end - t * nkb
        out.append((t, lo, hi))
        end = t * nkb + lo
    return out


def contributors(tiles: int, nkb: int, u: int, units: int, tile: int):
    """Units whose parked parts the finisher u of `tile` adds, in its order."""
    q, out = u - 1, []
    while q >= 0 and unit_range(tiles, nkb, q, units)[1] > tile * nkb:
        a, b = unit_range(tiles, nkb, q, units)
        if b > a:
            out.append(q)
        q -= 1
    return out


def check(tiles: int, nkb: int, units: int):
    finisher_of = {}
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
            if hi < nkb:
                assert i == 0, "a parked part is the first segment the unit processes"
                assert u not in parked
                parked[u] = t
            elif lo > 0:
                assert i == len(segs) - 1, "a finished split tile is the unit's last segment"
                finisher_of[t] = u
    assert len(covered) == tiles * nkb
    for t, u in finisher_of.items():
        got = contributors(tiles, nkb, u, units, t)
        assert sorted(got) == sorted(q for q, tt in parked.items() if tt == t)
        assert all(q < u for q in got), "every wait points to an earlier unit"
    for q, t in parked.items():
        assert t in finisher_of and finisher_of[t] > q


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
                    if lo > 0 and hi == nkb:
                        assert len(contributors(tiles, nkb, u, units, t)) == 1


def test_no_wait_before_own_park():
    """A unit that parks does so before any wait of its own: its parked part
    is processed first and a finisher segment last, and one unit cannot be
    both the parker and the finisher of a single segment."""
    for tiles, nkb, units in ((77, 40, 76), (3, 17, 7), (80, 152, 76), (1, 153, 74)):
        for u in range(units):
            segs = segments(tiles, nkb, u, units)
            kinds = ["park" if hi < nkb else ("finish" if lo > 0 else "whole") for _, lo, hi in segs]
            if "park" in kinds:
                assert kinds.index("park") == 0
            if "finish" in kinds:
                assert kinds.index("finish") == len(kinds) - 1
                assert len(kinds) > 1 or kinds[0] == "finish"
