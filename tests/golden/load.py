"""Reader for the hand-derived fixtures in this folder."""

from __future__ import annotations

import os

HERE = os.path.dirname(os.path.abspath(__file__))


def _num(tok: str) -> float:
    t = tok.strip()
    if "0x" in t.lower():
        return float.fromhex(t)
    return float(t)


def quant_rows():
    """(name, row floats, scale float, codes ints) per case."""
    cases = []
    cur = None
    with open(os.path.join(HERE, "quant_rows.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest.strip()}
                cases.append(cur)
            elif key == "row":
                cur["row"] = [_num(t) for t in rest.split()]
            elif key == "scale":
                cur["scale"] = _num(rest)
            elif key == "codes":
                cur["codes"] = [int(t) for t in rest.split()]
    return [(c["name"], c["row"], c["scale"], c["codes"]) for c in cases]


def _cases(fname):
    cases, cur = [], None
    with open(os.path.join(HERE, fname)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest.strip()}
                cases.append(cur)
            else:
                cur[key] = rest.strip()
    return cases


def fp8_rows():
    """(name, row floats, scale float, codes ints) per FP8 case."""
    return [(c["name"], [_num(t) for t in c["row"].split()], _num(c["scale"]),
             [int(t, 16) for t in c["codes"].split()]) for c in _cases("fp8_rows.txt")]


def w4_groups():
    """(name, row floats zero-padded to whole groups, scales, codes per
    group, leading packed bytes) per group-128 int4 case.  "@k" in a row
    moves to position k."""
    out = []
    for c in _cases("w4_groups.txt"):
        row = []
        for t in c["row"].split():
            if t.startswith("@"):
                row.extend([0.0] * (int(t[1:]) - len(row)))
            else:
                row.append(_num(t))
        row.extend([0.0] * (-len(row) % 128))
        groups = [[int(v) for v in g.split()] for g in c["codes"].split("|")]
        out.append((c["name"], row, [_num(t) for t in c["scales"].split()], groups,
                    [int(t, 16) for t in c["bytes"].split()]))
    return out
