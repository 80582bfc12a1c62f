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
