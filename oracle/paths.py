"""Irreps strings, path enumeration and tensor layouts for the oracle (test infrastructure only).

Irreps grammar: terms ``MULxLP`` joined by ``+``, P in {e, o}; e.g. ``"128x0e+128x1o"``.

Path enumeration (the plainest reading of "all parity-allowed UVU paths with l3 <= lmax_out"):
for each x irrep i1 in string order, each SH irrep i2 in string order, and each l3 ascending over
|l1-l2| .. min(l1+l2, lmax_out), one path p = (i1, i2, l3) whose output parity is p1 * p2.
Every triangle-allowed l3 is kept, including outputs whose parity is not (-1)^l3.

Layouts (row-major):
    x   [N][U][D_x]     D_x  = sum_{i1} (2 l1 + 1), l1 blocks in string order
    Y   [E][D_Y]        D_Y  = sum_{i2} (2 l2 + 1), l2 blocks in string order
    w   [E][P][U]
    out [N][U][D_out]   D_out = sum_p (2 l3_p + 1), path blocks in path order
The channel-wise (UVU) structure needs every x irrep to share one multiplicity U and every SH
irrep to have multiplicity 1 ("Receiver-streaming convolutions for channel-wise UVU tensor
products", opening post: one (receiver, channel) pair per owner).
"""

from __future__ import annotations

import re
from dataclasses import dataclass

_TERM = re.compile(r"^\s*(\d+)x(\d+)([eo])\s*$")


def parse_irreps(s: str) -> list[tuple[int, int, int]]:
    """Return [(mul, l, parity)] with parity +1 for 'e' and -1 for 'o'."""
    out = []
    for term in s.split("+"):
        m = _TERM.match(term)
        if not m:
            raise ValueError(f"bad irreps term {term!r} in {s!r}")
        out.append((int(m.group(1)), int(m.group(2)), 1 if m.group(3) == "e" else -1))
    return out


@dataclass(frozen=True)
class Path:
    l1: int
    l2: int
    l3: int
    parity: int
    xoff: int  # offset of the l1 block inside a channel's x row
    yoff: int  # offset of the l2 block inside an edge's Y row
    ooff: int  # offset of the l3 block inside a channel's out row


@dataclass(frozen=True)
class Layout:
    mul: int
    dim_x: int
    dim_y: int
    dim_out: int
    paths: tuple[Path, ...]


def layout(irreps_x: str, irreps_sh: str, lmax_out: int) -> Layout:
    xs = parse_irreps(irreps_x)
    ys = parse_irreps(irreps_sh)
    muls = {m for m, _, _ in xs}
    if len(muls) != 1:
        raise ValueError("UVU needs one multiplicity for every x irrep")
    if any(m != 1 for m, _, _ in ys):
        raise ValueError("SH irreps must have multiplicity 1")
    mul = muls.pop()
    paths = []
    xoff = 0
    ooff = 0
    for _, l1, p1 in xs:
        yoff = 0
        for _, l2, p2 in ys:
            for l3 in range(abs(l1 - l2), min(l1 + l2, lmax_out) + 1):
                paths.append(Path(l1, l2, l3, p1 * p2, xoff, yoff, ooff))
                ooff += 2 * l3 + 1
            yoff += 2 * l2 + 1
        xoff += 2 * l1 + 1
    dim_y = sum(2 * l + 1 for _, l, _ in ys)
    return Layout(mul, xoff, dim_y, ooff, tuple(paths))
