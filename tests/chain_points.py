"""A point set whose first Boruvka round hooks every point into one chain.

The merge of page "HDBSCAN" ("The algorithm on the device": find each
component's cheapest edge, "then merge") must stay fast when the hooks form
long chains.  This builds the worst case for a root walk: n points on a folded
path in 6 dimensions with integer coordinates, where step i (from point i - 1
to point i) has squared length exactly G0 + i.  So the steps grow strictly
along the path, every point's nearest other point is its predecessor, and in
the first round point i hooks onto point i - 1: one chain of depth n - 1.

Construction:

* step i's squared length G0 + i is split as a^2 + (b^2 + c^2 + e^2 + g^2)
  with a = floor(sqrt(G0 + i)) and the rest, at most 2a, a sum of four
  squares (every non-negative integer is one, by Lagrange's theorem);
* the path runs along x in rows of ``row`` steps of length about a, turns
  upward for ``turn`` steps (rows lie ``turn`` steps apart, farther than any
  step), then runs back; the small parts (b, c, e, g) go to four more
  dimensions with signs alternating step by step, so they do not drift;
* all coordinates are integers below 2^24 and every squared step length is
  below 2^24, so float32 holds them and a step's distance exactly.

With G0 = 10^6 the steps are 1000 to about 1060 long while any two points two
or more steps apart are at least about 1400 apart; the minimum spanning tree
of the mutual-reachability distance (min_samples 2) is therefore the path,
edge (i - 1, i) of weight sqrt(G0 + i) (the cycle property: every other pair
is longer than every step between them).  A test pins this against the
oracle on a prefix of the path.
"""

from __future__ import annotations

from math import isqrt

import numpy as np

G0 = 1_000_000


def _four_squares(r: int) -> tuple[int, int, int, int]:
    """Some (b, c, e, g) with b^2 + c^2 + e^2 + g^2 = r (always exists)."""
    for b in range(isqrt(r), -1, -1):
        for c in range(isqrt(r - b * b), -1, -1):
            rc = r - b * b - c * c
            for e in range(isqrt(rc), -1, -1):
                g2 = rc - e * e
                g = isqrt(g2)
                if g * g == g2:
                    return b, c, e, g
    raise AssertionError(r)


def chain(n: int, row: int = 14_000, turn: int = 4) -> np.ndarray:
    """float32 ``[6, n]`` points of the folded path (see the module text)."""
    P = np.zeros((n, 6), dtype=np.int64)
    x = y = 0
    extra = np.zeros(4, dtype=np.int64)
    direction = 1
    pos = 0  # steps taken in the current row, then in the current turn
    turning = False
    for i in range(1, n):
        T = G0 + i
        a = isqrt(T)
        sign = 1 if i % 2 else -1
        extra += sign * np.array(_four_squares(T - a * a), dtype=np.int64)
        if turning:
            y += a
            pos += 1
            if pos == turn:
                turning, pos, direction = False, 0, -direction
        else:
            x += direction * a
            pos += 1
            if pos == row:
                turning, pos = True, 0
        P[i] = (x, y, *extra)
    assert np.abs(P).max() < (1 << 24)
    return np.ascontiguousarray(P.astype(np.float32).T)


def tree(n: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The path as the library writes a tree: ``(lo, hi, w float32)`` in (w, lo, hi) order."""
    i = np.arange(1, n, dtype=np.int64)
    w = np.sqrt((G0 + i).astype(np.float32))
    return i - 1, i, w
