"""Closed forms of ChunkAttention, Knowl 4 (capacity gain and fragmentation).

sharing ratio       r = n_s / (n_p + n_c)
capacity multiplier ~ 1 / (1 - r)       (memory-bound batch capacity gain)
memory loss         <= (c - 1) / n       (leaf-chunk internal fragmentation)

The exact counterparts used by the tests:

* chunks a batch of b sequences of n tokens sharing n_s leading tokens needs,
  with chunk-aligned n_s: n_s / c + b * ceil((n - n_s) / c); without sharing:
  b * ceil(n / c).  Their ratio tends to 1 / (1 - r) as b grows.
* slots wasted by a sequence of n tokens: c * ceil(n / c) - n, at most c - 1.
"""
from __future__ import annotations

import math


def sharing_ratio(n_s: int, n_p: int, n_c: int = 0) -> float:
    return n_s / (n_p + n_c)


def capacity_multiplier(r: float) -> float:
    return 1.0 / (1.0 - r)


def fragmentation_bound(c: int, n: int) -> float:
    return (c - 1) / n


def chunks_shared(b: int, n: int, n_s: int, c: int) -> int:
    """Chunks used by b sequences of n tokens whose first n_s (a multiple of c) are common."""
    if n_s % c:
        raise ValueError("n_s must be chunk aligned")
    return n_s // c + b * math.ceil((n - n_s) / c)


def chunks_unshared(b: int, n: int, c: int) -> int:
    return b * math.ceil(n / c)


def wasted_slots(n: int, c: int) -> int:
    return c * math.ceil(n / c) - n
