"""Chunked-prefill block schedule (Chunked Prefill, section 3 "The hole chunking leaves").

A prompt longer than the chunk width W runs as full W-row blocks followed by
one block holding the remainder; a prompt of at most W rows runs as one block.
The page's own examples: 1137 rows at W = 512 -> 512, 512, 113; 1200 -> 512,
512, 176.
"""
from __future__ import annotations

from typing import List


def prefill_blocks(n_rows: int, width: int) -> List[int]:
    if width < 1:
        raise ValueError("width must be positive")
    if n_rows < 0:
        raise ValueError("negative row count")
    full, rem = divmod(n_rows, width)
    return [width] * full + ([rem] if rem else [])
