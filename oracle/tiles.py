"""Virtual expert tiles (oracle; test infrastructure only).

"Nanite for Experts" §5.4: expert tensors are cut into 256 KiB virtual tiles;
the tile is a scheduling unit, not a lossy representation (reassembled tiles
give the same output). The page's tiled-transfer run moved 1.61 GB over 7,504
tiles, about 214 KB per tile, so the last tile of a tensor is partial.

Reading: each matrix's packed bytes (quant plane then scale plane) are cut into
ceil(bytes / tile) tiles, the last one partial; tiles never span matrices.
"""
from __future__ import annotations

from typing import List, Tuple

from .formats import Q8_0


def matrix_bytes(rows: int, k: int, quant: int) -> int:
    return rows * (k // 32) * (34 if quant == Q8_0 else 18)


def tile_partition(hidden: int, inter: int, quant: int,
                   tile_bytes: int = 262144) -> List[Tuple[int, int]]:
    """(offset, length) of every tile of one expert payload, in payload order."""
    tiles = []
    off = 0
    for rows, k in ((inter, hidden), (inter, hidden), (hidden, inter)):
        n = matrix_bytes(rows, k, quant)
        t = 0
        while t < n:
            ln = min(tile_bytes, n - t)
            tiles.append((off + t, ln))
            t += ln
        off += n
    return tiles
