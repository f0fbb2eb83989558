"""Routing metadata by its definition.

Test infrastructure only (see the package docstring).

The flashinfer_ops page names the metadata the routing kernel writes
(``FlashInferOps.slot``: total padded tokens, expanded->permuted index,
permuted->token index, expert counts, the tile->expert and tile->row-limit
tables and the number of live tiles), keeps the buffers -1-filled
(``FlashInferOps.prepare_from_metadata``), and bounds the padded rows
(``gemm2_rows``: ``tile * (min(E, R) + (R - min(E, R)) // tile)`` for R
routes). The kernel itself is not on the pages; the order of routes inside an
expert's rows is this project's reading (open point 4): ascending expanded
index j = t * K + k, which makes the result unique.

    counts[e]    = #{(t, k) : ids[t, k] == e}
    padded[e]    = ceil(counts[e] / tile) * tile
    offsets      = exclusive prefix sum of padded, ascending e; offsets[E] =
                   total padded rows
    expanded_to_permuted[t, k] = offsets[e] + (rank of j among the routes of
                   e, ascending j); -1 where ids[t, k] == -1 (not routed: the
                   muse_moe_runner page, ``_finalize_native``, reads such
                   routes as zero rows)
    permuted_to_token[p] = t on an expert's live rows, -1 on padding rows and
                   on rows past the total
    tiles        = (e ascending, i ascending) over ceil(counts[e]/tile) tiles;
                   tile_expert = e, tile_row_limit = offsets[e] + counts[e];
                   tile tau covers permuted rows [tau*tile, (tau+1)*tile);
                   entries past the live tiles are -1
    totals       = (number of live tiles, total padded rows)

Parity: pinned (brute force sort by (e, j) and invariants in the tests).
"""
from __future__ import annotations

import numpy as np


def max_padded_rows(T: int, K: int, E: int, tile: int) -> int:
    """Upper bound of the padded permuted rows (``gemm2_rows`` without its
    128 KiB floor)."""
    R = T * K
    F = min(E, R)
    return tile * (F + (R - F) // tile)


def max_tiles(T: int, K: int, E: int, tile: int) -> int:
    return max_padded_rows(T, K, E, tile) // tile


def route_metadata(topk_ids: np.ndarray, E: int, tile: int) -> dict[str, np.ndarray]:
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, K = ids.shape
    flat = ids.reshape(-1)
    if np.any((flat < -1) | (flat >= E)):
        raise ValueError("expert id out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        if e >= 0:
            counts[e] += 1
    padded = -(-counts // tile) * tile
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    total = int(offsets[E])

    P = max_padded_rows(T, K, E, tile)
    expanded_to_permuted = np.full(T * K, -1, dtype=np.int64)
    permuted_to_token = np.full(P, -1, dtype=np.int64)
    cursor = offsets[:E].copy()
    for j in range(T * K):  # ascending expanded index
        e = flat[j]
        if e < 0:
            continue
        p = cursor[e]
        cursor[e] += 1
        expanded_to_permuted[j] = p
        permuted_to_token[p] = j // K

    MT = P // tile
    tile_expert = np.full(MT, -1, dtype=np.int64)
    tile_row_limit = np.full(MT, -1, dtype=np.int64)
    n = 0
    for e in range(E):
        for _ in range(int(padded[e] // tile)):
            tile_expert[n] = e
            tile_row_limit[n] = offsets[e] + counts[e]
            n += 1
    assert n * tile == total <= P
    i32 = lambda a: np.asarray(a, dtype=np.int32)  # noqa: E731
    return {
        "expert_counts": i32(counts),
        "expert_offsets": i32(offsets),
        "expanded_to_permuted": i32(expanded_to_permuted.reshape(T, K)),
        "permuted_to_token": i32(permuted_to_token),
        "tile_expert": i32(tile_expert),
        "tile_row_limit": i32(tile_row_limit),
        "totals": i32([n, total]),
    }
