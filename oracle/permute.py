"""Token permutation into per-expert groups.

Pair p = t * k + j is token t's j-th routed expert.  The groups are laid out
expert by expert (ascending id); inside a group pairs keep ascending p (a
stable order).  counts[e] = #pairs routed to e, offsets = exclusive prefix sum
with offsets[E] = P, sorted_pair[offsets[e] + r] = the r-th pair routed to e,
inv_pos[p] = the position of pair p in sorted_pair.

The pages do not describe this step; it is the plain reading of "group tokens
by expert" that makes the result unique.
"""
from __future__ import annotations

import numpy as np


def permute(ids: np.ndarray, E: int):
    """ids int [T, k] (or [P]) -> (offsets int32 [E+1], sorted_pair int32 [P], inv_pos int32 [P])."""
    flat = np.asarray(ids).reshape(-1)
    P = flat.shape[0]
    counts = [0] * E
    for p in range(P):
        e = int(flat[p])
        if not (0 <= e < E):
            raise ValueError("expert id out of range")
        counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:E]
    fill = list(fill)
    sorted_pair = [0] * P
    inv_pos = [0] * P
    for p in range(P):
        e = int(flat[p])
        pos = fill[e]
        fill[e] += 1
        sorted_pair[pos] = p
        inv_pos[p] = pos
    return (np.asarray(offsets, dtype=np.int32), np.asarray(sorted_pair, dtype=np.int32),
            np.asarray(inv_pos, dtype=np.int32))
