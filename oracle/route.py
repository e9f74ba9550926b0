"""Router: softmax over expert logits, top-k selection, renormalisation (fp64).

MoE activates only a few experts per token ([P3] "为什么 MoE 模型适合做 CPU–GPU
协同"; [P4] 局限, expert-activation sparsity).  The pages do not spell out the
router, so the oracle takes the plain MoE reading:

1. p = softmax(logits) over all E experts;
2. the k experts with the largest logits are selected, in descending logit
   order, ties broken toward the lower expert id (softmax is monotone, so this
   is the same set as the k largest probabilities, and deciding on the logits
   themselves keeps the integer decision independent of exp rounding);
3. w_j = p_{id_j} / sum over the selected of p.
"""
from __future__ import annotations

import numpy as np


def route(logits: np.ndarray, k: int):
    """logits float [T, E] -> (ids int32 [T, k], w fp64 [T, k])."""
    lg = np.asarray(logits, dtype=np.float64)
    T, E = lg.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    if not np.all(np.isfinite(lg)):
        raise ValueError("router logits must be finite")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        row = lg[t]
        p = np.exp(row - row.max())
        p = p / p.sum()
        # descending logit, then ascending id
        order = sorted(range(E), key=lambda e: (-row[e], e))[:k]
        sel = p[order]
        ids[t] = order
        w[t] = sel / sel.sum()
    return ids, w
