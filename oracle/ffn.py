"""Expert FFN (gate/up projection, SwiGLU, down projection) and the weighted combine, fp64.

[P5] §五: experts ("ExpertFFN") hold over 90% of an MoE model's weights.  The
pages name the FFN but not its formula; the oracle takes the standard SwiGLU
expert:

    g = W_gate x,  u = W_up x,  h = silu(g) * u,  y = W_down h,
    silu(g) = g / (1 + exp(-g)).

Weights are stored row-major with the reduction dimension last: w13 [2I, H]
(rows [0, I) gate, [I, 2I) up) and w2 [H, I] (reading).  Everything is kept in
fp64 (the CUDA path rounds h and y to bf16; the layer tolerance covers that).
"""
from __future__ import annotations

import numpy as np


def silu(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_ffn(X: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """X fp64 [n, H]; w13 fp64 [2I, H]; w2 fp64 [H, I] -> Y fp64 [n, H]."""
    I2, H = w13.shape
    I = I2 // 2
    assert X.shape[1] == H and w2.shape == (H, I)
    g = X @ w13[:I].T
    u = X @ w13[I:].T
    h = silu(g) * u
    return h @ w2.T


def expert_ffn(x: np.ndarray, k: int, offsets: np.ndarray, sorted_pair: np.ndarray,
               dequant_w13, dequant_w2, experts=None) -> np.ndarray:
    """Grouped FFN over the permuted pairs.

    x fp64 [T, H]; dequant_w13(e) -> fp64 [2I, H]; dequant_w2(e) -> fp64 [H, I].
    Returns y_perm fp64 [P, H]: row r holds expert e's output for the token of
    pair sorted_pair[r], where offsets[e] <= r < offsets[e+1].  ``experts``
    restricts the work to a subset (rows of other experts are left NaN)."""
    E = len(offsets) - 1
    P = len(sorted_pair)
    H = x.shape[1]
    y = np.full((P, H), np.nan)
    for e in range(E) if experts is None else experts:
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        tok = np.asarray(sorted_pair[a:b]) // k
        y[a:b] = swiglu_ffn(x[tok], dequant_w13(e), dequant_w2(e))
    return y


def combine(y_perm: np.ndarray, w: np.ndarray, inv_pos: np.ndarray, shared_y=None) -> np.ndarray:
    """out[t] = sum over j ascending of w[t, j] * y_perm[inv_pos[t*k + j]] (+ shared_y[t])."""
    T, k = w.shape
    H = y_perm.shape[1]
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            out[t] += w[t, j] * y_perm[inv_pos[t * k + j]]
    if shared_y is not None:
        out += shared_y
    return out
