"""The block-scaled (MX) reading of the MXFP4 layer, fp64: activations quantized to MXFP8.

The spec kernel list runs the MXFP4 prefill on block-scaled tensor-core MMA, which
multiplies E2M1 weights by FP8 activations, each with an E8M0 scale per 32 elements.  The
pages name no activation format; the reading here is the OCP Microscaling Formats v1.0
MXFP8 (E4M3) conversion applied to each 32-element block of a row along the reduction
dimension:

* shared exponent  u = floor(log2(max |v|)) - 8  (8 = the exponent of E4M3's largest
  normal, 448 = 1.75 * 2^8), clamped to the E8M0 range [-127, 127]; an all-zero block
  takes u = 0;
* each element becomes the E4M3 value nearest to v / 2^u (ties to the even code),
  saturating at +-448, and decodes back to E4M3 * 2^u.

Applied to x before the gate/up projection and to h before the down projection (both
are MMA B operands in that variant); everything else is the exact layer of layer.py.
TEST INFRASTRUCTURE, like the rest of the oracle.
"""
from __future__ import annotations

import numpy as np

from .ffn import combine, silu
from .formats import decode_blocks
from .permute import permute
from .route import route

_E4M3_MAX = 448.0


def _e4m3_grid() -> np.ndarray:
    """The non-negative finite E4M3 values in code order: code c = 8e + m, e in 0..15,
    m in 0..7, excluding the NaN code 127; e = 0 is subnormal (m / 8 * 2^-6)."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, np.exp2(e - 7.0) * (1.0 + m / 8.0))


_GRID = _e4m3_grid()


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value (ties to the even code), saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), _E4M3_MAX)
    hi = np.clip(np.searchsorted(_GRID, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo, dhi = a - _GRID[lo], _GRID[hi] - a
    c = np.where(dhi < dlo, hi, lo)
    c = np.where((dhi == dlo) & (hi != lo), np.where(lo % 2 == 0, lo, hi), c)
    return np.copysign(_GRID[c], v)


def mx_e4m3_quantize(X: np.ndarray, block: int = 32) -> np.ndarray:
    """Rows of X (fp64 [n, K], K % block == 0) through MXFP8 (see the module docstring);
    returns the decoded values (fp64, same shape)."""
    X = np.asarray(X, dtype=np.float64)
    n, K = X.shape
    b = X.reshape(n, K // block, block)
    amax = np.max(np.abs(b), axis=2)
    with np.errstate(divide="ignore"):
        u = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8.0, 0.0)
    u = np.clip(u, -127, 127)
    s = np.exp2(u)[..., None]
    return (e4m3_round(b / s) * s).reshape(n, K)


def blockscaled_ffn(X: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """SwiGLU expert with MXFP8 activations on both projections."""
    I = w13.shape[0] // 2
    Xq = mx_e4m3_quantize(X)
    g = Xq @ w13[:I].T
    u = Xq @ w13[I:].T
    h = mx_e4m3_quantize(silu(g) * u)
    return h @ w2.T


def layer_blockscaled(x_bits, logits, k, qtype, w13, w2):
    """The layer of layer.py with each expert's activations quantized to MXFP8."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    E = w13.shape[0]
    ids, w = route(logits, k)
    offsets, sorted_pair, inv_pos = permute(ids, E)
    P = len(sorted_pair)
    y = np.full((P, x.shape[1]), np.nan)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        tok = np.asarray(sorted_pair[a:b]) // k
        y[a:b] = blockscaled_ffn(x[tok], decode_blocks(w13[e], qtype), decode_blocks(w2[e], qtype))
    return dict(ids=ids, out=combine(y, w, inv_pos))
