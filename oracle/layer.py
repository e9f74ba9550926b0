"""The whole MoE expert layer: route -> permute -> expert FFN -> combine (+ shared expert).

The shared (always-on) expert is an FFN of the same shape applied to every token
with weight 1 and no gate (reading: the pages describe no shared expert; the
large-layer workload adds one).
"""
from __future__ import annotations

import numpy as np

from .ffn import combine, expert_ffn, swiglu_ffn
from .formats import decode_blocks
from .permute import permute
from .route import route


def _x_fp64(x_bf16_bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values."""
    b = np.asarray(x_bf16_bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _dec(blocks, qtype, ts, name, e):
    """Expert e's matrix `name` decoded; ts (NVFP4: {name: float32 [E]}) gives its tensor scale."""
    return decode_blocks(blocks[e], qtype, None if ts is None else ts[name][e])


def layer(x_bits, logits, k, qtype, w13, w2, shared_w13=None, shared_w2=None, ts=None):
    """Full layer on all tokens.

    x_bits uint16 bf16 [T, H]; logits float32 [T, E]; w13 uint8 [E, 2I, H/bs, blk];
    w2 uint8 [E, H, I/bs, blk]; ts: NVFP4's per-matrix tensor scales
    {"w13": [E], "w2": [E], "shared_w13": [1], "shared_w2": [1]} (None otherwise).
    Returns a dict with ids, w, offsets, sorted_pair, inv_pos, y_perm [P, H] and
    out [T, H] (fp64)."""
    x = _x_fp64(x_bits)
    E = w13.shape[0]
    ids, w = route(logits, k)
    offsets, sorted_pair, inv_pos = permute(ids, E)
    y = expert_ffn(x, k, offsets, sorted_pair,
                   lambda e: _dec(w13, qtype, ts, "w13", e), lambda e: _dec(w2, qtype, ts, "w2", e))
    sh = None
    if shared_w13 is not None:
        sh = swiglu_ffn(x, _dec(shared_w13, qtype, ts, "shared_w13", 0),
                        _dec(shared_w2, qtype, ts, "shared_w2", 0))
    out = combine(y, w, inv_pos, sh)
    return dict(ids=ids, w=w, offsets=offsets, sorted_pair=sorted_pair, inv_pos=inv_pos,
                y_perm=y, out=out, shared_y=sh)


def layer_rows(x_bits, logits, k, qtype, w13, w2, rows, shared_w13=None, shared_w2=None, ts=None):
    """Layer output for a subset of tokens, by the per-token definition.

    A token's output depends only on its own activations and logits:
    out[t] = sum_j w[t, j] * FFN_{ids[t, j]}(x[t]) (+ FFN_shared(x[t])).
    The experts are visited one at a time (decoded once, applied to every sampled token
    that selected it) so that only one expert's fp64 weights are held at a time.
    Returns (ids [n, k], w [n, k], out fp64 [n, H]) for the tokens in ``rows``."""
    rows = np.asarray(rows, dtype=np.int64)
    x = _x_fp64(np.asarray(x_bits)[rows])
    ids, w = route(np.asarray(logits)[rows], k)
    n, H = x.shape
    out = np.zeros((n, H))
    for e in np.unique(ids):
        sel_i, sel_j = np.nonzero(ids == e)
        y = swiglu_ffn(x[sel_i], _dec(w13, qtype, ts, "w13", e), _dec(w2, qtype, ts, "w2", e))
        for r, (i, j) in enumerate(zip(sel_i, sel_j)):
            out[i] += w[i, j] * y[r]
    if shared_w13 is not None:
        out += swiglu_ffn(x, _dec(shared_w13, qtype, ts, "shared_w13", 0),
                          _dec(shared_w2, qtype, ts, "shared_w2", 0))
    return ids, w, out
