"""Pins for the oracle FFN, combine and whole layer (no GPU).

FFN: small-integer weights and activations make both projections exact integer
matmuls; they are recomputed here with Python integers and math.exp, and the
down projection with math.fsum.  Layer: closed forms (identical experts make
the output independent of the routing weights), permutation equivariance and
the per-token definition against the grouped one.
"""
import math

import numpy as np

from oracle import combine, layer, layer_rows, swiglu_ffn
from oracle.formats import decode_blocks
from synth import make_layer


def test_swiglu_exact_small_integers():
    rng = np.random.default_rng(11)
    n, H, I = 5, 12, 7
    X = rng.integers(-3, 4, size=(n, H))
    W13 = rng.integers(-2, 3, size=(2 * I, H))
    W2 = rng.integers(-2, 3, size=(H, I))
    got = swiglu_ffn(X.astype(float), W13.astype(float), W2.astype(float))
    for r in range(n):
        xs = [int(v) for v in X[r]]
        g = [sum(int(W13[i, c]) * xs[c] for c in range(H)) for i in range(I)]
        u = [sum(int(W13[I + i, c]) * xs[c] for c in range(H)) for i in range(I)]
        h = [g[i] / (1.0 + math.exp(-g[i])) * u[i] for i in range(I)]
        for o in range(H):
            want = math.fsum(int(W2[o, i]) * h[i] for i in range(I))
            assert abs(got[r, o] - want) <= 1e-12 * (1 + abs(want))


def test_zero_gate_gives_zero():
    X = np.ones((2, 4))
    W13 = np.vstack([np.zeros((3, 4)), np.ones((3, 4))])
    assert np.all(swiglu_ffn(X, W13, np.ones((4, 3))) == 0.0)


def test_combine_closed_form():
    y = np.arange(12, dtype=float).reshape(3, 4)
    # token 0 routed to rows 2 and 0 with weights 0.25 / 0.75
    out = combine(y, np.array([[0.25, 0.75]]), np.array([2, 0]))
    assert np.allclose(out, 0.25 * y[2] + 0.75 * y[0])


def _tiny(**kw):
    args = dict(H=64, I=32, E=4, k=2, T=16, qtype="q4_0", seed=5)
    args.update(kw)
    return make_layer(**args)


def test_identical_experts_make_output_weight_independent():
    L = _tiny()
    w13 = np.broadcast_to(L.w13[:1], L.w13.shape).copy()
    w2 = np.broadcast_to(L.w2[:1], L.w2.shape).copy()
    r = layer(L.x, L.logits, L.k, L.qtype, w13, w2)
    x = (L.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    want = swiglu_ffn(x, decode_blocks(w13[0], "q4_0"), decode_blocks(w2[0], "q4_0"))
    assert np.allclose(r["out"], want, rtol=1e-12, atol=1e-14)


def test_token_permutation_equivariance():
    L = _tiny(qtype="mxfp4")
    r = layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    perm = np.random.default_rng(2).permutation(L.T)
    r2 = layer(L.x[perm], L.logits[perm], L.k, L.qtype, L.w13, L.w2)
    assert np.allclose(r2["out"], r["out"][perm], rtol=1e-12, atol=1e-15)


def test_per_token_definition_matches_grouped_and_shared_expert_adds():
    L = _tiny(shared=True)
    r = layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, L.shared_w13, L.shared_w2)
    rows = [0, 3, 7, 15]
    ids, w, out = layer_rows(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, rows, L.shared_w13, L.shared_w2)
    assert np.array_equal(ids, r["ids"][rows])
    assert np.allclose(out, r["out"][rows], rtol=1e-12, atol=1e-15)
    r0 = layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    assert np.allclose(r["out"] - r0["out"], r["shared_y"], rtol=1e-10, atol=1e-14)


def test_silu_identities():
    """silu(x) = x * sigmoid(x) pinned by facts that do not retype it: silu(x) - silu(-x)
    = x (sigmoid(x) + sigmoid(-x) = 1), silu(0) = 0, the tanh form of the sigmoid, and
    the limits x (x -> +inf) and 0 (x -> -inf)."""
    from oracle import silu
    x = np.linspace(-30.0, 30.0, 1201)
    assert np.allclose(silu(x) - silu(-x), x, rtol=0, atol=1e-12)
    assert silu(np.array([0.0]))[0] == 0.0
    xm = np.linspace(-8.0, 8.0, 321)  # (1 + tanh) cancels for large negative x
    assert np.allclose(silu(xm), xm * 0.5 * (1.0 + np.tanh(0.5 * xm)), rtol=1e-12, atol=1e-15)
    assert abs(silu(np.array([60.0]))[0] - 60.0) < 1e-20 and abs(silu(np.array([-60.0]))[0]) < 1e-24


def test_gate_rows_come_first_and_up_multiplies():
    """w13 holds the gate rows first: with gate rows giving 2 and up rows giving 3 the
    hidden value is silu(2) * 3, not silu(3) * 2 (a swapped half would give the latter)."""
    H, I = 4, 2
    X = np.ones((1, H))
    W13 = np.vstack([np.full((I, H), 0.5), np.full((I, H), 0.75)])  # gate 2, up 3
    W2 = np.eye(H, I)  # y[o] = h[o] for o < I
    y = swiglu_ffn(X, W13, W2)[0]
    s2 = 2.0 * 0.5 * (1.0 + math.tanh(1.0))  # silu(2) in the tanh form
    assert abs(y[0] - 3.0 * s2) < 1e-12 and abs(y[1] - 3.0 * s2) < 1e-12
    assert abs(y[0] - 2.0 * 3.0 * 0.5 * (1.0 + math.tanh(1.5))) > 0.1
