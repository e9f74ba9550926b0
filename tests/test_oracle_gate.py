"""Pins of the router-gate oracle against facts that do not depend on it: a one-hot
hidden vector reads out one column of the gate matrix (catches a transposed operand),
small-integer inputs give exact integer logits equal to a brute-force triple loop,
the map is linear in x and in Wg, and bf16 decoding is exact."""
import numpy as np

import oracle


def _bits(a):
    a = np.asarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)  # exact for bf16-representable values


def test_one_hot_rows_read_out_gate_columns():
    rng = np.random.default_rng(1)
    E, H = 5, 7
    wg = rng.integers(-8, 8, size=(E, H)).astype(np.float32)
    for h in range(H):
        x = np.zeros((1, H), np.float32)
        x[0, h] = 1.0
        got = oracle.gate(_bits(x), _bits(wg))
        assert np.array_equal(got[0], wg[:, h].astype(np.float64))


def test_small_integers_exact_against_brute_force():
    rng = np.random.default_rng(2)
    T, E, H = 3, 4, 64
    x = rng.integers(-16, 17, size=(T, H)).astype(np.float32)
    wg = rng.integers(-16, 17, size=(E, H)).astype(np.float32)
    got = oracle.gate(_bits(x), _bits(wg))
    for t in range(T):
        for e in range(E):
            s = 0
            for h in range(H):
                s += int(x[t, h]) * int(wg[e, h])
            assert got[t, e] == s


def test_linear_in_x_and_in_wg():
    rng = np.random.default_rng(3)
    T, E, H = 4, 6, 32
    x1 = rng.integers(-4, 5, size=(T, H)).astype(np.float32)
    x2 = rng.integers(-4, 5, size=(T, H)).astype(np.float32)
    wg = rng.integers(-4, 5, size=(E, H)).astype(np.float32)
    a = oracle.gate(_bits(x1), _bits(wg)) + oracle.gate(_bits(x2), _bits(wg))
    b = oracle.gate(_bits(x1 + x2), _bits(wg))
    assert np.array_equal(a, b)
    assert np.array_equal(oracle.gate(_bits(x1), _bits(2 * wg)), 2 * oracle.gate(_bits(x1), _bits(wg)))


def test_bf16_bits_decode_exactly():
    # 1.0, -2.5, the smallest normal 2^-126, the largest finite bf16
    bits = np.array([[0x3F80, 0xC020, 0x0080, 0x7F7F]], dtype=np.uint16)
    one = np.array([[0x3F80, 0, 0, 0], [0, 0x3F80, 0, 0], [0, 0, 0x3F80, 0], [0, 0, 0, 0x3F80]],
                   dtype=np.uint16)
    got = oracle.gate(bits, one)[0]
    assert got[0] == 1.0 and got[1] == -2.5 and got[2] == 2.0 ** -126
    assert got[3] == (2 - 2 ** -7) * 2.0 ** 127
