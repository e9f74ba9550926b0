"""Pins for the oracle's block decoders (no GPU).

Q4_0: every fp16 scale pattern x every code, against Python's own half-float
decoder (struct 'e', independent of numpy) and the definition w = (q - 8) * d.
MXFP4: every E8M0 byte x every E2M1 code, against the OCP MX v1.0 element table
written out as literals and math.ldexp for the scale.  Nibble order is pinned by
blocks whose low and high nibbles differ.
"""
import math
import struct

import numpy as np

from oracle import decode_mxfp4, decode_q4_0, e2m1_value, e8m0_scale
from synth import quantize_mxfp4, quantize_q4_0

# element i < 16 in the low nibble of code byte i, i >= 16 in the high nibble of byte i - 16
Q_OF_ELEM = [i for i in range(16)] + [15 - i for i in range(16)]


def _code_bytes(q_of_elem):
    return bytes((q_of_elem[i] & 0xF) | ((q_of_elem[i + 16] & 0xF) << 4) for i in range(16))


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    return bool(np.all(both_nan | (a.view(np.int64) == b.view(np.int64))))


def test_q4_0_every_scale_every_code():
    qs = _code_bytes(Q_OF_ELEM)
    raw = bytearray()
    dvals = []
    for bits in range(65536):
        db = struct.pack("<H", bits)
        raw += db + qs
        dvals.append(struct.unpack("<e", db)[0])
    blocks = np.frombuffer(bytes(raw), dtype=np.uint8).reshape(65536, 1, 18)
    got = decode_q4_0(blocks)  # [65536, 32]
    d = np.array(dvals, dtype=np.float64)
    q = np.array(Q_OF_ELEM, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        want = (q[None, :] - 8.0) * d[:, None]
    assert got.shape == (65536, 32)
    assert _same(got, want)


def test_q4_0_unit_scale_gives_centered_codes():
    blk = struct.pack("<e", 1.0) + _code_bytes(Q_OF_ELEM)
    got = decode_q4_0(np.frombuffer(blk, dtype=np.uint8).reshape(1, 18))
    assert got.tolist() == [float(q - 8) for q in Q_OF_ELEM]
    assert got.min() == -8.0 and got.max() == 7.0


def test_q4_0_shape_concatenates_blocks_along_k():
    rng = np.random.default_rng(1)
    b = rng.integers(0, 256, size=(3, 5, 4, 18), dtype=np.uint8)
    b[..., 1] &= 0x3B  # keep scales finite
    w = decode_q4_0(b)
    assert w.shape == (3, 5, 128)
    assert _same(w[1, 2, 64:96], decode_q4_0(b[1, 2, 2:3]))


OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_matches_ocp_table():
    got = e2m1_value(np.arange(16))
    assert _same(got, OCP_E2M1)


def test_e8m0_scales():
    got = e8m0_scale(np.arange(256))
    want = [math.ldexp(1.0, b - 127) for b in range(255)] + [math.nan]
    assert _same(got, want)


def test_mxfp4_every_scale_every_code():
    raw = bytearray()
    for e in range(256):
        raw += bytes([e]) + _code_bytes(Q_OF_ELEM)
    got = decode_mxfp4(np.frombuffer(bytes(raw), dtype=np.uint8).reshape(256, 1, 17))
    want = np.empty((256, 32))
    for e in range(256):
        for i, c in enumerate(Q_OF_ELEM):
            want[e, i] = math.nan if e == 255 else OCP_E2M1[c] * math.ldexp(1.0, e - 127)
    assert _same(got, want)


def test_q4_0_encode_decode_error_bound():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[3, 32:64] = 0.0  # an all-zero block
    blocks = quantize_q4_0(w)
    back = decode_q4_0(blocks)
    d = np.abs(blocks[..., 0:2].copy().view("<f2")[..., 0].astype(np.float64))
    dd = np.repeat(d, 32, axis=-1)
    # codes 0..14: half a step; code 15 also absorbs values up to 8 steps above the
    # centre (the range is -8..7), so at most one step; plus fp16 rounding of d (|q-8| <= 8)
    q = np.concatenate([blocks[..., 2:18] & 15, blocks[..., 2:18] >> 4], axis=-1).reshape(64, 256)
    step = np.where(q == 15, 1.0, 0.5)
    bound = dd * (step + 8 * 2.0 ** -11) * (1 + 2.0 ** -10) + 1e-12
    assert np.all(np.abs(back - w) <= bound)
    assert np.all(back[3, 32:64] == 0.0)


def test_mxfp4_encode_decode_error_bound():
    rng = np.random.default_rng(8)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    blocks = quantize_mxfp4(w)
    back = decode_mxfp4(blocks)
    scale = np.repeat(np.exp2(blocks[..., 0].astype(np.float64) - 127), 32, axis=-1)
    # E2M1 grid spacing is at most 2 (between 4 and 6) below the largest code; values
    # scaled into [6, 8) saturate to 6 (error < 2 * scale)
    assert np.all(np.abs(back - w) <= 2.0 * scale)
    # every block's largest element lands on a code in [4, 6]
    amax_code = np.max(np.abs(back / scale).reshape(64, 8, 32), axis=-1)
    assert np.all((amax_code >= 4) & (amax_code <= 6))
