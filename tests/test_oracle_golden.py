"""The oracle's block decoders against stored fixtures under tests/golden/: the E2M1
and E8M0 tables of the OCP MX v1.0 specification, and Q4_0 / MXFP4 blocks worked out
from the formats' definitions (see each file's header).  The pages themselves print no
worked example; these values are fixed by the format definitions they name."""
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _blocks(name):
    rows = _rows(name)
    out = []
    for blk, wts in zip(rows[0::2], rows[1::2]):
        assert blk[0] == "block" and wts[0] == "weights"
        out.append((np.frombuffer(bytes.fromhex(blk[1]), dtype=np.uint8), np.array(wts[1:], dtype=np.float64)))
    return out


def test_e2m1_table():
    for code, val in _rows("e2m1_codes.txt"):
        got = float(oracle.e2m1_value(int(code)))
        assert got == float(val) and np.signbit(got) == np.signbit(float(val)), code


def test_e8m0_table():
    for byte, val in _rows("e8m0_scales.txt"):
        got = float(oracle.e8m0_scale(int(byte)))
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val), byte


def test_q4_0_blocks():
    for blk, want in _blocks("q4_0_blocks.txt"):
        got = oracle.decode_q4_0(blk.reshape(1, 18))
        assert np.array_equal(got, want)


def test_mxfp4_blocks():
    for blk, want in _blocks("mxfp4_blocks.txt"):
        got = oracle.decode_mxfp4(blk.reshape(1, 17))
        assert np.array_equal(got, want)


def test_nvfp4_blocks():
    rows = _rows("nvfp4_blocks.txt")
    ts = float(rows[0][1])
    for blk, want in [(np.frombuffer(bytes.fromhex(rows[1][1]), dtype=np.uint8),
                       np.array(rows[2][1:], dtype=np.float64))]:
        got = oracle.decode_nvfp4(blk.reshape(1, 9), ts)
        assert np.array_equal(got, want)


def test_mxfp8_blocks():
    for blk, want in _blocks("mxfp8_blocks.txt"):
        got = oracle.decode_mxfp8(blk.reshape(1, 33))
        assert np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))
