"""Pins of the oracle's decoders for the next bank formats (NVFP4, MXFP8), which the
CUDA kernels do not read yet: E4M3 against PyTorch's own float8_e4m3fn conversion
(an independent implementation of the OCP FP8 format) for every byte, every MXFP8
scale x element pair and every NVFP4 scale x code pair against that conversion and the
OCP E2M1 table in tests/golden/, and the synthetic encoders' error bounds."""
import os

import numpy as np
import torch

import oracle
from synth import quantize_mxfp8, quantize_nvfp4

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _torch_e4m3(b):
    return torch.from_numpy(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _e2m1_table():
    with open(os.path.join(GOLDEN, "e2m1_codes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    return np.array([float(v) for _, v in rows])


def _same(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return np.all((np.isnan(a) & np.isnan(b)) | (a == b))


def test_e4m3_every_byte_matches_library():
    b = np.arange(256, dtype=np.uint8)
    assert _same(oracle.e4m3_value(b), _torch_e4m3(b))
    assert oracle.e4m3_value(0x7E) == 448.0 and np.isnan(oracle.e4m3_value(0x7F))


def test_mxfp8_every_scale_every_element():
    s, c = np.meshgrid(np.arange(256), np.arange(256), indexing="ij")
    blocks = np.zeros((256 * 256, 33), dtype=np.uint8)
    blocks[:, 0] = s.reshape(-1)
    blocks[:, 1] = c.reshape(-1)
    got = oracle.decode_mxfp8(blocks[:, None, :])[:, 0]
    scale = np.where(s.reshape(-1) == 255, np.nan, np.ldexp(1.0, s.reshape(-1) - 127))
    assert _same(got, _torch_e4m3(c.reshape(-1)) * scale)
    # the rest of each block decodes code 0 to (signed) zero times the scale
    assert _same(oracle.decode_mxfp8(blocks[:, None, :])[:, 1:], np.zeros((256 * 256, 31)) * scale[:, None])


def test_nvfp4_every_scale_every_code():
    table = _e2m1_table()
    for ts in (1.0, 0.125, 3.0517578125e-05):
        s = np.repeat(np.arange(256), 16)
        c = np.tile(np.arange(16), 256)
        blocks = np.zeros((s.size, 9), dtype=np.uint8)
        blocks[:, 0] = s
        blocks[:, 1] = c  # element 0 in the low nibble of the first code byte
        got = oracle.decode_nvfp4(blocks[:, None, :], ts)
        assert _same(got[:, 0], table[c] * _torch_e4m3(s) * ts)
        blocks[:, 1] = c << 4  # element 8 in the high nibble
        assert _same(oracle.decode_nvfp4(blocks[:, None, :], ts)[:, 8], table[c] * _torch_e4m3(s) * ts)


def test_encoders_round_trip_within_format_error():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    w[0, :16] = 0.0  # an all-zero NVFP4 block
    b, ts = quantize_nvfp4(w)
    d = oracle.decode_nvfp4(b, ts).reshape(8, 256)
    blk = np.abs(w.reshape(-1, 16)).max(axis=1).repeat(16).reshape(8, 256)
    # E2M1 steps are at most 1/3 of the block maximum's code (4 -> 6 at the top), and
    # the E4M3 block scale adds at most 1/16 of relative rounding
    assert np.all(np.abs(d - w) <= blk * (1 / 6 + 1 / 16) + 1e-30)
    assert np.all(d[0, :16] == 0.0)
    m = quantize_mxfp8(w)
    d8 = oracle.decode_mxfp8(m).reshape(8, 256)
    amax = np.abs(w.reshape(-1, 32)).max(axis=1).repeat(32).reshape(8, 256)
    # E4M3 keeps 4 significant bits; elements above 448 x 2^u saturate (OCP scale rule)
    assert np.all(np.abs(d8 - w) <= np.maximum(np.abs(w) / 16, amax * (1 - 448 / 512)) + 1e-30)
