"""Block decode of the expert banks' 4-bit formats, in fp64.

[P5] §五 lists GGUF Q4_0 and MXFP4 among the expert-bank formats and §六 the
GGUF dequant kernels.  The bit layouts are the formats' own definitions:

* Q4_0: 32 weights per block, fp16 scale d, weight = (q - 8) * d.
* MXFP4 (OCP MX v1.0): 32 E2M1 elements share one E8M0 scale 2^(e - 127);
  scale byte 0xFF is NaN.

Reading (the pages give no byte order): a block stores its scale first, then 16
code bytes; element i < 16 is the low nibble of code byte i and element i >= 16
the high nibble of code byte i - 16 (the GGUF order), for both formats.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32


def _codes(qs: np.ndarray) -> np.ndarray:
    """16 code bytes [..., 16] -> 32 four-bit codes [..., 32] in element order."""
    lo = qs & 0x0F
    hi = qs >> 4
    return np.concatenate([lo, hi], axis=-1).astype(np.int64)


def decode_q4_0(blocks: np.ndarray) -> np.ndarray:
    """Q4_0 blocks uint8 [..., nb, 18] -> weights fp64 [..., nb * 32].

    d = little-endian fp16 in bytes 0..1 (widened exactly to fp64);
    weight_i = (q_i - 8) * d."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    assert blocks.shape[-1] == 18
    d = np.ascontiguousarray(blocks[..., 0:2]).view("<f2")[..., 0].astype(np.float64)
    q = _codes(blocks[..., 2:18])
    with np.errstate(invalid="ignore"):
        w = (q - 8).astype(np.float64) * d[..., None]
    return w.reshape(*blocks.shape[:-2], blocks.shape[-2] * BLOCK)


def e2m1_value(code) -> np.ndarray:
    """E2M1 code (bit 3 sign, bits 2..1 exponent, bit 0 mantissa; bias 1) -> fp64.

    exponent field 0 is subnormal: m * 0.5; otherwise 2^(e - 1) * (1 + m / 2)."""
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.exp2(e - 1.0) * (1.0 + 0.5 * m))
    return np.where(s == 1, -mag, mag)


def e8m0_scale(byte) -> np.ndarray:
    """E8M0 scale byte -> 2^(byte - 127) in fp64; 0xFF -> NaN."""
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.exp2(b.astype(np.float64) - 127.0))


def decode_mxfp4(blocks: np.ndarray) -> np.ndarray:
    """MXFP4 blocks uint8 [..., nb, 17] -> weights fp64 [..., nb * 32]."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    assert blocks.shape[-1] == 17
    scale = e8m0_scale(blocks[..., 0])
    v = e2m1_value(_codes(blocks[..., 1:17]))
    w = v * scale[..., None]
    return w.reshape(*blocks.shape[:-2], blocks.shape[-2] * BLOCK)


def decode_blocks(blocks: np.ndarray, qtype: str) -> np.ndarray:
    if qtype == "q4_0":
        return decode_q4_0(blocks)
    if qtype == "mxfp4":
        return decode_mxfp4(blocks)
    raise ValueError(f"unknown qtype {qtype!r}")
