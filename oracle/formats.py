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


# ----------------------------------------------------------------------------- next formats
# The architecture walkthrough §五/§六 lists more bank formats than the two the layer
# runs on.  These decoders are the oracle side of two of them; the CUDA kernels do
# not read them yet.
#
# * NVFP4 (reading): 16 E2M1 elements share one E4M3 scale byte, and a whole weight
#   matrix shares one fp32 tensor scale; weight = E2M1(c) * E4M3(s) * tensor_scale.
#   A block stores its scale byte, then 8 code bytes: element i < 8 is the low nibble
#   of code byte i and i >= 8 the high nibble of byte i - 8 (the Q4_0 order at half
#   the block length).
# * MXFP8 (OCP MX v1.0, E4M3 elements): 32 E4M3 elements share one E8M0 scale;
#   a block stores the scale byte, then the 32 element bytes in order.
NVFP4_BLOCK = 16


def e4m3_value(byte) -> np.ndarray:
    """E4M3 byte (OCP FP8 E4M3: bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0
    mantissa; no infinities, exponent and mantissa all ones is NaN) -> fp64.
    Exponent field 0 is subnormal: m / 8 * 2^-6."""
    b = np.asarray(byte, dtype=np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, np.exp2(e - 7.0) * (1.0 + m / 8.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def decode_nvfp4(blocks: np.ndarray, tensor_scale: float) -> np.ndarray:
    """NVFP4 blocks uint8 [..., nb, 9] and the matrix's fp32 tensor scale ->
    weights fp64 [..., nb * 16]."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    assert blocks.shape[-1] == 9
    qs = blocks[..., 1:9]
    codes = np.concatenate([qs & 0x0F, qs >> 4], axis=-1).astype(np.int64)
    w = e2m1_value(codes) * e4m3_value(blocks[..., 0])[..., None] * float(np.float32(tensor_scale))
    return w.reshape(*blocks.shape[:-2], blocks.shape[-2] * NVFP4_BLOCK)


def decode_mxfp8(blocks: np.ndarray) -> np.ndarray:
    """MXFP8 (E4M3) blocks uint8 [..., nb, 33] -> weights fp64 [..., nb * 32]."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    assert blocks.shape[-1] == 33
    w = e4m3_value(blocks[..., 1:33]) * e8m0_scale(blocks[..., 0])[..., None]
    return w.reshape(*blocks.shape[:-2], blocks.shape[-2] * BLOCK)


def decode_blocks(blocks: np.ndarray, qtype: str, tensor_scale=None) -> np.ndarray:
    """Blocks of one format -> fp64 weights; NVFP4 also takes its matrix's tensor scale."""
    if qtype == "q4_0":
        return decode_q4_0(blocks)
    if qtype == "mxfp4":
        return decode_mxfp4(blocks)
    if qtype == "nvfp4":
        return decode_nvfp4(blocks, tensor_scale)
    if qtype == "mxfp8":
        return decode_mxfp8(blocks)
    raise ValueError(f"unknown qtype {qtype!r}")
