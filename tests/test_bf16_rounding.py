"""Pins for the test-side round-to-nearest-even bf16 conversion (tests/_util.rne_bf16_bits)
that the tensor-core operand tests take their expected values from: hand cases worked
from the bf16 format (8 significant bits, exponent bias 127, subnormals below 2^-126) and
PyTorch's float32 -> bfloat16 conversion, an independent implementation, on random bits."""
import numpy as np
import torch

from tests._util import canonical_bf16, rne_bf16_bits


def test_hand_cases():
    cases = [
        (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
        (1.0 + 2.0 ** -8, 0x3F80),              # tie -> even (1.0)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),          # tie -> even (1 + 2^-6)
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),  # above the tie -> up
        (3.0 * 2.0 ** -133, 0x0003),            # subnormal, exact
        (5.0 * 2.0 ** -134, 0x0002),            # 2.5 x 2^-133 -> tie -> even (2)
        (2.0 ** -134, 0x0000),                  # half the smallest subnormal -> 0 (even)
        (3.0 * 2.0 ** -134, 0x0002),            # 1.5 x 2^-133 -> 2 x 2^-133
        (2.0 ** -126, 0x0080),                  # smallest normal
        (255.0 / 128 * 2.0 ** 127, 0x7F7F),     # largest finite
        ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),  # tie between max and 2^128 -> even -> inf
        (2.0 ** 200, 0x7F80), (-np.inf, 0xFF80), (np.nan, 0x7FC0),
        (-7.0 * 65504.0, 0xC8E0),               # -458528 -> nearest multiple of 2^11: -458752
    ]
    for v, b in cases:
        assert int(rne_bf16_bits(np.array([v]))[0]) == b, (v, hex(int(rne_bf16_bits(np.array([v]))[0])), hex(b))


def test_matches_torch_on_random_float32():
    rng = np.random.default_rng(0)
    u = rng.integers(0, 2 ** 32, size=1 << 18, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = rne_bf16_bits(f.astype(np.float64))
    assert np.array_equal(canonical_bf16(got), canonical_bf16(want))


def test_matches_torch_on_products_of_q4_codes_and_fp16_scales():
    """The values the Q4_0 operand test rounds: (q - 8) * d, exact in fp32, for many d."""
    d = np.arange(0, 65536, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
    d = d[np.isfinite(d)]
    v = (np.arange(16)[:, None] - 8.0) * d[None, :]
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(canonical_bf16(rne_bf16_bits(v)), canonical_bf16(want))
