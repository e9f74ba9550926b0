"""Pins for the MXFP8 activation reading (oracle/blockscaled.py): the E4M3 grid against
PyTorch's float8_e4m3fn conversion (an independent implementation of the format) on
random values, the OCP MX shared-exponent rule on hand blocks, and exactness on values
the format holds."""
import numpy as np
import torch

from oracle.blockscaled import e4m3_round, mx_e4m3_quantize


def test_e4m3_round_matches_torch_float8_e4m3fn():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(1 << 16) * s for s in (1e-3, 0.1, 1.0, 30.0, 300.0)])
    v = v[np.abs(v) <= 448.0].astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(e4m3_round(v.astype(np.float64)), want)


def test_shared_exponent_and_saturation():
    # amax = 1.0 -> u = -8, scale 2^-8: 1.0 -> 256 (exact); 0.004 -> 1.024 -> E4M3 1.0 -> 2^-8
    blk = np.zeros((1, 32))
    blk[0, 0], blk[0, 1] = 1.0, 0.004
    q = mx_e4m3_quantize(blk)
    assert q[0, 0] == 1.0 and q[0, 1] == 2.0 ** -8 and np.all(q[0, 2:] == 0)
    # amax = 1.9 -> u = -8: 1.9 * 256 = 486.4 > 448 saturates to 448 / 256 = 1.75
    blk[0, 0] = 1.9
    assert mx_e4m3_quantize(blk)[0, 0] == 1.75
    assert np.all(mx_e4m3_quantize(np.zeros((2, 64))) == 0)


def test_values_the_format_holds_pass_unchanged():
    rng = np.random.default_rng(1)
    # E4M3 values times one power of two per block, with the block max at 2^(u+8) .. 448 * 2^u
    grid = np.array([m / 8 * 2.0 ** -6 for m in range(8)] + [2.0 ** (e - 7) * (1 + m / 8) for e in range(1, 16)
                                                            for m in range(8)][:-1])
    vals = rng.choice(grid[grid <= 448], size=(4, 64)) * rng.choice([-1, 1], size=(4, 64))
    vals[:, ::32] = 448.0  # block max 448 -> u = 0
    scaled = vals * np.exp2(rng.integers(-20, 20, size=(4, 1)))
    assert np.array_equal(mx_e4m3_quantize(scaled), scaled)
