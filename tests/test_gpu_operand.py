"""GPU: the tensor-core operands that the tcgen05 kernels build from the 4-bit weight
records, through ftmoe_dequant_operand, which runs the kernels' own decode functions.

* Prefill GEMM A tile: every weight rounded once to bf16, which must equal the
  round-to-nearest-even of the oracle's exact fp64 decode, bit for bit (zero signs
  and NaN payloads aside), for every fp16 Q4_0 scale x every code and every E8M0
  MXFP4 scale x every code (including the subnormal scale e = 0, overflow at e >= 254
  and NaN at e = 255).
* Decode GEMM A operand: the unscaled code (q - 8, or the E2M1 value), exact.
"""
import struct

import numpy as np
import pytest

import oracle
from tests._util import canonical_bf16, ensure_built, rne_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    return F, torch, cuda_device


def _operand_gpu(env, qtype, which, canon, E, N, K):
    F, torch, dev = env
    src = torch.from_numpy(canon.reshape(-1).copy()).to(dev)
    tiles = torch.empty(F.ftmoe_tiled_bytes(qtype, E, N, K), dtype=torch.uint8, device=dev)
    F.ftmoe_repack(qtype, src, tiles, E, N, K)
    out = torch.full((E, N, K), 0x7FFF, dtype=torch.int16, device=dev)  # NaN marker: unwritten
    F.ftmoe_dequant_operand(qtype, which, tiles, E, N, K, out)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


Q_OF_ELEM = list(range(16)) + [15 - i for i in range(16)]


def _codes16():
    return bytes((Q_OF_ELEM[i] & 15) | ((Q_OF_ELEM[i + 16] & 15) << 4) for i in range(16))


def _same(got, want):
    return np.array_equal(canonical_bf16(got), canonical_bf16(want))


def test_prefill_operand_q4_0_every_scale_every_code(env):
    F = env[0]
    raw = bytearray()
    for bits in range(65536):
        raw += struct.pack("<H", bits) + _codes16()
    canon = np.frombuffer(bytes(raw), dtype=np.uint8).reshape(1, 2048, 32, 18)
    got = _operand_gpu(env, "q4_0", F.OPERAND_PREFILL, canon, 1, 2048, 1024)
    want = rne_bf16_bits(oracle.decode_q4_0(canon))
    assert _same(got, want)
    # the rounding is not vacuous: many products need more than bf16's 8 bits
    exact = oracle.decode_q4_0(canon)
    fin = np.isfinite(exact)
    assert np.count_nonzero(exact[fin].astype(np.float32) != (got[fin].astype(np.uint32) << 16).view(np.float32)) > 10000


def test_prefill_operand_mxfp4_every_scale_every_code(env):
    F = env[0]
    raw = bytearray()
    for e in range(256):
        raw += bytes([e]) + _codes16()
    canon = np.frombuffer(bytes(raw), dtype=np.uint8).reshape(1, 16, 16, 17)
    got = _operand_gpu(env, "mxfp4", F.OPERAND_PREFILL, canon, 1, 16, 512)
    exact = oracle.decode_mxfp4(canon)
    want = rne_bf16_bits(exact)
    assert _same(got, want)
    # what this covers: bf16 subnormal results (e = 0, 1), overflow to inf (e >= 254), NaN
    mag = np.abs(exact[np.isfinite(exact)])
    assert np.any((mag > 0) & (mag < 2.0 ** -126))
    assert np.any(mag >= 2.0 ** 128) and np.isnan(exact).any()


def _unit_scales(canon, qtype):
    c = canon.copy()
    if qtype == "q4_0":
        c[..., 0], c[..., 1] = 0x00, 0x3C  # fp16 1.0
    else:
        c[..., 0] = 127                    # 2^0
    return c


@pytest.mark.parametrize("qtype,E,N,K", [("q4_0", 2, 48, 96), ("mxfp4", 3, 160, 224),
                                         ("q4_0", 1, 256, 2048), ("mxfp4", 2, 2048, 768)])
def test_operands_random_blocks_ragged_tiles(env, qtype, E, N, K):
    """Random block bytes (finite scales) on shapes with a partial 128-row tile (N = 48,
    160) and a half-filled last 64-element slab (K = 96, 224): both operands, every
    element."""
    F = env[0]
    rng = np.random.default_rng(E * N + K)
    blk = 18 if qtype == "q4_0" else 17
    canon = rng.integers(0, 256, size=(E, N, K // 32, blk), dtype=np.uint8)
    if qtype == "q4_0":
        canon[..., 1] &= 0x7B  # finite fp16 scales
    else:
        canon[..., 0] = np.minimum(canon[..., 0], 254)
    got = _operand_gpu(env, qtype, F.OPERAND_PREFILL, canon, E, N, K)
    assert _same(got, rne_bf16_bits(oracle.decode_blocks(canon, qtype)))
    codes = _operand_gpu(env, qtype, F.OPERAND_CODES, canon, E, N, K)
    want = oracle.decode_blocks(_unit_scales(canon, qtype), qtype)
    assert np.array_equal(want, (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64))


def test_operand_rejects_bad_arguments(env):
    F, torch, dev = env
    tiles = torch.zeros(F.ftmoe_tiled_bytes("q4_0", 1, 16, 64), dtype=torch.uint8, device=dev)
    out = torch.zeros(16 * 64 + 8, dtype=torch.int16, device=dev)
    for which, o in ((7, out), (F.OPERAND_PREFILL, out[1:])):
        with pytest.raises(F.FtmoeError) as ei:
            F.ftmoe_dequant_operand("q4_0", which, tiles, 1, 16, 64, o)
        assert ei.value.status == 1
