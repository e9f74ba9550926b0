"""Router gate on the GPU (ftmoe_gate) against the fp64 oracle.

Bar: every logit within (H/16 + 16) * 2^-23 * sum_h |x_h * wg_h| of the exact value
(products of two bf16 values are exact in fp32; along the longest chain of the
fixed summation order there are at most H/16 + 16 fp32 additions, each off by at
most 2^-23 of a partial sum bounded by sum |x w|, allowing truncation instead of
rounding).  Also: a token's logits are the same bits alone and in a batch, one-hot
inputs read out gate columns exactly, and the router's integer decision on the GPU
logits equals the oracle's on the same values.
"""
import numpy as np
import pytest

import oracle
from synth import gen_gate_weights, gen_x_bf16
from tests._util import bf16_tensor, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    return F, torch, cuda_device


def _f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _gate_gpu(env, x_bits, wg_bits):
    F, torch, dev = env
    T, H = x_bits.shape
    E = wg_bits.shape[0]
    out = torch.full((max(T, 1), E), float("nan"), dtype=torch.float32, device=dev)
    F.ftmoe_gate(bf16_tensor(x_bits, dev), bf16_tensor(wg_bits, dev), T, H, E, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()[:T]


def _check(got, x_bits, wg_bits):
    want = oracle.gate(x_bits, wg_bits)
    H = x_bits.shape[1]
    bound = (H / 16 + 16) * 2.0 ** -23 * (np.abs(_f64(x_bits)) @ np.abs(_f64(wg_bits)).T)
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= bound), float((err / np.maximum(bound, 1e-300)).max())


# (T, H, E): decode, ragged tiles, the large layer's gate, a prefill chunk
@pytest.mark.parametrize("T,H,E", [(64, 2048, 128), (37, 2048, 100), (1, 7168, 256), (32, 7168, 256),
                                   (4096, 2048, 128)])
def test_gate_matches_oracle(env, T, H, E):
    x = gen_x_bf16(21, T, H, "gate_x")
    wg = gen_gate_weights(22, E, H)
    _check(_gate_gpu(env, x, wg), x, wg)


def test_gate_batch_invariance(env):
    T, H, E = 64, 2048, 128
    x = gen_x_bf16(23, T, H, "gate_x")
    wg = gen_gate_weights(24, E, H)
    full = _gate_gpu(env, x, wg)
    for t in (0, 17, 63):
        alone = _gate_gpu(env, x[t:t + 1], wg)
        assert np.array_equal(alone[0].view(np.uint32), full[t].view(np.uint32))


def test_gate_one_hot_reads_columns(env):
    H, E = 256, 40
    wg = gen_gate_weights(25, E, H)
    hs = [0, 5, 100, 255]
    x = np.zeros((len(hs), H), dtype=np.uint16)
    for i, h in enumerate(hs):
        x[i, h] = 0x3F80  # 1.0
    got = _gate_gpu(env, x, wg)
    for i, h in enumerate(hs):
        assert np.array_equal(got[i].astype(np.float64), _f64(wg[:, h]))


def test_gate_then_route_integer_decision(env):
    F, torch, dev = env
    T, H, E, k = 64, 2048, 128, 8
    x = gen_x_bf16(26, T, H, "gate_x")
    wg = gen_gate_weights(27, E, H)
    lg = _gate_gpu(env, x, wg)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    F.ftmoe_route(torch.from_numpy(lg).to(dev), T, E, k, ids, w)
    torch.cuda.synchronize()
    rids, _ = oracle.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), rids)
