"""GPU: the MXFP8 expert bank (the pages' block-scaled FP8 bank, [P5] §五 / §六 "FP8 block
linear", read as OCP MX v1.0 MXFP8: 32 E4M3 elements sharing an E8M0 scale).

* exact decode (ftmoe_dequant, fp32) of every E8M0 scale x every E4M3 code against the
  oracle's decode (beyond fp32's range: +-inf);
* the prefill GEMM operand: round-to-nearest-even bf16 of E4M3 x 2^(e - 127) for every
  scale x every finite code; the grouped GEMV's operand: each finite E4M3 value, exact
  (the fast paths do not special-case the NaN code S.1111.111, which weight banks never
  hold; the exact decode maps it to NaN);
* the layer against the oracle through the grouped GEMV (decode sizes; the decode GEMM
  declines the format) and the tcgen05 GEMM (prefill, sampled rows), ragged shapes with a
  shared expert, and cache-slot blobs through a pointer table.
"""
import numpy as np
import pytest

import oracle
from synth import CONFIGS, make_layer
from tests._util import bf16_tensor, bf16_to_f64, canonical_bf16, ensure_built, rel_l2, rne_bf16_bits

pytestmark = pytest.mark.gpu
LAYER_TOL = 1e-2


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    return F, torch, cuda_device


def _every_scale_every_code():
    """256 rows (one per E8M0 scale byte) x 256 elements (every E4M3 code, in order)."""
    b = np.zeros((256, 8, 33), dtype=np.uint8)
    b[:, :, 0] = np.arange(256, dtype=np.uint8)[:, None]
    b[:, :, 1:] = np.arange(256, dtype=np.uint8).reshape(8, 32)[None]
    return b.reshape(1, 256, 8, 33)


def _tiles(env, canon, E, N, K):
    F, torch, dev = env
    src = torch.from_numpy(canon.reshape(-1).copy()).to(dev)
    tiles = torch.empty(F.ftmoe_tiled_bytes("mxfp8", E, N, K), dtype=torch.uint8, device=dev)
    F.ftmoe_repack("mxfp8", src, tiles, E, N, K)
    return tiles


def test_mxfp8_exact_decode_every_scale_every_code(env):
    F, torch, dev = env
    canon = _every_scale_every_code()
    tiles = _tiles(env, canon, 1, 256, 256)
    out = torch.full((1, 256, 256), 7.0, dtype=torch.float32, device=dev)
    F.ftmoe_dequant("mxfp8", tiles, 1, 256, 256, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ex = oracle.decode_mxfp8(canon)
    over = np.isfinite(ex) & (np.abs(ex) >= 2.0 ** 128)
    want = np.where(over, np.copysign(np.inf, ex), np.where(over, 0.0, ex)).astype(np.float32)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert np.all(same)


def test_mxfp8_operands_every_scale_every_finite_code(env):
    F, torch, dev = env
    canon = _every_scale_every_code()
    tiles = _tiles(env, canon, 1, 256, 256)
    finite_code = (np.arange(256) & 0x7F) != 0x7F
    ex = oracle.decode_mxfp8(canon)[0]
    out = torch.full((1, 256, 256), 0x7FFF, dtype=torch.int16, device=dev)
    F.ftmoe_dequant_operand("mxfp8", F.OPERAND_PREFILL, tiles, 1, 256, 256, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)[0]
    assert np.array_equal(canonical_bf16(got[:, finite_code]), canonical_bf16(rne_bf16_bits(ex[:, finite_code])))
    # the rounding is exercised: scales near the ends of the range leave bf16's
    assert np.any(np.abs(ex[:, finite_code]) < 2.0 ** -133) and np.any(np.abs(ex[:, finite_code]) >= 2.0 ** 128)
    F.ftmoe_dequant_operand("mxfp8", F.OPERAND_CODES, tiles, 1, 256, 256, out)
    torch.cuda.synchronize()
    codes = (out.cpu().numpy().view(np.uint16)[0].astype(np.uint32) << 16).view(np.float32)
    e4m3 = oracle.e4m3_value(np.arange(256))
    assert np.array_equal(codes[:, finite_code], np.broadcast_to(e4m3[finite_code], (256, finite_code.sum())))


def _layer(env, L, path=0):
    F, torch, dev = env
    from quantized_expert_ffn_layer_b300 import MoELayer
    m = MoELayer(L.qtype, L.E, L.H, L.I, L.w13, L.w2, L.shared_w13, L.shared_w2, device=dev)
    old = F.ftmoe_set_ffn_path(path)
    try:
        ids = torch.empty((L.T, L.k), dtype=torch.int32, device=dev)
        out = m.forward(torch.from_numpy(L.logits).to(dev), bf16_tensor(L.x, dev), L.k, ids_out=ids)
        torch.cuda.synchronize()
    finally:
        F.ftmoe_set_ffn_path(old)
    assert F.ftmoe_device_status() == 0
    return m, bf16_to_f64(out), ids.cpu().numpy()


@pytest.mark.parametrize("T", [1, 64, 256])
def test_mxfp8_decode_layer_parity(env, T):
    c = dict(CONFIGS["decode"])
    c.update(T=T, qtype="mxfp8")
    L = make_layer(**c)
    _, out, ids = _layer(env, L)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


@pytest.mark.parametrize("path", [1, 2])
def test_mxfp8_ragged_shared_expert_both_paths(env, path):
    L = make_layer(H=224, I=96, E=5, k=3, T=300, qtype="mxfp8", seed=9, shared=True)
    _, out, ids = _layer(env, L, path)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, L.shared_w13, L.shared_w2)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


def test_mxfp8_prefill_layer_sampled(env):
    c = dict(CONFIGS["prefill"])
    c.update(qtype="mxfp8")
    L = make_layer(**c)
    _, out, ids = _layer(env, L)
    rows = np.random.default_rng(3).choice(L.T, size=32, replace=False)
    rids, _, rout = oracle.layer_rows(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, rows)
    assert np.array_equal(ids[rows], rids)
    assert rel_l2(out[rows], rout) <= LAYER_TOL


@pytest.mark.parametrize("path", [1, 2])
def test_mxfp8_expert_blob_table(env, path):
    F, torch, dev = env
    L = make_layer(H=256, I=128, E=8, k=2, T=200, qtype="mxfp8", seed=21)
    m, ref, _ = _layer(env, L, path)
    blobs = torch.cat([m.w13.view(L.E, -1), m.w2.view(L.E, -1)], dim=1).contiguous()
    nb = blobs.shape[1]
    assert nb == F.ftmoe_expert_blob_bytes("mxfp8", L.H, L.I)
    slots = torch.flip(blobs, dims=[0]).contiguous()
    wt = F.make_weights("mxfp8", L.E, L.H, L.I,
                        expert_blob=[slots.data_ptr() + (L.E - 1 - e) * nb for e in range(L.E)])
    old = F.ftmoe_set_ffn_path(path)
    try:
        ws = m.workspace(L.T, L.k)
        out = torch.empty((L.T, L.H), dtype=torch.bfloat16, device=dev)
        F.ftmoe_layer(wt, torch.from_numpy(L.logits).to(dev), bf16_tensor(L.x, dev), L.T, L.k, out,
                      None, None, ws, ws.numel())
        torch.cuda.synchronize()
    finally:
        F.ftmoe_set_ffn_path(old)
    assert np.array_equal(bf16_to_f64(out), ref)
