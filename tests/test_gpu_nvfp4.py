"""GPU: the NVFP4 expert bank ([P5] §五 lists NVFP4 among the bank formats and §六 an NVFP4
fused MoE kernel): 16 E2M1 codes per block with an E4M3 scale, one fp32 tensor scale per
expert matrix.

* exact decode (ftmoe_dequant, fp32) of every E4M3 scale byte x every code, against the
  oracle's decode: E2M1 x E4M3 is exact and the tensor scale rounds once;
* the prefill GEMM operand: E2M1 x E4M3 as bf16 (exact; the tensor scale multiplies the
  accumulators), for every scale byte x code;
* the layer against the oracle on the decode shape (grouped GEMV, also at 8 to 16 rows
  per expert, where the decode GEMM declines the format), the prefill shape (tcgen05
  GEMM, sampled rows), ragged shapes with a shared expert, and through a pointer table.
"""
import numpy as np
import pytest

import oracle
from synth import CONFIGS, make_layer
from tests._util import canonical_bf16, ensure_built, rel_l2, rne_bf16_bits

pytestmark = pytest.mark.gpu
LAYER_TOL = 1e-2


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    return F, torch, cuda_device


def _tiles(env, blocks, ts, E, N, K):
    F, torch, dev = env
    raw = np.concatenate([blocks.reshape(-1), np.asarray(ts, dtype="<f4").view(np.uint8)])
    src = torch.from_numpy(raw).to(dev)
    tiles = torch.empty(F.ftmoe_tiled_bytes("nvfp4", E, N, K), dtype=torch.uint8, device=dev)
    F.ftmoe_repack("nvfp4", src, tiles, E, N, K)
    return tiles


def _every_scale_every_code():
    """256 rows (one per E4M3 scale byte) x 32 elements: each 16-element block holds the 16
    codes (the second block in reverse order)."""
    b = np.zeros((256, 2, 9), dtype=np.uint8)
    codes = np.arange(16, dtype=np.uint8)
    for s in range(256):
        for blk, c in enumerate((codes, codes[::-1])):
            b[s, blk, 0] = s
            b[s, blk, 1:] = c[:8] | (c[8:] << 4)
    return b.reshape(1, 256, 2, 9)


@pytest.mark.parametrize("ts", [1.0, 0.0123, -3.5])
def test_nvfp4_exact_decode_every_scale_every_code(env, ts):
    F, torch, dev = env
    blocks = _every_scale_every_code()
    tiles = _tiles(env, blocks, [ts], 1, 256, 32)
    out = torch.full((1, 256, 32), float("nan"), dtype=torch.float32, device=dev)
    F.ftmoe_dequant("nvfp4", tiles, 1, 256, 32, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = oracle.decode_nvfp4(blocks[0], np.float32(ts))[None].astype(np.float32)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert np.all(same)


def test_nvfp4_prefill_operand_every_scale_every_code(env):
    F, torch, dev = env
    blocks = _every_scale_every_code()
    tiles = _tiles(env, blocks, [7.0], 1, 256, 32)
    out = torch.full((1, 256, 32), 0x7FFF, dtype=torch.int16, device=dev)
    F.ftmoe_dequant_operand("nvfp4", F.OPERAND_PREFILL, tiles, 1, 256, 32, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    want = rne_bf16_bits(oracle.decode_nvfp4(blocks[0], 1.0))[None]  # tensor scale not in the operand
    assert np.array_equal(canonical_bf16(got), canonical_bf16(want))
    # every finite E2M1 x E4M3 product is exact in bf16
    ex = oracle.decode_nvfp4(blocks[0], 1.0)
    fin = np.isfinite(ex)
    assert np.array_equal((got[0][fin].astype(np.uint32) << 16).view(np.float32).astype(np.float64), ex[fin])


def _layer(env, L, path=0):
    F, torch, dev = env
    from quantized_expert_ffn_layer_b300 import MoELayer
    from tests._util import bf16_tensor, bf16_to_f64
    m = MoELayer(L.qtype, L.E, L.H, L.I, L.w13, L.w2, L.shared_w13, L.shared_w2, device=dev, ts=L.ts)
    old = F.ftmoe_set_ffn_path(path)
    try:
        ids = torch.empty((L.T, L.k), dtype=torch.int32, device=dev)
        out = m.forward(torch.from_numpy(L.logits).to(dev), bf16_tensor(L.x, dev), L.k, ids_out=ids)
        torch.cuda.synchronize()
    finally:
        F.ftmoe_set_ffn_path(old)
    assert F.ftmoe_device_status() == 0
    return m, bf16_to_f64(out), ids.cpu().numpy()


@pytest.mark.parametrize("T", [1, 4, 64, 256])
def test_nvfp4_decode_layer_parity(env, T):
    c = dict(CONFIGS["decode"])
    c.update(T=T, qtype="nvfp4")
    L = make_layer(**c)
    assert np.all(L.w13_ts > 0) and len(set(L.w13_ts.tolist())) > 1
    _, out, ids = _layer(env, L)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, ts=L.ts)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


@pytest.mark.parametrize("path", [1, 2])
def test_nvfp4_ragged_shared_expert_both_paths(env, path):
    """H = 224, I = 96 (partial tiles, half-filled last slab), a shared expert, several rows
    per expert: grouped GEMV (1) and tcgen05 GEMM (2)."""
    L = make_layer(H=224, I=96, E=5, k=3, T=300, qtype="nvfp4", seed=9, shared=True)
    _, out, ids = _layer(env, L, path)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, L.shared_w13, L.shared_w2, ts=L.ts)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


def test_nvfp4_prefill_layer_sampled(env):
    c = dict(CONFIGS["prefill"])
    c.update(qtype="nvfp4")
    L = make_layer(**c)
    _, out, ids = _layer(env, L)
    rows = np.random.default_rng(2).choice(L.T, size=32, replace=False)
    rids, _, rout = oracle.layer_rows(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, rows, ts=L.ts)
    assert np.array_equal(ids[rows], rids)
    assert rel_l2(out[rows], rout) <= LAYER_TOL


@pytest.mark.parametrize("path", [1, 2])
def test_nvfp4_expert_blob_table(env, path):
    """Cache-slot blobs (w13 tiles + trailer, then w2 tiles + trailer) through a pointer
    table give the same bits as contiguous weights."""
    F, torch, dev = env
    from tests._util import bf16_tensor
    L = make_layer(H=256, I=128, E=8, k=2, T=200, qtype="nvfp4", seed=21)
    m, ref, _ = _layer(env, L, path)
    blobs = torch.cat([m.w13.view(L.E, -1), m.w2.view(L.E, -1)], dim=1).contiguous()
    nb = blobs.shape[1]
    assert nb == F.ftmoe_expert_blob_bytes("nvfp4", L.H, L.I)
    slots = torch.flip(blobs, dims=[0]).contiguous()
    wt = F.make_weights("nvfp4", L.E, L.H, L.I,
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
    from tests._util import bf16_to_f64
    assert np.array_equal(bf16_to_f64(out), ref)
