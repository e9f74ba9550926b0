"""GPU parity: every libftmoe kernel against the fp64 oracle on the same seeded inputs.

Integer work (decode of the 4-bit formats, expert ids, permutation) must be
bit-exact; floating-point outputs must match within the layer tolerance
(rel-L2 <= 1e-2 on bf16 activations; observed ~3e-3 from bf16 rounding of h, y
and out) and the router weights within fp32 rounding (1e-6 relative).
"""
import struct

import numpy as np
import pytest

import oracle
from synth import CONFIGS, gen_logits, gen_x_bf16, make_layer
from tests._util import bf16_tensor, bf16_to_f64, ensure_built, rel_l2

pytestmark = pytest.mark.gpu

LAYER_TOL = 1e-2
W_RTOL = 1e-6


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    return F, torch, cuda_device


def _same_f32(got, want64):
    """got (fp32) equals the exact fp64 decode, where a value of magnitude >= 2^128 (MXFP4
    codes times 2^127 or 2^126 at E8M0 254 / 253 ... beyond fp32) is expected as +-inf:
    every decoded weight is either exact in fp32 or at least 2^128, so the fp32 result of
    the kernel's exact product is the value itself or an overflow to infinity."""
    want64 = np.asarray(want64, dtype=np.float64)
    over = np.isfinite(want64) & (np.abs(want64) >= 2.0 ** 128)
    want = np.where(over, np.copysign(np.inf, want64), np.where(over, 0.0, want64)).astype(np.float32)
    got = np.asarray(got, dtype=np.float32)
    nan = np.isnan(got) & np.isnan(want)
    return np.all(nan | (got.view(np.uint32) == want.view(np.uint32)))


# ------------------------------------------------------------------ dequant / repack
def _dequant_gpu(env, qtype, canon, E, N, K):
    F, torch, dev = env
    src = torch.from_numpy(canon.reshape(-1).copy()).to(dev)
    tiles = torch.empty(F.ftmoe_tiled_bytes(qtype, E, N, K), dtype=torch.uint8, device=dev)
    F.ftmoe_repack(qtype, src, tiles, E, N, K)
    out = torch.full((E, N, K), float("nan"), dtype=torch.float32, device=dev)
    F.ftmoe_dequant(qtype, tiles, E, N, K, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


Q_OF_ELEM = list(range(16)) + [15 - i for i in range(16)]


def _codes16():
    return bytes((Q_OF_ELEM[i] & 15) | ((Q_OF_ELEM[i + 16] & 15) << 4) for i in range(16))


def test_q4_0_decode_every_scale_every_code(env):
    raw = bytearray()
    for bits in range(65536):
        raw += struct.pack("<H", bits) + _codes16()
    canon = np.frombuffer(bytes(raw), dtype=np.uint8).reshape(1, 2048, 32, 18)
    got = _dequant_gpu(env, "q4_0", canon, 1, 2048, 1024)
    assert _same_f32(got, oracle.decode_q4_0(canon))


def test_mxfp4_decode_every_scale_every_code(env):
    raw = bytearray()
    for e in range(256):
        raw += bytes([e]) + _codes16()
    canon = np.frombuffer(bytes(raw), dtype=np.uint8).reshape(1, 16, 16, 17)
    got = _dequant_gpu(env, "mxfp4", canon, 1, 16, 512)
    assert _same_f32(got, oracle.decode_mxfp4(canon))


@pytest.mark.parametrize("qtype,E,N,K", [("q4_0", 3, 48, 96), ("mxfp4", 2, 32, 160), ("q4_0", 2, 16, 2048),
                                         ("mxfp4", 1, 64, 7168)])
def test_random_blocks_every_position(env, qtype, E, N, K):
    rng = np.random.default_rng(E * N + K)
    blk = 18 if qtype == "q4_0" else 17
    canon = rng.integers(0, 256, size=(E, N, K // 32, blk), dtype=np.uint8)
    if qtype == "q4_0":
        canon[..., 1] &= 0x7B  # finite fp16 scales
    got = _dequant_gpu(env, qtype, canon, E, N, K)
    assert _same_f32(got, oracle.decode_blocks(canon, qtype))


# ------------------------------------------------------------------ route
def _route_gpu(env, logits, k):
    F, torch, dev = env
    T, E = logits.shape
    lg = torch.from_numpy(logits).to(dev)
    ids = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    w = torch.zeros((T, k), dtype=torch.float32, device=dev)
    F.ftmoe_route(lg, T, E, k, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,k,zipf", [(64, 8, 2, 0.0), (1, 128, 8, 0.0), (333, 128, 8, 0.0),
                                        (4096, 128, 8, 1.0), (257, 256, 8, 1.0), (50, 1000, 32, 0.0),
                                        (20, 3, 3, 0.0), (9, 33, 1, 0.0)])
def test_route_matches_oracle(env, T, E, k, zipf):
    lg = gen_logits(11, T, E, zipf=zipf)
    ids, w = _route_gpu(env, lg, k)
    rids, rw = oracle.route(lg, k)
    assert np.array_equal(ids, rids)
    assert np.allclose(w, rw, rtol=W_RTOL, atol=1e-7)


def test_route_ties_go_to_lower_id(env):
    lg = np.zeros((5, 64), dtype=np.float32)
    lg[0, [3, 7, 40]] = 1.0
    lg[1, :] = 2.0
    lg[2, ::3] = -1.0
    lg[3, 63] = 5.0
    lg[3, 31] = 5.0
    lg[4, 32:] = 0.5
    for k in (1, 3, 8):
        ids, w = _route_gpu(env, lg, k)
        rids, rw = oracle.route(lg, k)
        assert np.array_equal(ids, rids)
        assert np.allclose(w, rw, rtol=W_RTOL)


# ------------------------------------------------------------------ permute
def _permute_gpu(env, ids, E):
    F, torch, dev = env
    T, k = ids.shape
    P = T * k
    d_ids = torch.from_numpy(ids.astype(np.int32)).to(dev)
    off = torch.full((E + 1,), -5, dtype=torch.int32, device=dev)
    sp = torch.full((max(P, 1),), -5, dtype=torch.int32, device=dev)
    inv = torch.full((max(P, 1),), -5, dtype=torch.int32, device=dev)
    nws = F.ftmoe_permute_workspace_bytes(T, k, E)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    F.ftmoe_permute(d_ids, T, k, E, off, sp, inv, ws, nws)
    torch.cuda.synchronize()
    assert F.ftmoe_device_status() == 0
    return off.cpu().numpy(), sp.cpu().numpy()[:P], inv.cpu().numpy()[:P]


@pytest.mark.parametrize("T,E,k", [(1, 128, 8), (64, 8, 2), (64, 128, 8), (2048, 8, 8), (2049, 128, 8),
                                   (4096, 128, 8), (2048, 256, 8), (1000, 1024, 32), (3000, 3, 2)])
def test_permute_matches_oracle(env, T, E, k):
    lg = gen_logits(5, T, E, zipf=1.0)
    ids, _ = oracle.route(lg, k)
    off, sp, inv = _permute_gpu(env, ids, E)
    r_off, r_sp, r_inv = oracle.permute(ids, E)
    assert np.array_equal(off, r_off)
    assert np.array_equal(sp, r_sp)
    assert np.array_equal(inv, r_inv)


def test_permute_empty(env):
    off, sp, inv = _permute_gpu(env, np.zeros((0, 4), np.int32), 16)
    assert off.tolist() == [0] * 17


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("T,k,H,shared", [(64, 2, 256, False), (37, 8, 2048, True), (5, 1, 7168, True)])
def test_combine_matches_oracle(env, T, k, H, shared):
    F, torch, dev = env
    rng = np.random.default_rng(T + k + H)
    P = T * k
    ybits = gen_x_bf16(3, P, H)
    perm = rng.permutation(P).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    sh = gen_x_bf16(4, T, H) if shared else None
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    F.ftmoe_combine(bf16_tensor(ybits, dev), torch.from_numpy(w).to(dev), torch.from_numpy(perm).to(dev),
                    bf16_tensor(sh, dev) if shared else None, T, k, H, out)
    torch.cuda.synchronize()
    f64 = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    want = oracle.combine(f64(ybits), w.astype(np.float64), perm, f64(sh) if shared else None)
    got = bf16_to_f64(out)
    # fp32 accumulation then one bf16 rounding: within 2^-8 relative per element
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30)


# ------------------------------------------------------------------ layer
def _layer_gpu(env, L, path=0):
    F, torch, dev = env
    from quantized_expert_ffn_layer_b300 import MoELayer
    m = MoELayer(L.qtype, L.E, L.H, L.I, L.w13, L.w2, L.shared_w13, L.shared_w2, device=dev, ts=L.ts)
    old = F.ftmoe_set_ffn_path(path)
    try:
        T = L.T
        ids = torch.empty((T, L.k), dtype=torch.int32, device=dev)
        w = torch.empty((T, L.k), dtype=torch.float32, device=dev)
        out = m.forward(torch.from_numpy(L.logits).to(dev), bf16_tensor(L.x, dev), L.k,
                        ids_out=ids, w_out=w)
        torch.cuda.synchronize()
    finally:
        F.ftmoe_set_ffn_path(old)
    assert F.ftmoe_device_status() == 0
    return m, bf16_to_f64(out), ids.cpu().numpy(), w.cpu().numpy()


def test_tiny_layer_full_parity(env):
    c = dict(CONFIGS["tiny"])
    L = make_layer(**c)
    _, out, ids, w = _layer_gpu(env, L)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    assert np.array_equal(ids, r["ids"])
    assert np.allclose(w, r["w"], rtol=W_RTOL)
    err = rel_l2(out, r["out"])
    assert err <= LAYER_TOL, err


@pytest.mark.parametrize("qtype", ["q4_0", "mxfp4"])
@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_decode_layer_parity(env, qtype, T):
    c = dict(CONFIGS["decode"])
    c.update(T=T, qtype=qtype)
    L = make_layer(**c)
    _, out, ids, w = _layer_gpu(env, L)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    assert np.array_equal(ids, r["ids"])
    err = rel_l2(out, r["out"])
    assert err <= LAYER_TOL, err


@pytest.mark.parametrize("qtype", ["q4_0", "mxfp4"])
@pytest.mark.parametrize("T", [128, 256])
def test_decode_layer_parity_mid_batches(env, qtype, T):
    """Decode layer shape at 8 to 16 rows per expert, where the default path is the
    tcgen05 decode GEMM (8 E <= T k < 32 E): every output against the oracle."""
    c = dict(CONFIGS["decode"])
    c.update(T=T, qtype=qtype)
    assert 8 * c["E"] <= T * c["k"] < 32 * c["E"]
    L = make_layer(**c)
    _, out, ids, _ = _layer_gpu(env, L)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    assert np.array_equal(ids, r["ids"])
    err = rel_l2(out, r["out"])
    assert err <= LAYER_TOL, err


def test_ragged_shapes_and_shared_expert(env):
    # H, I multiples of 32 but not 64 (ragged last record), several token groups per expert
    L = make_layer(H=224, I=96, E=5, k=3, T=77, qtype="mxfp4", seed=9, shared=True)
    _, out, ids, _ = _layer_gpu(env, L)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, L.shared_w13, L.shared_w2)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


@pytest.mark.parametrize("path", [1, 3])
def test_decode_batch_invariance(env, path):
    """A token's output does not depend on the other tokens of the batch (bit-exact),
    for the mma.sync grouped GEMV (1) and the tensor-memory tcgen05 decode GEMM (3)."""
    c = dict(CONFIGS["decode"])
    c.update(T=64)
    L = make_layer(**c)
    F, torch, dev = env
    m, out64, _, _ = _layer_gpu(env, L, path=path)
    for t in (0, 17, 63):
        x1 = bf16_tensor(L.x[t:t + 1], dev)
        lg1 = torch.from_numpy(L.logits[t:t + 1].copy()).to(dev)
        old = F.ftmoe_set_ffn_path(path)
        o1 = m.forward(lg1, x1, L.k)
        F.ftmoe_set_ffn_path(old)
        assert np.array_equal(bf16_to_f64(o1)[0], out64[t])


@pytest.mark.parametrize("qtype", ["q4_0", "mxfp4"])
def test_gemm_decode_path_ragged_shared_and_multi_tile(env, qtype):
    """Decode GEMM on ragged H / I (partial 128-row tiles, half-filled last block), a shared
    expert, and experts with more rows than one token tile."""
    L = make_layer(H=224, I=96, E=5, k=3, T=60, qtype=qtype, seed=13, shared=True, zipf=1.0)
    _, out, ids, _ = _layer_gpu(env, L, path=3)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, L.shared_w13, L.shared_w2)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


@pytest.mark.parametrize("qtype", ["q4_0", "mxfp4"])
def test_prefill_layer_sampled_parity(env, qtype):
    c = dict(CONFIGS["prefill"])
    c.update(qtype=qtype)
    L = make_layer(**c)
    _, out, ids, _ = _layer_gpu(env, L)
    rows = np.random.default_rng(1).choice(L.T, size=48, replace=False)
    rids, _, rout = oracle.layer_rows(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, rows)
    assert np.array_equal(ids[rows], rids)
    assert rel_l2(out[rows], rout) <= LAYER_TOL


# ------------------------------------------------------------------ tensor-core grouped GEMM
@pytest.mark.parametrize("qtype", ["q4_0", "mxfp4"])
@pytest.mark.parametrize("T", [64, 300])
def test_gemm_path_decode_shape_full_parity(env, qtype, T):
    """The tcgen05 path on the decode layer shape: few rows per expert (narrow MMA N)."""
    c = dict(CONFIGS["decode"])
    c.update(T=T, qtype=qtype)
    L = make_layer(**c)
    _, out, ids, _ = _layer_gpu(env, L, path=2)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


@pytest.mark.parametrize("qtype", ["q4_0", "mxfp4"])
def test_gemm_path_several_token_tiles_per_expert(env, qtype):
    """Experts with 300-400 rows: two 256-row token tiles each, the second one ragged."""
    L = make_layer(H=256, I=128, E=4, k=2, T=700, qtype=qtype, seed=4, zipf=0.5)
    _, out, ids, _ = _layer_gpu(env, L, path=2)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL
    # per-row check too: every row of the output within tolerance, not only on average
    num = np.linalg.norm(out - r["out"], axis=1)
    den = np.linalg.norm(r["out"], axis=1)
    assert np.all(num <= 2e-2 * den)


def test_gemm_path_ragged_shapes_and_shared_expert(env):
    """H = 224, I = 96: partial 128-row weight tiles and a half-filled last reduction block."""
    L = make_layer(H=224, I=96, E=5, k=3, T=300, qtype="mxfp4", seed=9, shared=True)
    _, out, ids, _ = _layer_gpu(env, L, path=2)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, L.shared_w13, L.shared_w2)
    assert np.array_equal(ids, r["ids"])
    assert rel_l2(out, r["out"]) <= LAYER_TOL


@pytest.mark.parametrize("path", [1, 2, 3])
def test_expert_blob_table_matches_contiguous_weights(env, path):
    """Weights reached through a per-expert pointer table (cache slots) give the same bits."""
    F, torch, dev = env
    from quantized_expert_ffn_layer_b300 import MoELayer
    L = make_layer(H=256, I=128, E=8, k=2, T=200, qtype="q4_0", seed=21)
    m = MoELayer(L.qtype, L.E, L.H, L.I, L.w13, L.w2, device=dev)
    blobs = torch.cat([m.w13.view(L.E, -1), m.w2.view(L.E, -1)], dim=1).contiguous()
    nb = blobs.shape[1]
    assert nb == F.ftmoe_expert_blob_bytes(L.qtype, L.H, L.I)
    # reverse the slot order so that the table is not the identity layout
    slots = torch.flip(blobs, dims=[0]).contiguous()
    ptrs = [slots.data_ptr() + (L.E - 1 - e) * nb for e in range(L.E)]
    wt = F.make_weights(L.qtype, L.E, L.H, L.I, expert_blob=ptrs)
    lg = torch.from_numpy(L.logits).to(dev)
    x = bf16_tensor(L.x, dev)
    old = F.ftmoe_set_ffn_path(path)
    try:
        ref = m.forward(lg, x, L.k)
        ws = m.workspace(L.T, L.k)
        out = torch.empty_like(ref)
        F.ftmoe_layer(wt, lg, x, L.T, L.k, out, None, None, ws, ws.numel())
        torch.cuda.synchronize()
    finally:
        F.ftmoe_set_ffn_path(old)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
