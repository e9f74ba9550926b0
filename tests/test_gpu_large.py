"""Large MoE layer (hidden 7168, expert intermediate 2048, 256 routed experts top-8 plus an
always-on shared expert, MXFP4, Zipf-skewed routing): one 2048-token prefill chunk (the
tensor-core path) and a 32-token decode step (the grouped-GEMV path), each checked on
sampled tokens against the fp64 oracle.  The 256 experts hold copies of 8 distinct
weight draws so that generating the 6 GB bank stays within a test's time."""
import numpy as np
import pytest

import oracle
from synth import CONFIGS, gen_logits, gen_x_bf16, make_layer
from tests._util import bf16_tensor, bf16_to_f64, ensure_built, rel_l2

pytestmark = pytest.mark.gpu
LAYER_TOL = 1e-2


@pytest.fixture(scope="module")
def large(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import MoELayer
    c = dict(CONFIGS["large"])
    L = make_layer(**c, distinct=8)
    m = MoELayer(L.qtype, L.E, L.H, L.I, L.w13, L.w2, L.shared_w13, L.shared_w2, device=cuda_device)
    yield L, m, torch, cuda_device
    del m
    torch.cuda.empty_cache()


def _run_and_check(L, m, torch, dev, x_bits, logits, nrows, seed):
    T = x_bits.shape[0]
    ids = torch.empty((T, L.k), dtype=torch.int32, device=dev)
    out = m.forward(torch.from_numpy(logits).to(dev), bf16_tensor(x_bits, dev), L.k, ids_out=ids)
    torch.cuda.synchronize()
    got = bf16_to_f64(out)
    rows = np.random.default_rng(seed).choice(T, size=nrows, replace=False)
    rids, _, rout = oracle.layer_rows(x_bits, logits, L.k, L.qtype, L.w13, L.w2, rows,
                                      L.shared_w13, L.shared_w2)
    assert np.array_equal(ids.cpu().numpy()[rows], rids)
    err = rel_l2(got[rows], rout)
    assert err <= LAYER_TOL, err


def test_large_prefill_chunk_sampled(large):
    L, m, torch, dev = large
    _run_and_check(L, m, torch, dev, L.x, L.logits, 8, 3)


def test_large_decode_step_sampled(large):
    L, m, torch, dev = large
    T = CONFIGS["large"]["decode_T"]
    x = gen_x_bf16(0, T, L.H, "decode_x")
    lg = gen_logits(0, T, L.E, zipf=1.0, tag="decode_logits")
    _run_and_check(L, m, torch, dev, x, lg, 8, 4)
