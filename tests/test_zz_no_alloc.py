"""ftmoe_permute_noalloc against ftmoe_permute, through the C ABI.

The no-allocation entry point serves callers that can neither call cudaMalloc nor
hand the library a workspace (a host that owns all device memory in its own fixed
pool, a plugin API without a workspace hook); its scratch is a fixed device array
inside the library.  Its results must be the same as the workspace form's, bit for
bit, and stay so on a second call that reuses the array.  This file is collected
last so that a failure here stops a -x run only after every other test ran.
"""
import numpy as np
import pytest

from synth import gen_logits
from tests._util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    return F, torch, cuda_device


def _ids(T, E, k, seed):
    lg = gen_logits(seed, T, E, zipf=1.0)
    return np.argsort(-lg, axis=1, kind="stable")[:, :k].astype(np.int32)


def _buffers(torch, dev, E, P):
    return (torch.full((E + 1,), -5, dtype=torch.int32, device=dev),
            torch.full((max(P, 1),), -5, dtype=torch.int32, device=dev),
            torch.full((max(P, 1),), -5, dtype=torch.int32, device=dev))


# (T, E, k): single-CTA size, just past it, the prefill size, exactly at the scratch limit
@pytest.mark.parametrize("T,E,k", [(64, 128, 8), (2049, 128, 8), (4096, 128, 8), (32768, 1024, 8)])
def test_noalloc_matches_workspace_form_twice(env, T, E, k):
    F, torch, dev = env
    P = T * k
    ids = torch.from_numpy(_ids(T, E, k, 3)).to(dev)
    off, sp, inv = _buffers(torch, dev, E, P)
    nws = F.ftmoe_permute_workspace_bytes(T, k, E)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    F.ftmoe_permute(ids, T, k, E, off, sp, inv, ws, nws)
    torch.cuda.synchronize()
    want = [t.cpu().numpy() for t in (off, sp, inv)]
    for call in range(2):
        # a different problem in between must not leak into the next call's result
        other = torch.from_numpy(_ids(T, E, k, 100 + call)).to(dev)
        o2, s2, i2 = _buffers(torch, dev, E, P)
        F.ftmoe_permute_noalloc(other, T, k, E, o2, s2, i2)
        off_n, sp_n, inv_n = _buffers(torch, dev, E, P)
        F.ftmoe_permute_noalloc(ids, T, k, E, off_n, sp_n, inv_n)
        torch.cuda.synchronize()
        got = [t.cpu().numpy() for t in (off_n, sp_n, inv_n)]
        for g, w in zip(got, want):
            assert np.array_equal(g, w), f"call {call}"
    assert F.ftmoe_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_fixed_scratch(env):
    F, torch, dev = env
    # ceil(300000 * 8 / 1024) * 1024 experts > 262144 entries
    T, k, E = 300000, 8, 1024
    off, sp, inv = _buffers(torch, dev, E, 16)
    with pytest.raises(F.FtmoeError) as ei:
        F.ftmoe_permute_noalloc(sp, T, k, E, off, sp, inv)
    assert ei.value.status == 7  # FTMOE_ERR_WORKSPACE: nothing was enqueued
    torch.cuda.synchronize()
