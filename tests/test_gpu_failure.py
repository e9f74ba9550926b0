"""Failure detection on the GPU without a GPU fault.

A bounded wait that runs out (a barrier nothing arrives on) must end in the
wait-ran-out code in the device status word with the kernel returning normally, and
the context must stay usable: the next call still gives the oracle's result.  An
out-of-range expert id must be reported in the status word and skipped, while every
valid pair is still grouped exactly as the definition says.
"""
import numpy as np
import pytest

import oracle
from synth import gen_logits
from tests._util import ensure_built

pytestmark = pytest.mark.gpu

DEV_BAD_EXPERT_ID, DEV_WAIT_TIMEOUT = 1, 2


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    F.ftmoe_device_status()  # start from a clear status word
    return F, torch, cuda_device


def _permute(F, torch, dev, ids, E, k):
    T = ids.shape[0]
    P = T * k
    ids_d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(dev)
    offs = torch.full((E + 1,), -5, dtype=torch.int32, device=dev)
    sp = torch.full((P,), -5, dtype=torch.int32, device=dev)
    inv = torch.full((P,), -5, dtype=torch.int32, device=dev)
    n = F.ftmoe_permute_workspace_bytes(T, k, E)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    F.ftmoe_permute(ids_d, T, k, E, offs, sp, inv, ws, n)
    torch.cuda.synchronize()
    return offs.cpu().numpy(), sp.cpu().numpy(), inv.cpu().numpy()


def test_wait_that_runs_out_reports_status_and_context_survives(env):
    F, torch, dev = env
    waited = torch.full((1,), 7, dtype=torch.int32, device=dev)
    F.ftmoe_check_wait_timeout(2_000_000, waited)  # 2 ms
    torch.cuda.synchronize()
    assert int(waited.item()) == 0
    assert F.ftmoe_device_status() == DEV_WAIT_TIMEOUT
    assert F.ftmoe_device_status() == 0  # reading clears it
    # the context still works: a permutation equals the oracle's, status stays clear
    T, E, k = 64, 128, 8
    lg = gen_logits(5, T, E, zipf=1.0)
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :k].astype(np.int32)
    offs, sp, inv = _permute(F, torch, dev, ids, E, k)
    want = oracle.permute(ids, E)
    assert np.array_equal(offs, want[0]) and np.array_equal(sp, want[1]) and np.array_equal(inv, want[2])
    assert F.ftmoe_device_status() == 0


def test_wait_limit_outside_range_is_rejected_on_the_host(env):
    F, torch, dev = env
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(F.FtmoeError) as ei:
            F.ftmoe_check_wait_timeout(bad)
        assert ei.value.status == 1  # FTMOE_ERR_INVALID_ARG
    assert F.ftmoe_device_status() == 0


@pytest.mark.parametrize("T", [16, 4096])  # single-CTA and multi-CTA permutation
def test_out_of_range_expert_id_is_reported_and_skipped(env, T):
    F, torch, dev = env
    E, k = 128, 8
    lg = gen_logits(9, T, E, zipf=1.0)
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :k].astype(np.int32)
    ids[3, 2] = E
    ids[T - 1, 0] = -1
    offs, sp, inv = _permute(F, torch, dev, ids, E, k)
    assert F.ftmoe_device_status() & DEV_BAD_EXPERT_ID
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    nv = int(valid.sum())
    assert nv == T * k - 2
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(np.bincount(flat[valid], minlength=E))]))
    # the valid pairs, grouped by expert and ascending within a group
    pairs = np.nonzero(valid)[0]
    want_sp = pairs[np.argsort(flat[pairs], kind="stable")]
    assert np.array_equal(sp[:nv], want_sp)
    assert np.array_equal(inv[want_sp], np.arange(nv))
    assert F.ftmoe_device_status() == 0
