"""Run by tests/test_gpu_checks.py in a child process with FTMOE_LIBRARY=checks, so that
the binding loads libftmoe_checks.so (every FFN and combine kernel bound-checks the
indices it reads).  Exits 0 when every case holds; prints what failed otherwise."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from synth import make_layer  # noqa: E402
from tests._util import bf16_tensor, bf16_to_f64, rel_l2  # noqa: E402
from quantized_expert_ffn_layer_b300 import MoELayer  # noqa: E402
from quantized_expert_ffn_layer_b300 import ftmoe as F  # noqa: E402

assert os.path.basename(F.LIB_PATH) == "libftmoe_checks.so", F.LIB_PATH
dev = torch.device("cuda:0")
TOL = 1e-2


def layer_case(L, path):
    m = MoELayer(L.qtype, L.E, L.H, L.I, L.w13, L.w2, L.shared_w13, L.shared_w2, device=dev, ts=L.ts)
    old = F.ftmoe_set_ffn_path(path)
    out = m.forward(torch.from_numpy(L.logits).to(dev), bf16_tensor(L.x, dev), L.k)
    torch.cuda.synchronize()
    F.ftmoe_set_ffn_path(old)
    r = oracle.layer(L.x, L.logits, L.k, L.qtype, L.w13, L.w2, L.shared_w13, L.shared_w2, ts=L.ts)
    err = rel_l2(bf16_to_f64(out), r["out"])
    st = F.ftmoe_device_status()
    assert st == 0 and err <= TOL, (L.qtype, L.T, path, st, err)


def malformed_case(path, qtype):
    """ftmoe_expert_ffn with host-made tables: offsets[E] beyond P (the last expert's rows
    run past the pairs) and one sorted_pair entry outside [0, T k).  The checks build
    clamps the rows to [0, P), reads token 0 for the bad pair, reports DEV_BAD_INDEX (8),
    and every other row equals the oracle's."""
    L = make_layer(H=256, I=128, E=8, k=2, T=100, qtype=qtype, seed=17)
    E, k, T, H, I = L.E, L.k, L.T, L.H, L.I
    P = T * k
    ids, _ = oracle.route(L.logits, k)
    offsets, sorted_pair, _ = oracle.permute(ids, E)
    bad_row = int(offsets[3]) + 1
    sp = sorted_pair.astype(np.int32).copy()
    sp[bad_row] = P + 7
    off = offsets.astype(np.int32).copy()
    off[E] = P + 100
    m = MoELayer(L.qtype, E, H, I, L.w13, L.w2, device=dev, ts=L.ts)
    ws_n = F.ftmoe_ffn_workspace_bytes(T, k, E, H, I)
    ws = torch.zeros(max(ws_n, 256), dtype=torch.uint8, device=dev)
    y = torch.zeros((P, H), dtype=torch.bfloat16, device=dev)
    old = F.ftmoe_set_ffn_path(path)
    F.ftmoe_expert_ffn(m.weights, bf16_tensor(L.x, dev), T, k, torch.from_numpy(off).to(dev),
                       torch.from_numpy(sp).to(dev), y, ws, ws_n)
    torch.cuda.synchronize()
    F.ftmoe_set_ffn_path(old)
    st = F.ftmoe_device_status()
    assert st & 8, (path, qtype, st)
    from oracle.formats import decode_blocks
    x = (L.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ts = L.ts or {"w13": [None] * E, "w2": [None] * E}
    want = oracle.expert_ffn(x, k, offsets, sorted_pair, lambda e: decode_blocks(L.w13[e], qtype, ts["w13"][e]),
                             lambda e: decode_blocks(L.w2[e], qtype, ts["w2"][e]))
    got = bf16_to_f64(y)
    keep = np.ones(P, dtype=bool)
    keep[bad_row] = False
    assert rel_l2(got[keep], want[keep]) <= TOL, (path, qtype, rel_l2(got[keep], want[keep]))


def main():
    F.ftmoe_device_status()
    layer_case(make_layer(H=256, I=128, E=8, k=2, T=64, qtype="q4_0", seed=0), 0)
    layer_case(make_layer(H=224, I=96, E=5, k=3, T=77, qtype="mxfp4", seed=9, shared=True), 1)
    layer_case(make_layer(H=224, I=96, E=5, k=3, T=300, qtype="q4_0", seed=9, shared=True), 2)
    layer_case(make_layer(H=224, I=96, E=5, k=3, T=60, qtype="mxfp4", seed=13, shared=True), 3)
    layer_case(make_layer(H=224, I=96, E=5, k=3, T=90, qtype="nvfp4", seed=3, shared=True), 0)
    for path in (1, 2, 3):
        malformed_case(path, "q4_0")
    malformed_case(1, "nvfp4")
    print("checks ok")


if __name__ == "__main__":
    main()
