"""Test helpers: build-on-demand of libftmoe, device upload of synthetic inputs, metrics."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ftmoe.h")


def ensure_built():
    from quantized_expert_ffn_layer_b300.build import build
    return build()


def header_functions():
    """Names of the functions ftmoe.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ftmoe_[a-z0-9_]+)\s*\(", src)))


def rel_l2(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def bf16_tensor(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_f64(t):
    import torch
    return t.detach().to("cpu").view(torch.int16).numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)
