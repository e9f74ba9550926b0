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


def rne_bf16_bits(x):
    """bf16 bit patterns (uint16) of float64 values rounded once to the nearest bf16, ties
    to even: the spacing of bf16 numbers at |x| is 2^(max(floor(log2|x|), -126) - 7) (8
    significant bits, subnormals below 2^-126); a result of magnitude >= 2^128 is +-inf;
    NaN -> the quiet NaN 0x7FC0.  Written from the definition (numpy's rint rounds half to
    even); every bf16 value is an fp32 value, so the bits are the top half of its fp32."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    a = np.abs(x)
    fin = np.isfinite(x) & (a > 0)
    _, ex = np.frexp(a[fin])                       # a = f * 2^ex, f in [0.5, 1)
    ulp = np.exp2(np.maximum(ex - 1, -126) - 7)
    v = np.rint(a[fin] / ulp) * ulp
    with np.errstate(over="ignore"):
        bits = (np.where(v >= 2.0 ** 128, np.inf, v).astype(np.float32).view(np.uint32) >> 16)
    out[fin] = bits.astype(np.uint16)
    out[np.isinf(x)] = 0x7F80
    out[np.isnan(x)] = 0x7FC0
    out |= np.where(np.signbit(x) & ~np.isnan(x), np.uint16(0x8000), np.uint16(0))
    return out


def canonical_bf16(bits):
    """bf16 bit patterns with every NaN mapped to 0x7FC0 and -0 to +0, so that an equality
    test compares values (IEEE zero signs and NaN payloads carry no value)."""
    b = np.asarray(bits, dtype=np.uint16).copy()
    nan = ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
    b[nan] = 0x7FC0
    b[b == 0x8000] = 0
    return b
