"""Router gate: expert logits from the hidden state (fp64).

The step right before the router: each token's hidden vector x (bf16) is scored
against every expert's gate vector, logits[t, e] = sum over h of x[t, h] * Wg[e, h].
The pages describe MoE routing only by what it selects ([P3] "为什么 MoE 模型适合做
CPU–GPU 协同": a few experts per token), not the gate itself, so the oracle takes
the plain reading: a bias-free linear map H -> E with the gate matrix Wg stored as
E rows of H bf16 values (the same orientation as the expert weights, the reduction
dimension last).  The product is exact in fp64 up to the matmul's rounding, which is
far below the fp32 result it is compared with.
"""
from __future__ import annotations

import numpy as np


def _bf16_fp64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def gate(x_bits: np.ndarray, wg_bits: np.ndarray) -> np.ndarray:
    """x_bits uint16 bf16 [T, H], wg_bits uint16 bf16 [E, H] -> logits fp64 [T, E]."""
    x = _bf16_fp64(x_bits)
    wg = _bf16_fp64(wg_bits)
    if x.ndim != 2 or wg.ndim != 2 or x.shape[1] != wg.shape[1]:
        raise ValueError("need x [T, H] and wg [E, H]")
    return x @ wg.T
