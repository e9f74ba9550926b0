"""fp64 CPU oracle of the quantized MoE expert layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product path (``quantized_expert_ffn_layer_b300``) never touches it; the two share
no code.  Every function is the plain definition of one stage written out in
numpy fp64, with no blocking, fusion or reordering beyond what the definition
states, so that it can be checked against the definitions by eye.

Sources (page title, section):

* [P5] "深入FreeToken架构从HTTP API到CUDA内核的本地MoE推理引擎全链路剖析",
  §五 (MoE engine: ExpertFFN banks in GGUF Q4_0 / MXFP4, pinned-host cold
  experts, global LRU, double-buffered prefill) and §六 (GGUF dequant + Q4_0 MoE
  kernels, pinned tensors, batched async copies).
* [P3] "从双缓冲 Prefill、带宽自适应 CPU–GPU 协同到 Agent 状态复用…", 机制一
  (full-layer double buffering) and 机制四 (global LRU expert cache); also
  "为什么 MoE 模型适合做 CPU–GPU 协同" (only a subset of experts is active per token).
* [P4] "FreeToken：高效的边缘原生 MoE 服务与带宽自适应执行", 方法 (pipelined
  loading; expert caching) and 核心洞察 (CUDA-graph-compatible LRU).
* [P1] "FreeToken：在桌面运行大规模模型的本地推理引擎", 开源生态中的位置
  (GGUF is llama.cpp's quantized format).
* OCP Microscaling Formats (MX) v1.0 for the E2M1 element and E8M0 scale encodings.

The pages only name the stages; where they leave a step open the oracle takes
the plain reading listed in each function's docstring.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, exhaustive enumeration, library routines or brute force.
"""
from .formats import (decode_blocks, decode_mxfp4, decode_mxfp8, decode_nvfp4,  # noqa: F401
                      decode_q4_0, e2m1_value, e4m3_value, e8m0_scale)
from .route import route  # noqa: F401
from .permute import permute  # noqa: F401
from .ffn import combine, expert_ffn, silu, swiglu_ffn  # noqa: F401
from .layer import layer, layer_rows  # noqa: F401
from .cache import LRUSim  # noqa: F401
from .gate import gate  # noqa: F401
