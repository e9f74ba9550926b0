"""Quantized MoE expert layer for NVIDIA B300 (sm_103a): libftmoe and its binding.

``ftmoe`` mirrors the C ABI of ``include/ftmoe.h`` (ctypes, argument
marshalling only); ``layer`` holds device-resident weights and workspaces for
repeated calls.  All arithmetic runs in libftmoe's CUDA kernels.
"""
from . import ftmoe  # noqa: F401  (raises ImportError when libftmoe.so is missing)
from .layer import MoELayer  # noqa: F401
