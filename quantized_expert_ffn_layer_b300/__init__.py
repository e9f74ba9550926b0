"""Quantized MoE expert layer for NVIDIA B300 (sm_103a): libftmoe and its binding.

``ftmoe`` mirrors the C ABI of ``include/ftmoe.h`` (ctypes, argument
marshalling only); ``layer`` holds device-resident weights and workspaces for
repeated calls.  All arithmetic runs in libftmoe's CUDA kernels; importing
``ftmoe`` (directly or through ``MoELayer``) raises ImportError when
libftmoe.so has not been built (``python -m quantized_expert_ffn_layer_b300.build``).
"""


import importlib


def __getattr__(name):
    if name == "ftmoe":
        return importlib.import_module(__name__ + ".ftmoe")
    if name == "MoELayer":
        return importlib.import_module(__name__ + ".layer").MoELayer
    raise AttributeError(name)
