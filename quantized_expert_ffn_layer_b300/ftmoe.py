"""Thin ctypes binding of libftmoe (include/ftmoe.h).

Functions carry the C names and arguments; the only work done here is argument
marshalling: torch tensors become device/host pointers, ``stream=None`` becomes
torch's current CUDA stream, and a non-OK status raises :class:`FtmoeError`.
Every step of the layer runs in the library's CUDA kernels; there is no other
implementation to fall back to, and importing this module fails loudly when the
shared library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# FTMOE_LIBRARY=checks selects the bounds-checking build (libftmoe_checks.so)
LIB_PATH = os.path.join(_HERE, "libftmoe_checks.so" if os.environ.get("FTMOE_LIBRARY") == "checks"
                        else "libftmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libftmoe.so not found at {LIB_PATH}; build it with "
        "`python -m quantized_expert_ffn_layer_b300.build`")

lib = C.CDLL(LIB_PATH)

FTMOE_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "NO_SLOT",
                5: "TIMEOUT", 6: "DEVICE_CHECK", 7: "WORKSPACE"}
Q4_0, MXFP4, NVFP4, MXFP8 = 1, 2, 3, 4
QTYPES = {"q4_0": Q4_0, "mxfp4": MXFP4, "nvfp4": NVFP4, "mxfp8": MXFP8}
PATH_AUTO, PATH_GEMV, PATH_GEMM, PATH_GEMM_DECODE = 0, 1, 2, 3
OPERAND_PREFILL, OPERAND_CODES = 0, 1
LRU_PER_LAYER, LRU_GLOBAL = 0, 1


class FtmoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = lib.ftmoe_status_string(status).decode()
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({msg})")


class ftmoe_weights(C.Structure):
    _fields_ = [("qtype", C.c_int), ("E", C.c_int), ("H", C.c_int), ("I", C.c_int),
                ("w13", C.c_void_p), ("w2", C.c_void_p),
                ("expert_blob", C.POINTER(C.c_void_p)),
                ("shared_w13", C.c_void_p), ("shared_w2", C.c_void_p)]


class ftmoe_cache_desc(C.Structure):
    _fields_ = [("layers", C.c_int), ("E", C.c_int), ("blob_bytes", C.c_size_t),
                ("bank", C.c_void_p), ("pool", C.c_void_p), ("slots_per_layer", C.c_int),
                ("policy", C.c_int), ("copy_stream", C.c_void_p)]


class ftmoe_cache_stats(C.Structure):
    _fields_ = [("lookups", C.c_uint64), ("hits", C.c_uint64), ("misses", C.c_uint64),
                ("prefetch_lookups", C.c_uint64), ("prefetch_copies", C.c_uint64),
                ("h2d_bytes", C.c_uint64), ("h2d_ms", C.c_double)]


_vp, _i, _sz = C.c_void_p, C.c_int, C.c_size_t
_SIGS = {
    "ftmoe_status_string": (C.c_char_p, [_i]),
    "ftmoe_version": (_i, []),
    "ftmoe_tiled_bytes": (_sz, [_i, _i, _i, _i]),
    "ftmoe_repack": (_i, [_i, _vp, _vp, _i, _i, _i, _vp]),
    "ftmoe_dequant": (_i, [_i, _vp, _i, _i, _i, _vp, _vp]),
    "ftmoe_dequant_operand": (_i, [_i, _i, _vp, _i, _i, _i, _vp, _vp]),
    "ftmoe_route": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp]),
    "ftmoe_permute_workspace_bytes": (_sz, [_i, _i, _i]),
    "ftmoe_permute": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ftmoe_permute_noalloc": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "ftmoe_expert_blob_bytes": (_sz, [_i, _i, _i]),
    "ftmoe_ffn_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "ftmoe_layer_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "ftmoe_expert_ffn": (_i, [C.POINTER(ftmoe_weights), _vp, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ftmoe_set_ffn_path": (_i, [_i]),
    "ftmoe_combine": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
    "ftmoe_layer": (_i, [C.POINTER(ftmoe_weights), _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ftmoe_device_status": (_i, [C.POINTER(_i), _vp]),
    "ftmoe_check_wait_timeout": (_i, [C.c_longlong, _vp, _vp]),
    "ftmoe_gate": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "ftmoe_cache_create": (_i, [C.POINTER(ftmoe_cache_desc), C.POINTER(_vp)]),
    "ftmoe_cache_prefetch": (_i, [_vp, _i, _vp, _i, _vp, _vp]),
    "ftmoe_cache_acquire": (_i, [_vp, _i, _vp, _i, _vp, C.POINTER(_vp), _vp, _vp]),
    "ftmoe_cache_prefetch_history": (_i, [_vp, _i, _vp, C.POINTER(_i), _vp, _vp]),
    "ftmoe_cache_release": (_i, [_vp, _i, _vp]),
    "ftmoe_cache_stats_get": (_i, [_vp, C.POINTER(ftmoe_cache_stats)]),
    "ftmoe_cache_destroy": (_i, [_vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def _p(x):
    """Tensor / int / None -> pointer value."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, status):
    if status != FTMOE_OK:
        raise FtmoeError(fn, status)


def _qt(q):
    return QTYPES[q] if isinstance(q, str) else int(q)


# ------------------------------------------------------------------ plain C calls
def ftmoe_version():
    return lib.ftmoe_version()


def ftmoe_tiled_bytes(qtype, E, N, K):
    return lib.ftmoe_tiled_bytes(_qt(qtype), E, N, K)


def ftmoe_repack(qtype, canon, tiles, E, N, K, stream=None):
    _check("ftmoe_repack", lib.ftmoe_repack(_qt(qtype), _p(canon), _p(tiles), E, N, K, _s(stream)))


def ftmoe_dequant(qtype, tiles, E, N, K, out, stream=None):
    _check("ftmoe_dequant", lib.ftmoe_dequant(_qt(qtype), _p(tiles), E, N, K, _p(out), _s(stream)))


def ftmoe_dequant_operand(qtype, which, tiles, E, N, K, out, stream=None):
    _check("ftmoe_dequant_operand", lib.ftmoe_dequant_operand(_qt(qtype), int(which), _p(tiles), E, N, K,
                                                              _p(out), _s(stream)))


def ftmoe_route(logits, T, E, k, ids, w, stream=None):
    _check("ftmoe_route", lib.ftmoe_route(_p(logits), T, E, k, _p(ids), _p(w), _s(stream)))


def ftmoe_permute_workspace_bytes(T, k, E):
    return lib.ftmoe_permute_workspace_bytes(T, k, E)


def ftmoe_permute(ids, T, k, E, offsets, sorted_pair, inv_pos, ws, ws_bytes, stream=None):
    _check("ftmoe_permute", lib.ftmoe_permute(_p(ids), T, k, E, _p(offsets), _p(sorted_pair),
                                              _p(inv_pos), _p(ws), ws_bytes, _s(stream)))


def ftmoe_permute_noalloc(ids, T, k, E, offsets, sorted_pair, inv_pos, stream=None):
    _check("ftmoe_permute_noalloc", lib.ftmoe_permute_noalloc(_p(ids), T, k, E, _p(offsets),
                                                              _p(sorted_pair), _p(inv_pos),
                                                              _s(stream)))


def ftmoe_expert_blob_bytes(qtype, H, I):
    return lib.ftmoe_expert_blob_bytes(_qt(qtype), H, I)


def ftmoe_ffn_workspace_bytes(T, k, E, H, I):
    return lib.ftmoe_ffn_workspace_bytes(T, k, E, H, I)


def ftmoe_layer_workspace_bytes(T, k, E, H, I, has_shared):
    return lib.ftmoe_layer_workspace_bytes(T, k, E, H, I, int(bool(has_shared)))


def ftmoe_set_ffn_path(path):
    return lib.ftmoe_set_ffn_path(int(path))


def make_weights(qtype, E, H, I, w13=None, w2=None, expert_blob=None, shared_w13=None,
                 shared_w2=None):
    """Fill an ftmoe_weights struct; expert_blob is a sequence of E device pointers."""
    wts = ftmoe_weights(_qt(qtype), E, H, I, _p(w13), _p(w2), None, _p(shared_w13), _p(shared_w2))
    if expert_blob is not None:
        arr = (C.c_void_p * E)(*[int(p) if p else None for p in expert_blob])
        wts.expert_blob = C.cast(arr, C.POINTER(C.c_void_p))
        wts._blob_keepalive = arr
    return wts


def ftmoe_expert_ffn(wts, x, T, k, offsets, sorted_pair, y_perm, ws, ws_bytes, stream=None):
    _check("ftmoe_expert_ffn", lib.ftmoe_expert_ffn(C.byref(wts), _p(x), T, k, _p(offsets),
                                                    _p(sorted_pair), _p(y_perm), _p(ws), ws_bytes,
                                                    _s(stream)))


def ftmoe_combine(y_perm, w, inv_pos, shared_y, T, k, H, out, stream=None):
    _check("ftmoe_combine", lib.ftmoe_combine(_p(y_perm), _p(w), _p(inv_pos), _p(shared_y), T, k, H,
                                              _p(out), _s(stream)))


def ftmoe_layer(wts, logits, x, T, k, out, ids_out, w_out, ws, ws_bytes, stream=None):
    _check("ftmoe_layer", lib.ftmoe_layer(C.byref(wts), _p(logits), _p(x), T, k, _p(out), _p(ids_out),
                                          _p(w_out), _p(ws), ws_bytes, _s(stream)))


def ftmoe_device_status(stream=None):
    code = C.c_int(0)
    _check("ftmoe_device_status", lib.ftmoe_device_status(C.byref(code), _s(stream)))
    return code.value


def ftmoe_gate(x, wg, T, H, E, logits, stream=None):
    _check("ftmoe_gate", lib.ftmoe_gate(_p(x), _p(wg), T, H, E, _p(logits), _s(stream)))


def ftmoe_check_wait_timeout(limit_ns, waited_ok=None, stream=None):
    _check("ftmoe_check_wait_timeout", lib.ftmoe_check_wait_timeout(int(limit_ns), _p(waited_ok),
                                                                    _s(stream)))


# ------------------------------------------------------------------ cache
class ExpertCache:
    """Owns one ftmoe_cache handle; methods are the ftmoe_cache_* calls."""

    def __init__(self, layers, E, blob_bytes, bank, pool, slots_per_layer, policy, copy_stream):
        self.E = E
        d = ftmoe_cache_desc(layers, E, blob_bytes, _p(bank), _p(pool), slots_per_layer, policy,
                             _s(copy_stream))
        h = C.c_void_p()
        _check("ftmoe_cache_create", lib.ftmoe_cache_create(C.byref(d), C.byref(h)))
        self.h = h
        self._blob = (C.c_void_p * E)()

    @staticmethod
    def _ids(ids):
        arr = (C.c_int32 * len(ids))(*[int(i) for i in ids])
        return arr

    def prefetch(self, layer, ids):
        a = self._ids(ids)
        slots = (C.c_int32 * len(ids))()
        copied = (C.c_uint8 * len(ids))()
        _check("ftmoe_cache_prefetch", lib.ftmoe_cache_prefetch(self.h, layer, a, len(ids), slots, copied))
        return list(slots), [bool(c) for c in copied]

    def prefetch_history(self, layer):
        """Prefetch what `layer` asked for at its last acquire; returns (ids, slots, copied)."""
        ids = (C.c_int32 * self.E)()
        slots = (C.c_int32 * self.E)()
        copied = (C.c_uint8 * self.E)()
        n = C.c_int(0)
        _check("ftmoe_cache_prefetch_history",
               lib.ftmoe_cache_prefetch_history(self.h, layer, ids, C.byref(n), slots, copied))
        k = n.value
        return list(ids)[:k], list(slots)[:k], [bool(c) for c in list(copied)[:k]]

    def acquire(self, layer, ids, compute_stream=None):
        a = self._ids(ids)
        slots = (C.c_int32 * len(ids))()
        copied = (C.c_uint8 * len(ids))()
        _check("ftmoe_cache_acquire", lib.ftmoe_cache_acquire(self.h, layer, a, len(ids), _s(compute_stream),
                                                              self._blob, slots, copied))
        return list(self._blob), list(slots), [bool(c) for c in copied]

    def release(self, layer, compute_stream=None):
        _check("ftmoe_cache_release", lib.ftmoe_cache_release(self.h, layer, _s(compute_stream)))

    def stats(self):
        s = ftmoe_cache_stats()
        _check("ftmoe_cache_stats_get", lib.ftmoe_cache_stats_get(self.h, C.byref(s)))
        return {f: getattr(s, f) for f, _ in ftmoe_cache_stats._fields_}

    def close(self):
        if self.h:
            _check("ftmoe_cache_destroy", lib.ftmoe_cache_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
