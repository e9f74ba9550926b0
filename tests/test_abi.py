"""The C-ABI library builds for sm_103a, loads, and exports every function ftmoe.h
declares; host-side argument checks answer without a GPU."""
import ctypes

import pytest

from tests._util import ensure_built, header_functions


@pytest.fixture(scope="module")
def F():
    ensure_built()
    from quantized_expert_ffn_layer_b300 import ftmoe
    return ftmoe


def test_every_declared_symbol_is_exported(F):
    names = header_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(F.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding wraps exactly the declared functions
    assert sorted(F.EXPORTED) == names


def test_sizes(F):
    assert F.ftmoe_expert_blob_bytes("q4_0", 2048, 768) == 2654208
    assert F.ftmoe_tiled_bytes("q4_0", 128, 1536, 2048) == 128 * 96 * 32 * 576
    assert F.ftmoe_tiled_bytes("mxfp4", 1, 16, 96) == 2 * 544  # ragged K: 2 records
    assert F.ftmoe_tiled_bytes("q4_0", 1, 8, 64) == 0           # N not a multiple of 16
    assert F.ftmoe_tiled_bytes("nvfp4", 1, 16, 64) == 576 + 16  # one record + tensor-scale trailer
    assert F.ftmoe_tiled_bytes("nvfp4", 3, 32, 96) == 3 * (2 * 2 * 576 + 16)
    assert F.ftmoe_tiled_bytes(9, 1, 16, 64) == 0                # unknown format
    assert F.ftmoe_permute_workspace_bytes(64, 8, 128) == 0
    assert F.ftmoe_permute_workspace_bytes(4096, 8, 128) == 32 * 128 * 4
    assert F.ftmoe_layer_workspace_bytes(64, 8, 128, 2048, 768, 0) > 64 * 8 * 2048 * 2


def test_invalid_arguments_rejected_on_host(F):
    with pytest.raises(F.FtmoeError) as ei:
        F.ftmoe_route(0, 4, 8, 9, 0, 0, stream=0)  # k > E
    assert ei.value.status == 1
    with pytest.raises(F.FtmoeError):
        F.ftmoe_route(0, 4, 2000, 2, 0, 0, stream=0)  # E too large
    with pytest.raises(F.FtmoeError):
        F.ftmoe_repack("q4_0", 0, 0, 1, 16, 64, stream=0)  # null pointers
    w = F.make_weights("q4_0", 8, 250, 128, 1, 1)  # H not a multiple of 32
    with pytest.raises(F.FtmoeError):
        F.ftmoe_layer(w, 1, 1, 4, 2, 1, None, None, 1, 1 << 30, stream=0)
    # T == 0 is a successful no-op for route
    F.ftmoe_route(0, 0, 8, 2, 0, 0, stream=0)
    assert F.ftmoe_status_string(4) if hasattr(F, "ftmoe_status_string") else True
    assert F.ftmoe_set_ffn_path(0) in (0, 1, 2, 3)
    # gate: H must be a multiple of 32, E in [1, 1024]; T == 0 is a no-op
    for T, H, E in ((4, 48, 8), (4, 64, 0), (4, 64, 1025), (-1, 64, 8)):
        with pytest.raises(F.FtmoeError) as ei:
            F.ftmoe_gate(1, 1, T, H, E, 1, stream=0)
        assert ei.value.status == 1
    with pytest.raises(F.FtmoeError):
        F.ftmoe_gate(0, 0, 4, 64, 8, 0, stream=0)  # null pointers
    F.ftmoe_gate(0, 0, 0, 64, 8, 0, stream=0)


def test_cache_descriptor_checked_on_host(F):
    """A malformed cache descriptor is refused before anything touches the GPU."""
    good = dict(layers=2, E=8, blob_bytes=1024, bank=1, pool=1, slots_per_layer=2, policy=0,
                copy_stream=1)
    bad = [dict(layers=0), dict(E=0), dict(slots_per_layer=0), dict(bank=None), dict(pool=None),
           dict(blob_bytes=0), dict(blob_bytes=1000), dict(copy_stream=None), dict(policy=2)]
    for b in bad:
        d = dict(good, **b)
        desc = F.ftmoe_cache_desc(d["layers"], d["E"], d["blob_bytes"], d["bank"], d["pool"],
                                  d["slots_per_layer"], d["policy"], d["copy_stream"])
        h = ctypes.c_void_p()
        assert F.lib.ftmoe_cache_create(ctypes.byref(desc), ctypes.byref(h)) == 1, b
        assert not h.value
    assert F.lib.ftmoe_cache_create(None, None) == 1
    # the other cache calls refuse a null handle
    n = ctypes.c_int(0)
    assert F.lib.ftmoe_cache_prefetch_history(None, 0, None, ctypes.byref(n), None, None) == 1
    assert F.lib.ftmoe_cache_release(None, 0, None) == 1
    assert F.lib.ftmoe_cache_destroy(None) == 1


def test_workspace_sizes_grow_with_the_problem(F):
    a = F.ftmoe_layer_workspace_bytes(64, 8, 128, 2048, 768, 0)
    b = F.ftmoe_layer_workspace_bytes(4096, 8, 128, 2048, 768, 0)
    c = F.ftmoe_layer_workspace_bytes(64, 8, 128, 2048, 768, 1)  # with a shared expert
    assert 0 < a < b and c > a
    assert F.ftmoe_ffn_workspace_bytes(64, 8, 128, 2048, 768) <= a
    # the FFN scratch holds h ([T*k][I] bf16) and, for the tensor-core prefill path, x in
    # the permuted order ([T*k][H] bf16)
    P = 4096 * 8
    assert F.ftmoe_ffn_workspace_bytes(4096, 8, 128, 2048, 768) >= P * 768 * 2 + P * 2048 * 2
