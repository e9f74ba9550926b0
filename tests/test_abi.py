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
    assert F.ftmoe_tiled_bytes(3, 1, 16, 64) == 0
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
