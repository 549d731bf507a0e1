"""TLR-output entry points on the host (no GPU): workspace sizing and argument
checks that run before any device use.

The recompression ("TLR Matrix Multiplication", section "Introduction: TLR
GEMM", the TLR-output cases) keeps per tile a sketch Y and basis Q (b x s), the
projection B (s x b), the core G = B B^T and its eigenvectors W (s x s), the
eigenvalues (s) and the tile's energy (fp64): the workspace for t tiles must
hold t copies of that, and must grow by the same amount for every tile.
"""
import ctypes

import numpy as np
import pytest


@pytest.fixture(scope="module")
def g():
    from gemm_tlr_gb300.build import build
    build()
    import gemm_tlr_gb300
    gemm_tlr_gb300.lib()
    return gemm_tlr_gb300


@pytest.mark.parametrize("b,s", [(1024, 128), (64, 64), (200, 16), (10, 2)])
def test_workspace_holds_each_tiles_scratch_and_grows_per_tile(g, b, s):
    per_tile_floor = 4 * (2 * b * s + 2 * s * s + s) + 8   # Q, B, G, W, eigenvalues, energy
    one = g.tlr_compress_workspace_bytes(b, s, 1)
    assert one >= per_tile_floor
    steps = [g.tlr_compress_workspace_bytes(b, s, t + 1) - g.tlr_compress_workspace_bytes(b, s, t)
             for t in range(1, 6)]
    assert len(set(steps)) == 1 and steps[0] >= per_tile_floor
    big = g.tlr_compress_workspace_bytes(b, s, 992)
    assert big >= 992 * per_tile_floor
    # zero tiles sizes the same as one (a compression always needs one tile's scratch)
    assert g.tlr_compress_workspace_bytes(b, s, 0) == one


@pytest.mark.parametrize("b,s,tiles", [(0, 16, 1), (-5, 16, 1), (64, 0, 1), (64, -2, 1), (64, 16, -1)])
def test_workspace_sizing_refuses_bad_sizes(g, b, s, tiles):
    with pytest.raises(g.TLRError) as e:
        g.tlr_compress_workspace_bytes(b, s, tiles)
    assert g._abi.STATUS[e.value.code] == "INVALID_ARG"


def test_workspace_sizing_refuses_a_null_result_pointer(g):
    assert g.lib().tlr_compress_workspace_bytes(64, 16, 1, None) == 1   # TLR_STATUS_INVALID_ARG


def test_compress_and_pack_refuse_a_null_handle(g):
    """Both entry points check the handle first, so these calls touch no device."""
    lib = g.lib()
    P = ctypes.c_void_p
    st = lib.tlr_compress(P(0), P(0), 64, 64, 64, 64, 0, ctypes.c_float(0.1), 8, P(0), 16,
                          P(0), P(0), P(0), P(0), P(0), P(0), 0)
    assert st == 1
    ranks = np.zeros((1, 1), dtype=np.int32)
    st = lib.tlr_pack(P(0), 64, 64, 8, P(ranks.ctypes.data), P(0), P(0), P(0), P(0), P(0), P(0),
                      P(0), P(0), P(0), P(0), P(0))
    assert st == 1
