"""The attention's launch-shape choice on the host (tsd_tree_attn_plan,
tsd_tree_attn_launches, tsd_tree_attn_workspace_bytes), without a GPU: for
the benchmark workloads and edge shapes, the key-range pieces cover every key
exactly once in whole 128-key tiles, the kernel and block size agree, the
device plan is used exactly where its rule says, rows go straight to the
output only with one piece (and then no workspace and one launch), and the
grid holds every work item."""

import ctypes

import numpy as np
import pytest

TILE = 128


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import tree_speculative_decoding_virtual_gb300 as tsd
    return tsd.lib


def _plan(L, B, N, Hq, Hkv, D, S):
    info = (ctypes.c_int32 * 8)()
    rc = L.tsd_tree_attn_plan(B, N, Hq, Hkv, D, S, info)
    return rc, list(info)


SHAPES = [
    # B, N_max, Hq, Hkv, D, max_slots
    (1, 4, 4, 4, 64, 128 + 4),            # tiny
    (4, 63, 32, 8, 128, 4096 + 63),       # 8B
    (64, 16, 32, 8, 128, 9000),           # ragged-like batch
    (4, 64, 64, 8, 128, 32768 + 64),      # 70B long context
    (8, 256, 32, 8, 128, 2048 + 256),     # budgeted N=256
    (8, 16, 32, 8, 128, 2048 + 16),       # budgeted N=16
    (2, 20, 16, 1, 128, 200000),          # very long prefix: most pieces
    (65, 8, 8, 8, 64, 3000),              # more sequences than the device plan takes
    (1, 1, 1, 1, 64, 1),                  # one key
]


@pytest.mark.parametrize("shape", SHAPES)
def test_plan_invariants(L, shape):
    B, N, Hq, Hkv, D, S = shape
    rc, info = _plan(L, B, N, Hq, Hkv, D, S)
    assert rc == 0
    mode, dual, rows, row_blocks, pieces, keys, grid, direct = info
    g = Hq // Hkv
    assert mode in (1, 2) and dual in (0, 1) and rows in (128, 256)
    if dual and N * g > 128:
        assert rows == 128  # the two-blocks-per-SM kernel holds 128 rows a block
    # (when every row fits one 128-row block the report gives the 256-row pitch)
    assert row_blocks == -(-N * g // rows)
    # pieces of whole tiles cover the key range exactly once
    assert keys % TILE == 0 and 1 <= pieces <= 32 and keys <= 64 * TILE
    assert (pieces - 1) * keys < S <= pieces * keys
    # the device plan: batches of 2..64 whose pieces would walk >= 16 tiles
    assert (mode == 2) == (2 <= B <= 64 and keys // TILE >= 16)
    assert direct == (1 if (mode == 1 and pieces == 1) else 0)
    units = B * Hkv * row_blocks
    if mode == 1:
        assert grid == units * pieces
    else:
        assert units * pieces <= grid <= units * 32
    ws = L.tsd_tree_attn_workspace_bytes(B, N, Hq, Hkv, D, S)
    assert (ws == 0) == bool(direct)
    launches = L.tsd_tree_attn_launches(B, N, Hq, Hkv, D, S)
    assert launches == (3 if mode == 2 else 1 if direct else 2)


def test_plan_rejections(L):
    info = (ctypes.c_int32 * 8)()
    assert L.tsd_tree_attn_plan(1, 8, 4, 4, 96, 100, info) != 0     # head dim
    assert L.tsd_tree_attn_plan(1, 8, 6, 4, 128, 100, info) != 0    # Hq not a multiple of Hkv
    assert L.tsd_tree_attn_plan(1, 300, 4, 4, 128, 100, info) != 0  # N_max above 256
    assert L.tsd_tree_attn_launches(1, 8, 4, 4, 96, 100) == 0


def test_more_keys_never_fewer_tiles(L):
    """Along growing key ranges the pieces always cover the range, and the
    chosen piece count is what it takes for the chosen piece size."""
    for S in list(range(1, 600, 37)) + list(range(4000, 262145, 15013)) + [262144]:
        rc, info = _plan(L, 4, 32, 32, 8, 128, S)
        assert rc == 0
        pieces, keys = info[4], info[5]
        assert pieces == -(-S // keys)
    # beyond 32 pieces of 64 tiles of 128 keys the call is refused
    assert _plan(L, 4, 32, 32, 8, 128, 262145)[0] == -2  # TSD_ERR_LIMIT
