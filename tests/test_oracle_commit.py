"""Pins for the oracle's KV commit (prefix-sharing fast reorder).

The expected cache is built independently: before the call, the K/V entry
of draft node j is read from slot P + j; after the call, slot P + k must hold
the entry of node path[k] - 1 (the k-th node of the accepted path), every
slot below P must be unchanged, and every block that sequence b does not own
must be unchanged.
"""

import numpy as np
import pytest

import gen
from oracle import build_ancestors, commit_path, verify_greedy

PAGE = 16


def _slot(cache, table, b, t):
    return cache[..., table[b, t // PAGE], :, t % PAGE, :]


def _check(k0, v0, k1, v1, table, prefix, A, path, err, new_len, moved, n_nodes):
    B = len(prefix)
    owned = set()
    for b in range(B):
        P = int(prefix[b])
        nb = int(n_nodes[b])
        for blk in table[b, :(P + nb + PAGE - 1) // PAGE]:
            owned.add(int(blk))
        if err[b]:
            assert new_len[b] == P and moved[b] == 0
        else:
            assert new_len[b] == P + A[b] + 1
            assert moved[b] == sum(1 for k in range(A[b] + 1) if path[b, k] - 1 != k)
        for t in range(P):
            assert np.array_equal(_slot(k1, table, b, t), _slot(k0, table, b, t))
        upto = P + (A[b] + 1 if not err[b] else 0)
        for k in range(P, upto):
            node = int(path[b, k - P]) - 1
            assert np.array_equal(_slot(k1, table, b, k), _slot(k0, table, b, P + node))
            assert np.array_equal(_slot(v1, table, b, k), _slot(v0, table, b, P + node))
    nblocks = k0.shape[-4]
    for blk in range(nblocks):
        if blk not in owned:
            assert np.array_equal(k1[..., blk, :, :, :], k0[..., blk, :, :, :])
            assert np.array_equal(v1[..., blk, :, :, :], v0[..., blk, :, :, :])


def test_overlap_hazard_example():
    """Accepted path of real ids 0, 2, 5: slot P+1 <- P+2 and P+2 <- P+5.  The
    second move's destination is the first move's source, so every source
    must be read before any write."""
    rng = np.random.default_rng(0)
    P, n, D, H = 5, 6, 4, 2
    prefix = np.array([P], dtype=np.int32)
    nn_ = np.array([n], dtype=np.int32)
    cache = gen.paged_cache(rng, prefix, nn_, H, D, shuffle=True, spare_blocks=2)
    path = np.array([[1, 3, 6, 0, 0]], dtype=np.int32)
    A = np.array([2], dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    k1, v1, new_len, moved = commit_path(cache.k, cache.v, cache.block_table, prefix, A, path, err)
    t = cache.block_table
    assert np.array_equal(_slot(k1, t, 0, P + 1), _slot(cache.k, t, 0, P + 2))
    assert np.array_equal(_slot(k1, t, 0, P + 2), _slot(cache.k, t, 0, P + 5))
    assert np.array_equal(_slot(k1, t, 0, P), _slot(cache.k, t, 0, P))
    assert new_len[0] == P + 3 and moved[0] == 2


def test_chain_path_moves_nothing():
    """Length-based commit: a path that is already in slot order moves no
    bytes and leaves the cache bit-identical."""
    rng = np.random.default_rng(1)
    prefix = np.array([33, 0], dtype=np.int32)
    nn_ = np.array([9, 4], dtype=np.int32)
    cache = gen.paged_cache(rng, prefix, nn_, 2, 8, shuffle=True)
    path = np.array([[1, 2, 3, 4, 0], [1, 2, 0, 0, 0]], dtype=np.int32)
    A = np.array([3, 1], dtype=np.int32)
    err = np.zeros(2, dtype=np.int32)
    k1, v1, new_len, moved = commit_path(cache.k, cache.v, cache.block_table, prefix, A, path, err)
    assert np.array_equal(k1, cache.k) and np.array_equal(v1, cache.v)
    assert moved.tolist() == [0, 0] and new_len.tolist() == [37, 2]


@pytest.mark.parametrize("seed", range(6))
def test_random_verify_then_commit(seed):
    inp = gen.random_small(seed, B=4, N_max=40, Hq=2, Hkv=2, D=8, V=3, prefix_lo=0,
                           prefix_hi=50, max_depth=7, p_match=0.9)
    _, _, _, err = build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    err = err.copy()
    if seed % 2:
        err[1] = 1
    _, A, _, path, _ = verify_greedy(inp.logits, inp.tokens, inp.parent, inp.n_nodes, err,
                                     inp.D_max)
    c = inp.cache
    k1, v1, new_len, moved = commit_path(c.k, c.v, c.block_table, inp.prefix_len, A, path, err)
    _check(c.k, c.v, k1, v1, c.block_table, inp.prefix_len, A, path, err, new_len, moved,
           inp.n_nodes)


def test_layers_all_committed():
    rng = np.random.default_rng(3)
    prefix = np.array([20, 7], dtype=np.int32)
    nn_ = np.array([8, 8], dtype=np.int32)
    layers = [gen.paged_cache(np.random.default_rng(10 + l), prefix, nn_, 2, 8, shuffle=False)
              for l in range(3)]
    K = np.stack([c.k for c in layers])
    Vv = np.stack([c.v for c in layers])
    table = layers[0].block_table
    path = np.array([[1, 5, 7, 0], [1, 2, 8, 0]], dtype=np.int32)
    A = np.array([2, 2], dtype=np.int32)
    err = np.zeros(2, dtype=np.int32)
    k1, v1, new_len, moved = commit_path(K, Vv, table, prefix, A, path, err)
    _check(K, Vv, k1, v1, table, prefix, A, path, err, new_len, moved, nn_)
    assert moved.tolist() == [2, 1]
