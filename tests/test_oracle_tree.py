"""Pins for the oracle's safe tree tensors (virtual root, ancestor table,
bitmask, range / acyclicity / closure checks).

The expected values come from the pages' example trees (golden fixtures), from
hand-made malformed trees whose error bits follow from the definitions, and
from networkx as an independent graph library."""

import json
import os

import networkx as nx
import numpy as np
import pytest

import gen
import oracle
from oracle import (ERR_CLOSURE, ERR_COUNT, ERR_CYCLE, ERR_RANGE, ERR_ROOT, ERR_TOO_DEEP,
                    build_ancestors)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("fixture", ["medusa_figure_tree.json", "three_paths_tree.json"])
def test_pages_example_trees(fixture):
    g = _load(fixture)
    parent = np.array([g["parent"]], dtype=np.int32)
    anc, depth, mask, err = build_ancestors(parent, None, g["d_max"])
    assert err[0] == 0
    assert anc[0].tolist() == g["anc"]
    assert depth[0].tolist() == g["depth"]
    assert mask[0, :, 0].tolist() == g["mask"]


def test_virtual_root_makes_every_index_safe():
    # every entry of the table is a valid row index [0, N]; row 0 is all zero
    rng = np.random.default_rng(5)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        parent = gen.relabel(rng, gen.random_tree(rng, n, 6))[None]
        anc, depth, mask, err = build_ancestors(parent, None, 6)
        assert err[0] == 0
        assert anc.min() >= 0 and anc.max() <= n
        assert (anc[0, 0] == 0).all()


def _nx_tree(parent, n):
    G = nx.DiGraph()
    G.add_nodes_from(range(n))
    for i in range(1, n):
        G.add_edge(int(parent[i]), i)
    return G


def test_against_networkx_random_trees():
    """Depth, ancestor rows and masks agree with networkx's ancestors and
    shortest-path depth on random trees with shuffled ids and padding."""
    rng = np.random.default_rng(11)
    for trial in range(400):
        n_max = int(rng.integers(1, 70))
        B = 3
        d_max = int(rng.integers(3, 10))
        parent = np.zeros((B, n_max), dtype=np.int32)
        n_nodes = rng.integers(1, n_max, size=B, endpoint=True).astype(np.int32)
        for b in range(B):
            nb = int(n_nodes[b])
            p = gen.random_tree(rng, nb, d_max)
            if nb > 2:
                p = gen.relabel(rng, p)
            parent[b, :nb] = p
            parent[b, nb:] = rng.integers(-9, 200, size=n_max - nb)  # junk padding
        anc, depth, mask, err = build_ancestors(parent, n_nodes, d_max)
        W = (n_max + 31) // 32
        for b in range(B):
            nb = int(n_nodes[b])
            assert err[b] == 0
            G = _nx_tree(parent[b], nb)
            assert nx.is_arborescence(G)
            dist = nx.shortest_path_length(G, source=0)
            for i in range(nb):
                ancestors = nx.ancestors(G, i)
                assert depth[b, i] == dist[i] == len(ancestors)
                # row: ancestors ordered by depth, in safe ids, then zeros
                by_depth = sorted(ancestors | {i}, key=lambda x: dist[x])
                row = [x + 1 for x in by_depth] + [0] * (d_max + 1 - len(by_depth))
                assert anc[b, i + 1].tolist() == row
                bits = 0
                for a in ancestors | {i}:
                    bits |= 1 << a
                got = sum(int(mask[b, i, w]) << (32 * w) for w in range(W))
                assert got == bits
                # closure: the row of a node extends its parent's row by one
                if i > 0:
                    p = int(parent[b, i])
                    d = depth[b, i]
                    assert (anc[b, i + 1, :d] == anc[b, p + 1, :d]).all()
                    assert anc[b, i + 1, d] == i + 1
                assert bin(got).count("1") == depth[b, i] + 1
            assert (anc[b, nb + 1:] == 0).all()
            assert (mask[b, nb:] == 0).all()
            assert (depth[b, nb:] == 0).all()


BAD = [
    # (parent, n_nodes, d_max, expected bits) -- bits follow from the definitions
    ([-1, 1, 0], 3, 4, ERR_CYCLE),                 # self loop at node 1
    ([-1, 2, 1, 0], 4, 4, ERR_CYCLE),              # 1 <-> 2 cycle off the root
    ([-1, 0, -1], 3, 4, ERR_RANGE),                # second root
    ([-1, 0, 7], 3, 4, ERR_RANGE),                 # parent >= N_max
    ([-1, 0, -3], 3, 4, ERR_RANGE),                # parent < -1
    ([-1, 0, 3, 0], 3, 4, ERR_CLOSURE),            # valid node 2 points at padding node 3
    ([0, 0, 1], 3, 4, ERR_ROOT),                   # root has a parent
    ([2, 0, 1], 3, 4, ERR_ROOT),                   # root inside a cycle
    ([-1, 0, 1, 2, 3], 5, 3, ERR_TOO_DEEP),        # chain of depth 4 > D_max 3
    ([-1, 0, 1, 2], 4, 3, 0),                      # depth exactly D_max is fine
    ([-1, 0, 1], 0, 4, ERR_COUNT),                 # empty tree
    ([-1, 0, 1], 4, 4, ERR_COUNT),                 # more nodes than rows
    ([5, 9, -1], 3, 4, ERR_ROOT | ERR_RANGE),      # several structural bits at once
    ([-1, 0, 4, 2, 0], 4, 4, ERR_CLOSURE),         # padding slot junk is ignored, closure seen
]


@pytest.mark.parametrize("parent,nb,d_max,bits", BAD)
def test_malformed_trees_exact_bits(parent, nb, d_max, bits):
    n_max = len(parent)
    p = np.array([parent], dtype=np.int32)
    anc, depth, mask, err = build_ancestors(p, np.array([nb]), d_max)
    assert int(err[0]) == bits
    if bits:
        # fail closed: nothing usable is emitted for this sequence
        assert not anc.any() and not depth.any() and not mask.any()


def test_cycle_detection_matches_networkx():
    """Random functional graphs: CYCLE is set exactly when the parent graph of
    the valid nodes is not a tree rooted at 0 (given no structural errors)."""
    rng = np.random.default_rng(3)
    seen_cycle = seen_ok = 0
    for _ in range(3000):
        n = int(rng.integers(2, 9))
        par = np.concatenate([[-1], rng.integers(0, n, size=n - 1)]).astype(np.int32)
        _, _, _, err = build_ancestors(par[None], None, 32)
        G = _nx_tree(par, n)
        is_tree = nx.is_arborescence(G)
        assert (int(err[0]) == 0) == is_tree
        assert int(err[0]) in (0, ERR_CYCLE)
        seen_cycle += not is_tree
        seen_ok += is_tree
    assert seen_cycle > 100 and seen_ok > 100


def test_mask_width_spans_words():
    # a chain of 70 nodes needs 3 mask words; the last node sees all 70
    parent = gen.chain_tree(70)[None]
    anc, depth, mask, err = build_ancestors(parent, None, 69)
    assert err[0] == 0
    assert mask.shape == (1, 70, 3)
    assert mask[0, 69].tolist() == [0xFFFFFFFF, 0xFFFFFFFF, (1 << 6) - 1]
    assert depth[0, 69] == 69
    assert anc[0, 70].tolist() == list(range(1, 71))
