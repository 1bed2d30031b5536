"""Pins for the oracle's greedy tree verification.

* The pages' three-path example (golden fixture): the second path goes
  through, so two draft tokens are accepted and the bonus is the target's
  choice after E.
* Brute force: enumerate every root-to-node path with networkx, take its
  longest accepted prefix, keep the deepest (lowest id on ties); compare on
  thousands of random small trees with shuffled ids.
* Chains with independent per-token match probability alpha reproduce the
  page's expected tokens per cycle E = (1 - alpha^(gamma+1)) / (1 - alpha).
* argmax tie rules: first maximum; +0.0 == -0.0.
* Sequences with err != 0 are skipped.
"""

import json
import os

import networkx as nx
import numpy as np
import pytest

import gen
from oracle import build_ancestors, verify_greedy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _one_hot_logits(greedy, V, rng=None):
    n = len(greedy)
    L = np.zeros((1, n, V), dtype=np.float32)
    if rng is not None:
        L[0] = rng.standard_normal((n, V)).astype(np.float32)
    for i, t in enumerate(greedy):
        L[0, i, t] = L[0, i].max() + 1.0
    return L


def test_three_paths_example():
    with open(os.path.join(GOLDEN, "three_paths_tree.json")) as f:
        g = json.load(f)
    case = g["accept_case"]
    parent = np.array([g["parent"]], dtype=np.int32)
    tokens = np.array([case["tokens"]], dtype=np.int32)
    logits = _one_hot_logits(case["target_greedy"], case["vocab"], np.random.default_rng(0))
    _, _, _, err = build_ancestors(parent, None, g["d_max"])
    am, A, leaf, path, bonus = verify_greedy(logits, tokens, parent, None, err, g["d_max"])
    e = case["expect"]
    assert am[0].tolist() == case["target_greedy"]
    assert A[0] == e["accept_len"] and leaf[0] == e["leaf"]
    assert path[0, :len(e["path"])].tolist() == e["path"]
    assert bonus[0] == e["bonus"]


def _brute_force(parent, tokens, greedy, nb):
    """Longest accepted prefix over all root-to-node paths (networkx)."""
    G = nx.DiGraph()
    G.add_nodes_from(range(nb))
    for i in range(1, nb):
        G.add_edge(int(parent[i]), i)
    best_len, best_leaf = -1, None
    for node in range(nb):
        p = nx.shortest_path(G, 0, node)  # the unique path in a tree
        ok = 1
        while ok < len(p) and tokens[p[ok]] == greedy[p[ok - 1]]:
            ok += 1
        # the accepted prefix ends at p[ok-1]
        end = p[ok - 1]
        L = ok - 1
        if L > best_len or (L == best_len and end < best_leaf):
            best_len, best_leaf = L, end
    return best_len, best_leaf, [x + 1 for x in nx.shortest_path(G, 0, best_leaf)]


def test_brute_force_random_trees():
    rng = np.random.default_rng(21)
    hits = 0
    for trial in range(3000):
        nb = int(rng.integers(1, 10))
        V = int(rng.integers(2, 5))  # tiny vocab: many matches and sibling repeats
        parent = gen.random_tree(rng, nb, 5)
        if nb > 2:
            parent = gen.relabel(rng, parent)
        greedy = rng.integers(0, V, size=nb)
        tokens = rng.integers(0, V, size=nb).astype(np.int32)
        logits = _one_hot_logits(greedy, V)
        _, _, _, err = build_ancestors(parent[None], None, 5)
        am, A, leaf, path, bonus = verify_greedy(logits, tokens[None], parent[None], None, err, 5)
        L, lf, p = _brute_force(parent, tokens, greedy, nb)
        assert (A[0], leaf[0]) == (L, lf)
        assert path[0, :L + 1].tolist() == p and (path[0, L + 1:] == 0).all()
        assert bonus[0] == greedy[lf]
        hits += L > 0
    assert hits > 1000


@pytest.mark.parametrize("alpha", [0.3, 0.7])
def test_chain_expected_tokens_per_cycle(alpha):
    """gamma = 5 drafted tokens on a chain, each matching independently with
    probability alpha: E[A + 1] = (1 - alpha^6) / (1 - alpha)."""
    gamma, trials, V = 5, 20000, 16
    rng = np.random.default_rng(int(alpha * 100))
    n = gamma + 1
    parent = np.tile(gen.chain_tree(n), (trials, 1))
    greedy = rng.integers(0, V, size=(trials, n))
    match = rng.random((trials, n)) < alpha
    other = (greedy + 1 + rng.integers(0, V - 1, size=(trials, n))) % V
    tokens = np.zeros((trials, n), dtype=np.int32)
    tokens[:, 1:] = np.where(match[:, 1:], greedy[:, :-1], other[:, :-1])
    logits = np.zeros((trials, n, V), dtype=np.float32)
    logits[np.arange(trials)[:, None], np.arange(n)[None, :], greedy] = 1.0
    err = np.zeros(trials, dtype=np.int32)
    _, A, _, _, _ = verify_greedy(logits, tokens, parent, None, err, gamma)
    emitted = A + 1
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    se = emitted.std() / np.sqrt(trials)
    assert abs(emitted.mean() - expect) < 5 * se


def test_argmax_ties_and_signed_zero():
    V = 8
    logits = np.full((1, 4, V), -1.0, dtype=np.float32)
    logits[0, 0, [2, 5]] = 3.0            # tie -> 2
    logits[0, 1, [6]] = 0.0               # 0.0 at 6 and -0.0 at 1: equal -> 1
    logits[0, 1, [1]] = -0.0
    logits[0, 2, :] = -1e30               # a row of equal values -> 0
    logits[0, 3, [7]] = 1e-30             # a tiny positive beats zeros
    logits[0, 3, [0]] = 0.0
    parent = np.array([[-1, 0, 0, 0]], dtype=np.int32)
    tokens = np.zeros((1, 4), dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    am, *_ = verify_greedy(logits, tokens, parent, None, err, 1)
    assert am[0].tolist() == [2, 1, 0, 7]


def test_err_and_padding():
    inp = gen.random_small(4, B=3, N_max=10, Hq=2, Hkv=1, D=8, V=20, prefix_lo=0, prefix_hi=5,
                           max_depth=4)
    _, _, _, err = build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    err = err.copy()
    err[2] = 4
    am, A, leaf, path, bonus = verify_greedy(inp.logits, inp.tokens, inp.parent, inp.n_nodes, err,
                                             inp.D_max)
    assert (am[2] == -1).all() and A[2] == 0 and leaf[2] == -1 and bonus[2] == -1
    assert (path[2] == 0).all()
    for b in range(2):
        nb = int(inp.n_nodes[b])
        assert (am[b, nb:] == -1).all()
        assert (am[b, :nb] == inp.targets[b, :nb]).all()  # planted targets are the maxima
        assert path[b, 0] == 1  # the root is always accepted
