"""Pins for the oracle's best-first budgeted tree construction.

* Optimality (the page's claim): on tiny vocabularies, enumerate every
  prefix-closed tree of N nodes and check that none has a larger surrogate
  A_hat than the best-first tree.
* The best-first A_hat equals the sum of the N-1 largest path scores over all
  token sequences of length <= K (brute-force enumeration).
* Concavity: the marginal gain rho of the n-th inserted node is
  non-increasing in n.
* Structure: parents precede children, depths are parent depth + 1, each
  node's rho is the fp32 product of the marginals along its path, sibling
  tokens are distinct.
"""

import itertools

import numpy as np
import pytest

import gen
from oracle import best_first_tree, ranked_tokens


def _all_sequences(K, V):
    for d in range(1, K + 1):
        for seq in itertools.product(range(V), repeat=d):
            yield seq


def _score(q, seq):
    r = np.float32(1.0)
    for k, t in enumerate(seq):
        r = np.float32(r * q[k, t])
    return r


def _best_prefix_closed(q, N):
    """Max A_hat over all prefix-closed sets of N-1 non-root sequences."""
    K, V = q.shape
    seqs = list(_all_sequences(K, V))
    best = -1.0
    for combo in itertools.combinations(range(len(seqs)), N - 1):
        chosen = {seqs[c] for c in combo}
        if all(s[:-1] in chosen or len(s) == 1 for s in chosen):
            a = sum(float(_score(q, s)) for s in chosen)
            best = max(best, a)
    return best


@pytest.mark.parametrize("seed", range(4))
def test_optimal_against_exhaustive_trees(seed):
    rng = np.random.default_rng(seed)
    K, V = 3, 3
    z = rng.standard_normal((1, K, V)) * 1.5
    q = (np.exp(z) / np.exp(z).sum(-1, keepdims=True)).astype(np.float32)
    for N in range(1, 7):
        parent, tokens, depth, rho, ahat = best_first_tree(q, np.array([0]), N)
        if N == 1:
            assert ahat[0] == 0.0
            continue
        assert abs(ahat[0] - _best_prefix_closed(q[0], N)) < 1e-12


@pytest.mark.parametrize("seed", range(3))
def test_equals_top_scores_over_all_sequences(seed):
    rng = np.random.default_rng(100 + seed)
    K, V, N = 4, 4, 30
    z = rng.standard_normal((2, K, V)) * 1.4
    q = (np.exp(z) / np.exp(z).sum(-1, keepdims=True)).astype(np.float32)
    _, _, _, rho, ahat = best_first_tree(q, np.array([1, 2]), N)
    for b in range(2):
        scores = sorted((float(_score(q[b], s)) for s in _all_sequences(K, V)), reverse=True)
        assert abs(ahat[b] - sum(scores[:N - 1])) < 1e-12
        # the inserted scores are exactly the top N-1 as a multiset
        assert sorted(rho[b, 1:].astype(np.float64).tolist(), reverse=True) == scores[:N - 1]


def test_structure_and_concavity_at_scale():
    q, root = gen.bastion_marginals()
    q = q[:2, :, :2000].copy()
    q /= q.sum(-1, keepdims=True)
    N = 96
    parent, tokens, depth, rho, ahat = best_first_tree(q, root[:2], N)
    for b in range(2):
        assert parent[b, 0] == -1 and depth[b, 0] == 0 and rho[b, 0] == 1.0
        assert tokens[b, 0] == root[b]
        for n in range(1, N):
            p = parent[b, n]
            assert 0 <= p < n
            assert depth[b, n] == depth[b, p] + 1 <= q.shape[1]
            assert rho[b, n] == np.float32(rho[b, p] * q[b, depth[b, n] - 1, tokens[b, n]])
        gains = rho[b, 1:]
        assert (np.diff(gains.astype(np.float64)) <= 0).all()
        for p in range(N):
            kids = tokens[b][parent[b] == p]
            assert len(set(kids.tolist())) == len(kids)
            # siblings are a prefix of their position's ranked token list
            if len(kids):
                d = depth[b, p]
                ranked = ranked_tokens(q[b, d])[:len(kids)]
                assert sorted(kids.tolist()) == sorted(ranked.tolist())
        assert ahat[b] == sum(float(x) for x in rho[b, 1:])


def test_ranked_tokens_tie_rule():
    q = np.array([0.1, 0.3, 0.3, 0.05, 0.25], dtype=np.float32)
    assert ranked_tokens(q).tolist() == [1, 2, 4, 0, 3]
