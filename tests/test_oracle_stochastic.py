"""Pins for the stochastic tree verification oracle (CPU only).

What pins it, independently of its own code:

* Losslessness, exactly: for a node whose k children are independent draws
  from q, the emitted token (the accepted child's, else the node's draw) is
  distributed as p = softmax(logits) ([Blog], modified rejection sampling: the
  result is distributed as the target).  The distribution is integrated from
  the oracle used as a black box: every uniform enters through a threshold
  (accept iff u below it; the draw is monotone in its uniform), so each
  threshold is found by bisection to ~1e-15 and the masses summed over all
  child-token combinations weighted by q.  A residual that is not updated,
  not normalised, has the wrong sign, or a draw from p instead of the residual
  all miss p by far more than the tolerance.
* A chain (one child per node) reduces to the page's single-token rule,
  checked against the pinned ``modified_rejection_step``.
* The greedy limit: a one-hot target (huge logit gaps) turns acceptance into
  token equality, so on trees with distinct sibling tokens the path, accept
  length, leaf and bonus equal the greedy oracle's.
* p == q: no child is ever rejected, the walk follows first children.
* Skipped sequences and padding rows.
"""

import itertools

import numpy as np
import pytest

import oracle
from oracle import node_decision, tree_verify_stochastic, tree_verify_stochastic_all

ONE = 1.0 - 2.0 ** -53  # largest double below 1


def _threshold(pred):
    """sup{u in [0,1): pred(u)} for a predicate true on [0, t) and false on
    [t, 1); returns 1.0 when pred(ONE) holds, 0.0 when pred(0) fails."""
    if pred(ONE):
        return 1.0
    if not pred(0.0):
        return 0.0
    lo, hi = 0.0, ONE
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return hi


def _emitted_given_tokens(logits, q, toks):
    """Exact distribution of the token a node emits, given its children's
    tokens (children ids 1..k), from black-box calls of node_decision."""
    k, V = len(toks), len(q)
    ids = list(range(1, k + 1))
    out = np.zeros(V)
    reach = 1.0
    for j in range(k):
        def accepted(u, j=j):
            ua = np.zeros(k + 1)
            ua[1:j + 1] = ONE          # earlier children rejected (when possible)
            ua[j + 1] = u
            c, _, _, _ = node_decision(logits, q, ids, toks, ua, 0.5)
            return c == j + 1
        th = _threshold(accepted)
        out[toks[j]] += reach * th
        reach *= (1.0 - th)
        if reach == 0.0:
            return out
    ua = np.full(k + 1, ONE)
    tok_at = lambda ud: node_decision(logits, q, ids, toks, ua, ud)[1]
    lo = 0.0
    while lo < 1.0:
        t = tok_at(lo)
        end = _threshold(lambda u, t=t, lo=lo: u < lo or tok_at(u) == t)
        out[t] += reach * (end - lo)
        if end >= 1.0:
            break
        lo = end
    return out


def _emitted(logits, q, k):
    V = len(q)
    total = np.zeros(V)
    for toks in itertools.product(range(V), repeat=k):
        w = np.prod([q[x] for x in toks])
        if w > 0:
            total += w * _emitted_given_tokens(logits, q, list(toks))
    return total


@pytest.mark.parametrize("k,V,seed", [(0, 5, 0), (1, 4, 1), (2, 4, 2), (3, 3, 3), (2, 5, 4)])
def test_emitted_token_is_distributed_as_p(k, V, seed):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 1.5, size=V)
    p = np.exp(logits - logits.max())
    p /= p.sum()
    for q in (rng.dirichlet(np.ones(V)), rng.dirichlet(0.3 * np.ones(V)),
              np.roll(p, 1), p[::-1].copy()):
        got = _emitted(logits, q, k)
        np.testing.assert_allclose(got, p, rtol=0, atol=1e-12)


def test_emitted_with_zero_draft_mass():
    """q puts no mass on some tokens (the residual must supply them) and the
    draft can be degenerate (one-hot)."""
    logits = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    for q in (np.array([0.0, 0.5, 0.5, 0.0]), np.array([1.0, 0.0, 0.0, 0.0])):
        for k in (1, 2, 3):
            np.testing.assert_allclose(_emitted(logits, q, k), np.exp(logits), rtol=0, atol=1e-12)


def test_second_token_conditional():
    """Two-level tree: root with two children, each with two children.  Given
    the walk accepted a root child with token a, the next emitted token is
    distributed as that child's own target (its row of logits), whatever the
    root's decisions were: nodes are decided independently."""
    rng = np.random.default_rng(7)
    V = 4
    logits = rng.normal(0, 1, size=(7, V))
    q = rng.dirichlet(np.ones(V), size=7)
    parent = np.array([[-1, 0, 0, 1, 1, 2, 2]])
    p0 = np.exp(logits[0] - logits[0].max())
    p0 /= p0.sum()
    # root's first child: a token with p/q < 1 (can be rejected); second: one
    # where p > q (positive residual mass, so u = 0 accepts it)
    tokens = np.array([[0, int(np.argmin(p0 / q[0])), int(np.argmax(p0 - q[0])), 3, 0, 1, 3]])
    u_acc = np.zeros((1, 7))
    u_acc[0, 1] = 0.0   # child 1 accepted whenever its target mass is positive
    for child in (1, 2):
        if child == 2:
            u_acc[0, 1] = ONE   # force the root's first child to be rejected ...
            u_acc[0, 2] = 0.0   # ... and the second accepted
        kids = [3, 4] if child == 1 else [5, 6]
        expect = np.exp(logits[child] - logits[child].max())
        expect /= expect.sum()
        dist = np.zeros(V)
        for toks in itertools.product(range(V), repeat=2):
            tk = tokens.copy()
            tk[0, kids] = toks
            w = q[child][toks[0]] * q[child][toks[1]]
            dist += w * _emitted_given_tokens(logits[child], q[child], list(toks))
            nxt, drw, A, leaf, path, bonus = tree_verify_stochastic_all(
                logits[None], q[None], tk, parent, None, 3, u_acc, np.full((1, 7), 0.5))
            assert nxt[0, 0] == child and path[0, 1] == child + 1
            assert A[0] == (1 if nxt[0, child] < 0 else 2)
        np.testing.assert_allclose(dist, expect, rtol=0, atol=1e-12)


def test_chain_matches_single_token_rule():
    rng = np.random.default_rng(11)
    V, n = 6, 9
    parent = np.array([[-1] + list(range(n - 1))])
    for _ in range(40):
        logits = rng.normal(0, 2, size=(1, n, V))
        q = rng.dirichlet(np.ones(V), size=(1, n))
        tokens = rng.integers(0, V, size=(1, n))
        ua, ud = rng.random((1, n)), rng.random((1, n))
        nxt, drw, A, leaf, path, bonus = tree_verify_stochastic_all(logits, q, tokens, parent,
                                                                     None, n, ua, ud)
        for i in range(n - 1):
            p = np.exp(logits[0, i] - logits[0, i].max())
            p /= p.sum()
            ok, t = oracle.modified_rejection_step(p, q[0, i], int(tokens[0, i + 1]),
                                                   float(ua[0, i + 1]), float(ud[0, i]))
            assert (nxt[0, i] == i + 1) == ok
            if not ok:
                assert drw[0, i] == t
        # the walk stops at the first rejection
        stop = next((i for i in range(n) if nxt[0, i] < 0))
        assert A[0] == stop and leaf[0] == stop and bonus[0] == drw[0, stop]
        assert list(path[0, :stop + 1]) == list(range(1, stop + 2))


def _random_tree(rng, n, V, max_kids=4):
    """Random tree with distinct sibling tokens (ids in BFS order)."""
    parent = [-1]
    for i in range(1, n):
        parent.append(int(rng.integers(0, i)))
    tokens = np.zeros(n, dtype=np.int64)
    for i in range(n):
        kids = [j for j in range(1, n) if parent[j] == i]
        tokens[kids] = rng.choice(V, size=len(kids), replace=False)
    return np.array(parent), tokens


def test_greedy_limit_equals_greedy_verify():
    rng = np.random.default_rng(5)
    B, n, V, d_max = 6, 24, 50, 23
    parent = np.zeros((B, n), dtype=np.int64)
    tokens = np.zeros((B, n), dtype=np.int64)
    for b in range(B):
        parent[b], tokens[b] = _random_tree(rng, n, V)
    logits = rng.normal(0, 1, size=(B, n, V))
    # plant the target's choice: often the first or another child's token
    for b in range(B):
        for i in range(n):
            kids = [j for j in range(1, n) if parent[b, j] == i]
            a = int(tokens[b, rng.choice(kids)]) if kids and rng.random() < 0.8 else int(
                rng.integers(V))
            logits[b, i, a] = logits[b, i].max() + 1e4   # one-hot in fp64
    q = rng.dirichlet(np.ones(V), size=(B, n))
    ua, ud = rng.random((B, n)), rng.random((B, n))
    nxt, drw, A, leaf, path, bonus = tree_verify_stochastic_all(logits, q, tokens, parent, None,
                                                                d_max, ua, ud)
    g_am, g_A, g_leaf, g_path, g_bonus = oracle.verify_greedy(
        logits, tokens, parent, None, np.zeros(B, dtype=np.int32), d_max)
    assert np.array_equal(A, g_A) and np.array_equal(leaf, g_leaf)
    assert np.array_equal(path, g_path) and np.array_equal(bonus, g_bonus)
    assert (A > 0).any()


def test_equal_distributions_follow_first_children():
    rng = np.random.default_rng(9)
    n, V = 15, 30
    parent, tokens = _random_tree(rng, n, V)
    logits = rng.normal(0, 1, size=(1, n, V))
    p = np.exp(logits - logits.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    ua = np.full((1, n), ONE)
    nxt, drw, A, leaf, path, bonus = tree_verify_stochastic_all(
        logits, p, tokens[None], parent[None], None, n, ua, rng.random((1, n)))
    for i in range(n):
        kids = [j for j in range(1, n) if parent[j] == i]
        assert nxt[0, i] == (kids[0] if kids else -1)


def test_skipped_and_padding():
    rng = np.random.default_rng(2)
    n, V = 8, 10
    parent = np.array([[-1, 0, 0, 1, 1, 2, 0, 0], [-1, 0, 5, 0, 0, 0, 0, 0]])  # second: closure
    n_nodes = np.array([6, 4])
    logits = rng.normal(size=(2, n, V))
    q = rng.dirichlet(np.ones(V), size=(2, n))
    tokens = rng.integers(0, V, size=(2, n))
    nxt, drw, A, leaf, path, bonus = tree_verify_stochastic_all(
        logits, q, tokens, parent, n_nodes, 4, rng.random((2, n)), rng.random((2, n)))
    assert (nxt[0, 6:] == -1).all() and (drw[0, 6:] == -1).all()
    assert not ((nxt[0, :6] >= 0) & (drw[0, :6] >= 0)).any()
    internal = [i for i in range(6) if any(parent[0, j] == i for j in range(1, 6))]
    for i in range(6):
        if i in internal or i == leaf[0]:
            assert (nxt[0, i] >= 0) ^ (drw[0, i] >= 0)
        else:
            assert drw[0, i] == -1      # a leaf the walk does not reach draws nothing
    assert bonus[0] == drw[0, leaf[0]] >= 0
    assert (nxt[1] == -1).all() and (drw[1] == -1).all()
    assert A[1] == 0 and leaf[1] == -1 and bonus[1] == -1 and (path[1] == 0).all()


def test_draw_boundaries():
    """u_draw = 0 takes the first token of positive weight; the draw follows
    the cumulative weights in token order."""
    logits = np.array([-1e4, np.log(0.25), np.log(0.25), np.log(0.5)])  # token 0: weight 0
    q = np.full(4, 0.25)
    for u, t in ((0.0, 1), (0.2499, 1), (0.2501, 2), (0.4999, 2), (0.5001, 3), (ONE, 3)):
        c, tok, _, _ = node_decision(logits, q, [], [], np.zeros(1), u)
        assert c == -1 and tok == t


def test_out_of_range_child_is_skipped():
    """A child whose token lies outside [0, V) changes nothing: the result
    equals that of the same tree without it."""
    rng = np.random.default_rng(4)
    V = 6
    parent = np.array([[-1, 0, 0, 0, 1]])
    logits = rng.normal(size=(1, 5, V))
    q = rng.dirichlet(np.ones(V), size=(1, 5))
    for bad in (-1, V, 10 ** 6):
        for _ in range(20):
            ua, ud = rng.random((1, 5)), rng.random((1, 5))
            tokens = rng.integers(0, V, size=(1, 5))
            tokens[0, 2] = bad
            got = tree_verify_stochastic_all(logits, q, tokens, parent, None, 3, ua, ud)
            # the same tree with node 2 moved under node 4 (never reached at the root)
            par2 = parent.copy()
            par2[0, 2] = 4
            tok2 = tokens.copy()
            tok2[0, 2] = 0
            ref = tree_verify_stochastic_all(logits, q, tok2, par2, None, 3, ua, ud)
            assert got[0][0, 0] == ref[0][0, 0] and got[1][0, 0] == ref[1][0, 0]
            assert got[0][0, 0] != 2
