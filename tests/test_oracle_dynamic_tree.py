"""Pins of the oracle's dynamic draft trees ([Blog] EAGLE-2 section; reading:
confidence-driven expansion by path score, top-k frontier per level, rerank
of the N-1 best nodes).

Independent checks: brute-force enumeration of every path on tiny
vocabularies, the BASTION best-first construction (itself pinned by brute
force) in the case where both must agree, a greedy chain, path scores
recomputed along each path, closure under ties, and the qualitative behaviour
the page states (deep when confident, wide when uncertain)."""

import itertools

import numpy as np

import oracle
from oracle.dynamic_tree import dynamic_tree, pool_size


def softmax_rows(x):
    e = np.exp(x - x.max(-1, keepdims=True))
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def node_q(seed, V, temp=1.0):
    """A drafter stand-in: node (b, pool id) -> a distribution over V,
    seeded by (seed, b, pool id) so every node has its own row."""
    def q_of(b, pid):
        rng = np.random.default_rng([seed, b, pid])
        return softmax_rows(rng.standard_normal(V) / temp)
    return q_of


def path_of(parent, n):
    out = []
    while n >= 0:
        out.append(n)
        n = int(parent[n])
    return out[::-1]


def _brute_paths(q_of, V, L, exists):
    """Every token path of length 1..L that `exists` admits, with its fp32
    score recomputed along the path; exists(prefix_pid, token) -> pid or None."""
    out = []
    for length in range(1, L + 1):
        for toks in itertools.product(range(V), repeat=length):
            pid, s = 0, np.float32(1.0)
            for t in toks:
                s = np.float32(s * q_of(0, pid)[t])
                pid = exists(pid, t)
                if pid is None:
                    break
            if pid is not None:
                out.append((-float(s), length, toks))
    return out


def _kept_paths(par, tok, N):
    return {tuple(int(tok[0, m]) for m in path_of(par[0], n)[1:]) for n in range(1, N)}


def test_rerank_equals_brute_force_over_all_paths():
    """Two levels with k = V prune nothing: the pool holds every path of length
    <= 2, and the kept nodes must be the N-1 best paths by (score desc,
    length asc)."""
    V, L = 5, 2
    for seed in range(20):
        for N in (2, 6, 13, 31):
            q_of = node_q(100 + seed, V)
            pool, _, (par, tok, dep, sco) = dynamic_tree(q_of, [7], k=V, levels=L, N=N, V=V)
            child = {(int(pool[0][0][i]), int(pool[1][0][i])): i for i in range(1, pool_size(L, V))}
            scored = _brute_paths(q_of, V, L, lambda pid, t: child.get((pid, t)))
            assert len(scored) == V + V * V
            scored.sort(key=lambda x: (x[0], x[1]))
            assert _kept_paths(par, tok, N) == {toks for _, _, toks in scored[:N - 1]}


def test_beam_pruning_by_enumeration():
    """Three levels: a path exists iff each prefix of length >= 1 ranks in the
    k best of its level (by score, brute force over the level's paths) and
    each token ranks below k in its parent's row; the rerank keeps the N-1
    best existing paths."""
    V, k, L = 5, 3, 3
    for seed in range(10):
        q_of = node_q(300 + seed, V)
        pool, _, (par, tok, dep, sco) = dynamic_tree(q_of, [2], k=k, levels=L, N=12, V=V)
        # brute force, level by level, on token tuples
        score = {(): np.float32(1.0)}
        row_of = {(): q_of(0, 0)}
        pid_of = {(): 0}
        p_par, p_tok = pool[0][0], pool[1][0]
        kids = {(int(p_par[i]), int(p_tok[i])): i for i in range(1, pool_size(L, k))}
        frontier = [()]
        existing = []
        for level in range(1, L + 1):
            level_paths = []
            for pre in frontier:
                row = row_of[pre]
                order = sorted(range(V), key=lambda t: (-float(row[t]), t))[:k]
                for t in order:
                    path = pre + (t,)
                    score[path] = np.float32(score[pre] * row[t])
                    pid_of[path] = kids[(pid_of[pre], t)]
                    row_of[path] = q_of(0, pid_of[path])
                    level_paths.append(path)
            existing += level_paths
            frontier = sorted(level_paths, key=lambda p: (-float(score[p]), pid_of[p]))[:k]
        assert len(existing) == pool_size(L, k) - 1
        assert {pid_of[p] for p in existing} == set(range(1, pool_size(L, k)))
        ranked = sorted(existing, key=lambda p: (-float(score[p]), len(p), pid_of[p]))
        assert _kept_paths(par, tok, 12) == set(ranked[:11])


def test_equals_best_first_when_drafts_do_not_depend_on_the_path():
    """Path-independent drafts (row = the depth's marginal) and k >= N-1: the
    dynamic tree is BASTION's best-first tree, node for node."""
    rng = np.random.default_rng(5)
    B, K, V = 3, 5, 40
    q = softmax_rows(rng.standard_normal((B, K, V)) * 1.5)
    root = rng.integers(0, V, size=B)
    for N in (2, 7, 16, 30):
        # every node at depth d gets the marginal of position d + 1
        k = N - 1
        M = oracle.pool_size(K, k)
        pool = oracle.new_pool(B, M, root)
        frontier = np.zeros((B, 1), dtype=np.int32)
        for level in range(1, K + 1):
            F = frontier.shape[1]
            rows = np.stack([[q[b, level - 1] for _ in range(F)] for b in range(B)])
            frontier = oracle.expand_level(rows, frontier, pool, k, level)
        got = oracle.dynamic_tree_rerank(pool, M, N)
        ref = oracle.best_first_tree(q, root, N)
        for x, y, name in zip(got, ref[:4], ["parent", "tokens", "depth", "rho"]):
            assert np.array_equal(x, y), (N, name)


def test_top1_is_the_greedy_chain():
    V, L = 30, 6
    q_of = node_q(9, V)
    pool, fr, (par, tok, dep, sco) = dynamic_tree(q_of, [3, 4], k=1, levels=L, N=L + 1, V=V)
    for b in range(2):
        assert list(par[b]) == [-1] + list(range(L))
        assert list(dep[b]) == list(range(L + 1))
        pid = 0
        for n in range(1, L + 1):
            assert tok[b, n] == int(np.argmax(q_of(b, pid)))
            pid = n  # k = 1: level l's single node has pool id l


def test_scores_are_fp32_products_along_the_path_and_the_tree_is_closed():
    V, k, L, N = 50, 4, 5, 40
    q_of = node_q(21, V, temp=0.7)
    pool, frontiers, (par, tok, dep, sco) = dynamic_tree(q_of, [0, 1, 2], k=k, levels=L, N=N, V=V)
    for b in range(3):
        p_par, p_tok, p_dep, p_sco = (a[b] for a in pool)
        for pid in range(1, pool_size(L, k)):
            chain = path_of(p_par, pid)
            s = np.float32(1.0)
            for a, c in zip(chain, chain[1:]):
                s = np.float32(s * q_of(b, a)[p_tok[c]])
            assert s == p_sco[pid]
            assert p_dep[pid] == len(chain) - 1
        assert par[b, 0] == -1 and dep[b, 0] == 0 and sco[b, 0] == 1.0
        for n in range(1, N):
            assert 0 <= par[b, n] < n
            assert dep[b, n] == dep[b, par[b, n]] + 1
            assert sco[b, n] <= sco[b, par[b, n]]
        # scores non-increasing in output order
        assert np.all(np.diff(sco[b, 1:].astype(np.float64)) <= 0)


def test_frontier_is_the_k_best_of_each_level():
    V, k, L = 25, 3, 4
    q_of = node_q(33, V)
    pool, frontiers, _ = dynamic_tree(q_of, [5], k=k, levels=L, N=5, V=V)
    p_dep, p_sco = pool[2][0], pool[3][0]
    for level, fr in enumerate(frontiers, start=1):
        ids = [i for i in range(1, pool_size(L, k)) if p_dep[i] == level]
        assert len(ids) == (k if level == 1 else k * k)
        ranked = sorted(ids, key=lambda i: (-float(p_sco[i]), i))
        assert list(fr[0]) == ranked[:k]
        # each level's parents are exactly the previous frontier
        if level >= 2:
            assert {int(pool[0][0][i]) for i in ids} == set(int(x) for x in frontiers[level - 2][0])


def test_closure_under_ties():
    """Quantised draft probabilities make many equal scores; the tie rule
    (shallower first) still keeps every parent before its children."""
    V, k, L, N = 6, 3, 4, 20
    levels = np.float32([0.5, 0.25, 0.125, 0.0625, 0.0625])

    def q_of(b, pid):
        rng = np.random.default_rng([77, b, pid])
        row = np.zeros(V, dtype=np.float32)
        row[rng.permutation(V)[:5]] = levels
        return row

    _, _, (par, tok, dep, sco) = dynamic_tree(q_of, [0, 1], k=k, levels=L, N=N, V=V)
    for b in range(2):
        for n in range(1, N):
            assert 0 <= par[b, n] < n and dep[b, n] == dep[b, par[b, n]] + 1


def test_deep_when_confident_wide_when_uncertain():
    """The page's qualitative claim: peaked drafts give deep, narrow trees;
    flat drafts give wide, shallow ones."""
    V, k, L, N = 200, 8, 8, 48
    _, _, (_, _, dep_peak, _) = dynamic_tree(node_q(1, V, temp=0.15), [0], k, L, N, V)
    _, _, (_, _, dep_flat, _) = dynamic_tree(node_q(1, V, temp=3.0), [0], k, L, N, V)
    assert dep_peak.mean() > dep_flat.mean() + 1.0
    assert (dep_flat == 1).sum() > (dep_peak == 1).sum()
