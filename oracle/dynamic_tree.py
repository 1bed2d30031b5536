"""Dynamic draft trees: confidence-driven expansion and reranking (CPU only;
test infrastructure, never on the product path).

[Blog], EAGLE-2 section: dynamic draft trees grow deep and narrow where the
drafter is confident and wide with short branches where it is uncertain.  The
page gives that behaviour, not an algorithm.  The reading taken here (the
plainest one the pages support, with [BASTION] Methodology 1-2's path
confidence as the node score):

* Scores.  The root (the last emitted token, pool id 0, depth 0) has score 1; a
  child of node p with draft probability q for its token has score
  fl32(score(p) * q) -- the product of draft probabilities along the path, as
  an fp32 product so rankings reproduce bit for bit.
* Expansion, level by level.  Level 1: the root proposes its top-k tokens.
  Level l >= 2: each of the k frontier nodes of level l-1 proposes its top-k
  tokens (from its own draft distribution, which the drafter computes for that
  node).  A node's token rank sorts its q row descending, lower token id first
  on ties.  The frontier of a level is its k best nodes by (score desc, pool id
  asc).
* Pool ids.  Root 0; level 1 nodes 1..k (token rank j at 1 + j); level l >= 2
  nodes at 1 + k + (l-2) k^2 + f k + j for frontier slot f (in frontier order)
  and token rank j.
* Reranking.  The draft tree of N nodes keeps the root and the N-1 best non-root
  pool nodes by (score desc, depth asc, pool id asc), output in that order.
  A child's score never exceeds its parent's (q <= 1) and the parent is
  shallower, so every kept node's parent is kept and comes first.

Everything here is a plain scan over Python lists; no step is fused.
"""

from __future__ import annotations

import numpy as np

from .best_first import ranked_tokens


def pool_base(level: int, k: int) -> int:
    """First pool id of a level (level >= 1)."""
    return 1 if level == 1 else 1 + k + (level - 2) * k * k


def pool_size(levels: int, k: int) -> int:
    """Pool ids used by `levels` expansion levels, root included."""
    return 1 if levels == 0 else pool_base(levels, k) + (k if levels == 1 else k * k)


def new_pool(B: int, M: int, root_token):
    """Pool arrays with the root in place: parent, token, depth, score."""
    parent = np.full((B, M), -1, dtype=np.int32)
    token = np.zeros((B, M), dtype=np.int32)
    depth = np.zeros((B, M), dtype=np.int32)
    score = np.zeros((B, M), dtype=np.float32)
    token[:, 0] = np.asarray(root_token, dtype=np.int32)
    score[:, 0] = np.float32(1.0)
    return parent, token, depth, score


def expand_level(q_rows, frontier, pool, k: int, level: int):
    """One level of expansion.

    q_rows   float32 [B][F][V]: draft distribution of each frontier node
             (F = 1 at level 1, the root; F = k after).
    frontier int [B][F]: pool ids of the frontier nodes, in frontier order.
    pool     (parent, token, depth, score) arrays, updated in place.
    Returns the next frontier, int32 [B][k]: this level's k best nodes by
    (score desc, pool id asc).
    """
    parent, token, depth, score = pool
    q_rows = np.asarray(q_rows, dtype=np.float32)
    B, F, V = q_rows.shape
    base = pool_base(level, k)
    nxt = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        cands = []
        for f in range(F):
            p = int(frontier[b][f])
            ranks = ranked_tokens(q_rows[b, f])
            for j in range(k):
                tok = int(ranks[j])
                pid = base + f * k + j
                s = np.float32(score[b, p] * q_rows[b, f, tok])
                parent[b, pid] = p
                token[b, pid] = tok
                depth[b, pid] = level
                score[b, pid] = s
                cands.append((-float(s), pid))
        cands.sort()
        nxt[b] = [pid for _, pid in cands[:k]]
    return nxt


def rerank(pool, M: int, N: int):
    """The N-node draft tree: the root and the N-1 best non-root pool nodes
    among pool ids 1..M-1 by (score desc, depth asc, pool id asc), in that
    order, with parents re-indexed to output positions.
    Returns parent, tokens, depth (int32 [B][N]), score (float32 [B][N])."""
    p_par, p_tok, p_dep, p_sco = pool
    B = p_par.shape[0]
    parent = np.zeros((B, N), dtype=np.int32)
    tokens = np.zeros((B, N), dtype=np.int32)
    depth = np.zeros((B, N), dtype=np.int32)
    score = np.zeros((B, N), dtype=np.float32)
    for b in range(B):
        order = sorted(range(1, M), key=lambda i: (-float(p_sco[b, i]), int(p_dep[b, i]), i))
        keep = [0] + order[:N - 1]
        where = {pid: n for n, pid in enumerate(keep)}
        for n, pid in enumerate(keep):
            parent[b, n] = -1 if pid == 0 else where[int(p_par[b, pid])]
            tokens[b, n] = p_tok[b, pid]
            depth[b, n] = p_dep[b, pid]
            score[b, n] = p_sco[b, pid]
    return parent, tokens, depth, score


def dynamic_tree(q_of, root_token, k: int, levels: int, N: int, V: int):
    """Whole construction for tests: q_of(b, pool_id) -> float32 [V], the
    draft distribution the drafter gives at that node.  Returns the pool (after
    `levels` levels), the frontiers of every level, and the reranked tree."""
    B = len(root_token)
    M = pool_size(levels, k)
    pool = new_pool(B, M, root_token)
    frontier = np.zeros((B, 1), dtype=np.int32)
    frontiers = []
    for level in range(1, levels + 1):
        F = frontier.shape[1]
        q_rows = np.zeros((B, F, V), dtype=np.float32)
        for b in range(B):
            for f in range(F):
                q_rows[b, f] = q_of(b, int(frontier[b, f]))
        frontier = expand_level(q_rows, frontier, pool, k, level)
        frontiers.append(frontier.copy())
    return pool, frontiers, rerank(pool, M, N)
