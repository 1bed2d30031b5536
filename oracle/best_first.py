"""Best-first budgeted draft-tree construction from per-position marginals.

Follows [BASTION] Methodology 1 and 2: a block-diffusion drafter gives
per-position marginals q_k(.) for k = 1..K in one pass; node i at depth d(i)
has path score rho(i) = prod_{k=1}^{d(i)} q_k(x_ik); the acceptance surrogate
is A_hat(T) = sum_{i in T} rho(i); best-first expansion repeatedly adds the
valid node with the largest rho until the node budget is used.

Readings taken where the pages are silent:

* The budget N counts the root (the last emitted token, depth 0, rho = 1).
* rho is computed as an fp32 product, rho(child) = fl32(rho(parent) * q), so
  that rankings can be reproduced bit for bit.
* A "valid" node is a child of a node already in the tree, at depth <= K.
* Ties: candidates are ordered by (rho desc, depth asc, parent insertion index
  asc, token rank asc); a position's token rank orders q_k descending with the
  lower token id first on ties.
* Output order is insertion order, so every parent precedes its children.
* A_hat sums rho over the non-root nodes in fp64, in insertion order.

This is the plain scan: at every step, each inserted node's best
not-yet-inserted child is considered and the best of those is taken.
"""

from __future__ import annotations

import numpy as np


def ranked_tokens(q_row: np.ndarray) -> np.ndarray:
    """Token ids sorted by probability descending, lower id first on ties."""
    q_row = np.asarray(q_row, dtype=np.float32)
    ids = np.arange(len(q_row))
    return np.lexsort((ids, -q_row.astype(np.float64)))


def best_first_tree(q, root_token, N: int):
    """q: float32 [B][K][V] marginals; root_token: int [B]; N: node budget.
    Returns parent, tokens, depth (int32 [B][N]), rho (float32 [B][N]),
    ahat (float64 [B])."""
    q = np.asarray(q, dtype=np.float32)
    B, K, V = q.shape
    parent = np.full((B, N), -1, dtype=np.int32)
    tokens = np.zeros((B, N), dtype=np.int32)
    depth = np.zeros((B, N), dtype=np.int32)
    rho = np.zeros((B, N), dtype=np.float32)
    ahat = np.zeros(B, dtype=np.float64)
    for b in range(B):
        ranks = [ranked_tokens(q[b, k]) for k in range(K)]
        nodes_par = [-1]
        nodes_tok = [int(root_token[b])]
        nodes_dep = [0]
        nodes_rho = [np.float32(1.0)]
        nchild = [0]
        for _ in range(1, N):
            best = None
            best_key = None
            for p in range(len(nodes_par)):
                d = nodes_dep[p] + 1
                r = nchild[p]
                if d > K or r >= V:
                    continue
                tok = int(ranks[d - 1][r])
                cand = np.float32(nodes_rho[p] * q[b, d - 1, tok])
                key = (-float(cand), d, p, r)
                if best_key is None or key < best_key:
                    best_key = key
                    best = (p, d, r, tok, cand)
            if best is None:
                raise ValueError("budget larger than the number of valid nodes")
            p, d, r, tok, cand = best
            nodes_par.append(p)
            nodes_tok.append(tok)
            nodes_dep.append(d)
            nodes_rho.append(cand)
            nchild.append(0)
            nchild[p] += 1
        parent[b] = nodes_par
        tokens[b] = nodes_tok
        depth[b] = nodes_dep
        rho[b] = nodes_rho
        s = 0.0
        for n in range(1, N):
            s += float(nodes_rho[n])
        ahat[b] = s
    return parent, tokens, depth, rho, ahat
