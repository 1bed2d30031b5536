"""Greedy verification of a draft tree: per-node argmax, then the longest
accepted path.

Follows [Blog] on Medusa trees (the target evaluates all branches in one
parallel pass and the longest valid path is selected) and [EP-zh] lay summary
section 3 (several candidate paths are checked at once and one that goes
through is kept), with greedy (temperature 0) acceptance: a draft token is
accepted when it equals the target's most likely token at its parent.

Readings taken where the pages are silent:

* argmax: exact fp32 comparisons on the logits, the first (lowest) index
  wins ties; +0.0 and -0.0 compare equal.  Inputs must be finite.
* acc(root) = true; acc(i) = acc(parent(i)) and tokens[i] == argmax[parent(i)].
* leaf = the accepted node of maximal depth, lowest real id on ties.
* accept_len = depth(leaf) (accepted draft tokens, the root excluded).
* path[k] = safe id (real id + 1) of the depth-k ancestor of the leaf, for
  k <= accept_len, then 0 up to D_max.
* bonus = argmax[leaf] (the target's own next token after the accepted path).
* A sequence with err != 0 is skipped: argmax row -1, accept_len 0, leaf -1,
  path all 0, bonus -1.  Padding rows of argmax are -1.
"""

from __future__ import annotations

import numpy as np

from .tree import build_ancestors, ancestor_chain


def verify_greedy(logits, tokens, parent, n_nodes, err, d_max: int):
    logits = np.asarray(logits)
    B, n_max, V = logits.shape
    argmax = np.full((B, n_max), -1, dtype=np.int32)
    accept_len = np.zeros(B, dtype=np.int32)
    leaf = np.full(B, -1, dtype=np.int32)
    path = np.zeros((B, d_max + 1), dtype=np.int32)
    bonus = np.full(B, -1, dtype=np.int32)
    for b in range(B):
        if int(err[b]) != 0:
            continue
        nb = n_max if n_nodes is None else int(n_nodes[b])
        rows = logits[b, :nb, :]
        if not np.all(np.isfinite(rows)):
            raise ValueError("oracle requires finite logits")
        am = np.argmax(rows, axis=1).astype(np.int32)  # first maximum
        argmax[b, :nb] = am
        par = np.asarray(parent[b])
        chains = [ancestor_chain(par, i) for i in range(nb)]
        acc = [False] * nb
        # visit nodes by increasing depth so the parent is decided first
        for i in sorted(range(nb), key=lambda x: len(chains[x])):
            if i == 0:
                acc[i] = True
            else:
                p = int(par[i])
                acc[i] = acc[p] and int(tokens[b, i]) == int(am[p])
        best = 0
        for i in range(nb):
            if acc[i] and (len(chains[i]) > len(chains[best])
                           or (len(chains[i]) == len(chains[best]) and i < best)):
                best = i
        A = len(chains[best]) - 1
        leaf[b] = best
        accept_len[b] = A
        for k, node in enumerate(chains[best]):
            path[b, k] = node + 1
        bonus[b] = am[best]
    return argmax, accept_len, leaf, path, bonus


def verify_greedy_all(logits, tokens, parent, n_nodes, d_max):
    _, _, _, err = build_ancestors(parent, n_nodes, d_max)
    return verify_greedy(logits, tokens, parent, n_nodes, err, d_max)
