"""Stochastic verification of a draft tree by modified rejection sampling
(CPU only; test infrastructure, never on the product path).

Follows [Blog], section on classic speculative decoding and modified
rejection sampling: a drafted token x drawn from the draft distribution q is
accepted with probability min(1, p(x)/q(x)); on rejection a corrective token is
drawn from the normalised residual max(0, p - q); the emitted token is then
distributed exactly as the target p.  [Blog] on Medusa trees: the target scores
every branch of the tree in one pass and one path is kept.

The page gives the rule for one drafted token (a chain).  Readings taken for a
tree, where the pages are silent:

* Node i's children are candidates for the token that follows node i; they
  are taken to be independent draws from q_i (the draft distribution at node
  i, row i of ``q``) and are tried in increasing id order.  The first child is
  tested against r_0 = p_i = softmax(logits[i]); after each rejection the
  current distribution r is replaced by the page's residual
  norm(max(0, r - q_i)) and the next child is tested against it.  With
  independent draws this keeps the emitted token distributed as p_i (checked
  exactly by the pins).
* Acceptance of child c with token x: u_accept[c] * q_i(x) < r(x), the page's
  "u < min(1, r(x)/q(x))" without the division (the min is implied by u < 1;
  q_i(x) = 0 accepts iff r(x) > 0).
* A residual with no mass can only arise when r equals q_i (then no rejection
  is possible in exact arithmetic); the residual is then taken to be q_i.
* When every child is rejected (or node i is a leaf), node i draws a token
  from its current distribution r by inverse CDF in token order with the
  uniform u_draw[i]: the first token t whose cumulative weight exceeds
  u_draw[i] * (total weight); if rounding leaves none, the last token of
  positive weight.
* The walk starts at the root and follows each node's accepted child; it ends
  at the first node with none.  accept_len = the number of accepted draft
  nodes (depth of the last node), leaf = that node, bonus = its draw,
  path[k] = safe id (real id + 1) of the depth-k node of the walk, 0 beyond.
* A child whose token lies outside [0, V) is skipped: it is never accepted
  and leaves the residual unchanged (the kernel cannot index such a token).
* Every node is decided independently of whether the walk reaches it (the
  decisions use only the node's own row, children and uniforms), so
  ``next_child`` is defined for all valid nodes, and so is ``draw`` for every
  node whose children were all rejected.  A leaf draws only when it is the
  walk's last node (its draw is then the bonus token); the other leaves'
  draw entries are -1, since no token is ever taken from them.
* A sequence with err != 0 is skipped: rows of next_child and draw -1,
  accept_len 0, leaf -1, path 0, bonus -1.  Padding rows are -1.

Random numbers are inputs (uniforms in [0, 1)): u_accept[b][c] is used for the
test of child c at its parent, u_draw[b][i] for a draw at node i.  Arithmetic is
fp64; ``margins`` reports, per node, how far each used uniform lies from the
decision it feeds (relative), for callers comparing against another precision.
"""

from __future__ import annotations

import numpy as np

from .tree import build_ancestors


def _draw(w: np.ndarray, u: float):
    """Inverse CDF of the (unnormalised) weights w with uniform u.
    Returns (token, margin) where margin = distance of u * total from the
    nearest cumulative boundary of the chosen token, relative to the total."""
    c = np.cumsum(w)
    total = c[-1]
    tau = u * total
    hit = np.nonzero(c > tau)[0]
    if hit.size:
        t = int(hit[0])
    else:
        pos = np.nonzero(w > 0)[0]
        return (int(pos[-1]) if pos.size else len(w) - 1), 0.0
    lo = c[t - 1] if t > 0 else 0.0
    margin = min(tau - lo, c[t] - tau) / total
    return t, float(margin)


def node_decision(logits_row, q_row, child_ids, child_tokens, u_accept, u_draw):
    """Decide one node.  child_ids in increasing order; u_accept indexed by
    child id.  Returns (accepted child id or -1, drawn token or -1,
    acceptance margin, draw margin)."""
    l = np.asarray(logits_row, dtype=np.float64)
    q = np.asarray(q_row, dtype=np.float64)
    if not (np.all(np.isfinite(l)) and np.all(np.isfinite(q)) and np.all(q >= 0)):
        raise ValueError("oracle requires finite logits and finite non-negative q")
    w = np.exp(l - l.max())
    r = w / w.sum()
    acc_margin = np.inf
    for c, x in zip(child_ids, child_tokens):
        u = float(u_accept[c])
        lhs, rhs = u * q[x], r[x]
        scale = max(lhs, rhs)
        # both sides exactly zero (q(x) = 0 and r(x) underflowed): rejected
        # whatever u is, so no uniform is near this decision
        acc_margin = min(acc_margin, abs(lhs - rhs) / scale if scale > 0 else np.inf)
        if lhs < rhs:
            return int(c), -1, float(acc_margin), np.inf
        res = np.maximum(0.0, r - q)
        z = res.sum()
        if z > 0.0:
            r = res / z
        else:
            r = q / q.sum()
    tok, dm = _draw(r, float(u_draw))
    return -1, tok, float(acc_margin), dm


def tree_verify_stochastic(logits, q, tokens, parent, n_nodes, err, d_max: int, u_accept, u_draw,
                           return_margins: bool = False):
    """logits, q: [B][N_max][V]; tokens, parent: [B][N_max]; n_nodes: [B] or
    None; err: [B] (from the ancestor tables); u_accept, u_draw: [B][N_max].
    Returns (next_child, draw, accept_len, leaf, path, bonus) and, with
    return_margins, also (acc_margin, draw_margin) [B][N_max]."""
    logits = np.asarray(logits)
    q = np.asarray(q)
    B, n_max, V = logits.shape
    nxt = np.full((B, n_max), -1, dtype=np.int32)
    drw = np.full((B, n_max), -1, dtype=np.int32)
    acc_m = np.full((B, n_max), np.inf)
    drw_m = np.full((B, n_max), np.inf)
    accept_len = np.zeros(B, dtype=np.int32)
    leaf = np.full(B, -1, dtype=np.int32)
    path = np.zeros((B, d_max + 1), dtype=np.int32)
    bonus = np.full(B, -1, dtype=np.int32)
    for b in range(B):
        if int(err[b]) != 0:
            continue
        nb = n_max if n_nodes is None else int(n_nodes[b])
        par = [int(x) for x in parent[b][:nb]]
        for i in range(nb):
            kids = [j for j in range(1, nb) if par[j] == i and 0 <= int(tokens[b][j]) < V]
            toks = [int(tokens[b][j]) for j in kids]
            c, t, am, dm = node_decision(logits[b, i], q[b, i], kids, toks, u_accept[b],
                                         u_draw[b][i])
            nxt[b, i], drw[b, i], acc_m[b, i], drw_m[b, i] = c, t, am, dm
        walk = [0]
        while nxt[b, walk[-1]] >= 0:
            walk.append(int(nxt[b, walk[-1]]))
        for i in range(nb):
            leaf_node = not any(par[j] == i and 0 <= int(tokens[b][j]) < V for j in range(1, nb))
            if leaf_node and i != walk[-1]:
                drw[b, i] = -1
                drw_m[b, i] = np.inf
        if len(walk) - 1 > d_max:
            raise ValueError("walk deeper than D_max on a tree that passed the checks")
        accept_len[b] = len(walk) - 1
        leaf[b] = walk[-1]
        bonus[b] = drw[b, walk[-1]]
        for k, node in enumerate(walk):
            path[b, k] = node + 1
    out = (nxt, drw, accept_len, leaf, path, bonus)
    if return_margins:
        return out + (acc_m, drw_m)
    return out


def tree_verify_stochastic_all(logits, q, tokens, parent, n_nodes, d_max, u_accept, u_draw,
                               return_margins: bool = False):
    _, _, _, err = build_ancestors(parent, n_nodes, d_max)
    return tree_verify_stochastic(logits, q, tokens, parent, n_nodes, err, d_max, u_accept, u_draw,
                                  return_margins)


__all__ = ["node_decision", "tree_verify_stochastic", "tree_verify_stochastic_all"]
