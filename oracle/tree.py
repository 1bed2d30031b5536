"""Accelerator-safe tree tensors: virtual root, ancestor table, bitmask, checks.

Follows [EP-zh] 2.2 and [EP-pt] section 2 ("Semântica de Tensores em Árvore
Segura"): node ids are shifted so that a virtual root row sits at index 0, the
old root's parent sentinel -1 becomes 0, an ancestor index table A is built
whose every entry lies in [0, M], and range / acyclicity / validity-closure
checks run before any fused kernel.

Readings taken where the pages are silent:

* Input ids are real ids 0..N_b-1, node 0 is the tree root with parent -1.
  Safe ids are s = i + 1; row 0 of every safe table is the virtual root.
* depth(root) = 0, depth(i) = depth(parent(i)) + 1; anc[s][d] is the safe id
  of the depth-d ancestor of s (d <= depth), 0 beyond the node's depth.
* Parents may come in any order (acyclicity is a check, so topological order
  cannot be assumed).
* err[b] bits: 1 RANGE (a parent outside [0, N_max) for a non-root node,
  including a second -1), 2 CYCLE (the walk up does not reach the root within
  N_b steps), 4 TOO_DEEP (depth > D_max), 8 CLOSURE (a valid node whose parent
  is a padding node, N_b <= parent < N_max), 16 ROOT (parent[0] != -1),
  32 COUNT (n_nodes[b] outside [1, N_max]).  RANGE/CLOSURE/ROOT are checked
  first; CYCLE/TOO_DEEP only when those are clear.  A sequence with any bit set
  gets all-zero rows (fail closed).
* mask[b][i] is a bitmask over real ids: bit j set iff j is i or an ancestor
  of i.  Padding rows are zero.
"""

from __future__ import annotations

import numpy as np

ERR_RANGE = 1
ERR_CYCLE = 2
ERR_TOO_DEEP = 4
ERR_CLOSURE = 8
ERR_ROOT = 16
ERR_COUNT = 32


def _check_sequence(par: np.ndarray, nb: int, n_max: int, d_max: int):
    """Return (err, depths) for one sequence; depths only meaningful if err==0."""
    e = 0
    if int(par[0]) != -1:
        e |= ERR_ROOT
    for i in range(1, nb):
        p = int(par[i])
        if p < 0 or p >= n_max:
            e |= ERR_RANGE
        elif p >= nb:
            e |= ERR_CLOSURE
    depths = [0] * nb
    if e:
        return e, depths
    for i in range(nb):
        j, steps, cycle = i, 0, False
        while int(par[j]) != -1:
            if steps == nb:
                cycle = True
                break
            j = int(par[j])
            steps += 1
        if cycle:
            e |= ERR_CYCLE
        else:
            depths[i] = steps
            if steps > d_max:
                e |= ERR_TOO_DEEP
    return e, depths


def ancestor_chain(par: np.ndarray, i: int):
    """Real ids on the path from the root down to node i (root first).  The
    tree must already have passed the checks."""
    chain = [i]
    j = i
    while int(par[j]) != -1:
        j = int(par[j])
        chain.append(j)
    return chain[::-1]


def build_ancestors(parent, n_nodes, d_max: int):
    """Safe ancestor table, depth, ancestor bitmask and error bits.

    parent: int [B][N_max] real ids with -1 for the root.
    n_nodes: int [B] or None (then every sequence has N_max nodes).
    Returns anc int32 [B][N_max+1][d_max+1], depth int32 [B][N_max],
    mask uint32 [B][N_max][ceil(N_max/32)], err int32 [B].
    """
    parent = np.asarray(parent)
    B, n_max = parent.shape
    W = (n_max + 31) // 32
    anc = np.zeros((B, n_max + 1, d_max + 1), dtype=np.int32)
    depth = np.zeros((B, n_max), dtype=np.int32)
    mask = np.zeros((B, n_max, W), dtype=np.uint32)
    err = np.zeros(B, dtype=np.int32)
    for b in range(B):
        nb = n_max if n_nodes is None else int(n_nodes[b])
        if nb < 1 or nb > n_max:
            err[b] = ERR_COUNT
            continue
        par = parent[b]
        e, depths = _check_sequence(par, nb, n_max, d_max)
        if e:
            err[b] = e
            continue
        for i in range(nb):
            chain = ancestor_chain(par, i)  # chain[d] = depth-d ancestor
            depth[b, i] = depths[i]
            for d, a in enumerate(chain):
                anc[b, i + 1, d] = a + 1
                mask[b, i, a // 32] |= np.uint32(1 << (a % 32))
    return anc, depth, mask, err
