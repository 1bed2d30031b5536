"""Commit of the accepted path's K/V into the committed cache.

Follows [EP-zh] 2.1 (branchable KV cache: length-based commit keeps the prefix
and the first A steps of the chosen branch; path-index commit reorders the
cache along the accepted path; the prefix-sharing fast reorder moves only the
newly accepted segment, and only when needed) and [EP-pt] section 2 (the fast
reorder preserves the accepted prefix to avoid needless memory movement).

Readings taken where the pages are silent:

* Before the call, sequence b's draft tree K/V sit in the paged cache at slot
  P_b + i for real node i (the speculative tail after the committed prefix).
* For k = 0..A: slot P_b + k receives the entry of slot P_b + (path[k] - 1).
  An entry already in place (path[k] - 1 == k) is not copied.  The root
  (k = 0) is always in place.
* All sources are read before any destination is written (a destination can
  be the source of a later path element).
* new_len[b] = P_b + A + 1; moved[b] = number of k with path[k] - 1 != k.
* A sequence with err != 0 commits nothing: new_len = P_b, moved = 0.
* Slots >= new_len are unspecified afterwards.
* The cache may hold several layers: [L][num_blocks][Hkv][16][D]; every layer
  is committed with the same path.
* The tree may sit elsewhere than right after the prefix: with tail_base[b]
  given, real node i's K/V are at slot tail_base[b] + i and slot P_b + k
  receives the entry of slot tail_base[b] + (path[k] - 1) (no copy when the
  two slots coincide).

Deferred commit (the pages' conclusion names commit efficiency as future
work; the fast reorder moves only what is out of place).  Instead of moving
the accepted entries, commit_remap records where each one already is: the
logical slot P_b + k of the committed sequence is read from physical slot
tail_base[b] + path[k] - 1 until a later copy moves it.  The next step's
attention reads through that record, and the next tree is placed after the
current one (next_tail = tail_base + N_b) so that nothing recorded is
overwritten.
"""

from __future__ import annotations

import numpy as np

PAGE = 16


def commit_path(k_cache, v_cache, block_table, prefix_len, accept_len, path, err,
                tail_base=None):
    """Returns (k_new, v_new, new_len, moved); inputs are not modified."""
    k_new = np.array(k_cache, copy=True)
    v_new = np.array(v_cache, copy=True)
    layered = k_new.ndim == 5
    if not layered:
        k_new = k_new[None]
        v_new = v_new[None]
    B = len(prefix_len)
    new_len = np.zeros(B, dtype=np.int32)
    moved = np.zeros(B, dtype=np.int32)

    def where(b, slot):
        return int(block_table[b, slot // PAGE]), slot % PAGE

    for b in range(B):
        P = int(prefix_len[b])
        if int(err[b]) != 0:
            new_len[b] = P
            continue
        A = int(accept_len[b])
        T = P if tail_base is None else int(tail_base[b])
        copies = []
        for k in range(A + 1):
            src = T + int(path[b, k]) - 1
            dst = P + k
            if src != dst:
                copies.append((dst, src))
        # read every source first
        staged = []
        for dst, src in copies:
            pg, row = where(b, src)
            staged.append((dst, k_new[:, pg, :, row, :].copy(), v_new[:, pg, :, row, :].copy()))
        for dst, kk, vv in staged:
            pg, row = where(b, dst)
            k_new[:, pg, :, row, :] = kk
            v_new[:, pg, :, row, :] = vv
        new_len[b] = P + A + 1
        moved[b] = len(copies)
    if not layered:
        k_new = k_new[0]
        v_new = v_new[0]
    return k_new, v_new, new_len, moved


def commit_remap(prefix_len, n_nodes, accept_len, path, err, tail_base=None):
    """Deferred commit: nothing moves.  Returns (remap_src [B][len(path[0])]
    physical slots of logical P_b + k (-1 beyond the accepted path), remap_base
    [B] = P_b, remap_len [B] = A + 1, new_len [B] = P_b + A + 1, next_tail [B]
    = where the next tree's node 0 goes).  A sequence with err != 0 records
    nothing: remap_len 0, new_len P_b, next_tail its current tail base."""
    B = len(prefix_len)
    width = np.asarray(path).shape[1]
    remap_src = np.full((B, width), -1, dtype=np.int32)
    remap_base = np.zeros(B, dtype=np.int32)
    remap_len = np.zeros(B, dtype=np.int32)
    new_len = np.zeros(B, dtype=np.int32)
    next_tail = np.zeros(B, dtype=np.int32)
    for b in range(B):
        P = int(prefix_len[b])
        T = P if tail_base is None else int(tail_base[b])
        remap_base[b] = P
        if int(err[b]) != 0:
            new_len[b] = P
            next_tail[b] = T
            continue
        A = int(accept_len[b])
        for k in range(A + 1):
            remap_src[b, k] = T + int(path[b, k]) - 1
        remap_len[b] = A + 1
        new_len[b] = P + A + 1
        next_tail[b] = T + int(n_nodes[b])
    return remap_src, remap_base, remap_len, new_len, next_tail
