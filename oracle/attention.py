"""Tree-masked attention for all draft-tree nodes in one pass.

Follows [EP-zh] 2.3 (the teacher evaluates every speculative node at once
under a tree attention mask; node k attends only to the nodes on its own
ancestor path, itself included, with no leakage across branches), [EP-pt]
section 2 ("Execução do Professor com Máscara de Árvore Fundida") and [Blog]
on Medusa tree attention (parallel nodes attend only to their direct
ancestors).

Readings taken where the pages are silent:

* Every node sees the whole committed prefix, slots [0, P_b).  Tail slot
  P_b + j (the K/V of real node j) is visible to node i iff j is i or an
  ancestor of i.
* Scores are q . k * scale with scale = 1/sqrt(D) by default; softmax over the
  visible keys; output = sum softmax * v.  No positional rotation is applied
  here (the caller rotates with position P_b + depth(i)).
* GQA: query head h reads kv head h // (Hq // Hkv).
* lse is the natural log of the sum of exp(score) over visible keys.
* Rows that are not computed (sequence with err != 0, padding node) are
  reported as out = 0, lse = -inf.

The cache is paged: K, V are [num_blocks][Hkv][16][D] bf16 (as uint16 bits),
token slot t of sequence b lives in block block_table[b][t // 16], row t % 16.
All arithmetic is fp64 on the exact bf16 values.

Reading through a deferred commit (tree_attention_remapped): logical slot
s of the committed sequence is physical slot remap_src[b][s - remap_base[b]]
for s in [remap_base[b], remap_base[b] + remap_len[b]), else slot s; the tree's
node j is at physical slot tail_base[b] + j.  The keys a node sees, and their
order, are those of the sequence the copy commit would have produced.
"""

from __future__ import annotations

import numpy as np

from .tree import build_ancestors, ancestor_chain

PAGE = 16


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact conversion of bf16 bit patterns to fp64 (bf16 is the top half of
    an fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def gather_sequence_kv(cache: np.ndarray, block_table: np.ndarray, b: int, hkv: int,
                       n_slots: int) -> np.ndarray:
    """fp64 [n_slots][D] rows of one kv head of one sequence, slot order."""
    rows = []
    for t0 in range(0, n_slots, PAGE):
        page = int(block_table[b, t0 // PAGE])
        take = min(PAGE, n_slots - t0)
        rows.append(cache[page, hkv, :take, :])
    if not rows:
        return np.zeros((0, cache.shape[-1]), dtype=np.float64)
    return bf16_to_f64(np.concatenate(rows, axis=0))


def gather_slots_kv(cache: np.ndarray, block_table: np.ndarray, b: int, hkv: int,
                    slots) -> np.ndarray:
    """fp64 [len(slots)][D] rows of one kv head of one sequence, at the given
    physical slots, in that order."""
    rows = [cache[int(block_table[b, s // PAGE]), hkv, s % PAGE, :] for s in slots]
    if not rows:
        return np.zeros((0, cache.shape[-1]), dtype=np.float64)
    return bf16_to_f64(np.stack(rows, axis=0))


def tree_attention(q, k_cache, v_cache, block_table, prefix_len, n_nodes, parent, err,
                   scale: float, sample=None, remap=None):
    """Reference tree attention.

    q: uint16 [B][N_max][Hq][D]; k_cache, v_cache: uint16 [num_blocks][Hkv][16][D].
    parent: int [B][N_max]; err: int [B] (sequences with err != 0 are skipped).
    sample: optional iterable of (b, i, h) to compute; others stay 0 / -inf.
    remap: optional (remap_src, remap_base, remap_len, tail_base) of a deferred
    commit (see the module notes).
    Returns out fp64 [B][N_max][Hq][D], lse fp64 [B][N_max][Hq].
    """
    q = np.asarray(q)
    B, n_max, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, n_max, Hq, D), dtype=np.float64)
    lse = np.full((B, n_max, Hq), -np.inf, dtype=np.float64)

    wanted = None
    if sample is not None:
        wanted = {}
        for (b, i, h) in sample:
            wanted.setdefault(int(b), set()).add((int(i), int(h)))

    for b in range(B):
        if int(err[b]) != 0:
            continue
        if wanted is not None and b not in wanted:
            continue
        nb = n_max if n_nodes is None else int(n_nodes[b])
        P = int(prefix_len[b])
        par = np.asarray(parent[b])
        # visible[i][j]: tail slot P + j visible to node i
        visible = np.zeros((nb, nb), dtype=bool)
        for i in range(nb):
            for j in ancestor_chain(par, i):
                visible[i, j] = True
        for hkv in range(Hkv):
            heads = [hkv * g + x for x in range(g)]
            if wanted is not None and not any(h in heads for (_, h) in wanted[b]):
                continue
            if remap is None:
                K = gather_sequence_kv(k_cache, block_table, b, hkv, P + nb)
                V = gather_sequence_kv(v_cache, block_table, b, hkv, P + nb)
            else:
                slots = physical_slots(remap, b, P, nb)
                K = gather_slots_kv(k_cache, block_table, b, hkv, slots)
                V = gather_slots_kv(v_cache, block_table, b, hkv, slots)
            for h in heads:
                if wanted is not None:
                    nodes = sorted(i for (i, hh) in wanted[b] if hh == h and i < nb)
                else:
                    nodes = list(range(nb))
                if not nodes:
                    continue
                Q = bf16_to_f64(q[b, nodes, h, :])                 # [n][D]
                S = (Q @ K.T) * float(scale)                      # [n][P + nb]
                keep = np.ones_like(S, dtype=bool)
                keep[:, P:] = visible[nodes, :]
                S = np.where(keep, S, -np.inf)
                m = S.max(axis=1, keepdims=True)
                w = np.exp(S - m)
                l = w.sum(axis=1, keepdims=True)
                out[b, nodes, h, :] = (w @ V) / l
                lse[b, nodes, h] = (m + np.log(l))[:, 0]
    return out, lse


def physical_slots(remap, b: int, P: int, nb: int):
    """Physical slot of every logical key of sequence b, in logical order: the
    committed prefix [0, P) through the deferred commit's record, then the
    tree's nb nodes from tail_base."""
    remap_src, remap_base, remap_len, tail_base = remap
    rb, rl = int(remap_base[b]), int(remap_len[b])
    out = []
    for s in range(P):
        out.append(int(remap_src[b, s - rb]) if rb <= s < rb + rl else s)
    T = int(tail_base[b])
    out.extend(T + j for j in range(nb))
    return out


def tree_attention_all(q, k_cache, v_cache, block_table, prefix_len, n_nodes, parent, d_max,
                       scale):
    """Convenience: run the structural checks first, then attention."""
    _, _, _, err = build_ancestors(parent, n_nodes, d_max)
    return tree_attention(q, k_cache, v_cache, block_table, prefix_len, n_nodes, parent, err,
                          scale)
