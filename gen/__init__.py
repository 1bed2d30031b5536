"""Seeded synthetic inputs for the tree-verify hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no ancestor tables, no attention, no argmax, no
acceptance, no commit, no path scores).  Both the CPU oracle (through the
tests) and the CUDA path read the arrays it returns, so the two sides always
see identical bits.

Shapes follow the five verify workloads:

* ``tiny``    B=1, Hq=Hkv=4, D=64, prefix 128, 15-node random tree
              (depth <= 4, <= 3 children), V=1000, logits N(0,1), match 0.5.
* ``8b``      B=1, Hq=32, Hkv=8, D=128, prefix 4096, 63-node static
              level-order tree (depth 6), V=128256, logits N(0,2), match 0.7.
* ``ragged``  B=16, Hq=32, Hkv=8, D=128, prefix ~ U[512, 8192], 31-node random
              trees (depth <= 5), V=32000, logits N(0,1), match 0.6.
* ``70b``     B=4, Hq=64, Hkv=8, D=128, prefix 32768, 127-node random trees
              (depth <= 8), V=128256, logits N(0,2), match 0.7, paged cache
              with a shuffled block table.
* ``bastion`` B=8, K=16 draft positions, V=32000, draft marginals
              softmax(N(0,2)) in fp32; the verify layer is the 8B shape with
              prefix 2048.

N(0,2) is read as variance 2.  Every row of target logits carries one planted
target token whose logit is set to (row maximum + 1), so the target's greedy
choice for each node is known by construction; a draft token "matches" when
it equals the planted target of its parent.

bf16 tensors are returned as ``uint16`` bit patterns (round to nearest even
from an fp32 draw).
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

PAGE = 16  # tokens per KV-cache block

# --------------------------------------------------------------------------
# primitive draws
# --------------------------------------------------------------------------


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x)


def random_tree(rng: np.random.Generator, n: int, max_depth: int,
                max_children: Optional[int] = None) -> np.ndarray:
    """Parent array (root parent = -1).  Node i>0 picks its parent uniformly
    among earlier nodes whose depth is < max_depth and (optionally) that have
    fewer than max_children children."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = [0]
    kids = [0]
    for i in range(1, n):
        ok = [j for j in range(i)
              if depth[j] < max_depth and (max_children is None or kids[j] < max_children)]
        if not ok:
            raise ValueError("tree constraints leave no parent for node %d" % i)
        p = ok[int(rng.integers(len(ok)))]
        parent[i] = p
        depth.append(depth[p] + 1)
        kids.append(0)
        kids[p] += 1
    return parent


def level_order_tree(level_sizes: List[int], fanouts: List[List[int]]) -> np.ndarray:
    """Static tree given level sizes and, for each level, the child counts of
    that level's first nodes (the highest-ranked ones)."""
    assert level_sizes[0] == 1
    parent = [-1]
    prev = [0]
    nxt = 1
    for lvl in range(1, len(level_sizes)):
        counts = fanouts[lvl - 1]
        assert sum(counts) == level_sizes[lvl], (lvl, counts)
        cur = []
        for rank, c in enumerate(counts):
            for _ in range(c):
                parent.append(prev[rank])
                cur.append(nxt)
                nxt += 1
        prev = cur
    return np.asarray(parent, dtype=np.int32)


# Our own static shape for the 8B workload: level sizes 1, 8, 16, 16, 10, 8, 4.
STATIC_8B_LEVELS = [1, 8, 16, 16, 10, 8, 4]
STATIC_8B_FANOUT = [
    [8],
    [4, 3, 2, 2, 2, 1, 1, 1],
    [4, 3, 2, 2, 1, 1, 1, 1, 1],
    [3, 2, 2, 1, 1, 1],
    [2, 2, 1, 1, 1, 1],
    [1, 1, 1, 1],
]


def static_8b_tree() -> np.ndarray:
    return level_order_tree(STATIC_8B_LEVELS, STATIC_8B_FANOUT)


def chain_tree(n: int) -> np.ndarray:
    p = np.arange(-1, n - 1, dtype=np.int32)
    return p


def relabel(rng: np.random.Generator, parent: np.ndarray) -> np.ndarray:
    """Randomly permute the ids of nodes 1..n-1 (root stays 0), so parents may
    come after their children."""
    n = len(parent)
    perm = np.concatenate([[0], 1 + rng.permutation(n - 1)]).astype(np.int64)
    out = np.full(n, -1, dtype=np.int32)
    for old in range(1, n):
        out[perm[old]] = perm[parent[old]]
    return out


def plant_targets(logits: np.ndarray, targets: np.ndarray) -> None:
    """In place: for each row r, set logits[r, targets[r]] = max(row) + 1."""
    flat = logits.reshape(-1, logits.shape[-1])
    t = targets.reshape(-1)
    mx = flat.max(axis=1)
    flat[np.arange(flat.shape[0]), t] = mx + np.float32(1.0)


def draft_tokens(rng: np.random.Generator, parent: np.ndarray, targets: np.ndarray,
                 p_match: float, vocab: int) -> np.ndarray:
    """tokens[i] = targets[parent[i]] with probability p_match, else uniform.
    The root's token is uniform (it is the token emitted by the last step)."""
    n = len(parent)
    tok = rng.integers(0, vocab, size=n, dtype=np.int64)
    coin = rng.random(n)
    for i in range(1, n):
        if parent[i] >= 0 and coin[i] < p_match:
            tok[i] = targets[parent[i]]
    return tok.astype(np.int32)


# --------------------------------------------------------------------------
# paged KV cache
# --------------------------------------------------------------------------


@dataclasses.dataclass
class PagedCache:
    k: np.ndarray            # uint16 [num_blocks][Hkv][PAGE][D]
    v: np.ndarray            # uint16 [num_blocks][Hkv][PAGE][D]
    block_table: np.ndarray  # int32 [B][max_blocks]
    num_blocks: int
    max_blocks: int


def paged_cache(rng: np.random.Generator, prefix_len: np.ndarray, n_nodes: np.ndarray,
                hkv: int, d: int, shuffle: bool, spare_blocks: int = 0) -> PagedCache:
    """Cache pool holding, for each sequence b, slots [0, P_b + N_b): the
    committed prefix followed by the draft tree's own K/V (slot P_b + i holds
    real node i).  Every slot in the pool is N(0,1) bf16."""
    B = len(prefix_len)
    need = [(int(prefix_len[b]) + int(n_nodes[b]) + PAGE - 1) // PAGE for b in range(B)]
    max_blocks = max(need) if B else 1
    num_blocks = sum(need) + spare_blocks
    ids = np.arange(num_blocks, dtype=np.int32)
    if shuffle:
        ids = rng.permutation(num_blocks).astype(np.int32)
    table = np.zeros((B, max_blocks), dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :need[b]] = ids[pos:pos + need[b]]
        pos += need[b]
    k = normal_bf16(rng, (num_blocks, hkv, PAGE, d))
    v = normal_bf16(rng, (num_blocks, hkv, PAGE, d))
    return PagedCache(k=k, v=v, block_table=table, num_blocks=num_blocks, max_blocks=max_blocks)


def grow_cache(rng: np.random.Generator, cache: PagedCache, prefix_len: np.ndarray,
               n_nodes: np.ndarray, extra: int) -> PagedCache:
    """A copy of `cache` whose block table also covers `extra` more slots per
    sequence, past slot P_b + N_b: fresh blocks appended to the pool (N(0,1)
    bf16, in shuffled order), the existing blocks and table entries kept."""
    B = len(prefix_len)
    have = [(int(prefix_len[b]) + int(n_nodes[b]) + PAGE - 1) // PAGE for b in range(B)]
    need = [(int(prefix_len[b]) + int(n_nodes[b]) + extra + PAGE - 1) // PAGE for b in range(B)]
    add = [need[b] - have[b] for b in range(B)]
    num_blocks = cache.num_blocks + sum(add)
    fresh = (cache.num_blocks + rng.permutation(sum(add))).astype(np.int32)
    table = np.zeros((B, max(max(need), cache.max_blocks)), dtype=np.int32)
    table[:, :cache.block_table.shape[1]] = cache.block_table
    pos = 0
    for b in range(B):
        table[b, have[b]:need[b]] = fresh[pos:pos + add[b]]
        pos += add[b]
    hkv, d = cache.k.shape[1], cache.k.shape[3]
    k = np.concatenate([cache.k, normal_bf16(rng, (sum(add), hkv, PAGE, d))])
    v = np.concatenate([cache.v, normal_bf16(rng, (sum(add), hkv, PAGE, d))])
    return PagedCache(k=k, v=v, block_table=table, num_blocks=num_blocks,
                      max_blocks=table.shape[1])


def next_step_tree(rng: np.random.Generator, B: int, N_max: int, Hq: int, Hkv: int, D: int,
                   max_depth: int):
    """The next verify step's draft trees for a two-step scenario: node counts,
    parent arrays (random trees, arbitrary id order), queries, and the K/V rows
    of every node ([B][N_max][Hkv][D] bf16 bits each; the caller writes them
    wherever its commit left room)."""
    n_nodes = rng.integers(1, N_max, size=B, endpoint=True).astype(np.int32)
    parent = np.zeros((B, N_max), dtype=np.int32)
    for b in range(B):
        nb = int(n_nodes[b])
        p = random_tree(rng, nb, max_depth)
        if nb > 2:
            p = relabel(rng, p)
        parent[b, :nb] = p
        parent[b, nb:] = -1
    q = normal_bf16(rng, (B, N_max, Hq, D))
    k_rows = normal_bf16(rng, (B, N_max, Hkv, D))
    v_rows = normal_bf16(rng, (B, N_max, Hkv, D))
    return n_nodes, parent, q, k_rows, v_rows


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------


@dataclasses.dataclass
class VerifyInputs:
    name: str
    B: int
    N_max: int
    Hq: int
    Hkv: int
    D: int
    V: int
    D_max: int
    parent: np.ndarray       # int32 [B][N_max]
    n_nodes: np.ndarray      # int32 [B]
    prefix_len: np.ndarray   # int32 [B]
    tokens: np.ndarray       # int32 [B][N_max]
    logits: np.ndarray       # float32 [B][N_max][V]
    q: np.ndarray            # uint16 [B][N_max][Hq][D]
    cache: PagedCache
    targets: np.ndarray      # int32 [B][N_max] planted target token per node

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


WORKLOADS = {
    # name: (B, Hq, Hkv, D, prefix, N, V, D_max, logit_std, p_match)
    "tiny": (1, 4, 4, 64, 128, 15, 1000, 4, 1.0, 0.5),
    "8b": (1, 32, 8, 128, 4096, 63, 128256, 6, float(np.sqrt(2.0)), 0.7),
    "ragged": (16, 32, 8, 128, None, 31, 32000, 5, 1.0, 0.6),
    "70b": (4, 64, 8, 128, 32768, 127, 128256, 8, float(np.sqrt(2.0)), 0.7),
}
SEEDS = {"tiny": 0, "8b": 1, "ragged": 2, "70b": 3, "bastion": 4}


def _trees_for(name: str, rng: np.random.Generator, B: int, N: int) -> np.ndarray:
    if name == "tiny":
        return np.stack([random_tree(rng, N, 4, 3) for _ in range(B)])
    if name == "8b":
        return np.stack([static_8b_tree() for _ in range(B)])
    if name == "ragged":
        return np.stack([random_tree(rng, N, 5) for _ in range(B)])
    if name == "70b":
        return np.stack([random_tree(rng, N, 8) for _ in range(B)])
    raise KeyError(name)


def verify_workload(name: str, seed: Optional[int] = None, with_logits: bool = True) -> VerifyInputs:
    """One of the four fixed-tree verify workloads, fully materialised."""
    B, Hq, Hkv, D, prefix, N, V, D_max, lstd, pm = WORKLOADS[name]
    rng = np.random.default_rng(SEEDS[name] if seed is None else seed)
    parent = _trees_for(name, rng, B, N)
    n_nodes = np.full(B, N, dtype=np.int32)
    if prefix is None:
        prefix_len = rng.integers(512, 8192, size=B, endpoint=True).astype(np.int32)
    else:
        prefix_len = np.full(B, prefix, dtype=np.int32)
    targets = rng.integers(0, V, size=(B, N)).astype(np.int32)
    tokens = np.stack([draft_tokens(rng, parent[b], targets[b], pm, V) for b in range(B)])
    if with_logits:
        logits = rng.standard_normal(size=(B, N, V), dtype=np.float32)
        if lstd != 1.0:
            logits *= np.float32(lstd)
        plant_targets(logits, targets)
    else:
        logits = np.zeros((0,), dtype=np.float32)
    q = normal_bf16(rng, (B, N, Hq, D))
    cache = paged_cache(rng, prefix_len, n_nodes, Hkv, D, shuffle=(name == "70b"))
    return VerifyInputs(name=name, B=B, N_max=N, Hq=Hq, Hkv=Hkv, D=D, V=V, D_max=D_max,
                        parent=parent, n_nodes=n_nodes, prefix_len=prefix_len, tokens=tokens,
                        logits=logits, q=q, cache=cache, targets=targets)


def first_sequences(inp: VerifyInputs, n: int) -> VerifyInputs:
    """The first n sequences of a workload, with a pool holding only their
    cache blocks (ids renumbered in increasing order, so a shuffled table stays
    shuffled).  The same shapes at a smaller size, for profiling."""
    n = max(1, min(n, inp.B))
    table = inp.cache.block_table[:n]
    need = [(int(inp.prefix_len[b]) + int(inp.n_nodes[b]) + PAGE - 1) // PAGE for b in range(n)]
    used = np.unique(np.concatenate([table[b, :need[b]] for b in range(n)]))
    remap = {int(x): i for i, x in enumerate(used)}
    new_table = np.zeros_like(table)
    for b in range(n):
        new_table[b, :need[b]] = [remap[int(x)] for x in table[b, :need[b]]]
    cache = PagedCache(k=inp.cache.k[used], v=inp.cache.v[used], block_table=new_table,
                       num_blocks=len(used), max_blocks=new_table.shape[1])
    logits = inp.logits[:n] if inp.logits.ndim == 3 else inp.logits
    return VerifyInputs(name=inp.name, B=n, N_max=inp.N_max, Hq=inp.Hq, Hkv=inp.Hkv, D=inp.D,
                        V=inp.V, D_max=inp.D_max, parent=inp.parent[:n].copy(),
                        n_nodes=inp.n_nodes[:n].copy(), prefix_len=inp.prefix_len[:n].copy(),
                        tokens=inp.tokens[:n].copy(), logits=np.ascontiguousarray(logits),
                        q=inp.q[:n].copy(), cache=cache, targets=inp.targets[:n].copy())


# BASTION-style budgeted trees -------------------------------------------------

BASTION = dict(B=8, K=16, V=32000, Hq=32, Hkv=8, D=128, prefix=2048, p_match=0.6,
               budgets=(16, 32, 64, 128, 256))


def bastion_marginals(seed: Optional[int] = None):
    """Per-sequence draft marginals q[B][K][V] = softmax(z), z ~ N(0,2).  The
    softmax is taken in fp64 and rounded once to fp32; both sides read that
    fp32 array.  Also returns the root tokens (uniform)."""
    c = BASTION
    rng = np.random.default_rng(SEEDS["bastion"] if seed is None else seed)
    z = rng.standard_normal(size=(c["B"], c["K"], c["V"])) * np.sqrt(2.0)
    z -= z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    q = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    root = rng.integers(0, c["V"], size=c["B"]).astype(np.int32)
    return q, root


def shaped_marginals(seed: int, B: int, K: int, V: int, shape: str):
    """Draft marginals q[B][K][V] (fp32) of one of several shapes, for
    best-first trees of different forms: "sharp" (softmax of 4 z: deep,
    narrow trees), "flat" (softmax of 0.3 z: wide and deep), "tied" (softmax
    of round(2 z): many equal probabilities), "pow2" (every probability a power
    of two: many equal path scores), "dominant" (token 0 raised by 6: long
    chains), "tiny_tail" (token 0 at 1/2, the rest of the mass 1e-7 spread
    over the others: path scores spanning more than 2^53), "uniform" (every
    probability 1/V: every rank a tie).  z ~ N(0, 1); softmax in fp64, rounded
    once to fp32.  Also returns uniform root tokens."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(size=(B, K, V))
    if shape == "sharp":
        z = 4.0 * z
    elif shape == "flat":
        z = 0.3 * z
    elif shape == "tied":
        z = np.round(2.0 * z)
    elif shape == "dominant":
        z[..., 0] += 6.0
    elif shape == "uniform":
        z = np.zeros_like(z)
    elif shape not in ("pow2", "tiny_tail"):
        raise ValueError(shape)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    q = e / e.sum(axis=-1, keepdims=True)
    if shape == "pow2":
        q = np.exp2(np.round(np.log2(q)))
    if shape == "tiny_tail":
        q = np.where(np.arange(V) == 0, 0.5, 1e-7 * q / max(V - 1, 1))
    root = rng.integers(0, V, size=B).astype(np.int32)
    return q.astype(np.float32), root


def dynamic_draft_rows(seed: int, b: int, pool_ids, V: int, temp: float = 1.0) -> np.ndarray:
    """Stand-in for a drafter's per-node output in dynamic-tree construction:
    the row of node (b, pool id) is softmax(z / temp), z ~ N(0,1) drawn from
    a generator seeded by (seed, b, pool id), so every node has its own row and
    the same node always gets the same row.  Softmax in fp64, rounded once to
    fp32.  Returns float32 [len(pool_ids)][V]."""
    rows = np.empty((len(pool_ids), V), dtype=np.float32)
    for r, pid in enumerate(pool_ids):
        rng = np.random.default_rng([seed, b, int(pid)])
        z = rng.standard_normal(V) / temp
        e = np.exp(z - z.max())
        rows[r] = (e / e.sum()).astype(np.float32)
    return rows


def bastion_verify_inputs(parent: np.ndarray, tokens: np.ndarray, depth: np.ndarray,
                          draft_top1: np.ndarray, seed: Optional[int] = None) -> VerifyInputs:
    """Verify-layer inputs for a built budgeted tree.

    ``parent``/``tokens``/``depth`` describe the tree [B][N]; ``draft_top1``
    [B][K] is the draft's most likely token at each position (supplied by the
    caller).  For node i the planted target is draft_top1[depth(i)+1] with
    probability 0.6 (when that position exists), else a uniform token."""
    c = BASTION
    B, N = parent.shape
    rng = np.random.default_rng((SEEDS["bastion"] if seed is None else seed) * 1000 + N)
    targets = rng.integers(0, c["V"], size=(B, N)).astype(np.int32)
    coin = rng.random((B, N))
    for b in range(B):
        for i in range(N):
            pos = int(depth[b, i]) + 1
            if pos <= c["K"] and coin[b, i] < c["p_match"]:
                targets[b, i] = draft_top1[b, pos - 1]
    logits = rng.standard_normal(size=(B, N, c["V"]), dtype=np.float32) * np.float32(np.sqrt(2.0))
    plant_targets(logits, targets)
    q = normal_bf16(rng, (B, N, c["Hq"], c["D"]))
    prefix_len = np.full(B, c["prefix"], dtype=np.int32)
    n_nodes = np.full(B, N, dtype=np.int32)
    cache = paged_cache(rng, prefix_len, n_nodes, c["Hkv"], c["D"], shuffle=False)
    return VerifyInputs(name="bastion%d" % N, B=B, N_max=N, Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"],
                        V=c["V"], D_max=min(16, N - 1), parent=parent.astype(np.int32),
                        n_nodes=n_nodes, prefix_len=prefix_len, tokens=tokens.astype(np.int32),
                        logits=logits, q=q, cache=cache, targets=targets)


DYNAMIC = dict(B=8, V=32000, k=10, levels=6, N=64, temp=1.0, seed=5)


def dynamic_verify_inputs(parent: np.ndarray, tokens: np.ndarray, depth: np.ndarray,
                          seed: Optional[int] = None) -> VerifyInputs:
    """Verify-layer inputs (the 8B shape with prefix 2048, V = 32000) for a
    dynamic draft tree [B][N] in rank order.  The planted target of node i is,
    with probability 0.6, the token of its first child in the tree (a node's
    kept children are its best-ranked tokens, so the first is the drafter's
    top choice there); otherwise, and for leaves, a uniform token."""
    c = BASTION
    B, N = parent.shape
    rng = np.random.default_rng((DYNAMIC["seed"] if seed is None else seed) * 1000 + N)
    targets = rng.integers(0, c["V"], size=(B, N)).astype(np.int32)
    coin = rng.random((B, N))
    for b in range(B):
        first_child = {}
        for i in range(1, N):
            first_child.setdefault(int(parent[b, i]), i)
        for i in range(N):
            if i in first_child and coin[b, i] < c["p_match"]:
                targets[b, i] = tokens[b, first_child[i]]
    logits = rng.standard_normal(size=(B, N, c["V"]), dtype=np.float32) * np.float32(np.sqrt(2.0))
    plant_targets(logits, targets)
    q = normal_bf16(rng, (B, N, c["Hq"], c["D"]))
    prefix_len = np.full(B, c["prefix"], dtype=np.int32)
    n_nodes = np.full(B, N, dtype=np.int32)
    cache = paged_cache(rng, prefix_len, n_nodes, c["Hkv"], c["D"], shuffle=False)
    return VerifyInputs(name="dynamic%d" % N, B=B, N_max=N, Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"],
                        V=c["V"], D_max=max(1, int(depth.max())), parent=parent.astype(np.int32),
                        n_nodes=n_nodes, prefix_len=prefix_len, tokens=tokens.astype(np.int32),
                        logits=logits, q=q, cache=cache, targets=targets)


def random_small(seed: int, B: int, N_max: int, Hq: int, Hkv: int, D: int, V: int,
                 prefix_lo: int, prefix_hi: int, max_depth: int, p_match: float = 0.6,
                 ragged_nodes: bool = True, shuffle_blocks: bool = True,
                 relabel_ids: bool = True, logit_std: float = 1.0,
                 prefix_len: Optional[np.ndarray] = None) -> VerifyInputs:
    """Randomised small verify inputs for parity sweeps: ragged node counts
    (padding rows), arbitrary parent order, shuffled pages.  ``prefix_len``,
    when given, fixes the per-sequence prefix lengths instead of drawing them
    from [prefix_lo, prefix_hi]."""
    rng = np.random.default_rng(seed)
    if ragged_nodes:
        n_nodes = rng.integers(1, N_max, size=B, endpoint=True).astype(np.int32)
    else:
        n_nodes = np.full(B, N_max, dtype=np.int32)
    parent = np.full((B, N_max), 0, dtype=np.int32)
    for b in range(B):
        nb = int(n_nodes[b])
        p = random_tree(rng, nb, max_depth)
        if relabel_ids and nb > 2:
            p = relabel(rng, p)
        parent[b, :nb] = p
        # padding entries hold junk that must be ignored
        parent[b, nb:] = rng.integers(-5, 2 * N_max, size=N_max - nb)
    drawn = rng.integers(prefix_lo, prefix_hi, size=B, endpoint=True).astype(np.int32)
    prefix_len = drawn if prefix_len is None else np.asarray(prefix_len, dtype=np.int32).copy()
    targets = rng.integers(0, V, size=(B, N_max)).astype(np.int32)
    tokens = np.zeros((B, N_max), dtype=np.int32)
    for b in range(B):
        nb = int(n_nodes[b])
        tokens[b, :nb] = draft_tokens(rng, parent[b, :nb], targets[b, :nb], p_match, V)
        tokens[b, nb:] = rng.integers(0, V, size=N_max - nb)
    logits = rng.standard_normal(size=(B, N_max, V), dtype=np.float32) * np.float32(logit_std)
    plant_targets(logits, targets)
    q = normal_bf16(rng, (B, N_max, Hq, D))
    cache = paged_cache(rng, prefix_len, n_nodes, Hkv, D, shuffle=shuffle_blocks, spare_blocks=3)
    return VerifyInputs(name="random%d" % seed, B=B, N_max=N_max, Hq=Hq, Hkv=Hkv, D=D, V=V,
                        D_max=max_depth, parent=parent, n_nodes=n_nodes, prefix_len=prefix_len,
                        tokens=tokens, logits=logits, q=q, cache=cache, targets=targets)


# Stochastic verification ---------------------------------------------------


@dataclasses.dataclass
class StochasticInputs:
    B: int
    N_max: int
    V: int
    D_max: int
    parent: np.ndarray     # int32 [B][N_max]
    n_nodes: np.ndarray    # int32 [B]
    tokens: np.ndarray     # int32 [B][N_max]
    logits: np.ndarray     # float32 [B][N_max][V]  target logits
    q_draft: np.ndarray    # float32 [B][N_max][V]  draft probabilities
    u_accept: np.ndarray   # float32 [B][N_max]     uniforms in [0, 1)
    u_draw: np.ndarray     # float32 [B][N_max]
    seed: int = 0


def stochastic_inputs(seed: int, B: int, N_max: int, V: int, max_depth: int,
                      parents: Optional[np.ndarray] = None, ragged_nodes: bool = False,
                      logit_std: float = float(np.sqrt(2.0)), draft_noise: float = 1.0,
                      relabel_ids: bool = True) -> StochasticInputs:
    """Inputs for stochastic tree verification.

    Target logits ~ N(0, logit_std^2) in fp32.  The draft row of node i is a
    noisy copy of the target seen through the drafter: the normalised
    exponential of (logits[i] + N(0, draft_noise^2)), formed in fp64 and
    rounded once to fp32.  Each child's token is drawn from its parent's
    draft row (independent draws, repeats allowed).  Uniforms are fp32 in
    [0, 1).  ``parents`` [B][N_max] fixes the trees; otherwise random trees
    of depth <= max_depth (ids relabelled, padding entries junk)."""
    rng = np.random.default_rng(seed)
    if ragged_nodes:
        n_nodes = rng.integers(1, N_max, size=B, endpoint=True).astype(np.int32)
    else:
        n_nodes = np.full(B, N_max, dtype=np.int32)
    if parents is not None:
        parent = np.asarray(parents, dtype=np.int32).copy()
    else:
        parent = np.zeros((B, N_max), dtype=np.int32)
        for b in range(B):
            nb = int(n_nodes[b])
            p = random_tree(rng, nb, max_depth)
            if relabel_ids and nb > 2:
                p = relabel(rng, p)
            parent[b, :nb] = p
            parent[b, nb:] = rng.integers(-5, 2 * N_max, size=N_max - nb)
    logits = rng.standard_normal(size=(B, N_max, V), dtype=np.float32) * np.float32(logit_std)
    q_draft = np.zeros((B, N_max, V), dtype=np.float32)
    tokens = rng.integers(0, V, size=(B, N_max)).astype(np.int32)
    for b in range(B):
        nb = int(n_nodes[b])
        for i in range(nb):
            z = logits[b, i].astype(np.float64) + rng.standard_normal(V) * draft_noise
            e = np.exp(z - z.max())
            q64 = e / e.sum()
            q_draft[b, i] = q64.astype(np.float32)
            kids = np.nonzero(parent[b, :nb] == i)[0]
            kids = kids[kids > 0]
            if kids.size:
                tokens[b, kids] = rng.choice(V, size=kids.size, p=q64)
    u_accept = rng.random((B, N_max), dtype=np.float32)
    u_draw = rng.random((B, N_max), dtype=np.float32)
    return StochasticInputs(B=B, N_max=N_max, V=V, D_max=max_depth, parent=parent,
                            n_nodes=n_nodes, tokens=tokens, logits=logits, q_draft=q_draft,
                            u_accept=u_accept, u_draw=u_draw, seed=seed)


def redraw_uniforms(inp: StochasticInputs, rng: np.random.Generator, accept_idx, draw_idx) -> None:
    """In place: fresh uniforms at the given (b, node) index arrays."""
    ab, ai = accept_idx
    if len(ab):
        inp.u_accept[ab, ai] = rng.random(len(ab), dtype=np.float32)
    db, di = draw_idx
    if len(db):
        inp.u_draw[db, di] = rng.random(len(db), dtype=np.float32)


def stochastic_for(inp: VerifyInputs, seed: int = 0, draft_noise: float = 1.0):
    """Draft rows, child tokens and uniforms for stochastic verification of
    an existing verify workload (its trees and target logits): the draft row
    of node i is the normalised exponential of (logits[i] + N(0,
    draft_noise^2)) formed in fp64 and rounded to fp32; each child's token is
    drawn from its parent's draft row; uniforms fp32 in [0, 1).  Returns
    (q_draft [B][N][V], tokens [B][N], u_accept [B][N], u_draw [B][N])."""
    rng = np.random.default_rng(1000 + seed)
    B, N, V = inp.B, inp.N_max, inp.V
    q_draft = np.zeros((B, N, V), dtype=np.float32)
    tokens = inp.tokens.copy()
    for b in range(B):
        nb = int(inp.n_nodes[b])
        for i in range(nb):
            z = inp.logits[b, i].astype(np.float64) + rng.standard_normal(V) * draft_noise
            e = np.exp(z - z.max())
            q64 = e / e.sum()
            q_draft[b, i] = q64.astype(np.float32)
            kids = np.nonzero(inp.parent[b, :nb] == i)[0]
            kids = kids[kids > 0]
            if kids.size:
                c = np.cumsum(q64)
                tokens[b, kids] = np.minimum(np.searchsorted(c, rng.random(kids.size) * c[-1],
                                                             side="right"), V - 1)
    u_accept = rng.random((B, N), dtype=np.float32)
    u_draw = rng.random((B, N), dtype=np.float32)
    return q_draft, tokens, u_accept, u_draw
