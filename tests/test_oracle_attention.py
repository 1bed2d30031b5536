"""Pins for the oracle's tree attention.

* A chain tree with an empty prefix is causal attention: compared against
  torch's scaled_dot_product_attention(is_causal=True) in fp64.
* A single-node tree is plain decode attention over prefix + itself.
* A general tree equals SDPA with a boolean mask built from networkx's
  ancestor sets (an independent graph library), with GQA expanded by
  repeat_interleave, on paged caches with shuffled blocks.
* Perturbing the K/V of any node outside a node's ancestor path leaves that
  node's output unchanged (no leakage across branches).
* Identical keys: lse = s0 + log(#visible keys), out = mean of visible V
  (closed form; pins the visible-key count and the lse definition).
* Sampled evaluation equals full evaluation.
"""

import networkx as nx
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import gen
import oracle
from oracle import bf16_to_f64, build_ancestors, tree_attention

PAGE = 16


def _dense_kv(cache, table, b, hkv, n):
    rows = []
    for t in range(n):
        rows.append(cache[table[b, t // PAGE], hkv, t % PAGE])
    return bf16_to_f64(np.stack(rows))


def _sdpa_reference(inp, b):
    """Attention for sequence b through torch SDPA with an explicit mask."""
    nb = int(inp.n_nodes[b])
    P = int(inp.prefix_len[b])
    G = nx.DiGraph()
    G.add_nodes_from(range(nb))
    for i in range(1, nb):
        G.add_edge(int(inp.parent[b, i]), i)
    allow = np.zeros((nb, P + nb), dtype=bool)
    allow[:, :P] = True
    for i in range(nb):
        for j in nx.ancestors(G, i) | {i}:
            allow[i, P + j] = True
    g = inp.Hq // inp.Hkv
    K = np.stack([_dense_kv(inp.cache.k, inp.cache.block_table, b, h, P + nb) for h in range(inp.Hkv)])
    V = np.stack([_dense_kv(inp.cache.v, inp.cache.block_table, b, h, P + nb) for h in range(inp.Hkv)])
    Q = bf16_to_f64(inp.q[b, :nb]).transpose(1, 0, 2)  # [Hq][nb][D]
    Kt = torch.from_numpy(K).repeat_interleave(g, dim=0)
    Vt = torch.from_numpy(V).repeat_interleave(g, dim=0)
    out = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], Kt[None], Vt[None],
                                         attn_mask=torch.from_numpy(allow)[None, None])
    return out[0].numpy().transpose(1, 0, 2)  # [nb][Hq][D]


def _run_oracle(inp):
    _, _, _, err = build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    return tree_attention(inp.q, inp.cache.k, inp.cache.v, inp.cache.block_table, inp.prefix_len,
                          inp.n_nodes, inp.parent, err, inp.scale)


def test_chain_is_causal_attention():
    rng = np.random.default_rng(0)
    n, D, H = 12, 16, 2
    parent = gen.chain_tree(n)[None]
    prefix = np.array([0], dtype=np.int32)
    nn_ = np.array([n], dtype=np.int32)
    cache = gen.paged_cache(rng, prefix, nn_, H, D, shuffle=True, spare_blocks=2)
    q = gen.normal_bf16(rng, (1, n, H, D))
    _, _, _, err = build_ancestors(parent, nn_, n)
    out, lse = tree_attention(q, cache.k, cache.v, cache.block_table, prefix, nn_, parent, err,
                              1.0 / np.sqrt(D))
    for h in range(H):
        K = _dense_kv(cache.k, cache.block_table, 0, h, n)
        V = _dense_kv(cache.v, cache.block_table, 0, h, n)
        Q = bf16_to_f64(q[0, :, h])
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], torch.from_numpy(K)[None],
                                             torch.from_numpy(V)[None], is_causal=True)[0].numpy()
        np.testing.assert_allclose(out[0, :, h], ref, rtol=0, atol=1e-12)


def test_single_node_is_decode_attention():
    rng = np.random.default_rng(1)
    D, Hq, Hkv, P = 32, 4, 2, 37
    parent = np.array([[-1]], dtype=np.int32)
    prefix = np.array([P], dtype=np.int32)
    nn_ = np.array([1], dtype=np.int32)
    cache = gen.paged_cache(rng, prefix, nn_, Hkv, D, shuffle=True, spare_blocks=1)
    q = gen.normal_bf16(rng, (1, 1, Hq, D))
    _, _, _, err = build_ancestors(parent, nn_, 0)
    out, lse = tree_attention(q, cache.k, cache.v, cache.block_table, prefix, nn_, parent, err,
                              1.0 / np.sqrt(D))
    for h in range(Hq):
        K = _dense_kv(cache.k, cache.block_table, 0, h // 2, P + 1)
        V = _dense_kv(cache.v, cache.block_table, 0, h // 2, P + 1)
        Q = bf16_to_f64(q[0, :, h])
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], torch.from_numpy(K)[None],
                                             torch.from_numpy(V)[None])[0].numpy()
        np.testing.assert_allclose(out[0, 0, h], ref[0], rtol=0, atol=1e-12)
        s = (K @ Q[0]) / np.sqrt(D)
        assert abs(lse[0, 0, h] - torch.logsumexp(torch.from_numpy(s), 0).item()) < 1e-10


@pytest.mark.parametrize("seed,Hq,Hkv,D,P", [(0, 4, 4, 16, 0), (1, 8, 2, 32, 21),
                                             (2, 6, 3, 8, 50), (3, 4, 1, 16, 16)])
def test_tree_matches_masked_sdpa(seed, Hq, Hkv, D, P):
    inp = gen.random_small(seed, B=3, N_max=20, Hq=Hq, Hkv=Hkv, D=D, V=50,
                           prefix_lo=P, prefix_hi=P + 17, max_depth=6)
    out, lse = _run_oracle(inp)
    for b in range(inp.B):
        nb = int(inp.n_nodes[b])
        ref = _sdpa_reference(inp, b)
        np.testing.assert_allclose(out[b, :nb], ref, rtol=0, atol=1e-12)
        assert (out[b, nb:] == 0).all()
        assert np.isneginf(lse[b, nb:]).all()


def test_no_leakage_perturbation():
    inp = gen.random_small(7, B=2, N_max=24, Hq=4, Hkv=2, D=16, V=40, prefix_lo=5, prefix_hi=30,
                           max_depth=7, ragged_nodes=False)
    out0, lse0 = _run_oracle(inp)
    rng = np.random.default_rng(99)
    for b in range(inp.B):
        P = int(inp.prefix_len[b])
        nb = int(inp.n_nodes[b])
        target = int(rng.integers(nb))
        chain = set(oracle.ancestor_chain(inp.parent[b], target))
        outside = [j for j in range(nb) if j not in chain]
        if not outside:
            continue
        k2 = inp.cache.k.copy()
        v2 = inp.cache.v.copy()
        for j in outside:
            slot = P + j
            blk = inp.cache.block_table[b, slot // PAGE]
            k2[blk, :, slot % PAGE] = gen.bf16_bits(np.full(inp.D, 100.0, np.float32))
            v2[blk, :, slot % PAGE] = gen.bf16_bits(np.full(inp.D, -100.0, np.float32))
        _, _, _, err = build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
        out1, lse1 = tree_attention(inp.q, k2, v2, inp.cache.block_table, inp.prefix_len,
                                    inp.n_nodes, inp.parent, err, inp.scale)
        assert np.array_equal(out1[b, target], out0[b, target])
        assert np.array_equal(lse1[b, target], lse0[b, target])
        # and a node whose path does include a perturbed node does change
        changed = [i for i in range(nb) if set(oracle.ancestor_chain(inp.parent[b], i)) & set(outside)]
        if changed:
            assert not np.array_equal(out1[b, changed[0]], out0[b, changed[0]])


def test_identical_keys_closed_form():
    """All keys equal: every visible score is the same s0, so
    lse = s0 + log(P + depth + 1) and out = mean of the visible values."""
    rng = np.random.default_rng(4)
    D, H, P, n = 8, 2, 9, 10
    parent = gen.random_tree(rng, n, 4)[None]
    prefix = np.array([P], dtype=np.int32)
    nn_ = np.array([n], dtype=np.int32)
    cache = gen.paged_cache(rng, prefix, nn_, H, D, shuffle=False)
    key = gen.bf16_bits(np.linspace(-1, 1, D).astype(np.float32))
    cache.k[:] = key
    q = gen.normal_bf16(rng, (1, n, H, D))
    anc, depth, _, err = build_ancestors(parent, nn_, 4)
    out, lse = tree_attention(q, cache.k, cache.v, cache.block_table, prefix, nn_, parent, err, 0.5)
    kf = bf16_to_f64(key)
    for i in range(n):
        visible = list(range(P)) + [P + int(s) - 1 for s in anc[0, i + 1, :depth[0, i] + 1]]
        for h in range(H):
            s0 = 0.5 * float(bf16_to_f64(q[0, i, h]) @ kf)
            assert abs(lse[0, i, h] - (s0 + np.log(P + depth[0, i] + 1))) < 1e-12
            V = _dense_kv(cache.v, cache.block_table, 0, h, P + n)
            np.testing.assert_allclose(out[0, i, h], V[visible].mean(axis=0), rtol=0, atol=1e-12)


def test_sampled_equals_full_and_err_skips():
    inp = gen.random_small(9, B=3, N_max=12, Hq=4, Hkv=2, D=16, V=30, prefix_lo=0, prefix_hi=40,
                           max_depth=5)
    _, _, _, err = build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    err = err.copy()
    err[1] = 2  # pretend sequence 1 failed its checks
    full, lse = tree_attention(inp.q, inp.cache.k, inp.cache.v, inp.cache.block_table,
                               inp.prefix_len, inp.n_nodes, inp.parent, err, inp.scale)
    assert (full[1] == 0).all() and np.isneginf(lse[1]).all()
    sample = [(0, 0, 1), (2, int(inp.n_nodes[2]) - 1, 3), (0, int(inp.n_nodes[0]) - 1, 0)]
    part, plse = tree_attention(inp.q, inp.cache.k, inp.cache.v, inp.cache.block_table,
                                inp.prefix_len, inp.n_nodes, inp.parent, err, inp.scale,
                                sample=sample)
    for (b, i, h) in sample:
        # same arithmetic, different BLAS blocking: equal to rounding
        np.testing.assert_allclose(part[b, i, h], full[b, i, h], rtol=0, atol=1e-12)
        assert abs(plse[b, i, h] - lse[b, i, h]) < 1e-12
