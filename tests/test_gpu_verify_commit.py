"""The fused greedy verification + commit (tsd_tree_verify_greedy_commit),
bit-exact with the oracle's verify_greedy followed by commit_path ("Speculative
Decoding Hierárquico", Medusa section; "EAGLE-Pangu" technical summary 2.1):
the acceptance outputs, new lengths, moved counts and every byte of the K and V
pools (all blocks, all layers)."""

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsd():
    import torch
    import tree_speculative_decoding_virtual_gb300 as m
    torch.cuda.set_device(0)
    return m


def _run(tsd, inp, K, V, layers=None, err_override=None):
    import torch
    from _gpu_path import dev_tensor, to_np
    parent = dev_tensor(inp.parent)
    n_nodes = dev_tensor(inp.n_nodes)
    anc, depth, mask, err = tsd.tree_build_ancestors(parent, n_nodes, inp.D_max)
    if err_override is not None:
        err = dev_tensor(err_override)
    kd = dev_tensor(K, torch.bfloat16)
    vd = dev_tensor(V, torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    am, A, leaf, path, bonus, new_len, moved = tsd.tree_verify_greedy_commit(
        dev_tensor(inp.logits), dev_tensor(inp.tokens), parent, anc, depth, mask, n_nodes, err,
        inp.D_max, kd, vd, dev_tensor(inp.cache.block_table), dev_tensor(inp.prefix_len),
        status=status)
    torch.cuda.synchronize()
    return dict(argmax=to_np(am), accept_len=to_np(A), leaf=to_np(leaf), path=to_np(path),
                bonus=to_np(bonus), new_len=to_np(new_len), moved=to_np(moved),
                k=to_np(kd, np.uint16), v=to_np(vd, np.uint16), status=int(status.item()))


def _oracle(inp, K, V, err_override=None):
    _, _, _, err = oracle.build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    if err_override is not None:
        err = err_override
    am, A, leaf, path, bonus = oracle.verify_greedy(inp.logits, inp.tokens, inp.parent,
                                                    inp.n_nodes, err, inp.D_max)
    k1, v1, new_len, moved = oracle.commit_path(K, V, inp.cache.block_table, inp.prefix_len, A,
                                                path, err)
    return dict(argmax=am, accept_len=A, leaf=leaf, path=path, bonus=bonus, new_len=new_len,
                moved=moved, k=k1, v=v1)


def _check(g, o):
    for key in ["argmax", "accept_len", "leaf", "path", "bonus", "new_len", "moved"]:
        assert np.array_equal(g[key], o[key]), (key, g[key], o[key])
    assert np.array_equal(g["k"], o["k"]), "committed K cache"
    assert np.array_equal(g["v"], o["v"]), "committed V cache"


@pytest.mark.parametrize("name", ["tiny", "8b", "ragged"])
def test_fused_commit_workloads(tsd, name):
    inp = gen.verify_workload(name, seed=gen.SEEDS[name] + 40)
    g = _run(tsd, inp, inp.cache.k, inp.cache.v)
    o = _oracle(inp, inp.cache.k, inp.cache.v)
    _check(g, o)
    assert g["status"] == 0


@pytest.mark.parametrize("seed,D,Hkv,layers", [(11, 128, 2, 5), (12, 64, 4, 3), (13, 128, 8, 1),
                                              (14, 64, 1, 2)])
def test_fused_commit_layers(tsd, seed, D, Hkv, layers):
    """Layer-stacked pools and several kv heads: the block that finishes a
    sequence stages whole heads' sources before it writes their slots."""
    inp = gen.random_small(seed, B=4, N_max=40, Hq=Hkv * 2, Hkv=Hkv, D=D, V=30, prefix_lo=0,
                           prefix_hi=90, max_depth=12, p_match=0.97)
    rng = np.random.default_rng(seed)
    K = np.stack([gen.normal_bf16(rng, inp.cache.k.shape) for _ in range(layers)])
    V = np.stack([gen.normal_bf16(rng, inp.cache.v.shape) for _ in range(layers)])
    g = _run(tsd, inp, K, V)
    o = _oracle(inp, K, V)
    _check(g, o)
    assert o["moved"].sum() > 0
    assert g["status"] == 0


def test_fused_commit_deep_paths(tsd):
    """Accepted paths of depth 32 (33 entries): chains whose node ids run
    backwards, so every accepted entry is out of place and one head's moves
    fill the staging by themselves."""
    inp = gen.random_small(21, B=3, N_max=33, Hq=16, Hkv=8, D=128, V=8, prefix_lo=5,
                           prefix_hi=40, max_depth=32, p_match=1.0, ragged_nodes=False,
                           relabel_ids=False)
    rng = np.random.default_rng(21)
    for b in range(inp.B):
        # node 32 - d sits at depth d, except the root (node 0)
        order = [0] + list(range(32, 0, -1))
        par = np.full(33, -1, dtype=np.int32)
        for d in range(1, 33):
            par[order[d]] = order[d - 1]
        inp.parent[b] = par
        inp.tokens[b] = gen.draft_tokens(rng, par, inp.targets[b], 1.0, inp.V)
    g = _run(tsd, inp, inp.cache.k, inp.cache.v)
    o = _oracle(inp, inp.cache.k, inp.cache.v)
    _check(g, o)
    assert (o["accept_len"] == 32).all() and (o["moved"] >= 31).all()


def test_fused_commit_skips_failed_sequences(tsd):
    """A sequence with err != 0 commits nothing (new_len = P, moved = 0) while
    the others commit."""
    inp = gen.random_small(31, B=5, N_max=24, Hq=4, Hkv=2, D=64, V=20, prefix_lo=0, prefix_hi=50,
                           max_depth=8, p_match=0.97)
    _, _, _, err = oracle.build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    err = err.copy()
    err[1] = 1
    err[3] = 4
    g = _run(tsd, inp, inp.cache.k, inp.cache.v, err_override=err)
    o = _oracle(inp, inp.cache.k, inp.cache.v, err_override=err)
    _check(g, o)
    assert g["new_len"][1] == inp.prefix_len[1] and g["moved"][1] == 0
