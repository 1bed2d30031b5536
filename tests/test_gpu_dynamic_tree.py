"""GPU parity of dynamic draft-tree construction (expand level by level, then
rerank) against the oracle, bit for bit: every level's pool entries and
frontier, and the reranked tree; the tree then passes the ancestor checks."""

import numpy as np
import pytest

import gen
import oracle

from _gpu_path import dev_tensor, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # B, V, k, levels, N, drafter temperature
    (4, 32000, 10, 6, 64, 1.0),
    (2, 3000, 32, 4, 256, 0.5),
    (3, 500, 1, 8, 9, 1.0),
    (2, 1000, 5, 3, 31, 2.0),
    (1, 100, 3, 7, 40, 0.2),
    (5, 128256, 8, 5, 48, 1.0),
]


@pytest.fixture(scope="module")
def tsd():
    import torch
    import tree_speculative_decoding_virtual_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.mark.parametrize("case", range(len(CASES)))
def test_dynamic_tree_matches_oracle(tsd, case):
    import torch
    B, V, k, L, N, temp = CASES[case]
    seed = 900 + case
    root = np.random.default_rng(seed).integers(0, V, size=B).astype(np.int32)
    M = oracle.pool_size(L, k)
    M_max = M + 5  # room beyond the used ids is left untouched
    pool_g = tsd.dynamic_tree_new_pool(B, M_max, "cuda")
    pool_o = oracle.new_pool(B, M, root)
    root_g = dev_tensor(root)
    fr_g, fr_o = None, np.zeros((B, 1), dtype=np.int32)
    for level in range(1, L + 1):
        rows = np.stack([gen.dynamic_draft_rows(seed, b, fr_o[b], V, temp) for b in range(B)])
        fr_g = tsd.dynamic_tree_expand(dev_tensor(rows), k, level, pool_g, root_token=root_g,
                                       frontier=fr_g)
        fr_o = oracle.expand_level(rows, fr_o, pool_o, k, level)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(fr_g), fr_o), level
    for g, o, name in zip(pool_g, pool_o, ["parent", "token", "depth", "score"]):
        assert np.array_equal(to_np(g)[:, :M], o), name
    tree_g = tsd.dynamic_tree_rerank(pool_g, M, N)
    tree_o = oracle.dynamic_tree_rerank(pool_o, M, N)
    for g, o, name in zip(tree_g, tree_o, ["parent", "tokens", "depth", "score"]):
        assert np.array_equal(to_np(g), o), name
    # the reranked tree is a valid draft tree for verification
    anc, depth, mask, err = tsd.tree_build_ancestors(tree_g[0], None, max(L, 1))
    torch.cuda.synchronize()
    assert (to_np(err) == 0).all()
    assert np.array_equal(to_np(depth), tree_o[2])
