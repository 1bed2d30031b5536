"""Pins for the deferred commit ("EAGLE-Pangu" technical summary 2.1: the
fast reorder moves only the accepted segment and only when needed; its
conclusion names commit efficiency as future work).  Committing by record
instead of by copy must leave the next verify step's attention unchanged:
through the record, every node sees the same keys in the same order as after
the copy commit, so the fp64 oracle gives identical outputs.  A later copy
from the recorded places (the generalised commit with a tree base)
materialises the same cache the copy commits would have produced."""

import numpy as np
import pytest

import gen
import oracle


def _write_rows(cache, block_table, b, slot0, k_rows, v_rows, n):
    for j in range(n):
        s = slot0 + j
        pg, row = int(block_table[b, s // gen.PAGE]), s % gen.PAGE
        cache.k[pg, :, row, :] = k_rows[j]
        cache.v[pg, :, row, :] = v_rows[j]


def _two_steps(seed, B=3, N=12, Hq=8, Hkv=2, D=64, P=(0, 70)):
    rng = np.random.default_rng(seed)
    inp = gen.random_small(seed, B=B, N_max=N, Hq=Hq, Hkv=Hkv, D=D, V=40, prefix_lo=P[0],
                           prefix_hi=P[1], max_depth=4, p_match=0.9)
    _, _, _, err = oracle.build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    _, A, _, path, _ = oracle.verify_greedy(inp.logits, inp.tokens, inp.parent, inp.n_nodes, err,
                                            inp.D_max)
    n2, parent2, q2, k2, v2 = gen.next_step_tree(rng, B, N, Hq, Hkv, D, max_depth=4)
    big = gen.grow_cache(rng, inp.cache, inp.prefix_len, inp.n_nodes, extra=N)
    return inp, err, A, path, n2, parent2, q2, k2, v2, big


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_attention_through_the_record_equals_attention_after_the_copy(seed):
    inp, err, A, path, n2, parent2, q2, k2, v2, big = _two_steps(seed)
    table = big.block_table
    _, _, _, err2 = oracle.build_ancestors(parent2, n2, 4)
    # copy commit, then the next tree right after the new prefix
    k1, v1, new_len, _ = oracle.commit_path(big.k, big.v, table, inp.prefix_len, A, path, err)
    copied = gen.PagedCache(k=k1, v=v1, block_table=table, num_blocks=big.num_blocks,
                            max_blocks=big.max_blocks)
    for b in range(inp.B):
        _write_rows(copied, table, b, int(new_len[b]), k2[b], v2[b], int(n2[b]))
    out_c, lse_c = oracle.tree_attention(q2, copied.k, copied.v, table, new_len, n2, parent2, err2,
                                         inp.scale)
    # deferred commit, then the next tree after the current one
    src, base, length, new_len_r, next_tail = oracle.commit_remap(inp.prefix_len, inp.n_nodes, A,
                                                                   path, err)
    assert np.array_equal(new_len_r, new_len)
    rec = gen.PagedCache(k=big.k.copy(), v=big.v.copy(), block_table=table,
                         num_blocks=big.num_blocks, max_blocks=big.max_blocks)
    for b in range(inp.B):
        _write_rows(rec, table, b, int(next_tail[b]), k2[b], v2[b], int(n2[b]))
    out_r, lse_r = oracle.tree_attention(q2, rec.k, rec.v, table, new_len, n2, parent2, err2,
                                         inp.scale, remap=(src, base, length, next_tail))
    assert np.array_equal(out_r, out_c) and np.array_equal(lse_r, lse_c)
    assert (A > 0).any()  # the record is not the identity everywhere


def test_record_reads_the_accepted_entries():
    inp, err, A, path, n2, parent2, q2, k2, v2, big = _two_steps(7)
    src, base, length, new_len, next_tail = oracle.commit_remap(inp.prefix_len, inp.n_nodes, A,
                                                                 path, err)
    for b in range(inp.B):
        P, nb = int(inp.prefix_len[b]), int(inp.n_nodes[b])
        if err[b]:
            assert length[b] == 0 and new_len[b] == P
            continue
        # the k-th committed entry is the k-th node of the accepted path
        chain = oracle.ancestor_chain(inp.parent[b], int(path[b, A[b]]) - 1)  # root first
        assert [int(s) - P for s in src[b, :A[b] + 1]] == chain
        assert (src[b, A[b] + 1:] == -1).all()
        assert next_tail[b] == P + nb and length[b] == A[b] + 1
        slots = oracle.physical_slots((src, base, length, next_tail), b, int(new_len[b]), 3)
        assert slots[:P] == list(range(P)) and slots[P:P + A[b] + 1] == [P + c for c in chain]
        assert slots[-3:] == [P + nb, P + nb + 1, P + nb + 2]


def test_copy_from_the_record_materialises_the_copy_commit():
    """Materialising the record later (copy from the recorded tree base)
    gives the bytes the immediate copy commit gave, for every slot below the
    new length; the copy from a tree base equals the plain copy when the base
    is the prefix."""
    inp, err, A, path, n2, parent2, q2, k2, v2, big = _two_steps(9)
    table = big.block_table
    k1, v1, nl1, mv1 = oracle.commit_path(big.k, big.v, table, inp.prefix_len, A, path, err)
    k3, v3, nl3, mv3 = oracle.commit_path(big.k, big.v, table, inp.prefix_len, A, path, err,
                                          tail_base=inp.prefix_len)
    assert np.array_equal(k1, k3) and np.array_equal(v1, v3) and np.array_equal(mv1, mv3)
    # a tree placed 5 slots further: the same entries reach the same slots
    shifted = gen.PagedCache(k=big.k.copy(), v=big.v.copy(), block_table=table,
                             num_blocks=big.num_blocks, max_blocks=big.max_blocks)
    for b in range(inp.B):
        P, nb = int(inp.prefix_len[b]), int(inp.n_nodes[b])
        rows_k = [big.k[int(table[b, (P + j) // 16]), :, (P + j) % 16].copy() for j in range(nb)]
        rows_v = [big.v[int(table[b, (P + j) // 16]), :, (P + j) % 16].copy() for j in range(nb)]
        _write_rows(shifted, table, b, P + 5, rows_k, rows_v, nb)
    k4, v4, nl4, _ = oracle.commit_path(shifted.k, shifted.v, table, inp.prefix_len, A, path, err,
                                        tail_base=inp.prefix_len + 5)
    for b in range(inp.B):
        for s in range(int(nl1[b])):
            pg, row = int(table[b, s // 16]), s % 16
            assert np.array_equal(k4[pg, :, row], k1[pg, :, row])
            assert np.array_equal(v4[pg, :, row], v1[pg, :, row])
