"""Deferred commit on the GPU ("EAGLE-Pangu" technical summary 2.1, the fast
reorder; its conclusion names commit efficiency as future work).  Two verify
steps: after step one, either the copy commit moves the accepted entries and
the next tree is written right after the new prefix, or kv_commit_remap
records where the entries are (nothing moves) and the next tree is written
after the current one.  Step two's attention must be bit for bit the same
both ways, the record must equal the oracle's, and copying from the recorded
tree base later must give the copy commit's bytes.  Covers the
two-blocks-per-SM kernel with the uniform split, the device split plan, the
single-piece direct path and the 256-row kernel."""

import numpy as np
import pytest

import gen
import oracle

from _gpu_path import dev_tensor, to_np

pytestmark = pytest.mark.gpu

CASES = {
    # name: (random_small kwargs)
    "small": dict(B=3, N_max=24, Hq=8, Hkv=2, D=128, prefix_lo=0, prefix_hi=300, max_depth=5),
    "8b-shaped": dict(B=1, N_max=63, Hq=32, Hkv=8, D=128, prefix_lo=4096, prefix_hi=4096,
                      max_depth=6),
    "ragged plan": dict(B=16, N_max=31, Hq=32, Hkv=8, D=128, prefix_lo=2000, prefix_hi=8000,
                        max_depth=5),
    "direct": dict(B=40, N_max=31, Hq=32, Hkv=8, D=128, prefix_lo=100, prefix_hi=400,
                   max_depth=5),
    "256-row": dict(B=1, N_max=20, Hq=16, Hkv=1, D=128, prefix_lo=150000, prefix_hi=150000,
                    max_depth=5),
    "d64": dict(B=2, N_max=16, Hq=4, Hkv=4, D=64, prefix_lo=20, prefix_hi=200, max_depth=4),
}


@pytest.fixture(scope="module")
def tsd():
    import torch
    import tree_speculative_decoding_virtual_gb300 as m
    torch.cuda.set_device(0)
    return m


def _write_rows(k, v, table, base, n, k_rows, v_rows):
    """Device write of the next tree's K/V rows at slots base[b] + j."""
    import torch
    for b in range(len(base)):
        nb = int(n[b])
        slots = int(base[b]) + np.arange(nb)
        pages = torch.from_numpy(table[b, slots // gen.PAGE].astype(np.int64)).cuda()
        rows = torch.from_numpy((slots % gen.PAGE).astype(np.int64)).cuda()
        k.view(torch.int16)[pages, :, rows, :] = torch.from_numpy(k_rows[b, :nb].view(np.int16)).cuda()
        v.view(torch.int16)[pages, :, rows, :] = torch.from_numpy(v_rows[b, :nb].view(np.int16)).cuda()


@pytest.mark.parametrize("case", list(CASES))
def test_step_through_the_record_equals_step_after_the_copy(tsd, case):
    import torch
    kw = CASES[case]
    seed = 900 + list(CASES).index(case)
    rng = np.random.default_rng(seed)
    inp = gen.random_small(seed, V=64, p_match=0.9, ragged_nodes=case != "8b-shaped", **kw)
    B, N, Hq, Hkv, D, Dm = inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, inp.D_max
    big = gen.grow_cache(rng, inp.cache, inp.prefix_len, inp.n_nodes, extra=N)
    n2, parent2, q2, k2, v2 = gen.next_step_tree(rng, B, N, Hq, Hkv, D, max_depth=Dm)
    table = dev_tensor(big.block_table)
    prefix, n_nodes, parent = dev_tensor(inp.prefix_len), dev_tensor(inp.n_nodes), dev_tensor(inp.parent)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    # step one: the tree, its verification
    anc, depth, mask, err = tsd.tree_build_ancestors(parent, n_nodes, Dm)
    am, A, leaf, path, bonus = tsd.tree_verify_greedy(dev_tensor(inp.logits), dev_tensor(inp.tokens),
                                                      parent, anc, depth, mask, n_nodes, err, Dm)
    torch.cuda.synchronize()
    assert to_np(A).max() > 0

    # (a) copy commit; the next tree right after the new prefix
    kc, vc = dev_tensor(big.k, torch.bfloat16), dev_tensor(big.v, torch.bfloat16)
    new_len, _ = tsd.kv_commit_path(kc, vc, table, prefix, n_nodes, A, path, err, N, Dm,
                                    status=status)
    torch.cuda.synchronize()
    nl = to_np(new_len)
    _write_rows(kc, vc, big.block_table, nl, n2, k2, v2)
    # (b) deferred commit; the next tree after the current one
    kr, vr = dev_tensor(big.k, torch.bfloat16), dev_tensor(big.v, torch.bfloat16)
    src, rbase, rlen, nl_r, next_tail = tsd.kv_commit_remap(prefix, n_nodes, A, path, err, N, Dm,
                                                            status=status)
    torch.cuda.synchronize()
    o_rec = oracle.commit_remap(inp.prefix_len, inp.n_nodes, to_np(A), to_np(path), to_np(err))
    for got, want in zip([src, rbase, rlen, nl_r, next_tail], o_rec):
        assert np.array_equal(to_np(got), want)
    _write_rows(kr, vr, big.block_table, to_np(next_tail), n2, k2, v2)

    # step two on both layouts
    parent2_d, n2_d = dev_tensor(parent2), dev_tensor(n2)
    anc2, depth2, mask2, err2 = tsd.tree_build_ancestors(parent2_d, n2_d, Dm)
    q2_d = dev_tensor(q2, torch.bfloat16)
    max_slots = int((nl + n2).max())
    out_c, lse_c = tsd.tree_attn_fwd(q2_d, kc, vc, table, new_len, n2_d, mask2, err2, max_slots,
                                     status=status)
    out_r, lse_r = tsd.tree_attn_fwd(q2_d, kr, vr, table, nl_r, n2_d, mask2, err2, max_slots,
                                     status=status, remap=(src, rbase, rlen, next_tail))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(to_np(out_r, np.uint16), to_np(out_c, np.uint16))
    assert np.array_equal(to_np(lse_r).view(np.uint32), to_np(lse_c).view(np.uint32))

    # the oracle through the record, on a sample of rows
    sample = sorted({(int(rng.integers(B)), int(rng.integers(N)), int(rng.integers(Hq)))
                     for _ in range(24)})
    sample = [(b, i, h) for (b, i, h) in sample if i < n2[b]]
    o_err2 = oracle.build_ancestors(parent2, n2, Dm)[3]
    ref, ref_lse = oracle.tree_attention(q2, to_np(kr, np.uint16), to_np(vr, np.uint16),
                                         big.block_table, nl, n2, parent2, o_err2, inp.scale,
                                         sample=sample, remap=(to_np(src), to_np(rbase),
                                                               to_np(rlen), to_np(next_tail)))
    got = oracle.bf16_to_f64(to_np(out_r, np.uint16))
    for (b, i, h) in sample:
        if o_err2[b] == 0:
            assert np.abs(got[b, i, h] - ref[b, i, h]).max() <= 1e-2
            assert abs(float(to_np(lse_r)[b, i, h]) - ref_lse[b, i, h]) <= 2e-3

    # materialising the record later: copy from the recorded tree base
    tail0 = dev_tensor(inp.prefix_len)
    nl_m, _ = tsd.kv_commit_path(kr, vr, table, prefix, n_nodes, A, path, err, N, Dm,
                                 tail_base=tail0, status=status)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(nl_m), nl)
    kc_h, vc_h, kr_h, vr_h = (to_np(x, np.uint16) for x in (kc, vc, kr, vr))
    for b in range(B):
        for s in range(int(nl[b])):
            pg, row = int(big.block_table[b, s // gen.PAGE]), s % gen.PAGE
            assert np.array_equal(kr_h[pg, :, row], kc_h[pg, :, row])
            assert np.array_equal(vr_h[pg, :, row], vc_h[pg, :, row])


def test_commit_from_a_shifted_tree_base(tsd):
    """The generalised copy: a tree written 37 slots past the prefix commits
    to the same bytes as the plain copy commit of the tree at the prefix."""
    import torch
    rng = np.random.default_rng(31)
    inp = gen.random_small(31, B=4, N_max=20, Hq=8, Hkv=2, D=128, V=64, prefix_lo=10,
                           prefix_hi=90, max_depth=5, p_match=0.9)
    big = gen.grow_cache(rng, inp.cache, inp.prefix_len, inp.n_nodes, extra=64)
    table = dev_tensor(big.block_table)
    B, N, Dm = inp.B, inp.N_max, inp.D_max
    parent, n_nodes, prefix = dev_tensor(inp.parent), dev_tensor(inp.n_nodes), dev_tensor(inp.prefix_len)
    anc, depth, mask, err = tsd.tree_build_ancestors(parent, n_nodes, Dm)
    _, A, _, path, _ = tsd.tree_verify_greedy(dev_tensor(inp.logits), dev_tensor(inp.tokens),
                                              parent, anc, depth, mask, n_nodes, err, Dm)
    k1, v1 = dev_tensor(big.k, torch.bfloat16), dev_tensor(big.v, torch.bfloat16)
    nl1, mv1 = tsd.kv_commit_path(k1, v1, table, prefix, n_nodes, A, path, err, N, Dm)
    k2, v2 = dev_tensor(big.k, torch.bfloat16), dev_tensor(big.v, torch.bfloat16)
    def rows_of(cache):  # the tree's rows as generated, [B][N][Hkv][D]
        return np.stack([np.stack([cache[int(big.block_table[b, (int(inp.prefix_len[b]) + j) // 16]),
                                         :, (int(inp.prefix_len[b]) + j) % 16] for j in range(N)])
                         for b in range(B)])
    rows_k, rows_v = rows_of(big.k), rows_of(big.v)
    shifted = inp.prefix_len + 37
    _write_rows(k2, v2, big.block_table, shifted, inp.n_nodes, rows_k, rows_v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nl2, mv2 = tsd.kv_commit_path(k2, v2, table, prefix, n_nodes, A, path, err, N, Dm,
                                  tail_base=dev_tensor(shifted.astype(np.int32)), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and np.array_equal(to_np(nl2), to_np(nl1))
    # every accepted entry moved, the root included
    o = oracle.commit_path(big.k, big.v, big.block_table, inp.prefix_len, to_np(A), to_np(path),
                           to_np(err), tail_base=shifted)
    assert np.array_equal(to_np(mv2), o[3])
    a_h, b_h = to_np(k1, np.uint16), to_np(k2, np.uint16)
    for b in range(B):
        for s in range(int(to_np(nl1)[b])):
            pg, row = int(big.block_table[b, s // 16]), s % 16
            assert np.array_equal(a_h[pg, :, row], b_h[pg, :, row])
