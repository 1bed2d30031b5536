"""The allocation-free verify entry point, for callers that cannot allocate
device memory (e.g. a plugin inside an engine that owns all device memory, or
a path where an allocation's implicit device synchronisation is not
allowed).  It must give the oracle's results (and the workspace entry
point's), call after call, although every call reuses the same fixed device
array: on two workloads in a row, at exactly the array's capacity, and after
a batch with malformed trees.

This file is collected last on purpose: it must pass in a fresh process and
after every other test."""

import ctypes

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


def _inputs_on_device(inp):
    from _gpu_path import dev_tensor
    return dict(logits=dev_tensor(inp.logits), tokens=dev_tensor(inp.tokens),
                parent=dev_tensor(inp.parent), n_nodes=dev_tensor(inp.n_nodes))


def _call_static_through_abi(tsd, d, anc, depth, mask, err, inp):
    """The allocation-free entry point, called directly through the C ABI."""
    import torch
    B, N, V, Dm = inp.B, inp.N_max, inp.V, inp.D_max
    outs = dict(argmax=torch.empty((B, N), dtype=torch.int32, device="cuda"),
                accept_len=torch.empty((B,), dtype=torch.int32, device="cuda"),
                leaf=torch.empty((B,), dtype=torch.int32, device="cuda"),
                path=torch.empty((B, Dm + 1), dtype=torch.int32, device="cuda"),
                bonus=torch.empty((B,), dtype=torch.int32, device="cuda"))
    rc = tsd.lib.tsd_tree_verify_greedy_static(
        d["logits"].data_ptr(), d["tokens"].data_ptr(), d["parent"].data_ptr(), anc.data_ptr(),
        depth.data_ptr(), mask.data_ptr(), d["n_nodes"].data_ptr(), err.data_ptr(), B, N, V, Dm,
        outs["argmax"].data_ptr(), outs["accept_len"].data_ptr(), outs["leaf"].data_ptr(),
        outs["path"].data_ptr(), outs["bonus"].data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    return outs


NAMES = ["argmax", "accept_len", "leaf", "path", "bonus"]


def _check_against_oracle_and_workspace(tsd, inp):
    import torch
    from _gpu_path import to_np
    d = _inputs_on_device(inp)
    anc, depth, mask, err = tsd.tree_build_ancestors(d["parent"], d["n_nodes"], inp.D_max)
    ref = tsd.tree_verify_greedy(d["logits"], d["tokens"], d["parent"], anc, depth, mask,
                                 d["n_nodes"], err, inp.D_max)
    got = _call_static_through_abi(tsd, d, anc, depth, mask, err, inp)
    torch.cuda.synchronize()
    _, _, _, o_err = oracle.build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    want = oracle.verify_greedy(inp.logits, inp.tokens, inp.parent, inp.n_nodes, o_err, inp.D_max)
    for name, r, o in zip(NAMES, ref, want):
        assert np.array_equal(to_np(got[name]), o), ("oracle", name)
        assert np.array_equal(to_np(got[name]), to_np(r)), ("workspace entry point", name)
    return o_err


def test_static_scratch_matches_oracle_call_after_call():
    import torch
    import tree_speculative_decoding_virtual_gb300 as tsd
    torch.cuda.set_device(0)
    assert tsd.tree_verify_static_capacity() == 1 << 20
    # two calls in a row on different workloads: the shared array must not
    # carry anything from the first call into the second
    for inp in (gen.verify_workload("8b"), gen.verify_workload("ragged")):
        _check_against_oracle_and_workspace(tsd, inp)


def test_static_scratch_at_capacity_and_after_malformed_trees():
    import torch
    import tree_speculative_decoding_virtual_gb300 as tsd
    torch.cuda.set_device(0)
    # 511 sequences x 256 rows: 2048 bytes of tickets (511 rounded up to 256-byte
    # alignment) + 511 * 256 8-byte keys = exactly 1 MiB, the array's size
    inp = gen.random_small(511, B=511, N_max=256, Hq=1, Hkv=1, D=64, V=48, prefix_lo=0,
                           prefix_hi=1, max_depth=8, p_match=0.7, ragged_nodes=False)
    # a self-loop and a second root: the ancestors kernel flags these sequences
    inp.parent[3, 200] = 200
    inp.parent[400, 17] = -1
    o_err = _check_against_oracle_and_workspace(tsd, inp)
    assert o_err[3] != 0 and o_err[400] != 0 and (o_err == 0).sum() == 509
    # the next call, on a well-formed batch, still matches
    _check_against_oracle_and_workspace(tsd, gen.verify_workload("tiny", seed=5))


def test_static_scratch_rejects_oversized_batches():
    import tree_speculative_decoding_virtual_gb300 as tsd
    # one sequence more than the capacity case: 2048 + 512 * 256 * 8 bytes > 1 MiB
    rc = tsd.lib.tsd_tree_verify_greedy_static(1, 1, 1, 1, 1, 1, None, None, 512, 256, 48, 8,
                                               1, 1, 1, 1, 1, None)
    assert rc == -2  # TSD_ERR_LIMIT, nothing launched
    rc = tsd.lib.tsd_tree_verify_greedy_static(1, 1, 1, 1, 1, 1, None, None, 65535, 256, 128256,
                                               8, 1, 1, 1, 1, 1, None)
    assert rc == -2
