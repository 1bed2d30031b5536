"""The allocation-free verify entry point, for callers that cannot allocate
device memory (e.g. a plugin inside an engine that owns all device memory, or
a path where an allocation's implicit device synchronisation is not
allowed).  It must give the same results as the workspace entry point, call
after call, although every call reuses the same fixed device array.

This file is collected last on purpose: it must pass in a fresh process and
after every other test."""

import ctypes

import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


def _inputs_on_device(inp):
    from _gpu_path import dev_tensor
    return dict(logits=dev_tensor(inp.logits), tokens=dev_tensor(inp.tokens),
                parent=dev_tensor(inp.parent), n_nodes=dev_tensor(inp.n_nodes))


def _call_static_through_abi(tsd, d, anc, depth, mask, err, inp):
    """The new entry point, called directly through the C ABI."""
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


def test_static_scratch_matches_workspace_entry_point():
    import torch
    import tree_speculative_decoding_virtual_gb300 as tsd
    from _gpu_path import to_np
    torch.cuda.set_device(0)
    assert tsd.tree_verify_static_capacity() == 1 << 20
    # two calls in a row on different workloads: the shared array must not
    # carry anything from the first call into the second
    for inp in (gen.verify_workload("8b"), gen.verify_workload("ragged")):
        d = _inputs_on_device(inp)
        anc, depth, mask, err = tsd.tree_build_ancestors(d["parent"], d["n_nodes"], inp.D_max)
        ref = tsd.tree_verify_greedy(d["logits"], d["tokens"], d["parent"], anc, depth, mask,
                                     d["n_nodes"], err, inp.D_max)
        got = _call_static_through_abi(tsd, d, anc, depth, mask, err, inp)
        torch.cuda.synchronize()
        for name, r in zip(["argmax", "accept_len", "leaf", "path", "bonus"], ref):
            assert np.array_equal(to_np(got[name]), to_np(r)), name


def test_static_scratch_rejects_oversized_batches():
    import tree_speculative_decoding_virtual_gb300 as tsd
    # 65535 sequences x 256 rows of 8-byte argmax keys cannot fit in 1 MiB
    rc = tsd.lib.tsd_tree_verify_greedy_static(1, 1, 1, 1, 1, 1, None, None, 65535, 256, 128256, 8,
                                               1, 1, 1, 1, 1, None)
    assert rc == -2  # TSD_ERR_LIMIT, nothing launched
