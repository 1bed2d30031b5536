"""Failure detection without a GPU fault: every wait inside the tree-attention
kernel is bounded.  With the test stall on, the kernel's MMA thread first
waits on a barrier that nothing signals; with a 1 ms limit that wait runs
out, and the kernel must report TSD_STATUS_TIMEOUT through its status word,
drain what it issued, free its tensor memory and return.  The context must
stay usable: the next call with the normal settings is correct."""

import numpy as np
import pytest

import gen

from _gpu_path import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_wait_limit_expiry_reports_timeout_and_recovers():
    import torch
    import tree_speculative_decoding_virtual_gb300 as tsd
    from _gpu_path import dev_tensor
    torch.cuda.set_device(0)
    inp = gen.random_small(31, B=2, N_max=24, Hq=8, Hkv=2, D=128, V=100, prefix_lo=200,
                           prefix_hi=600, max_depth=6)
    c = inp.cache
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    parent, n_nodes = dev_tensor(inp.parent), dev_tensor(inp.n_nodes)
    anc, depth, mask, err = tsd.tree_build_ancestors(parent, n_nodes, inp.D_max)
    old = tsd.get_option(tsd.OPT_WAIT_LIMIT_NS)
    try:
        tsd.set_option(tsd.OPT_WAIT_LIMIT_NS, 1_000_000)
        tsd.set_option(tsd.OPT_TEST_STALL, 1)
        tsd.tree_attn_fwd(dev_tensor(inp.q, torch.bfloat16), dev_tensor(c.k, torch.bfloat16),
                          dev_tensor(c.v, torch.bfloat16), dev_tensor(c.block_table),
                          dev_tensor(inp.prefix_len), n_nodes, mask, err,
                          int((inp.prefix_len + inp.n_nodes).max()), status=status)
        torch.cuda.synchronize()  # returns: no hang, no fault
        assert int(status.item()) & tsd.STATUS_TIMEOUT
    finally:
        tsd.set_option(tsd.OPT_TEST_STALL, 0)
        tsd.set_option(tsd.OPT_WAIT_LIMIT_NS, old)
    # the context is healthy: the same inputs give the oracle's answer
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    compare(inp, g, o)
    assert g["status"] == 0


def test_options_are_validated():
    import tree_speculative_decoding_virtual_gb300 as tsd
    with pytest.raises(tsd.TsdError):
        tsd.set_option(99, 1)
    with pytest.raises(tsd.TsdError):
        tsd.set_option(tsd.OPT_WAIT_LIMIT_NS, -5)
    assert tsd.get_option(tsd.OPT_TEST_STALL) == 0
    with pytest.raises(tsd.TsdError):
        tsd.set_option(tsd.OPT_TEST_STALL, 2)
