"""No leakage across branches, on the GPU: a node sees its ancestors and
itself in the tree tail, nothing else ("EAGLE-Pangu" technical summary 2.3,
fused tree-masked teacher execution; "Speculative Decoding Hierárquico",
Medusa tree attention mask).  Overwriting every tail K/V entry that is not an
ancestor of a chosen node (nor the node) with +-100 must leave that node's
output and lse bit-identical, and the outputs of its ancestors and of every
other sequence too; every node whose own slot was overwritten must change.

Runs the three kernel layouts: the 8B shape (two blocks per SM, splits
merged by the merge kernel), the ragged batch (device split plan) and the
70B shape (256-row blocks)."""

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu

BF16_100 = 0x42C8  # +100.0 as bf16 bits; the sign bit gives -100


@pytest.fixture(scope="module")
def tsd():
    import torch
    import tree_speculative_decoding_virtual_gb300 as m
    torch.cuda.set_device(0)
    return m


def _chain(parent_row, i):
    out = [i]
    while parent_row[out[-1]] >= 0:
        out.append(int(parent_row[out[-1]]))
    return set(out)


@pytest.mark.parametrize("workload", ["8b", "ragged", "70b"])
def test_non_ancestor_kv_cannot_leak(tsd, workload):
    import torch
    from _gpu_path import dev_tensor, to_np
    inp = gen.verify_workload(workload)
    c = inp.cache
    b = 0
    nb, P = int(inp.n_nodes[b]), int(inp.prefix_len[b])
    depths = [len(_chain(inp.parent[b], j)) - 1 for j in range(nb)]
    i = int(np.argmax(depths))  # the deepest node (lowest id): the longest kept path
    keep = _chain(inp.parent[b], i)
    pert = [j for j in range(nb) if j not in keep]
    assert len(pert) > 0

    parent, n_nodes = dev_tensor(inp.parent), dev_tensor(inp.n_nodes)
    anc, depth, mask, err = tsd.tree_build_ancestors(parent, n_nodes, inp.D_max)
    q = dev_tensor(inp.q, torch.bfloat16)
    k = dev_tensor(c.k, torch.bfloat16)
    v = dev_tensor(c.v, torch.bfloat16)
    table, prefix = dev_tensor(c.block_table), dev_tensor(inp.prefix_len)
    max_slots = int((inp.prefix_len + inp.n_nodes).max())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def attend():
        out, lse = tsd.tree_attn_fwd(q, k, v, table, prefix, n_nodes, mask, err, max_slots,
                                     status=status)
        torch.cuda.synchronize()
        return to_np(out, np.uint16), to_np(lse).view(np.uint32)

    out1, lse1 = attend()
    rng = np.random.default_rng(17)
    kv = k.view(torch.int16), v.view(torch.int16)
    for j in pert:
        slot = P + j
        blk, row = int(c.block_table[b, slot // gen.PAGE]), slot % gen.PAGE
        for t in kv:
            signs = rng.integers(0, 2, size=(inp.Hkv, inp.D)).astype(np.uint16) << 15
            t[blk, :, row, :] = torch.from_numpy((signs | BF16_100).view(np.int16)).cuda()
    out2, lse2 = attend()
    assert int(status.item()) == 0

    for j in sorted(keep):  # the node and its ancestors: bit for bit
        assert np.array_equal(out2[b, j], out1[b, j]), ("out", j)
        assert np.array_equal(lse2[b, j], lse1[b, j]), ("lse", j)
    assert np.array_equal(out2[b + 1:], out1[b + 1:]) and np.array_equal(lse2[b + 1:], lse1[b + 1:])
    for j in pert:  # its own slot was overwritten: its output moves
        assert not np.array_equal(out2[b, j], out1[b, j]), ("unchanged", j)

    # the overwritten keys score far above the rest (about 100 * |q| / sqrt(D))
    # and their values are +-100; a few such rows still match the oracle on the
    # perturbed cache, within the tolerance scaled to the row's magnitude (the
    # bf16 rounding of the output and of P is relative)
    k_h, v_h = to_np(k, np.uint16), to_np(v, np.uint16)
    sample = [(b, j, h) for j in pert[:2] for h in (0, inp.Hq - 1)] + [(b, i, 0)]
    ref, ref_lse = oracle.tree_attention(inp.q, k_h, v_h, c.block_table, inp.prefix_len,
                                         inp.n_nodes, inp.parent, np.zeros(inp.B, np.int32),
                                         inp.scale, sample=sample)
    got = oracle.bf16_to_f64(out2)
    for (bb, j, h) in sample:
        scale = max(1.0, float(np.abs(ref[bb, j, h]).max()))
        assert np.abs(got[bb, j, h] - ref[bb, j, h]).max() <= 1e-2 * scale
        r = ref_lse[bb, j, h]
        assert abs(float(lse2[bb, j, h].view(np.float32)) - r) <= 2e-3 + 1e-5 * abs(r)
