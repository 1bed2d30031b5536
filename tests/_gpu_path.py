"""Helpers for the GPU parity tests: run the CUDA path through the binding and
the oracle on the same seeded inputs, and compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL_MAX = 1e-2   # attention: max-abs over valid elements (bf16 in, fp32 accumulate)
ATOL_MEAN = 2e-3  # attention: mean-abs over valid elements
LSE_ATOL = 2e-3   # lse: fp32 sums of O(P) terms, relative error ~1e-6; absolute bound


def dev_tensor(a, dtype=None, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


def to_np(t, dtype=None):
    a = t.detach().cpu()
    if a.dtype == torch.bfloat16:
        a = a.view(torch.int16)
    a = a.numpy()
    return a.view(dtype) if dtype is not None else a


def run_gpu(tsd, inp, sample_attention=None, with_lse=True, max_slots=None):
    """Whole hot path on the GPU; returns a dict of numpy arrays (cache after
    commit included).  ``max_slots`` is the host bound passed to the attention
    (default: the exact largest prefix + nodes)."""
    c = inp.cache
    parent = dev_tensor(inp.parent)
    n_nodes = dev_tensor(inp.n_nodes)
    prefix = dev_tensor(inp.prefix_len)
    table = dev_tensor(c.block_table)
    k = dev_tensor(c.k, torch.bfloat16)
    v = dev_tensor(c.v, torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    anc, depth, mask, err = tsd.tree_build_ancestors(parent, n_nodes, inp.D_max)
    if max_slots is None:
        max_slots = int((inp.prefix_len + inp.n_nodes).max())
    out, lse = tsd.tree_attn_fwd(dev_tensor(inp.q, torch.bfloat16), k, v, table, prefix, n_nodes,
                                 mask, err, max_slots, want_lse=with_lse, status=status)
    am, A, leaf, path, bonus = tsd.tree_verify_greedy(dev_tensor(inp.logits),
                                                      dev_tensor(inp.tokens), parent, anc, depth,
                                                      mask, n_nodes, err, inp.D_max)
    new_len, moved = tsd.kv_commit_path(k, v, table, prefix, n_nodes, A, path, err, inp.N_max,
                                        inp.D_max, status=status)
    torch.cuda.synchronize()
    return dict(anc=to_np(anc), depth=to_np(depth), mask=to_np(mask, np.uint32), err=to_np(err),
                out=to_np(out, np.uint16), lse=None if lse is None else to_np(lse),
                argmax=to_np(am), accept_len=to_np(A), leaf=to_np(leaf), path=to_np(path),
                bonus=to_np(bonus), new_len=to_np(new_len), moved=to_np(moved),
                k=to_np(k, np.uint16), v=to_np(v, np.uint16), status=int(status.item()))


def run_oracle(inp, sample_attention=None):
    c = inp.cache
    anc, depth, mask, err = oracle.build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    out, lse = oracle.tree_attention(inp.q, c.k, c.v, c.block_table, inp.prefix_len, inp.n_nodes,
                                     inp.parent, err, inp.scale, sample=sample_attention)
    am, A, leaf, path, bonus = oracle.verify_greedy(inp.logits, inp.tokens, inp.parent,
                                                    inp.n_nodes, err, inp.D_max)
    k1, v1, new_len, moved = oracle.commit_path(c.k, c.v, c.block_table, inp.prefix_len, A, path,
                                                err)
    return dict(anc=anc, depth=depth, mask=mask, err=err, out=out, lse=lse, argmax=am,
                accept_len=A, leaf=leaf, path=path, bonus=bonus, new_len=new_len, moved=moved,
                k=k1, v=v1)


def attention_rows(inp, err, sample=None, attn_skip=()):
    """Boolean [B][N_max][Hq] of rows to compare (valid nodes of sequences
    without errors and not in ``attn_skip``, restricted to the sample if
    given)."""
    sel = np.zeros((inp.B, inp.N_max, inp.Hq), dtype=bool)
    for b in range(inp.B):
        if err[b] == 0 and b not in attn_skip:
            sel[b, :int(inp.n_nodes[b]), :] = True
    if sample is not None:
        only = np.zeros_like(sel)
        for (b, i, h) in sample:
            only[b, i, h] = True
        sel &= only
    return sel


def compare(inp, g, o, sample=None, check_lse=True, attn_skip=()):
    """``attn_skip``: sequences the attention alone must skip (a key range
    beyond the max_slots bound): their rows are checked to be zero / -inf."""
    for key in ["anc", "depth", "mask", "err"]:
        assert np.array_equal(g[key], o[key]), key
    for key in ["argmax", "accept_len", "leaf", "path", "bonus", "new_len", "moved"]:
        assert np.array_equal(g[key], o[key]), (key, g[key], o[key])
    assert np.array_equal(g["k"], o["k"]), "committed K cache"
    assert np.array_equal(g["v"], o["v"]), "committed V cache"
    sel = attention_rows(inp, o["err"], sample, attn_skip)
    got = oracle.bf16_to_f64(g["out"])
    diff = np.abs(got - o["out"])[sel]
    if diff.size:
        assert diff.max() <= ATOL_MAX, ("attention max-abs", diff.max())
        assert diff.mean() <= ATOL_MEAN, ("attention mean-abs", diff.mean())
    # skipped / padding rows are zero and -inf
    skip = attention_rows(inp, o["err"], None, attn_skip) == False  # noqa: E712
    assert (g["out"][skip] == 0).all()
    if check_lse and g["lse"] is not None:
        d = np.abs(g["lse"].astype(np.float64)[sel] - o["lse"][sel])
        if d.size:
            assert d.max() <= LSE_ATOL, ("lse", d.max())
        assert np.isneginf(g["lse"][skip]).all()
    return float(diff.max()) if diff.size else 0.0, float(diff.mean()) if diff.size else 0.0
