"""GPU parity of stochastic tree verification against the oracle.

The kernel computes in fp32, the oracle in fp64.  Every acceptance test and
every draw is a comparison of a uniform with a threshold; where the uniform
lies within rounding of the threshold either outcome is correct, so the
inputs are made unambiguous first: the oracle reports how far each used
uniform lies from its threshold (relative to the larger side for
acceptances, to the total weight for draws), and uniforms closer than the
margins below are drawn again.  Then every node's accepted child and drawn
token, and every sequence's walk, must match exactly.

Margins: the kernel's weights carry a relative error of a few fp32 ulps
(expf, the division by the normaliser) and its cumulative sums over up to
2^18 tokens a relative error below 40 ulps of the total (sums of at most
~80 terms per thread, then warp, block and cluster trees); 2e-5 of the
total for draws and 1e-3 relative for acceptances leave a factor of at
least eight.
"""

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu

EPS_ACCEPT = 1e-3
EPS_DRAW = 2e-5


@pytest.fixture(scope="module")
def tsd():
    import torch
    import tree_speculative_decoding_virtual_gb300 as m
    torch.cuda.set_device(0)
    return m


def _children(parent, nb, i):
    return [j for j in range(1, nb) if int(parent[j]) == i]


def unambiguous(inp, max_iter=60):
    """Redraw uniforms until no decision lies within the margins; returns
    the oracle's result on the final inputs."""
    rng = np.random.default_rng(inp.seed + 12345)
    for _ in range(max_iter):
        out = oracle.tree_verify_stochastic_all(inp.logits, inp.q_draft, inp.tokens, inp.parent,
                                                inp.n_nodes, inp.D_max, inp.u_accept, inp.u_draw,
                                                return_margins=True)
        am, dm = out[6], out[7]
        bad = np.argwhere((am < EPS_ACCEPT) | (dm < EPS_DRAW))
        if bad.size == 0:
            return out[:6]
        ab, ai, db, di = [], [], [], []
        for b, i in bad:
            for c in _children(inp.parent[b], int(inp.n_nodes[b]), int(i)):
                ab.append(b)
                ai.append(c)
            db.append(b)
            di.append(i)
        gen.redraw_uniforms(inp, rng, (np.array(ab, dtype=np.int64), np.array(ai, dtype=np.int64)),
                            (np.array(db, dtype=np.int64), np.array(di, dtype=np.int64)))
    raise AssertionError("could not draw unambiguous uniforms")


def run_gpu(tsd, inp, repeat=1):
    import torch
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    parent, n_nodes, tokens = d(inp.parent), d(inp.n_nodes), d(inp.tokens)
    logits, q = d(inp.logits), d(inp.q_draft)
    ua, ud = d(inp.u_accept), d(inp.u_draw)
    anc, depth, mask, err = tsd.tree_build_ancestors(parent, n_nodes, inp.D_max)
    ws = torch.zeros(max(tsd.tree_verify_stochastic_workspace_bytes(inp.B, inp.N_max, inp.V), 1),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(repeat):
        r = tsd.tree_verify_stochastic(logits, q, tokens, parent, n_nodes, err, ua, ud, inp.D_max,
                                       workspace=ws)
        torch.cuda.synchronize()
        outs.append([x.cpu().numpy() for x in r])
    assert not ws[:4 * inp.B].any().item(), "tickets not left zero-filled"
    return outs if repeat > 1 else outs[0]


NAMES = ["next", "draw", "accept_len", "leaf", "path", "bonus"]


def compare(got, ref):
    for name, g, r in zip(NAMES, got, ref):
        if not np.array_equal(g, r):
            idx = np.argwhere(g != r)[:5]
            raise AssertionError("%s differs at %s: gpu %s oracle %s" % (
                name, idx.tolist(), [g[tuple(i)] for i in idx], [r[tuple(i)] for i in idx]))


CASES = [
    # seed, B, N_max, V, depth, ragged
    (1, 3, 33, 1000, 8, True),
    (2, 2, 64, 257, 12, True),     # V not a multiple of 4: scalar loads
    (3, 4, 17, 4099, 5, False),
    (4, 2, 256, 300, 32, True),    # the node limit, deep trees
    (5, 2, 1, 50, 0, False),       # a lone root: a draw from p
    (6, 3, 31, 32000, 5, True),
    (7, 1, 9, 262144, 4, False),   # the vocabulary limit: eight CTAs of 32768
    (8, 2, 40, 3, 6, False),       # fewer tokens than CTAs could take
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_random_trees(tsd, case):
    seed, B, N, V, depth, ragged = case
    inp = gen.stochastic_inputs(seed, B, N, V, depth, ragged_nodes=ragged)
    ref = unambiguous(inp)
    compare(run_gpu(tsd, inp), ref)


def test_8b_shape(tsd):
    """The 8B-shaped verify layer: the 63-node static tree, V = 128256."""
    B, N, V = 1, 63, 128256
    parents = np.stack([gen.static_8b_tree()])
    inp = gen.stochastic_inputs(21, B, N, V, 6, parents=parents)
    ref = unambiguous(inp)
    got = run_gpu(tsd, inp)
    compare(got, ref)
    assert got[2][0] >= 0


def test_70b_shape(tsd):
    """Four sequences of 127-node random trees (depth <= 8), V = 128256."""
    inp = gen.stochastic_inputs(22, 4, 127, 128256, 8)
    ref = unambiguous(inp)
    compare(run_gpu(tsd, inp), ref)


def test_low_acceptance_many_rejections(tsd):
    """A draft far from the target: most children rejected, so many nodes
    run several residual rounds before settling or drawing."""
    inp = gen.stochastic_inputs(23, 3, 48, 5000, 3, logit_std=2.0, draft_noise=4.0)
    ref = unambiguous(inp)
    got = run_gpu(tsd, inp)
    compare(got, ref)
    n_draw_internal = sum(int((got[1][b] >= 0).sum()) for b in range(3))
    assert n_draw_internal > 0


def test_star_tree(tsd):
    """A root with 255 children (up to 255 residual rounds in one cluster)."""
    N = 256
    parents = np.zeros((1, N), dtype=np.int32)
    parents[0, 0] = -1
    inp = gen.stochastic_inputs(24, 1, N, 700, 1, parents=parents, draft_noise=3.0)
    inp.u_accept[:] = np.float32(0.999)   # reject nearly everything
    ref = unambiguous(inp)
    compare(run_gpu(tsd, inp), ref)


def test_equal_distributions_accept_first_children(tsd):
    """q equal to the target distribution (rounded to fp32): with uniforms
    below 1 - 1e-3 every first child is accepted."""
    inp = gen.stochastic_inputs(25, 2, 40, 3000, 7)
    l = inp.logits.astype(np.float64)
    e = np.exp(l - l.max(axis=2, keepdims=True))
    inp.q_draft[:] = (e / e.sum(axis=2, keepdims=True)).astype(np.float32)
    inp.u_accept[:] = np.minimum(inp.u_accept, np.float32(0.998))
    ref = unambiguous(inp)
    got = run_gpu(tsd, inp)
    compare(got, ref)
    for b in range(2):
        for i in range(40):
            kids = _children(inp.parent[b], 40, i)
            assert got[0][b, i] == (kids[0] if kids else -1)


def test_zero_mass_residual(tsd):
    """Target and draft one-hot on the same token a; the first child's token
    b != a has q(b) = 0 = p(b) and is rejected; the residual max(0, p - q)
    is then empty and is replaced by q, so the next child (token a) is
    accepted, and a node whose children are all rejected draws a."""
    V, N = 64, 6
    parent = np.array([[-1, 0, 0, 1, 1, 3]], dtype=np.int32)
    inp = gen.stochastic_inputs(26, 1, N, V, 5, parents=parent)
    a = 17
    inp.logits[:] = -1000.0
    inp.logits[:, :, a] = 0.0
    inp.q_draft[:] = 0.0
    inp.q_draft[:, :, a] = 1.0
    inp.tokens[0] = [0, 5, a, 9, 8, a]   # root: b then a; node 1: b, b; node 3: a
    inp.u_accept[:] = 0.5
    ref = unambiguous(inp)
    got = run_gpu(tsd, inp)
    compare(got, ref)
    assert got[0][0, 0] == 2 and got[0][0, 1] == -1 and got[1][0, 1] == a


def test_skipped_padding_and_bad_tokens(tsd):
    import torch
    inp = gen.stochastic_inputs(27, 4, 20, 900, 6, ragged_nodes=True)
    inp.parent[1, 0] = 3            # root with a parent: TREE_ROOT
    inp.n_nodes[2] = 0              # TREE_COUNT
    nb = int(inp.n_nodes[3])
    if nb > 2:
        inp.tokens[3, 1] = -7       # out-of-range child tokens are skipped
        inp.tokens[3, nb - 1] = 900
    ref = unambiguous(inp)
    got = run_gpu(tsd, inp)
    compare(got, ref)
    for b in (1, 2):
        assert got[2][b] == 0 and got[3][b] == -1 and got[5][b] == -1
        assert (got[0][b] == -1).all() and (got[1][b] == -1).all()


def test_repeat_calls_identical(tsd):
    inp = gen.stochastic_inputs(28, 3, 50, 2000, 6, ragged_nodes=True)
    ref = unambiguous(inp)
    outs = run_gpu(tsd, inp, repeat=3)
    for got in outs:
        compare(got, ref)


def test_host_checks(tsd):
    import torch
    inp = gen.stochastic_inputs(29, 2, 8, 100, 3)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    parent, n_nodes, tokens = d(inp.parent), d(inp.n_nodes), d(inp.tokens)
    logits, q = d(inp.logits), d(inp.q_draft)
    ua, ud = d(inp.u_accept), d(inp.u_draw)
    _, _, _, err = tsd.tree_build_ancestors(parent, n_nodes, inp.D_max)
    # an output aliasing an input
    with pytest.raises(tsd.TsdError):
        tsd.tree_verify_stochastic(logits, q, tokens, parent, n_nodes, err, ua, ud, inp.D_max,
                                   next=tokens)
    # err is required
    with pytest.raises(tsd.TsdError):
        tsd.tree_verify_stochastic(logits, q, tokens, parent, n_nodes, None, ua, ud, inp.D_max)
    # the vocabulary limit
    big = torch.zeros((1, 1, 262148), dtype=torch.float32, device="cuda")
    with pytest.raises(tsd.TsdError):
        tsd.tree_verify_stochastic(big, big.clone(), tokens[:1, :1].contiguous(),
                                   parent[:1, :1].contiguous(), None, err[:1].contiguous(),
                                   ua[:1, :1].contiguous(), ud[:1, :1].contiguous(), 0)
    for V in (3, 1000, 32000, 128256, 262144):
        C, S = tsd.tree_verify_stochastic_plan(1, 63, V)
        assert 1 <= C <= 8 and C * S >= V and S % 4 == 0


def test_commit_after_stochastic_verify(tsd):
    """The walk's accept_len and path feed the commit unchanged (the layout
    of the greedy verify's result)."""
    import torch
    from _gpu_path import dev_tensor, to_np
    base = gen.random_small(31, B=3, N_max=30, Hq=8, Hkv=2, D=64, V=500, prefix_lo=5,
                            prefix_hi=70, max_depth=6, ragged_nodes=True)
    inp = gen.stochastic_inputs(31, 3, 30, 500, 6, parents=base.parent)
    inp.n_nodes = base.n_nodes.copy()   # the same trees and node counts as the cache
    ref = unambiguous(inp)
    got = run_gpu(tsd, inp)
    compare(got, ref)
    c = base.cache
    k = dev_tensor(c.k, torch.bfloat16)
    v = dev_tensor(c.v, torch.bfloat16)
    bt, pl, nn = dev_tensor(c.block_table), dev_tensor(base.prefix_len), dev_tensor(base.n_nodes)
    _, _, _, err = tsd.tree_build_ancestors(dev_tensor(base.parent), nn, base.D_max)
    new_len, moved = tsd.kv_commit_path(k, v, bt, pl, nn, torch.from_numpy(got[2]).cuda(),
                                        torch.from_numpy(got[4]).cuda(), err, base.N_max,
                                        base.D_max)
    torch.cuda.synchronize()
    rk, rv, rlen, rmoved = oracle.commit_path(c.k, c.v, c.block_table, base.prefix_len, got[2],
                                              got[4], np.zeros(3, dtype=np.int32))
    assert np.array_equal(to_np(new_len), rlen) and np.array_equal(to_np(moved), rmoved)
    assert np.array_equal(to_np(k, np.uint16), rk) and np.array_equal(to_np(v, np.uint16), rv)
