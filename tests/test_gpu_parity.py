"""GPU parity: the CUDA path through the C ABI against the oracle on the same
seeded inputs.  Bit-exact for ancestors, masks, error bits, argmax, accepted
length / leaf / path / bonus, commit lengths and the whole committed cache
pool; attention within max-abs 1e-2 and mean-abs 2e-3 over valid elements.

Covers the five verify workloads at their full sizes (the 70B-shaped one on a
sample of attention rows the oracle computes one by one), randomised small
shapes across tile boundaries, node counts and prefixes, and the degenerate
and fail-closed cases."""

import numpy as np
import pytest

import gen
import oracle

from _gpu_path import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsd():
    import torch
    import tree_speculative_decoding_virtual_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.mark.parametrize("name", ["tiny", "8b", "ragged"])
def test_workload_full(tsd, name):
    inp = gen.verify_workload(name)
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    mx, mean = compare(inp, g, o)
    assert g["status"] == 0
    assert o["accept_len"].min() >= 0


@pytest.mark.parametrize("seed", [5, 8])
def test_tiny_shape_with_accepted_moves(tsd, seed):
    """The tiny workload's shapes with seeds whose trees accept two and four
    draft tokens, so the commit moves entries (seed 0, the workload's own,
    accepts none)."""
    inp = gen.verify_workload("tiny", seed=seed)
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    compare(inp, g, o)
    assert g["status"] == 0
    assert o["accept_len"].min() >= 2 and o["moved"].min() >= 2


def test_workload_70b_sampled(tsd):
    inp = gen.verify_workload("70b")
    rng = np.random.default_rng(0)
    sample = set()
    for b in range(inp.B):
        for h in rng.choice(inp.Hq, size=6, replace=False):
            for i in range(inp.N_max):
                sample.add((b, i, int(h)))
        for _ in range(64):
            sample.add((b, int(rng.integers(inp.N_max)), int(rng.integers(inp.Hq))))
    sample = sorted(sample)
    g = run_gpu(tsd, inp)
    o = run_oracle(inp, sample_attention=sample)
    compare(inp, g, o, sample=sample)
    assert g["status"] == 0


def _plant_jump(inp, b, node, h, scale, slots):
    """Set the keys at `slots` of sequence b (in the kv head of q-head h) to
    `scale` times the query of (node, h): with |q|^2 ~ D their scores exceed
    the other keys' by about 16 * scale in log2 units."""
    c = inp.cache
    hkv = h // (inp.Hq // inp.Hkv)
    qf = (inp.q[b, node, h].astype(np.uint32) << 16).view(np.float32)
    kbits = gen.bf16_bits(qf * np.float32(scale))
    for s in slots:
        c.k[c.block_table[b, s // gen.PAGE], hkv, s % gen.PAGE] = kbits


@pytest.mark.parametrize("workload,scale", [("8b", 2.0), ("8b", 16.0), ("70b", 5.0)])
def test_scores_far_above_the_first_tile(tsd, workload, scale):
    """Keys late in a split's range that score far above its first tile (by
    about 30, 260 and 80 in log2 units): the kernels weigh P against the first
    tile's max while a tile sums to at most 2^64 and otherwise take the max
    again and rescale; the planted rows and their neighbours match the oracle
    (the 8B shape runs the two-blocks-per-SM kernel, the 70B shape 256-row
    blocks)."""
    inp = gen.verify_workload(workload)
    P0 = int(inp.prefix_len[0])
    slots = [P0 // 3, P0 // 2 + 37, (2 * P0) // 3 + 70, P0 - 5]
    for h in (0, inp.Hq // inp.Hkv):  # a q-head of each of the first two kv heads
        _plant_jump(inp, 0, 0, h, scale, slots)
    sample = {(0, i, h) for i in range(min(inp.N_max, 8)) for h in range(inp.Hq)}
    sample |= {(b, 0, 0) for b in range(inp.B)}
    sample = sorted(sample)
    g = run_gpu(tsd, inp)
    o = run_oracle(inp, sample_attention=sample)
    compare(inp, g, o, sample=sample)
    assert g["status"] == 0


@pytest.mark.parametrize("N", [16, 32, 64, 128, 256])
def test_bastion_budget(tsd, N):
    import torch
    from _gpu_path import dev_tensor, to_np
    q, root = gen.bastion_marginals()
    bf = tsd.best_first_tree_build(dev_tensor(q), dev_tensor(root), N)
    torch.cuda.synchronize()
    got = [to_np(x) for x in bf]
    ref = oracle.best_first_tree(q, root, N)
    for name, x, y in zip(["parent", "tokens", "depth", "rho", "ahat"], got, ref):
        assert np.array_equal(x, y), name
    # verify the built tree on the 8B-shaped layer
    top1 = np.stack([[oracle.ranked_tokens(q[b, k])[0] for k in range(q.shape[1])]
                     for b in range(q.shape[0])])
    inp = gen.bastion_verify_inputs(ref[0], ref[1], ref[2], top1)
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    compare(inp, g, o)


def test_long_context_many_splits(tsd):
    """Prefixes of 150k-200k keys: the split count reaches its largest values
    (the merge takes its widest form), a GQA group of 16 heads fills 320 rows
    (a full 256-row block plus a 64-row block that runs its two softmax groups
    on alternate key tiles); sampled rows against the oracle."""
    inp = gen.random_small(4242, B=2, N_max=20, Hq=16, Hkv=1, D=128, V=500, prefix_lo=150000,
                           prefix_hi=200000, max_depth=5, ragged_nodes=False)
    rng = np.random.default_rng(1)
    sample = sorted({(b, int(rng.integers(inp.N_max)), int(rng.integers(inp.Hq)))
                     for b in range(inp.B) for _ in range(40)})
    g = run_gpu(tsd, inp)
    o = run_oracle(inp, sample_attention=sample)
    compare(inp, g, o, sample=sample)
    assert g["status"] == 0


@pytest.mark.parametrize("case", ["70b-shaped", "kv2"])
def test_single_sequence_long_context(tsd, case):
    """One sequence with a long prefix and the host's uniform split: the 70B
    shape with B = 1 (eight 128-row blocks per kv head), and on the 256-row
    kernel a GQA group of 16 over 20 nodes (a 256-row block and a 64-row block
    whose two softmax groups take alternate key tiles) with a 150k-key prefix
    cut into 32 pieces."""
    if case == "70b-shaped":
        inp = gen.random_small(77, B=1, N_max=127, Hq=64, Hkv=8, D=128, V=300, prefix_lo=32768,
                               prefix_hi=32768, max_depth=8, ragged_nodes=False)
    else:
        inp = gen.random_small(78, B=1, N_max=20, Hq=16, Hkv=1, D=128, V=300, prefix_lo=150000,
                               prefix_hi=150000, max_depth=5, ragged_nodes=False)
    max_slots = int((inp.prefix_len + inp.n_nodes).max())
    plan = tsd.tree_attn_plan(1, inp.N_max, inp.Hq, inp.Hkv, inp.D, max_slots)
    assert plan["mode"] == 1 and plan["splits"] > 1
    if case == "kv2":
        assert plan["rows_per_block"] == 256 and plan["two_blocks_per_sm"] == 0
    rng = np.random.default_rng(5)
    sample = sorted({(0, int(rng.integers(inp.N_max)), int(rng.integers(inp.Hq)))
                     for _ in range(60)} | {(0, inp.N_max - 1, h) for h in range(inp.Hq)})
    g = run_gpu(tsd, inp)
    o = run_oracle(inp, sample_attention=sample)
    compare(inp, g, o, sample=sample)
    assert g["status"] == 0


# Skewed prefix lengths: one long sequence among short ones (and an empty
# prefix), so the device split plan cuts the long key ranges into many pieces
# and the short ones into one or two.
SKEWED_PREFIX = [20000, 150, 900, 40, 3000, 0, 7000, 260]


@pytest.mark.parametrize("loose", [False, True])
def test_ragged_split_plan(tsd, loose):
    """Ragged batch through the device split plan, with the exact host bound
    on prefix + nodes and with a loose one (4x): both must give the oracle's
    result; the loose bound only changes the grid the plan may use."""
    inp = gen.random_small(31337, B=8, N_max=24, Hq=16, Hkv=2, D=128, V=300, prefix_lo=0,
                           prefix_hi=1, max_depth=6, prefix_len=np.array(SKEWED_PREFIX))
    exact = int((inp.prefix_len + inp.n_nodes).max())
    g = run_gpu(tsd, inp, max_slots=4 * exact if loose else exact)
    o = run_oracle(inp)
    compare(inp, g, o)
    assert g["status"] == 0


def test_split_plan_edges(tsd):
    """Device split plan at its limits: 64 sequences (the most it plans), with
    ragged node counts, one empty prefix, one sequence far longer than the
    rest, and malformed trees whose sequences the plan must leave out (their
    rows zero) while the others are still split and merged correctly."""
    rng = np.random.default_rng(64)
    prefix = rng.integers(1, 400, size=64)
    prefix[7] = 0
    prefix[40] = 12000
    inp = gen.random_small(6464, B=64, N_max=12, Hq=8, Hkv=2, D=128, V=200, prefix_lo=0,
                           prefix_hi=1, max_depth=5, prefix_len=prefix)
    for b in (3, 41):  # a self-loop and a second root: the ancestors kernel flags both
        nb = int(inp.n_nodes[b])
        if nb > 1:
            inp.parent[b, nb - 1] = nb - 1 if b == 3 else -1
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    assert (o["err"][[3, 41]] != 0).any()
    compare(inp, g, o)
    assert g["status"] == 0


@pytest.mark.parametrize("D,N,Hq,Hkv", [(64, 30, 32, 8), (128, 32, 32, 8), (128, 9, 8, 8)])
def test_two_blocks_per_sm_path(tsd, D, N, Hq, Hkv):
    """Ragged batches with long key ranges whose kv heads each have at most
    128 query rows run the two-blocks-per-SM kernel (64-key tiles,
    double-buffered S): head dims 64 and 128, exactly 128 rows, tree tails
    that end mid-tile, shuffled blocks; attention on a sample of rows."""
    rng = np.random.default_rng(D + N)
    prefix = rng.integers(2500, 9000, size=16)
    inp = gen.random_small(700 + N, B=16, N_max=N, Hq=Hq, Hkv=Hkv, D=D, V=120, prefix_lo=0,
                           prefix_hi=1, max_depth=6, prefix_len=prefix)
    assert tsd.tree_attn_launches(16, N, Hq, Hkv, D, int((inp.prefix_len + inp.n_nodes).max())) == 3
    sample = sorted({(b, int(rng.integers(inp.n_nodes[b])), int(rng.integers(Hq)))
                     for b in range(16) for _ in range(12)}
                    | {(3, i, h) for i in range(int(inp.n_nodes[3])) for h in range(Hq)})
    g = run_gpu(tsd, inp)
    o = run_oracle(inp, sample_attention=sample)
    compare(inp, g, o, sample=sample)
    assert g["status"] == 0


def test_multi_wave_partials_kept_in_l2(tsd):
    """More blocks than fit at once (80 sequences, three pieces per key
    range): the partials are stored with an evict-last L2 policy and the
    merge kernel drops each line once it has read it, so every row of every
    piece must still be read before its line goes.  All rows against the
    oracle."""
    import torch
    rng = np.random.default_rng(8080)
    prefix = rng.integers(4300, 4990, size=80)
    inp = gen.random_small(8080, B=80, N_max=6, Hq=4, Hkv=2, D=64, V=40, prefix_lo=0,
                           prefix_hi=1, max_depth=4, prefix_len=prefix)
    max_slots = int((inp.prefix_len + inp.n_nodes).max())
    plan = tsd.tree_attn_plan(inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, max_slots)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan["mode"] == 1 and plan["direct"] == 0 and plan["two_blocks_per_sm"] == 1, plan
    assert plan["grid_blocks"] > 2 * nsm, plan
    g = run_gpu(tsd, inp, max_slots=max_slots)
    o = run_oracle(inp)
    compare(inp, g, o)
    assert g["status"] == 0


def test_attention_launch_count(tsd):
    """The launch count the library reports: split + merge, plus the plan
    kernel for ragged-capable batches with long blocks, and a single launch
    (no workspace) when every key range is one piece, which the host plan
    also prefers when a second piece would save less than the merge costs
    (70 sequences of 300 keys)."""
    assert tsd.tree_attn_launches(1, 63, 32, 8, 128, 4159) == 2
    assert tsd.tree_attn_launches(16, 31, 32, 8, 128, 8078) == 3
    assert tsd.tree_attn_launches(70, 6, 4, 2, 64, 1300) == 2
    assert tsd.tree_attn_launches(70, 6, 4, 2, 64, 300) == 1
    assert tsd.tree_attn_launches(40, 31, 32, 8, 128, 431) == 1
    assert tsd.tree_attn_workspace_bytes(40, 31, 32, 8, 128, 431) == 0
    assert tsd.tree_attn_launches(1, 63, 32, 8, 96, 4159) == 0


@pytest.mark.parametrize("case", ["128-row blocks", "256-row blocks"])
def test_single_piece_key_ranges(tsd, case):
    """Enough (sequence, kv head) units to fill the GPU with one piece per key
    range: rows are normalised and written by the split kernel itself (no
    merge launch, no workspace), on the two-blocks-per-SM kernel (40
    sequences, short prefixes) and on the 256-row kernel (one sequence, 60
    kv heads, a 4500-key prefix, 320 rows per kv head: a full 256-row block
    and a 64-row block whose two softmax groups take alternate key tiles)."""
    if case == "128-row blocks":
        inp = gen.random_small(4040, B=40, N_max=31, Hq=32, Hkv=8, D=128, V=64, prefix_lo=100,
                               prefix_hi=400, max_depth=5)
    else:
        inp = gen.random_small(4041, B=1, N_max=20, Hq=960, Hkv=60, D=128, V=64, prefix_lo=4500,
                               prefix_hi=4500, max_depth=5, ragged_nodes=False)
    max_slots = int((inp.prefix_len + inp.n_nodes).max())
    plan = tsd.tree_attn_plan(inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, max_slots)
    assert plan["direct"] == 1 and plan["two_blocks_per_sm"] == (1 if case == "128-row blocks" else 0)
    assert tsd.tree_attn_workspace_bytes(inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, max_slots) == 0
    rng = np.random.default_rng(9)
    sample = sorted({(int(rng.integers(inp.B)), int(rng.integers(inp.N_max)), int(rng.integers(inp.Hq)))
                     for _ in range(120)} | {(0, i, h) for i in range(inp.N_max) for h in (0, inp.Hq - 1)})
    g = run_gpu(tsd, inp)
    o = run_oracle(inp, sample_attention=sample)
    compare(inp, g, o, sample=sample)
    assert g["status"] == 0


@pytest.mark.parametrize("prefix_hi,launches", [(300, 1), (1300, 2)])
def test_large_batch_uniform_split(tsd, prefix_hi, launches):
    """More sequences than the device plan takes (B = 70): the host's
    uniform split and its three-dimensional grid, with one piece per key
    range (rows written by the split kernel) and with two pieces and the
    merge kernel."""
    inp = gen.random_small(4711, B=70, N_max=6, Hq=4, Hkv=2, D=64, V=50, prefix_lo=0,
                           prefix_hi=prefix_hi, max_depth=3)
    max_slots = int((inp.prefix_len + inp.n_nodes).max())
    assert tsd.tree_attn_launches(inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, max_slots) == launches
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    compare(inp, g, o)
    assert g["status"] == 0


SWEEP = [
    # B, N_max, Hq, Hkv, D, V, P range, depth
    (2, 1, 4, 4, 64, 100, (0, 40), 1),
    (3, 2, 8, 2, 128, 257, (0, 3), 2),
    (2, 31, 32, 8, 128, 1000, (15, 17), 6),
    (2, 32, 8, 1, 64, 1001, (16, 16), 8),
    (3, 33, 16, 2, 128, 4099, (1, 130), 9),
    (2, 64, 8, 8, 64, 5000, (63, 65), 12),
    (1, 255, 4, 4, 128, 300, (0, 0), 20),
    (2, 256, 8, 1, 128, 2048, (100, 300), 32),
    (4, 47, 12, 3, 64, 777, (0, 700), 7),
]


@pytest.mark.parametrize("case", range(len(SWEEP)))
def test_random_sweep(tsd, case):
    B, N, Hq, Hkv, D, V, (plo, phi), dmax = SWEEP[case]
    inp = gen.random_small(1000 + case, B=B, N_max=N, Hq=Hq, Hkv=Hkv, D=D, V=V, prefix_lo=plo,
                           prefix_hi=phi, max_depth=dmax, p_match=0.8)
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    compare(inp, g, o)
    assert g["status"] == 0


def test_chain_and_single_node(tsd):
    """A chain tree at the depth limit (causal attention) and single-node
    trees (plain decode)."""
    rng = np.random.default_rng(3)
    for N in (1, 33):
        inp = gen.random_small(77 + N, B=2, N_max=N, Hq=8, Hkv=2, D=128, V=300, prefix_lo=0,
                               prefix_hi=90, max_depth=N - 1, ragged_nodes=False,
                               relabel_ids=False)
        inp.parent[:] = gen.chain_tree(N)
        inp.tokens[:] = np.stack([gen.draft_tokens(rng, inp.parent[b], inp.targets[b], 0.9, 300)
                                  for b in range(2)])
        g = run_gpu(tsd, inp)
        o = run_oracle(inp)
        compare(inp, g, o)


def test_malformed_trees_fail_closed(tsd):
    """Error bits match the oracle exactly; bad sequences are skipped by every
    downstream kernel (zero output, nothing accepted, nothing committed) and
    good sequences in the same batch are unaffected."""
    inp = gen.random_small(5, B=6, N_max=12, Hq=4, Hkv=2, D=64, V=64, prefix_lo=3, prefix_hi=40,
                           max_depth=4, ragged_nodes=False)
    inp.parent[1, 5] = 5                 # self loop
    inp.parent[2, 0] = 3                 # root with a parent
    inp.parent[3, 7] = 40                # out of range
    inp.n_nodes[4] = 0                   # empty tree
    inp.parent[5, :] = gen.chain_tree(12)  # depth 11 > D_max 4
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    assert o["err"][0] == 0 and (o["err"][1:] != 0).all()
    compare(inp, g, o)
    assert (g["accept_len"][1:] == 0).all() and (g["bonus"][1:] == -1).all()
    assert (g["new_len"][1:] == inp.prefix_len[1:]).all()


@pytest.mark.parametrize("B,N,Hq,Hkv,P,mode,direct,dual", [
    (6, 12, 4, 2, 40, 1, 1, 1),      # two blocks per SM, one piece per key range
    (6, 12, 8, 2, 2900, 1, 0, 1),    # two blocks per SM, uniform split (23 pieces)
    (7, 40, 64, 8, 3700, 1, 0, 1),   # the same with three row tiles per kv head
    (6, 12, 16, 8, 12200, 2, 0, 1),  # two blocks per SM, device plan
    (7, 40, 64, 8, 4300, 2, 0, 0)])  # 256-row blocks, device plan
def test_failed_sequences_every_attention_plan(tsd, B, N, Hq, Hkv, P, mode, direct, dual):
    """Failed sequences under each launch shape of the attention: a cyclic
    tree and an empty tree (err != 0: skipped by every kernel) and a
    sequence whose key range runs past the max_slots bound the caller
    passed (TSD_STATUS_BAD_LEN from the attention, which skips it; the
    verification and commit, which take no such bound, still run it).  The
    uniform split's blocks read their inputs before the grid dependency on
    the ancestors kernel resolves and the error words after it, so a stale
    err would show here as rows written for a failed tree."""
    prefix = np.full(B, P, dtype=np.int32)
    prefix[::2] -= 37          # ragged lengths
    prefix[3] = P + 300        # past the bound below
    inp = gen.random_small(900 + B + N + P, B=B, N_max=N, Hq=Hq, Hkv=Hkv, D=128, V=80,
                           prefix_lo=0, prefix_hi=1, max_depth=6, prefix_len=prefix)
    inp.parent[1, int(inp.n_nodes[1]) - 1] = int(inp.n_nodes[1]) - 1  # self loop (or root cycle)
    inp.n_nodes[2] = 0
    others = [b for b in range(B) if b != 3]
    max_slots = int((inp.prefix_len[others] + inp.n_nodes[others]).max())
    assert int(inp.prefix_len[3] + inp.n_nodes[3]) > max_slots
    plan = tsd.tree_attn_plan(B, N, Hq, Hkv, inp.D, max_slots)
    assert (plan["mode"], plan["direct"], plan["two_blocks_per_sm"]) == (mode, direct, dual), plan
    rng = np.random.default_rng(B * N)
    sample = sorted({(b, int(rng.integers(inp.N_max)), int(rng.integers(Hq)))
                     for b in range(B) for _ in range(10)}
                    | {(0, i, h) for i in range(int(inp.n_nodes[0])) for h in (0, Hq - 1)})
    g = run_gpu(tsd, inp, max_slots=max_slots)
    o = run_oracle(inp, sample_attention=sample)
    assert o["err"][1] != 0 and o["err"][2] != 0 and o["err"][3] == 0
    compare(inp, g, o, sample=sample, attn_skip=(3,))
    assert g["status"] == 2  # TSD_STATUS_BAD_LEN, from the attention alone
    assert g["accept_len"][3] == o["accept_len"][3] and g["new_len"][3] > inp.prefix_len[3]


def test_argmax_ties_across_chunks(tsd):
    """Maxima planted in several chunks of a long row: the lowest index wins;
    +0.0 and -0.0 tie; a non-multiple-of-4 vocabulary takes the scalar path."""
    import torch
    from _gpu_path import dev_tensor, to_np
    for V in (128256, 32003):
        B, N = 2, 5
        rng = np.random.default_rng(V)
        logits = rng.standard_normal((B, N, V)).astype(np.float32)
        logits[0, 0, [V - 1, 70000 % V, 12345]] = 9.0
        logits[0, 1, :] = -1.0
        logits[0, 1, [V - 3, 5]] = 0.0
        logits[0, 1, 5] = -0.0
        logits[0, 1, 2] = -0.0
        logits[1, 2, :] = 3.0
        parent = np.array([[-1, 0, 1, 2, 3]] * B, dtype=np.int32)
        tokens = np.zeros((B, N), dtype=np.int32)
        n_nodes = np.full(B, N, dtype=np.int32)
        anc, depth, mask, err = tsd.tree_build_ancestors(dev_tensor(parent), dev_tensor(n_nodes), 4)
        am, *_ = tsd.tree_verify_greedy(dev_tensor(logits), dev_tensor(tokens), dev_tensor(parent),
                                        anc, depth, mask, dev_tensor(n_nodes), err, 4)
        torch.cuda.synchronize()
        ref = oracle.verify_greedy(logits, tokens, parent, n_nodes, np.zeros(B, np.int32), 4)[0]
        assert np.array_equal(to_np(am), ref)
        assert to_np(am)[0, 0] == min(V - 1, 70000 % V, 12345)
        assert to_np(am)[0, 1] == 2 and to_np(am)[1, 2] == 0


def test_bad_block_id_is_reported(tsd):
    """A block id outside the pool is caught by the kernels' bounds checks:
    the status word says so and no memory outside the pool is touched."""
    inp = gen.random_small(8, B=2, N_max=8, Hq=4, Hkv=2, D=64, V=50, prefix_lo=20, prefix_hi=30,
                           max_depth=3, ragged_nodes=False, shuffle_blocks=False)
    inp.cache.block_table[1, 0] = inp.cache.num_blocks + 1000
    g = run_gpu(tsd, inp)
    assert g["status"] & 1  # TSD_STATUS_BAD_PAGE


def test_commit_layers_stacked(tsd):
    """All layers committed in one launch, bit-exact with the oracle."""
    import torch
    from _gpu_path import dev_tensor, to_np
    inp = gen.random_small(9, B=3, N_max=20, Hq=4, Hkv=2, D=128, V=30, prefix_lo=0, prefix_hi=60,
                           max_depth=6, p_match=0.95)
    L = 5
    rng = np.random.default_rng(1)
    K = np.stack([gen.normal_bf16(rng, inp.cache.k.shape) for _ in range(L)])
    Vv = np.stack([gen.normal_bf16(rng, inp.cache.v.shape) for _ in range(L)])
    anc, depth, mask, err = oracle.build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    _, A, _, path, _ = oracle.verify_greedy(inp.logits, inp.tokens, inp.parent, inp.n_nodes, err,
                                            inp.D_max)
    k1, v1, new_len, moved = oracle.commit_path(K, Vv, inp.cache.block_table, inp.prefix_len, A,
                                                path, err)
    kd = dev_tensor(K, torch.bfloat16)
    vd = dev_tensor(Vv, torch.bfloat16)
    nl, mv = tsd.kv_commit_path(kd, vd, dev_tensor(inp.cache.block_table),
                                dev_tensor(inp.prefix_len), dev_tensor(inp.n_nodes), dev_tensor(A),
                                dev_tensor(path), dev_tensor(err), inp.N_max, inp.D_max)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(kd, np.uint16), k1) and np.array_equal(to_np(vd, np.uint16), v1)
    assert np.array_equal(to_np(nl), new_len) and np.array_equal(to_np(mv), moved)
    assert moved.sum() > 0
