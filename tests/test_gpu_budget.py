"""GPU parity of the tree budget ([BASTION] Methodology 3) against the oracle:
the library's host-side cost model and calibration, and the device-side
choice of the tree size from best-first path scores.  The kernel takes the
choice in fp32 (a running sum of the path scores, a cross-multiplied
comparison), the oracle is the page's quotient in fp64; both read the same
fp32 cost table.  The chosen size must be the oracle's wherever every
comparison that decides it is further from a tie than the kernel's rounding
can move it, and S there must agree within that rounding.  Then the chosen
sizes drive the verify step on the truncated trees."""

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


@pytest.mark.parametrize("shape", [(1, 4, 4, 64, [128], 1000, 4, 15),
                                   (8, 32, 8, 128, [2048] * 8, 32000, 16, 256),
                                   (4, 64, 8, 128, [32768] * 4, 128256, 8, 127),
                                   (3, 8, 1, 64, [0, 9, 70000], 257, 0, 1)])
def test_cost_model_matches_oracle(tsd, shape):
    B, Hq, Hkv, D, P, V, D_max, N = shape
    for peaks in [(6757.2, 1888.4), (8000.0, 2250.0)]:
        got = tsd.verify_step_cost(B, Hq, Hkv, D, P, V, D_max, N, *peaks)
        ref = oracle.verify_step_cost(B, Hq, Hkv, D, P, V, D_max, N, *peaks)
        assert got == ref


def test_calibrate_matches_oracle(tsd):
    rng = np.random.default_rng(3)
    for n in (2, 5, 9):
        x = np.sort(rng.uniform(5, 400, size=n))
        y = 1.4 * x + 7.0 + rng.normal(0, 3, size=n)
        a, b = tsd.budget_calibrate(x, y)
        ra, rb = oracle.calibrate(x, y)
        assert a == pytest.approx(ra, rel=1e-12) and b == pytest.approx(rb, rel=1e-10, abs=1e-10)
    with pytest.raises(tsd.TsdError):
        tsd.budget_calibrate([1.0, 1.0], [2.0, 3.0])


def _cost(n_max, seed):
    # C(n) = T_draft + alpha * t_roof(n) + beta on the BASTION verify shape,
    # rounded to fp32 (the table the kernel reads; the oracle reads the same
    # values)
    c = gen.BASTION
    t_roof = lambda n: oracle.verify_step_cost(c["B"], 32, 8, 128, [2048] * c["B"], c["V"],
                                               min(16, max(n - 1, 0)), n, 6757.2, 1888.4)[2]
    return oracle.cost_table(1.3, 11.0 + seed, 20.0, t_roof, n_max).astype(np.float32)


U32 = 2.0 ** -24  # unit roundoff of fp32


def _fp32_margin(n_max):
    """Relative error bound of the kernel's two sides of S(n) < S(n-1): an
    fp32 running sum of at most n_max - 1 positive terms, then one product."""
    return 2.0 * (n_max + 2) * U32


def _allowed_within(S, n, margin):
    """Whether stopping at n is the rule's choice once comparisons within a
    relative `margin` of a tie may go either way: no clear decrease up to n,
    and no clear increase right after it."""
    for k in range(2, n + 1):
        if S[k - 1] < S[k - 2] * (1.0 - margin):
            return False
    return n == len(S) or S[n] < S[n - 1] * (1.0 + margin)


def _check_choice(rho, cost, l_ar, n_gpu, s_gpu):
    """Exact n where every deciding comparison clears the fp32 margin; S at
    the choice within the kernel's rounding.  Near-ties: a choice the margin
    allows.  Returns the rows checked exactly."""
    n_ref, s_ref = oracle.budget_select(rho, cost.astype(np.float64), l_ar)
    n_max = rho.shape[1]
    checked = 0
    for b in range(rho.shape[0]):
        S = oracle.speedup_curve(rho[b], cost.astype(np.float64), l_ar)
        top = min(int(n_ref[b]) + 1, n_max)
        gaps = [abs(S[n - 1] - S[n - 2]) / S[n - 2] for n in range(2, top + 1) if S[n - 2] > 0]
        if gaps and min(gaps) <= _fp32_margin(n_max):
            # a near-tie: either side of it is a correct fp32 choice
            assert _allowed_within(S, int(n_gpu[b]), _fp32_margin(n_max)), (b, int(n_gpu[b]))
            continue
        assert int(n_gpu[b]) == int(n_ref[b]), (b, int(n_gpu[b]), int(n_ref[b]))
        bound = (int(n_ref[b]) + 2) * U32 * abs(s_ref[b])
        assert abs(float(s_gpu[b]) - s_ref[b]) <= bound, (b, float(s_gpu[b]), s_ref[b])
        checked += 1
    return checked


@pytest.mark.parametrize("n_max", [16, 64, 256])
def test_select_on_best_first_scores(tsd, n_max):
    import torch
    from _gpu_path import dev_tensor, to_np
    q, root = gen.bastion_marginals()
    parent, tokens, depth, rho, ahat = tsd.best_first_tree_build(dev_tensor(q), dev_tensor(root),
                                                                 n_max)
    # the choice sits where S stops growing, so its deciding comparison is
    # often close to a tie; many cost tables give enough rows clear of it
    checked = total = 0
    for seed in range(12):
        cost = _cost(n_max, 5.0 * seed)
        for l_ar in (5.0, 400.0):
            n_opt, s_opt = tsd.budget_select(rho, torch.from_numpy(cost).cuda(), l_ar)
            torch.cuda.synchronize()
            checked += _check_choice(to_np(rho), cost, l_ar, to_np(n_opt), to_np(s_opt))
            total += q.shape[0]
    assert checked >= 0.4 * total, (checked, total)


def test_select_random_scores_and_edges(tsd):
    import torch
    from _gpu_path import to_np
    rng = np.random.default_rng(5)
    checked = total = 0
    for _ in range(20):
        B, n_max = int(rng.integers(1, 300)), int(rng.integers(1, 257))  # B up to 65535 allowed
        rho = np.sort(rng.random((B, n_max)).astype(np.float32), axis=1)[:, ::-1].copy()
        rho[:, 0] = 1.0
        rho[:, n_max // 2:] *= np.float32(rng.random())  # a drop, so some choices stop early
        cost = np.concatenate([[1.0], np.cumsum(rng.uniform(0.1, 5.0, size=n_max)) + 10.0])
        cost = cost.astype(np.float32)
        l_ar = float(rng.uniform(1, 100))
        n_opt, s_opt = tsd.budget_select(torch.from_numpy(rho).cuda(), torch.from_numpy(cost).cuda(),
                                         l_ar)
        torch.cuda.synchronize()
        checked += _check_choice(rho, cost, l_ar, to_np(n_opt), to_np(s_opt))
        total += B
    assert checked >= 0.9 * total, (checked, total)
    # host-side argument checks: nothing is launched
    rho_d = torch.from_numpy(rho).cuda()
    with pytest.raises(tsd.TsdError):
        tsd.budget_select(rho_d, torch.from_numpy(cost).cuda(), -1.0)
    with pytest.raises(tsd.TsdError):
        tsd.budget_select(rho_d, torch.from_numpy(cost[:2]).cuda(), 1.0)


def test_chosen_sizes_drive_the_verify_step(tsd):
    """Best-first tree of 256 nodes -> per-sequence size -> the verify step on
    the first n_opt nodes of each tree (a prefix of a best-first order is a
    tree), against the oracle on the same truncated trees."""
    import torch
    from _gpu_path import dev_tensor, to_np
    q, root = gen.bastion_marginals()
    n_max = 256
    parent, tokens, depth, rho, ahat = tsd.best_first_tree_build(dev_tensor(q), dev_tensor(root),
                                                                 n_max)
    cost = _cost(n_max, 0)
    n_opt, _ = tsd.budget_select(rho, torch.from_numpy(cost).cuda(), 60.0)
    torch.cuda.synchronize()
    n_opt = to_np(n_opt)
    assert (n_opt >= 1).all() and (n_opt <= n_max).all()
    top1 = np.stack([[oracle.ranked_tokens(q[b, k])[0] for k in range(q.shape[1])]
                     for b in range(q.shape[0])])
    inp = gen.bastion_verify_inputs(to_np(parent), to_np(tokens), to_np(depth), top1)
    inp.n_nodes = n_opt.astype(np.int32)
    g = run_gpu(tsd, inp)
    o = run_oracle(inp)
    compare(inp, g, o)
    assert (g["err"] == 0).all()
