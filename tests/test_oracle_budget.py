"""Pins for the oracle's tree-budget controller ([BASTION] Methodology 3):
the verify-step cost model, its least-squares calibration and the online
choice of the tree size.  Each check is independent of the formula it tests:
array sizes summed from actual buffers, a library line fit, exact rational
arithmetic, and closed forms."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import budget


def _buffers_nbytes(B, Hq, Hkv, D, P, V, D_max, N):
    """Bytes of every tensor one verify step must touch, from real buffers."""
    W = (N + 31) // 32
    i32 = np.int32
    tables = [np.zeros((B, N), i32), np.zeros((B,), i32), np.zeros((B, N + 1, D_max + 1), i32),
              np.zeros((B, N), i32), np.zeros((B, N, W), np.uint32), np.zeros((B,), i32)]
    kv = [np.zeros((p + N, Hkv, D), np.uint16) for p in P] * 2          # K and V of every sequence
    act = [np.zeros((B, N, Hq, D), np.uint16), np.zeros((B, N, Hq, D), np.uint16),
           np.zeros((B, N, Hq), np.float32), np.zeros((B, N, V), np.float32)]
    moved = [np.zeros((B, D_max, Hkv, D), np.uint16)] * 4                # K, V read and written
    return sum(a.nbytes for a in tables + kv + act + moved)


@pytest.mark.parametrize("shape", [(1, 4, 4, 64, [128], 1000, 4, 15),
                                   (3, 32, 8, 128, [512, 7, 4096], 32000, 5, 31),
                                   (2, 8, 1, 64, [0, 33], 257, 0, 40)])
def test_cost_bytes_match_the_buffers(shape):
    B, Hq, Hkv, D, P, V, D_max, N = shape
    nbytes, _, _ = budget.verify_step_cost(B, Hq, Hkv, D, P, V, D_max, N, 1000.0, 1000.0)
    assert nbytes == _buffers_nbytes(B, Hq, Hkv, D, P, V, D_max, N)


def test_cost_flops_reduce_to_decode_attention():
    # N = 1 and D_max = 0: every head of every sequence is plain decode over
    # P + 1 keys: a D-long dot product and a D-long weighted sum per key
    for P, Hq, D in [(0, 1, 4), (4096, 32, 128), (77, 12, 64)]:
        _, flops, _ = budget.verify_step_cost(2, Hq, 1, D, [P, P], 100, 0, 1, 1.0, 1.0)
        assert flops == 2 * Hq * (P + 1) * (2 * D + 2 * D)


def test_cost_roofline_takes_the_binding_roof():
    args = (4, 64, 8, 128, [32768] * 4, 128256, 8, 127)
    nbytes, flops, _ = budget.verify_step_cost(*args, 6757.2, 1888.4)
    # an unbounded tensor pipe leaves the HBM time, and the reverse
    assert budget.verify_step_cost(*args, 6757.2, 1e30)[2] == pytest.approx(nbytes / 6757.2e3)
    assert budget.verify_step_cost(*args, 1e30, 1888.4)[2] == pytest.approx(flops / 1888.4e6)
    # this 70B-shaped step is bound by the tensor pipe, a 1-node one by HBM
    t = budget.verify_step_cost(*args, 6757.2, 1888.4)[2]
    assert t == pytest.approx(flops / 1888.4e6)
    b1, f1, t1 = budget.verify_step_cost(4, 64, 8, 128, [32768] * 4, 128256, 0, 1, 6757.2, 1888.4)
    assert t1 == pytest.approx(b1 / 6757.2e3) and b1 / 6757.2e3 > f1 / 1888.4e6


def test_calibrate_recovers_an_exact_line_and_matches_polyfit():
    x = np.array([12.5, 20.0, 35.0, 61.0, 140.0])
    a, b = budget.calibrate(x, 1.75 * x + 4.25)
    assert a == pytest.approx(1.75, abs=1e-12) and b == pytest.approx(4.25, abs=1e-10)
    rng = np.random.default_rng(7)
    y = 1.3 * x + 9.0 + rng.normal(0, 2.0, size=x.size)
    a, b = budget.calibrate(x, y)
    pa, pb = np.polyfit(x, y, 1)
    assert a == pytest.approx(pa, rel=1e-10) and b == pytest.approx(pb, rel=1e-9)
    with pytest.raises(ValueError):
        budget.calibrate([3.0], [4.0])
    with pytest.raises(ValueError):
        budget.calibrate([3.0, 3.0], [4.0, 5.0])


def _first_local_max_exact(rho_row, cost, l_ar):
    """Brute force in exact rationals: every S(n), then the last n before the
    first strict decrease."""
    S = []
    for n in range(1, len(rho_row) + 1):
        a = sum((Fraction(float(r)) for r in rho_row[1:n]), Fraction(0))
        S.append(a * Fraction(float(l_ar)) / Fraction(float(cost[n])))
    n = 1
    while n < len(S) and S[n] >= S[n - 1]:
        n += 1
    return n, S[n - 1]


def _deciding_gap(rho_row, cost, l_ar, n_opt):
    """Smallest relative gap |S(n) - S(n-1)| / S(n-1) among the comparisons
    that decide n_opt (n = 2 .. n_opt + 1), in exact rationals."""
    S = []
    for n in range(1, len(rho_row) + 1):
        a = sum((Fraction(float(r)) for r in rho_row[1:n]), Fraction(0))
        S.append(a * Fraction(float(l_ar)) / Fraction(float(cost[n])))
    gaps = [abs(S[n - 1] - S[n - 2]) / S[n - 2] for n in range(2, min(n_opt + 1, len(S)) + 1)
            if S[n - 2] > 0]
    return float(min(gaps)) if gaps else float("inf")


def test_budget_select_matches_exact_brute_force():
    rng = np.random.default_rng(11)
    for _ in range(200):
        n_max = int(rng.integers(1, 40))
        # dyadic values with few significant bits: every sum and quotient's
        # comparison is exact, so the fp64 choice must match exact arithmetic
        rho = np.sort(rng.integers(0, 64, size=n_max) / 64.0)[::-1].astype(np.float32)
        rho[0] = 1.0
        cost = np.concatenate([[1.0], rng.integers(8, 512, size=n_max).astype(np.float64)])
        cost[1:] = np.sort(cost[1:])  # a verify step never gets cheaper with more nodes
        l_ar = float(rng.integers(1, 16))
        n_opt, s_opt = budget.budget_select(rho[None, :], cost, l_ar)
        n_ref, s_ref = _first_local_max_exact(rho, cost, l_ar)
        assert int(n_opt[0]) == n_ref
        assert s_opt[0] == pytest.approx(float(s_ref), rel=1e-12)


def test_budget_select_non_dyadic_matches_exact_brute_force():
    """Path scores that are products of draft probabilities (fp32, full
    significands), costs from an affine roofline model with a non-integer
    slope and offset, a non-integer L_AR: the choice equals the exact-rational
    one whenever the deciding comparisons are not within fp64 rounding of a
    tie (such draws are redrawn; they are rare)."""
    rng = np.random.default_rng(23)
    checked = 0
    while checked < 300:
        n_max = int(rng.integers(2, 80))
        q = rng.dirichlet(np.full(6, 0.7), size=n_max).max(axis=1)
        rho = np.empty(n_max, dtype=np.float32)
        rho[0] = 1.0
        for i in range(1, n_max):  # each node's score: its parent's times a probability
            rho[i] = np.float32(rho[int(rng.integers(0, i))] * np.float32(q[i]))
        rho[1:] = np.sort(rho[1:])[::-1]  # best-first insertion order
        t_roof = np.cumsum(rng.uniform(0.05, 3.0, size=n_max)) + rng.uniform(5.0, 50.0)
        cost = np.concatenate([[1.0], rng.uniform(1.0, 40.0) + rng.uniform(0.8, 4.0) * t_roof])
        l_ar = float(rng.uniform(0.3, 90.0))
        n_ref, s_ref = _first_local_max_exact(rho, cost, l_ar)
        if _deciding_gap(rho, cost, l_ar, n_ref) < 1e-12:
            continue
        n_opt, s_opt = budget.budget_select(rho[None, :], cost, l_ar)
        assert int(n_opt[0]) == n_ref
        assert s_opt[0] == pytest.approx(float(s_ref), rel=1e-12)
        checked += 1


def test_speedup_curve_against_exact_rationals():
    rng = np.random.default_rng(4)
    rho = np.concatenate([[1.0], rng.random(30)]).astype(np.float32)
    cost = np.concatenate([[1.0], 3.0 + np.cumsum(rng.random(31))])
    S = budget.speedup_curve(rho, cost, 7.25)
    for n in range(1, 32):
        exact = sum((Fraction(float(r)) for r in rho[1:n]), Fraction(0)) * Fraction(7.25) \
            / Fraction(float(cost[n]))
        assert S[n - 1] == pytest.approx(float(exact), rel=1e-13)
    assert S[0] == 0.0  # the root alone accepts nothing beyond the autoregressive token


def test_budget_select_closed_forms():
    n_max = 64
    # equal scores and an affine cost c0 + c1 n: S(n) = (n - 1) r L / (c0 + c1 n)
    # increases for all n, so the whole budget is used
    rho = np.full((1, n_max), 0.25, dtype=np.float32)
    rho[0, 0] = 1.0
    cost = np.array([10.0 + 0.5 * n for n in range(n_max + 1)])
    assert budget.budget_select(rho, cost, 3.0)[0][0] == n_max
    # scores that vanish after node m under a cost that grows: S peaks at m
    for m in (2, 5, 17):
        r = np.zeros((1, n_max), dtype=np.float32)
        r[0, 0] = 1.0
        r[0, 1:m] = 0.5
        assert budget.budget_select(r, cost, 3.0)[0][0] == m
    # equal values do not stop the growth: scores that vanish after node m
    # under a flat cost keep S constant from m on, so the whole budget is used
    flat = np.full(n_max + 1, 12.5)
    for m in (2, 9):
        r = np.zeros((1, n_max), dtype=np.float32)
        r[0, 0] = 1.0
        r[0, 1:m] = 0.3
        assert budget.budget_select(r, flat, 3.0)[0][0] == n_max
    # a single node: nothing to choose
    assert budget.budget_select(np.ones((2, 1), np.float32), np.array([1.0, 1.0]), 1.0)[0].tolist() == [1, 1]
