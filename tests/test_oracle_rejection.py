"""Pins for the modified rejection sampling rule (CPU only).

The page's identity: the emitted token is distributed exactly as the target
distribution p, because min(q, p) + (1 - sum min(p, q)) * residual = p.
Checked exactly in fp64, and by Monte-Carlo through the oracle's step
function with draft tokens drawn from q.
"""

import numpy as np

from oracle import modified_rejection_step, residual_distribution


def test_exact_identity():
    rng = np.random.default_rng(0)
    for _ in range(200):
        V = int(rng.integers(2, 12))
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V))
        accept_mass = np.minimum(p, q)
        reject_mass = 1.0 - accept_mass.sum()
        total = accept_mass + reject_mass * residual_distribution(p, q)
        np.testing.assert_allclose(total, p, rtol=0, atol=1e-15)


def test_monte_carlo_emits_p():
    rng = np.random.default_rng(0)
    V, n = 8, 200000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    xs = rng.choice(V, size=n, p=q)
    u = rng.random(n)
    w = rng.random(n)
    counts = np.zeros(V)
    acc = 0
    for x, a, r in zip(xs, u, w):
        ok, t = modified_rejection_step(p, q, int(x), float(a), float(r))
        counts[t] += 1
        acc += ok
    freq = counts / n
    assert (np.abs(freq - p) < 5 * np.sqrt(p * (1 - p) / n)).all()
    # acceptance rate is sum min(p, q)
    rate = np.minimum(p, q).sum()
    assert abs(acc / n - rate) < 5 * np.sqrt(rate * (1 - rate) / n)


def test_equal_distributions_never_reject():
    p = np.array([0.5, 0.25, 0.25])
    assert (residual_distribution(p, p) == 0).all()
    for x in range(3):
        ok, t = modified_rejection_step(p, p, x, 0.999999, 0.3)
        assert ok and t == x


def test_residual_skips_zero_mass():
    p = np.array([0.2, 0.5, 0.3])
    q = np.array([0.4, 0.2, 0.4])  # residual mass only on token 1
    for u in (0.0, 0.5, 0.999):
        ok, t = modified_rejection_step(p, q, 0, 0.99, u)
        assert not ok and t == 1
