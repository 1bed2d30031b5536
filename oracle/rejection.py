"""Modified rejection sampling for one drafted position (CPU only).

Follows [Blog], section on classic speculative decoding and modified
rejection sampling: a drafted token x (drawn from the draft distribution q)
is accepted with probability min(1, p(x)/q(x)); on rejection a corrective
token is drawn from the normalised residual max(0, p - q) / sum max(0, p - q).
The page states that the emitted token is then distributed exactly as p.

Random numbers are inputs: ``u_accept`` and ``u_residual`` are uniforms in
[0, 1).  The residual draw is an inverse-CDF lookup in token order.
"""

from __future__ import annotations

import numpy as np


def residual_distribution(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """max(0, p - q) normalised; all-zero when p == q (never sampled then)."""
    r = np.maximum(0.0, np.asarray(p, dtype=np.float64) - np.asarray(q, dtype=np.float64))
    s = r.sum()
    if s <= 0.0:
        return np.zeros_like(r)
    return r / s


def modified_rejection_step(p, q, x: int, u_accept: float, u_residual: float):
    """Returns (accepted, token)."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    ratio = p[x] / q[x]
    if u_accept < min(1.0, ratio):
        return True, int(x)
    r = residual_distribution(p, q)
    cdf = np.cumsum(r)
    tok = int(np.searchsorted(cdf, u_residual * cdf[-1], side="right"))
    return False, min(tok, len(p) - 1)
