"""The seeded marginal generators behave as their docstrings say (they feed
both the oracle and the GPU path, so a shape that silently lost its property
would make a test case prove less): non-negative fp32 rows summing to about
one, the same bits for the same seed, and each shape's defining property."""

import numpy as np
import pytest

import gen

SHAPES = ["sharp", "flat", "tied", "pow2", "dominant", "tiny_tail", "uniform"]


@pytest.mark.parametrize("shape", SHAPES)
def test_rows_are_distributions_and_reproducible(shape):
    q, root = gen.shaped_marginals(3, 2, 5, 40, shape)
    assert q.dtype == np.float32 and q.shape == (2, 5, 40)
    assert (q >= 0).all() and np.isfinite(q).all()
    s = q.astype(np.float64).sum(-1)
    assert np.allclose(s, 1.0, atol=1e-5) or shape in ("pow2", "tiny_tail")
    assert root.dtype == np.int32 and ((root >= 0) & (root < 40)).all()
    q2, root2 = gen.shaped_marginals(3, 2, 5, 40, shape)
    assert np.array_equal(q.view(np.uint32), q2.view(np.uint32)) and np.array_equal(root, root2)


def test_shape_properties():
    q, _ = gen.shaped_marginals(4, 1, 3, 64, "pow2")
    m, e = np.frexp(q.astype(np.float64))
    assert (m == 0.5).all()                                   # every value a power of two
    q, _ = gen.shaped_marginals(4, 1, 3, 64, "uniform")
    assert (q == q[..., :1]).all()                            # every rank a tie
    q, _ = gen.shaped_marginals(4, 1, 3, 64, "tied")
    assert len(np.unique(q[0, 0])) < 64                       # equal probabilities present
    q, _ = gen.shaped_marginals(4, 1, 3, 64, "tiny_tail")
    assert (q[..., 0] == np.float32(0.5)).all() and (q[..., 1:] < 1e-7).all()
    q, _ = gen.shaped_marginals(4, 1, 3, 64, "dominant")
    assert (q.argmax(-1) == 0).mean() > 0.9
    q_sharp, _ = gen.shaped_marginals(4, 1, 3, 64, "sharp")
    q_flat, _ = gen.shaped_marginals(4, 1, 3, 64, "flat")
    assert q_sharp.max(-1).mean() > 3 * q_flat.max(-1).mean()
    with pytest.raises(ValueError):
        gen.shaped_marginals(4, 1, 3, 64, "nonsense")


def test_bastion_marginals_shape():
    q, root = gen.bastion_marginals()
    c = gen.BASTION
    assert q.shape == (c["B"], c["K"], c["V"]) and q.dtype == np.float32
    assert np.allclose(q.astype(np.float64).sum(-1), 1.0, atol=1e-4)
