"""The tree budget's host functions ([BASTION] Methodology 3: a roofline cost
model of the verify step, calibrated against measured times) through the C
ABI without a GPU, against the oracle: the cost model bit for bit, the
calibration to rounding, and the refusals."""

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def tsd():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import tree_speculative_decoding_virtual_gb300 as m
    return m


@pytest.mark.parametrize("shape", [(1, 4, 4, 64, [128], 1000, 4, 15),
                                   (8, 32, 8, 128, [2048] * 8, 32000, 16, 256),
                                   (4, 64, 8, 128, [32768] * 4, 128256, 8, 127),
                                   (3, 8, 1, 64, [0, 9, 70000], 257, 0, 1),
                                   (5, 16, 2, 128, [1, 500, 4096, 77, 12345], 50000, 31, 200)])
def test_cost_model_matches_oracle(tsd, shape):
    B, Hq, Hkv, D, P, V, D_max, N = shape
    for peaks in [(6757.2, 1888.4), (8000.0, 2250.0), (3350.0, 989.0)]:
        got = tsd.verify_step_cost(B, Hq, Hkv, D, P, V, D_max, N, *peaks)
        ref = oracle.verify_step_cost(B, Hq, Hkv, D, P, V, D_max, N, *peaks)
        assert got == ref


def test_calibration_matches_oracle(tsd):
    rng = np.random.default_rng(11)
    for n in (2, 3, 7, 40):
        x = np.sort(rng.uniform(2, 900, size=n))
        y = 2.1 * x - 3.0 + rng.normal(0, 1, size=n)
        a, b = tsd.budget_calibrate(x, y)
        ra, rb = oracle.calibrate(x, y)
        assert a == pytest.approx(ra, rel=1e-12)
        assert b == pytest.approx(rb, rel=1e-10, abs=1e-10)
    # an exact line is recovered exactly enough
    x = np.array([10.0, 20.0, 40.0, 80.0])
    a, b = tsd.budget_calibrate(x, 3.0 * x + 5.0)
    assert a == pytest.approx(3.0, rel=1e-14) and b == pytest.approx(5.0, rel=1e-13)
    with pytest.raises(tsd.TsdError):
        tsd.budget_calibrate([1.0, 1.0], [2.0, 3.0])  # no spread in x
