"""The fp64 sum of A_hat (BASTION Methodology 2: the sum of the path scores of
a tree's non-root nodes, taken in insertion order) may be added in any order
when every partial sum is exact.  With at most 255 fp32 terms, all multiples of
2^b (b the lowest set bit over the terms) and each below 2^(e+1) (e the largest
term's exponent), every partial sum is an integer multiple of 2^b below
2^(e+9), so e + 9 - b <= 53 makes every fp64 addition exact.  Checked here
against the exactly rounded sum (math.fsum) and other orders; and the bound
is needed: without it the order changes the result."""

import math

import numpy as np


def _span_ok(v):
    v = v[v > 0].astype(np.float64)
    if v.size == 0:
        return True
    e_max = int(np.floor(np.log2(v.max())))
    lows = []
    for x in v:
        m, e = np.frexp(x)
        sig = int(m * 2.0 ** 53)
        lows.append(e - 53 + ((sig & -sig).bit_length() - 1))
    return e_max + 9 - min(lows) <= 53


def _seq(v):
    s = 0.0
    for x in v:
        s += float(x)
    return s


def test_any_order_is_exact_within_the_span():
    rng = np.random.default_rng(0)
    checked = 0
    for _ in range(400):
        n = int(rng.integers(1, 256))
        top = int(rng.integers(-20, 1))
        width = int(rng.integers(1, 45))
        expo = rng.integers(top - width, top + 1, size=n)
        v = (rng.random(n) * np.exp2(expo)).astype(np.float32)
        if not _span_ok(v):
            continue
        s = _seq(v)
        assert s == math.fsum(float(x) for x in v)
        assert s == _seq(v[::-1])
        assert s == _seq(rng.permutation(v))
        pair = v.astype(np.float64)
        while pair.size > 1:   # pairwise tree, as a warp adds
            if pair.size % 2:
                pair = np.append(pair, 0.0)
            pair = pair[0::2] + pair[1::2]
        assert s == float(pair[0])
        checked += 1
    assert checked > 100


def test_order_matters_beyond_the_span():
    v = np.array([1.0, 2.0 ** -53, 2.0 ** -53], dtype=np.float32)
    assert not _span_ok(v)
    assert _seq(v) != _seq(v[::-1])
