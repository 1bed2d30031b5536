"""Best-first budgeted trees (BASTION Methodology 1 and 2) on the GPU against
the oracle, bit for bit (parent, tokens, depth, rho, A_hat), on marginals of
several shapes: deep and narrow, wide, many equal probabilities, powers of
two (many equal path scores), long chains, path scores spanning more than
2^53 (A_hat then has to be summed in insertion order), uniform rows (every
rank a tie), the largest number of positions, vocabularies smaller than the
budget, the smallest budgets, and rows longer than the shared-memory-staged
top-M kernel takes."""

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsd():
    import torch
    import tree_speculative_decoding_virtual_gb300 as m
    torch.cuda.set_device(0)
    return m


def _needs_ordered_sum(rho):
    """True when the fp64 sum of these fp32 terms may depend on the order:
    the terms' bits span more than 53 - 9 positions (at most 255 terms)."""
    v = np.asarray(rho, dtype=np.float32)
    v = v[v > 0]
    if v.size == 0:
        return False
    e_max = int(np.floor(np.log2(np.float64(v.max()))))
    lows = []
    for x in v:
        m, e = np.frexp(np.float64(x))          # x = m * 2^e, 0.5 <= m < 1
        sig = int(m * 2.0 ** 53)
        lows.append(e - 53 + ((sig & -sig).bit_length() - 1))
    return e_max + 9 - min(lows) > 53


CASES = [
    # shape, seed, B, K, V, N
    ("sharp", 11, 3, 8, 40, 256),
    ("flat", 12, 2, 6, 30, 256),
    ("tied", 13, 3, 6, 24, 256),
    ("pow2", 14, 3, 10, 16, 180),
    ("dominant", 15, 2, 16, 300, 256),
    ("tiny_tail", 16, 2, 12, 20, 256),
    ("sharp", 17, 2, 64, 3, 256),      # the largest number of positions
    ("tied", 18, 2, 2, 7, 57),         # every one of the 56 valid nodes
    ("flat", 19, 3, 4, 5, 2),
    ("flat", 20, 3, 4, 5, 1),
    ("dominant", 21, 4, 16, 32000, 64),
    ("uniform", 22, 2, 4, 32000, 256),  # more ties at the filter's threshold than it keeps
    ("uniform", 23, 2, 3, 1500, 100),   # every candidate tied: the select reaches the index bits
    ("flat", 24, 2, 5, 40961, 64),      # a row longer than the staged kernel takes
    ("sharp", 25, 2, 6, 500, 65),       # 64 ranked tokens: two full runs of the final sort
    ("tied", 26, 2, 4, 1000, 33),       # 32 ranked tokens: one full run
]


@pytest.mark.parametrize("shape,seed,B,K,V,N", CASES)
def test_best_first_shapes(tsd, shape, seed, B, K, V, N):
    import torch
    from _gpu_path import dev_tensor, to_np
    q, root = gen.shaped_marginals(seed, B, K, V, shape)
    got = [to_np(x) for x in tsd.best_first_tree_build(dev_tensor(q), dev_tensor(root), N)]
    torch.cuda.synchronize()
    ref = oracle.best_first_tree(q, root, N)
    for name, x, y in zip(["parent", "tokens", "depth", "rho", "ahat"], got, ref):
        assert np.array_equal(x, y), (name, shape)
    if shape == "tiny_tail":
        # the case exists to take the insertion-order sum
        assert all(_needs_ordered_sum(ref[3][b, 1:]) for b in range(B))
