"""CPU checks of the two arguments the GPU best-first kernels rest on
(BASTION Methodology 2: best-first expansion adds the valid node with the
largest path score), each restated here in plain Python and compared with the
oracle or with brute force:

* Sibling runs.  A step may insert the best candidate (p, r) together with
  p's next-ranked children (p, r+1), (p, r+2), ... while each still beats
  both the best candidate outside p and the first child of (p, r); the
  insertion order is then the one-at-a-time order of the oracle.
* The top-M threshold.  With the row's elements dealt to 1024 threads in
  16-byte groups, 32 threads to a warp, tau = the least over warps of the
  warp's ceil(M/32)-th largest thread maximum has at least M elements at or
  above it, so every one of the M best (by value, then index) is >= tau."""

import numpy as np
import pytest

import gen
from oracle import best_first_tree, ranked_tokens


def _key(rho, depth, parent):
    # larger wins: (rho desc, depth asc, parent asc)
    return (float(rho), -depth, -parent)


def _runs_tree(q, root, N):
    q = np.asarray(q, dtype=np.float32)
    K, V = q.shape
    M = min(N - 1, V)
    tq = [q[k][ranked_tokens(q[k])[:M]] for k in range(K)]
    tt = [ranked_tokens(q[k])[:M] for k in range(K)]
    rho, dep, nch, par, tok = [np.float32(1.0)], [0], [0], [-1], [int(root)]

    def cand(node):  # (key, rank) of node's next child, or None
        d, r = dep[node] + 1, nch[node]
        if d > K or r >= M:
            return None
        return _key(np.float32(rho[node] * tq[d - 1][r]), d, node)

    steps = 0
    while len(par) < N:
        steps += 1
        keys = [(cand(x), x) for x in range(len(par))]
        keys = [(k, x) for k, x in keys if k is not None]
        (best, p) = max(keys)
        others = [k for k, x in keys if x != p]
        k2 = max(others) if others else None
        d, r = dep[p] + 1, nch[p]
        r0 = np.float32(rho[p] * tq[d - 1][r])
        fc0 = _key(np.float32(r0 * tq[d][0]), d + 1, len(par)) if d < K and M > 0 else None
        bound = max([k for k in (k2, fc0) if k is not None], default=None)
        run = 0
        while r + run < M and len(par) + run < N:
            rc = np.float32(rho[p] * tq[d - 1][r + run])
            if bound is not None and not _key(rc, d, p) > bound:
                break
            run += 1
        assert run >= 1
        for i in range(run):
            rho.append(np.float32(rho[p] * tq[d - 1][r + i]))
            dep.append(d)
            nch.append(0)
            par.append(p)
            tok.append(int(tt[d - 1][r + i]))
        nch[p] += run
    return par, tok, dep, rho, steps


@pytest.mark.parametrize("shape", ["sharp", "flat", "tied", "pow2", "dominant", "uniform"])
def test_sibling_runs_keep_the_insertion_order(shape):
    rng = np.random.default_rng(hash(shape) % 1000)
    runs_seen = 0
    for case in range(12):
        K, V = int(rng.integers(1, 7)), int(rng.integers(1, 24))
        total = sum(V ** d for d in range(1, K + 1))
        N = int(min(rng.integers(1, 120), total + 1))
        q, root = gen.shaped_marginals(1000 + case, 1, K, V, shape)
        par, tok, dep, rho, steps = _runs_tree(q[0], root[0], N)
        ref = best_first_tree(q, root, N)
        assert par == list(ref[0][0]) and tok == list(ref[1][0]) and dep == list(ref[2][0])
        assert np.array_equal(np.array(rho, dtype=np.float32), ref[3][0])
        runs_seen += (N - 1) - steps
    if shape in ("flat", "uniform", "tied", "pow2"):
        assert runs_seen > 0  # some step inserted more than one node


def _tau(row, M, threads=1024, warp=32):
    V = len(row)
    if V % 4 == 0:
        groups = row.reshape(-1, 4).max(axis=1)
        owner = np.arange(len(groups)) % threads
    else:
        groups = row
        owner = np.arange(V) % threads
    tmax = np.full(threads, -np.inf, dtype=np.float32)
    np.maximum.at(tmax, owner, groups)
    mw = (M + warp - 1) // warp
    per_warp = [np.sort(tmax[w * warp:(w + 1) * warp])[::-1][mw - 1] for w in range(threads // warp)]
    return min(per_warp)


@pytest.mark.parametrize("V", [3, 17, 500, 1023, 1024, 4096, 32000])
def test_threshold_keeps_every_one_of_the_m_best(V):
    rng = np.random.default_rng(V)
    for trial in range(6):
        kind = trial % 3
        if kind == 0:
            row = rng.random(V).astype(np.float32)
        elif kind == 1:
            row = np.round(rng.random(V) * 7).astype(np.float32) / 7  # many ties
        else:
            row = np.exp(3 * rng.standard_normal(V)).astype(np.float32)
        for M in sorted({1, min(15, V), min(31, V), min(32, V), min(255, V), min(511, V)}):
            tau = _tau(row, M)
            assert (row >= tau).sum() >= M
            best = np.lexsort((np.arange(V), -row.astype(np.float64)))[:M]
            assert (row[best] >= tau).all()


def test_threshold_count_is_tight():
    """Every warp holding the same thread maxima (one large value per thread,
    set by its lane) leaves exactly 32 * ceil(M/32) elements at or above tau:
    a smaller per-warp rank would keep fewer than M."""
    V = 32000
    rng = np.random.default_rng(9)
    row = (rng.random(V) * 0.5).astype(np.float32)
    for t in range(1024):
        row[4 * t] = np.float32(1.0 + (t % 32) / 32.0)   # thread t's first 16-byte group
    for M in (15, 32, 33, 255, 511):
        tau = _tau(row, M)
        assert (row >= tau).sum() == 32 * ((M + 31) // 32) >= M
