"""Hardware-aware tree budget: verify-step cost model, its calibration, and the
online choice of the tree size.

Follows [BASTION] Methodology 3 ("Controlador de Orçamento Online Consciente
de Hardware"): the verification latency T_verify(N) comes from a roofline
model (memory bandwidth and compute) calibrated against observed run times;
the controller grows the tree until the estimated speed-up
S(N) = A_hat(T_N) * L_AR / C(N) starts to decrease.

Readings taken where the page is silent:

* The roofline time of one verify step (a1-a4, one layer, the whole batch) is
  max(bytes / BW, flops / TC) over the step's algorithmic bytes and FLOPs:
  the ancestor tables; the attention's K/V over prefix and tree, q, out and
  lse; the logits; at most D_max moved entries per sequence for the commit.
  The attention FLOPs count 4*D per key for every (node, q head) row, over the
  prefix and at most D_max + 1 tree keys.
* Calibration is a least-squares line T_measured ~ alpha * T_roofline + beta
  (the scale corrects for fusion, the offset for launch and scheduling).
* C(N) = T_draft + T_verify(N); L_AR is the latency of one autoregressive step;
  A_hat(T_N) = the sum of rho over the non-root nodes among the first N
  inserted (best-first insertion order), accumulated in fp64 in that order.
* "Starts to decrease": the chosen N is the largest n such that
  S(1) <= S(2) <= ... <= S(n) (equal values do not stop the growth); when S
  never decreases, the whole budget.  S(n) is the page's quotient written
  out in fp64: A_hat(n) is the fp64 sum of the non-root path scores (as
  stored) in insertion order, S(n) = A_hat(n) * L_AR / C(n) with the step
  costs as given; s_opt is S at the chosen n.
"""

from __future__ import annotations

import numpy as np


def verify_step_cost(B, Hq, Hkv, D, prefix_len, V, D_max, N, hbm_gbs, tc_tflops):
    """(bytes, flops, roofline microseconds) of one verify step with N-node
    trees for every sequence."""
    P = [int(x) for x in prefix_len]
    assert len(P) == B
    W = (N + 31) // 32
    tables = 4 * (B * N + B + B * (N + 1) * (D_max + 1) + B * N + B * N * W + B)
    kv = 2 * 2 * Hkv * D * sum(p + N for p in P)             # K and V, bf16
    q_out = 2 * 2 * B * N * Hq * D                           # q and out, bf16
    lse = 4 * B * N * Hq
    logits = 4 * B * N * V
    commit = 2 * 2 * 2 * Hkv * D * B * D_max                 # read + write of K and V
    nbytes = tables + kv + q_out + lse + logits + commit
    keys = sum(N * p for p in P) + B * N * (D_max + 1)
    flops = 4.0 * D * Hq * keys
    t_us = max(nbytes / (hbm_gbs * 1e9), flops / (tc_tflops * 1e12)) * 1e6
    return float(nbytes), float(flops), float(t_us)


def calibrate(t_roof, t_meas):
    """Least-squares (alpha, beta) of t_meas ~ alpha * t_roof + beta."""
    x = np.asarray(t_roof, dtype=np.float64)
    y = np.asarray(t_meas, dtype=np.float64)
    if x.size < 2:
        raise ValueError("calibration needs at least two points")
    xm, ym = x.mean(), y.mean()
    sxx = float(((x - xm) ** 2).sum())
    if not sxx > 0.0:
        raise ValueError("calibration needs two distinct roofline times")
    alpha = float(((x - xm) * (y - ym)).sum()) / sxx
    beta = float(ym - alpha * xm)
    return alpha, beta


def speedup_curve(rho_row, cost, l_ar):
    """S(n) = A_hat(n) * L_AR / C(n) for n = 1..N_max, in fp64.  rho_row:
    [N_max] path scores in insertion order (rho_row[0] is the root, which
    A_hat leaves out); cost: [N_max + 1], cost[n] = C(n) > 0."""
    L = float(l_ar)
    S, a = [], 0.0
    for n in range(1, len(rho_row) + 1):
        if n >= 2:
            a += float(rho_row[n - 1])
        S.append(a * L / float(cost[n]))
    return np.array(S, dtype=np.float64)


def budget_select(rho, cost, l_ar):
    """rho: [B][N_max] path scores in insertion order (rho[b][0] is the root);
    cost: [N_max + 1] with cost[n] = C(n) > 0 for n = 1..N_max; l_ar: L_AR > 0.
    Returns (n_opt int32 [B], s_opt float64 [B]): the last n before S first
    decreases, and S there."""
    rho = np.asarray(rho)
    cost = np.asarray(cost)
    B, n_max = rho.shape
    if not float(l_ar) > 0.0 or not np.all(cost[1:n_max + 1] > 0):
        raise ValueError("L_AR and every step cost must be positive")
    n_opt = np.zeros(B, dtype=np.int32)
    s_opt = np.zeros(B, dtype=np.float64)
    for b in range(B):
        S = speedup_curve(rho[b], cost, l_ar)
        n = 1
        while n < n_max and not S[n] < S[n - 1]:
            n += 1
        n_opt[b] = n
        s_opt[b] = S[n - 1]
    return n_opt, s_opt


def cost_table(alpha, beta, t_draft, t_roof_of_n, n_max):
    """[n_max + 1] table of C(n) = t_draft + alpha * t_roof(n) + beta (entry 0
    unused, set to C(1)), in fp64; the choice reads it rounded to fp32."""
    c = np.zeros(n_max + 1, dtype=np.float64)
    for n in range(1, n_max + 1):
        c[n] = float(t_draft) + float(alpha) * float(t_roof_of_n(n)) + float(beta)
    c[0] = c[1]
    if not np.all(c[1:] > 0.0) or not np.all(np.isfinite(c)):
        raise ValueError("step costs must be positive and finite")
    return c


__all__ = ["verify_step_cost", "calibrate", "speedup_curve", "budget_select", "cost_table"]
