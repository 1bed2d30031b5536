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
  never decreases, the whole budget.  The choice is taken in fp32: A_hat is
  an fp32 running sum in insertion order, and S(n) < S(n-1) is tested as
  A_hat(n) * C(n-1) < A_hat(n-1) * C(n) (L_AR > 0 cancels), each product
  rounded to fp32; S at the chosen n is (A_hat * L_AR) / C, in fp32.
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


def budget_select(rho, cost, l_ar):
    """rho: [B][N_max] path scores in insertion order (rho[b][0] is the root);
    cost: [N_max + 1] with cost[n] = C(n) > 0 for n = 1..N_max; l_ar: L_AR.
    Returns (n_opt int32 [B], s_opt float32 [B])."""
    f32 = np.float32
    rho = np.asarray(rho, dtype=f32)
    cost = np.asarray(cost, dtype=f32)
    l_ar = f32(l_ar)
    B, n_max = rho.shape
    n_opt = np.zeros(B, dtype=np.int32)
    s_opt = np.zeros(B, dtype=f32)
    for b in range(B):
        a_prev, c_prev = f32(0.0), cost[1]
        best = 1
        for n in range(2, n_max + 1):
            a = f32(a_prev + rho[b, n - 1])
            c = cost[n]
            if f32(a * c_prev) < f32(a_prev * c):  # S(n) < S(n - 1)
                break
            a_prev, c_prev, best = a, c, n
        n_opt[b] = best
        s_opt[b] = f32(f32(a_prev * l_ar) / c_prev)
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


__all__ = ["verify_step_cost", "calibrate", "budget_select", "cost_table"]
